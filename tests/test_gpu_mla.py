"""pa_mla_decode (absorbed MLA, 128 heads on a 576-wide latent) on the GPU
against the fp64 oracle: the DeepSeek-shaped batch on sampled sequences,
ragged small contexts across page and tile edges, forced splits, and bad
metadata."""
import numpy as np
import pytest
import torch

from paged_kv_attention_16_gb300 import inputs, pa
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_attention_16_gb300 import build
    build.build()
    pa.pa_get_device_status()


def gpu_mla(m, expect_status=0):
    d = pa.to_device(m)
    out = pa.mla_decode(d)
    status = pa.pa_get_device_status()
    assert status == expect_status, f"device status {status:#x}, expected {expect_status:#x}"
    return out.float().cpu().numpy().astype(np.float64)


def test_mla_deepseek_batch_sampled():
    """Twelve of the 64 sequences: the longest and the shortest context and
    ten spread over the batch (most of them cut into several pieces by the
    per-cluster work runs, so their rows go through the merge)."""
    m = inputs.mla_decode_batch()
    ctx = m.seq_lens.numpy()
    seqs = sorted({int(ctx.argmax()), int(ctx.argmin()), 0, 5, 11, 17, 26, 33, 41, 48, 55, 63})
    rows = np.concatenate([np.arange(s * 128, (s + 1) * 128) for s in seqs]).astype(np.int64)
    got = gpu_mla(m)
    want = parity.oracle_mla(m, rows=rows)
    parity.compare(got, want, "bf16", rows=rows, what="mla deepseek")


@pytest.mark.parametrize("block_size", [64, 32, 128])
def test_mla_ragged_contexts(block_size):
    m = inputs.mla_batch([1, 31, 32, 33, 64, 100, 2049, 700], block_size=block_size,
                         seed=block_size)
    got = gpu_mla(m)
    parity.compare(got, parity.oracle_mla(m), "bf16", what=f"mla bs{block_size}")


@pytest.mark.parametrize("kvs", [32, 96, 512])
def test_mla_forced_splits(kvs):
    m = inputs.mla_batch([3000, 65, 1], seed=kvs, kv_split_tokens=kvs)
    got = gpu_mla(m)
    parity.compare(got, parity.oracle_mla(m), "bf16", what=f"mla kvs {kvs}")


def test_mla_bad_block_zeroes_its_sequence():
    m = inputs.mla_batch([300, 200, 90], seed=9)
    want = parity.oracle_mla(m)
    m.block_table[1, 1] = m.num_blocks + 3
    got = gpu_mla(m, expect_status=pa.PA_DEV_BAD_BLOCK)
    assert np.all(got[1] == 0.0)
    parity.compare(got[[0, 2]], want[[0, 2]], "bf16", what="healthy sequences")


def test_mla_seq_len_above_bound_is_flagged():
    m = inputs.mla_batch([300, 200], seed=10)
    want = parity.oracle_mla(m)
    m.max_seq_len = 250
    got = gpu_mla(m, expect_status=pa.PA_DEV_BAD_SEQLEN)
    assert np.all(got[0] == 0.0)
    parity.compare(got[1:], want[1:], "bf16", what="healthy sequence")


def test_mla_graph_replay():
    m = inputs.mla_batch([700, 1500, 64], seed=11, max_seq_len=4096)
    d = pa.to_device(m)
    out = torch.empty((3, 128, 512), dtype=torch.bfloat16, device="cuda")
    pa.pa_reserve(pa.pa_mla_decode_workspace_bytes(3, 128, 512, 4096))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pa.mla_decode(d, out=out, stream=s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            pa.mla_decode(d, out=out, stream=s)
    torch.cuda.synchronize()
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert pa.pa_get_device_status() == 0
    parity.compare(out.float().cpu().numpy().astype(np.float64), parity.oracle_mla(m), "bf16",
                   what="mla graph replay")


def test_mla_split_not_multiple_of_32_is_refused():
    """A KV split must start on a 32-position tile (tiles never cross a page)."""
    m = pa.to_device(inputs.mla_batch([300, 65], seed=5))
    out = torch.empty((m.num_seqs, m.num_heads, m.kv_lora_rank), dtype=torch.bfloat16,
                      device="cuda")
    st = pa.pa_mla_decode(m.q, m.kv_cache, m.block_table, m.seq_lens, m.num_heads,
                          m.kv_lora_rank, m.rope_dim, m.block_size, m.scale, out,
                          max_seq_len=m.max_seq_len, kv_split_tokens=48, check=False)
    assert st == pa.PA_ERR_UNSUPPORTED
