"""Decode-only batches declared with max_query_len == 1 (pa_forward_ex): up to
1024 requests, one row-kernel launch that sizes the KV splits from seq_lens
and merges a row's splits in the thread block that finishes last (more
requests, fp32, or a looser bound keep the planned path, which the same
calls check too).  Checked against the fp64 oracle on the decode workloads,
with the model variants, both layouts, every GQA group the row kernel
takes, split counts up to the 64 a row allows, repeated and graph-replayed
calls (the split counters must return to zero), and bad metadata."""
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
    pa.lib()
    pa.pa_get_device_status()  # clear


def fast(b, expect_status=0, **kw):
    return parity.gpu_forward(b, max_query_len=1, expect_status=expect_status, **kw)


def test_llama_decode_b1_and_b64():
    for batch in (1, 64):
        b = inputs.llama_decode(batch)
        parity.compare(fast(b), parity.oracle_forward(b), "bf16", what=f"fast b{batch}")


@pytest.mark.parametrize("group", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("head_dim", [64, 128])
def test_groups_and_head_dims(group, head_dim):
    Hk = 2
    ctx = [1, 15, 16, 17, 700, 3000, 5000, 64]
    b = inputs.paged_batch([1] * len(ctx), ctx, Hk * group, Hk, head_dim, 16, dtype="bf16",
                           seed=group * 10 + head_dim)
    parity.compare(fast(b), parity.oracle_forward(b), "bf16", what=f"fast G{group} D{head_dim}")


def test_forced_short_splits_merge_in_kernel():
    b = inputs.paged_batch([1] * 5, [4000, 1, 2048, 333, 7000], 32, 8, 128, 16, dtype="bf16",
                           seed=31)
    got = fast(b, kv_split_tokens=256)
    parity.compare(got, parity.oracle_forward(b), "bf16", what="fast kvs 256")


def test_variants_and_hnd_layout():
    b = inputs.paged_batch([1] * 6, [900, 40, 2500, 1, 4100, 777], 32, 8, 128, 16, dtype="bf16",
                           seed=32)
    H = b.num_heads
    var = dict(sliding_window=300, sinks=np.linspace(-1.0, 2.0, H).astype(np.float32),
               alibi_slopes=(2.0 ** (-8.0 * np.arange(1, H + 1) / H)).astype(np.float32))
    want = parity.oracle_forward(b, **var)
    parity.compare(fast(b, **var), want, "bf16", what="fast variants")
    h = inputs.as_hnd(b)
    parity.compare(fast(h, **var), want, "bf16", what="fast variants hnd")


def test_repeated_calls_and_graph_replay():
    """Counters return to zero after every call: several calls in a row and a
    captured call replayed with new contents all stay correct."""
    H, Hk, D, bs = 32, 8, 128, 16
    b1 = inputs.paged_batch([1] * 6, [500, 1200, 64, 3000, 17, 800], H, Hk, D, bs, seed=33,
                            max_seq_len=4096, pool_pages=700)
    b2 = inputs.paged_batch([1] * 6, [4000, 20, 2222, 1, 999, 3500], H, Hk, D, bs, seed=34,
                            max_seq_len=4096, pool_pages=700)
    mb = max(b1.max_blocks_per_seq, b2.max_blocks_per_seq)

    def pad(t):
        o = torch.full((6, mb), -1, dtype=torch.int32)
        o[:, :t.shape[1]] = t
        return o

    b1.block_table, b2.block_table = pad(b1.block_table), pad(b2.block_table)
    for _ in range(3):
        parity.compare(fast(b1), parity.oracle_forward(b1), "bf16", what="fast repeat")
    d = pa.to_device(b1)
    out = torch.empty_like(d.q)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pa.forward(d, out=out, stream=s, max_query_len=1)  # warm-up: workspace and counters
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            pa.forward(d, out=out, stream=s, max_query_len=1)
    torch.cuda.synchronize()
    for b in (b2, b1, b2):
        d.q.copy_(b.q.cuda())
        d.k_cache.copy_(b.k_cache.cuda())
        d.v_cache.copy_(b.v_cache.cuda())
        d.block_table.copy_(b.block_table.cuda())
        d.seq_lens.copy_(b.seq_lens.cuda())
        g.replay()
        torch.cuda.synchronize()
        assert pa.pa_get_device_status() == 0
        got = out.float().cpu().numpy().astype(np.float64)
        parity.compare(got, parity.oracle_forward(b), "bf16", what="fast graph replay")


def test_bad_metadata_zeroes_only_its_request():
    b = inputs.paged_batch([1, 1, 1], [300, 2000, 90], 32, 8, 128, 16, dtype="bf16", seed=35)
    want = parity.oracle_forward(b)
    b.block_table[1, 5] = b.num_blocks + 3  # a visible page of request 1
    got = fast(b, expect_status=pa.PA_DEV_BAD_BLOCK)
    assert np.all(got[1] == 0.0)
    parity.compare(got[[0, 2]], want[[0, 2]], "bf16", what="fast healthy rows")
    b = inputs.paged_batch([1, 1], [300, 40], 32, 8, 128, 16, dtype="bf16", seed=36)
    want = parity.oracle_forward(b)
    b.max_seq_len = 200  # request 0 is longer than the bound
    got = fast(b, expect_status=pa.PA_DEV_BAD_SEQLEN)
    assert np.all(got[0] == 0.0)
    parity.compare(got[1:], want[1:], "bf16", what="fast healthy row")


def test_query_start_loc_must_be_the_identity():
    b = inputs.paged_batch([1, 1, 1], [300, 200, 100], 32, 8, 128, 16, dtype="bf16", seed=37)
    want = parity.oracle_forward(b)
    b.query_start_loc = torch.tensor([0, 1, 1, 3], dtype=torch.int32)  # request 1 empty, 2 two
    got = fast(b, expect_status=pa.PA_DEV_BAD_QSL)
    assert np.all(got[1] == 0.0) and np.all(got[2] == 0.0)
    parity.compare(got[:1], want[:1], "bf16", what="fast identity row")


def test_fp32_and_mixed_batches_take_the_planned_path():
    """max_query_len == 1 on a batch the one-launch path does not take (fp32)
    still runs the planned path; a larger bound does too."""
    b = inputs.tiny_decode_f32()
    parity.compare(fast(b), parity.oracle_forward(b), "f32", what="fast flag on fp32")
    b = inputs.paged_batch([1, 30, 1], [500, 64, 40], 32, 8, 128, 16, dtype="bf16", seed=38)
    got = parity.gpu_forward(b, max_query_len=30)
    parity.compare(got, parity.oracle_forward(b), "bf16", what="bound 30")


def test_requests_above_the_bound_are_bad_metadata():
    """A request with more new tokens than max_query_len is flagged
    PA_DEV_BAD_QLEN and its rows are zeros; the others stay exact (planned
    path: decode-only bound on a batch with one 3-token request, whose tile
    launch is skipped; and a bound of 30 on a batch with a 40-token extend)."""
    ctx = [300 + 37 * k for k in range(64)]
    q_lens = [1] * 64
    q_lens[40] = 3
    b = inputs.paged_batch(q_lens, ctx, 32, 8, 128, 16, dtype="bf16", seed=39)
    want = parity.oracle_forward(b)
    got = parity.gpu_forward(b, max_query_len=1, expect_status=pa.PA_DEV_BAD_QLEN)
    qsl = b.query_start_loc.numpy()
    bad = np.arange(qsl[40], qsl[41])
    keep = np.setdiff1d(np.arange(b.num_tokens), bad)
    assert np.all(got[bad] == 0.0)
    parity.compare(got[keep], want[keep], "bf16", what="bound 1, healthy rows")
    b = inputs.paged_batch([1, 40, 12, 1], [500, 900, 64, 40], 32, 8, 128, 16, dtype="bf16",
                           seed=40)
    want = parity.oracle_forward(b)
    got = parity.gpu_forward(b, max_query_len=30, expect_status=pa.PA_DEV_BAD_QLEN)
    qsl = b.query_start_loc.numpy()
    bad = np.arange(qsl[1], qsl[2])
    keep = np.setdiff1d(np.arange(b.num_tokens), bad)
    assert np.all(got[bad] == 0.0)
    parity.compare(got[keep], want[keep], "bf16", what="bound 30, healthy rows")


def test_large_batch_one_launch():
    """300 requests x 8 KV heads (more row groups than resident blocks)."""
    rng = np.random.default_rng(41)
    ctx = [int(x) for x in rng.integers(1, 6000, 300)]
    b = inputs.paged_batch([1] * 300, ctx, 32, 8, 128, 16, dtype="bf16", seed=41)
    parity.compare(fast(b), parity.oracle_forward(b), "bf16", what="fast 300 requests")


def test_up_to_64_splits_a_row():
    """kv_split_tokens 1024 on a 60K context: 59 splits, merged in-kernel."""
    b = inputs.paged_batch([1] * 3, [60000, 100, 33000], 16, 2, 128, 64, dtype="bf16", seed=42)
    parity.compare(fast(b, kv_split_tokens=1024), parity.oracle_forward(b), "bf16",
                   what="fast 59 splits")


@pytest.mark.parametrize("n", [1024, 1025])
def test_request_count_bound(n):
    """1024 requests run as one launch, 1025 on the planned path."""
    rng = np.random.default_rng(n)
    ctx = [int(x) for x in rng.integers(1, 300, n)]
    b = inputs.paged_batch([1] * n, ctx, 8, 2, 64, 16, dtype="bf16", seed=n)
    parity.compare(fast(b), parity.oracle_forward(b), "bf16", what=f"fast {n} requests")


def test_alternating_caches_reuse_no_stale_maps():
    """The decode row maps are reused while the caches and extents stay the
    same: calls that alternate between two caches of different shapes (and
    a third with the first's shape at another address) each stay exact."""
    b1 = inputs.paged_batch([1] * 5, [700, 40, 2000, 1, 333], 32, 8, 128, 16, dtype="bf16", seed=43)
    b2 = inputs.paged_batch([1] * 3, [5000, 64, 900], 16, 2, 64, 64, dtype="bf16", seed=44)
    b3 = inputs.paged_batch([1] * 5, [100, 2500, 17, 800, 64], 32, 8, 128, 16, dtype="bf16", seed=45)
    want = {id(b): parity.oracle_forward(b) for b in (b1, b2, b3)}
    for b in (b1, b2, b1, b3, b2, b3, b1):
        parity.compare(fast(b), want[id(b)], "bf16", what="alternating caches")
