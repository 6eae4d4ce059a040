"""The head-major (HND) KV-cache layout on the GPU: pa_forward_ex over HND
caches against the oracle reading the same storage, and bit for bit against
the NHD result (the layout changes where bytes sit, not what the kernels
compute); pa_cache_write into HND caches bit-exact against the oracle."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from paged_kv_attention_16_gb300 import inputs, pa
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_attention_16_gb300 import build
    build.build()
    pa.lib()
    pa.pa_get_device_status()  # clear


def oracle_hnd(b, rows=None):
    return orc.paged_attention(
        inputs.storage_array(b.q), inputs.storage_array(b.k_cache),
        inputs.storage_array(b.v_cache), b.block_table.numpy(), b.seq_lens.numpy(),
        b.query_start_loc.numpy(), b.num_heads, b.num_kv_heads, b.head_dim, b.block_size,
        b.scale, rows=rows, kv_layout="hnd")


def both_layouts(b, kv_split_tokens=None):
    """(NHD output, HND output) as raw device tensors."""
    dn = pa.to_device(b)
    dh = pa.to_device(inputs.as_hnd(b))
    on = pa.forward(dn, kv_split_tokens=kv_split_tokens)
    oh = pa.forward(dh, kv_split_tokens=kv_split_tokens)
    assert pa.pa_get_device_status() == 0
    return on, oh


def bits(t):
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("group", [1, 4, 16])
def test_hnd_small_mixed(dtype, head_dim, group):
    Hk = 2
    b = inputs.paged_batch([1, 1, 37, 5, 1, 130, 0, 3], [1, 300, 37, 261, 17, 200, 9, 3],
                           Hk * group, Hk, head_dim, 16, dtype=dtype, seed=group * 3 + head_dim)
    on, oh = both_layouts(b)
    assert torch.equal(bits(on), bits(oh))
    got = oh.float().cpu().numpy().astype(np.float64)
    parity.compare(got, oracle_hnd(inputs.as_hnd(b)), dtype,
                   what=f"hnd {dtype} D{head_dim} G{group}")


@pytest.mark.parametrize("block_size", [16, 64, 256])
@pytest.mark.parametrize("kvs", [0, 48])
def test_hnd_block_sizes_and_splits(block_size, kvs):
    b = inputs.paged_batch([1, 9, 1, 70], [1000, 333, 64, 70], 16, 4, 128, block_size,
                           dtype="bf16", seed=block_size + kvs)
    on, oh = both_layouts(b, kv_split_tokens=kvs)
    assert torch.equal(bits(on), bits(oh))
    got = oh.float().cpu().numpy().astype(np.float64)
    parity.compare(got, oracle_hnd(inputs.as_hnd(b)), "bf16", what=f"hnd bs{block_size} kvs{kvs}")


def test_hnd_llama_decode_b64_full():
    b = inputs.llama_decode(64)
    on, oh = both_layouts(b)
    assert torch.equal(bits(on), bits(oh))
    got = oh.float().cpu().numpy().astype(np.float64)
    parity.compare(got, oracle_hnd(inputs.as_hnd(b)), "bf16", what="hnd llama b64")


def test_hnd_mixed_qwen3_sampled():
    b = inputs.mixed_qwen3()
    on, oh = both_layouts(b)
    assert torch.equal(bits(on), bits(oh))
    rows = parity.sample_rows(b, 512, seed=9)
    got = oh.float().cpu().numpy().astype(np.float64)
    parity.compare(got, oracle_hnd(inputs.as_hnd(b), rows=rows), "bf16", rows=rows,
                   what="hnd mixed")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("block_size", [16, 64])
def test_hnd_cache_write_bit_exact(dtype, block_size):
    b = inputs.as_hnd(inputs.paged_batch([1, 7, 0, 33, 1, 130], [1, 20, 5, 33, 300, 400], 8, 2,
                                          128, block_size, dtype=dtype, seed=block_size))
    g = torch.Generator().manual_seed(17)
    k_new = torch.randn((b.num_tokens, 2, 128), generator=g).to(b.k_cache.dtype)
    v_new = torch.randn((b.num_tokens, 2, 128), generator=g).to(b.k_cache.dtype)
    kc = torch.randn(b.k_cache.shape, generator=g).to(b.k_cache.dtype)
    vc = torch.randn(b.v_cache.shape, generator=g).to(b.v_cache.dtype)
    want_k, want_v, want_st = orc.cache_write(
        inputs.storage_array(k_new), inputs.storage_array(v_new), inputs.storage_array(kc),
        inputs.storage_array(vc), b.block_table.numpy(), b.seq_lens.numpy(),
        b.query_start_loc.numpy(), b.block_size, kv_layout="hnd")
    assert want_st == 0
    d_kc, d_vc = kc.cuda(), vc.cuda()
    pa.pa_cache_write(k_new.cuda(), v_new.cuda(), d_kc, d_vc, b.block_table.cuda(),
                      b.seq_lens.cuda(), b.query_start_loc.cuda(), b.block_size, kv_layout="hnd")
    assert pa.pa_get_device_status() == 0
    gk, gv = inputs.storage_array(d_kc.cpu()), inputs.storage_array(d_vc.cpu())
    assert np.array_equal(gk.view(np.uint8), want_k.view(np.uint8))
    assert np.array_equal(gv.view(np.uint8), want_v.view(np.uint8))
