"""pa_cache_write on the GPU against the oracle's cache write: the caches
must match bit for bit (a write copies bits), on decode, extend and prefill
rows, zero-length requests, page crossings and both block sizes; bad metadata
sets its status bit and skips exactly what the oracle skips; a write followed
by pa_forward gives the oracle's attention."""
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


def new_rows(b):
    """The new tokens' K and V rows, read out of a batch whose caches already
    hold them: [T, Hk, D] each (torch, on the host)."""
    qsl = b.query_start_loc.tolist()
    ctx = b.seq_lens.tolist()
    bs = b.block_size
    k = torch.empty((b.num_tokens, b.num_kv_heads, b.head_dim), dtype=b.k_cache.dtype)
    v = torch.empty_like(k)
    for s in range(b.num_seqs):
        q_len = qsl[s + 1] - qsl[s]
        for i in range(q_len):
            pos = ctx[s] - q_len + i
            page = int(b.block_table[s, pos // bs])
            k[qsl[s] + i] = b.k_cache[page, pos % bs]
            v[qsl[s] + i] = b.v_cache[page, pos % bs]
    return k, v


def run_both(b, k_new, v_new, seed, expect_status=0):
    """Stale random caches; the GPU write and the oracle's write of the same
    rows; returns (GPU caches, oracle caches) as host storage arrays."""
    g = torch.Generator().manual_seed(seed)
    kc = torch.randn(b.k_cache.shape, generator=g).to(b.k_cache.dtype)
    vc = torch.randn(b.v_cache.shape, generator=g).to(b.v_cache.dtype)
    want_k, want_v, want_st = orc.cache_write(
        inputs.storage_array(k_new), inputs.storage_array(v_new), inputs.storage_array(kc),
        inputs.storage_array(vc), b.block_table.numpy(), b.seq_lens.numpy(),
        b.query_start_loc.numpy(), b.block_size)
    assert want_st == expect_status
    d_kc, d_vc = kc.cuda(), vc.cuda()
    pa.pa_cache_write(k_new.cuda(), v_new.cuda(), d_kc, d_vc, b.block_table.cuda(),
                      b.seq_lens.cuda(), b.query_start_loc.cuda(), b.block_size)
    assert pa.pa_get_device_status() == expect_status
    return (inputs.storage_array(d_kc.cpu()), inputs.storage_array(d_vc.cpu())), (want_k, want_v)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("block_size", [16, 64])
@pytest.mark.parametrize("head_dim", [64, 128])
def test_cache_write_bit_exact(dtype, block_size, head_dim):
    b = inputs.paged_batch([1, 7, 0, 33, 1, 130], [1, 20, 5, 33, 300, 400], 8, 2, head_dim,
                           block_size, dtype=dtype, seed=block_size + head_dim)
    g = torch.Generator().manual_seed(7)
    k_new = torch.randn((b.num_tokens, 2, head_dim), generator=g).to(b.k_cache.dtype)
    v_new = torch.randn((b.num_tokens, 2, head_dim), generator=g).to(b.k_cache.dtype)
    (gk, gv), (wk, wv) = run_both(b, k_new, v_new, seed=11)
    assert np.array_equal(gk.view(np.uint8), wk.view(np.uint8))
    assert np.array_equal(gv.view(np.uint8), wv.view(np.uint8))


def test_write_then_attend():
    """Overwrite the new tokens' slots with NaN, write them back through
    pa_cache_write, then pa_forward: the caches are bit-identical to the
    original and the attention matches the oracle on the original batch."""
    b = inputs.paged_batch([1, 1, 24, 60, 1], [900, 65, 200, 60, 3], 16, 4, 128, 16,
                           dtype="bf16", seed=3)
    k_new, v_new = new_rows(b)
    d = pa.to_device(b)
    qsl, ctx = b.query_start_loc.tolist(), b.seq_lens.tolist()
    for s in range(b.num_seqs):
        q_len = qsl[s + 1] - qsl[s]
        for pos in range(ctx[s] - q_len, ctx[s]):
            page = int(b.block_table[s, pos // 16])
            d.k_cache[page, pos % 16] = float("nan")
            d.v_cache[page, pos % 16] = float("nan")
    pa.pa_cache_write(k_new.cuda(), v_new.cuda(), d.k_cache, d.v_cache, d.block_table,
                      d.seq_lens, d.query_start_loc, b.block_size)
    assert torch.equal(d.k_cache.cpu().view(torch.int16), b.k_cache.view(torch.int16))
    assert torch.equal(d.v_cache.cpu().view(torch.int16), b.v_cache.view(torch.int16))
    got = pa.forward(d).float().cpu().numpy().astype(np.float64)
    assert pa.pa_get_device_status() == 0
    parity.compare(got, parity.oracle_forward(b), "bf16", what="write then attend")


def _small():
    b = inputs.paged_batch([2, 3, 1], [6, 7, 40], 8, 2, 64, 16, dtype="f32", seed=5)
    g = torch.Generator().manual_seed(5)
    k_new = torch.randn((b.num_tokens, 2, 64), generator=g)
    v_new = torch.randn((b.num_tokens, 2, 64), generator=g)
    return b, k_new, v_new


def test_bad_block_skips_only_its_rows():
    b, k_new, v_new = _small()
    b.block_table[2, 2] = b.k_cache.shape[0] + 9  # the page of the decode token (pos 39)
    (gk, gv), (wk, wv) = run_both(b, k_new, v_new, seed=12, expect_status=pa.PA_DEV_BAD_BLOCK)
    assert np.array_equal(gk, wk) and np.array_equal(gv, wv)


def test_q_len_above_context_skips_its_request():
    b, k_new, v_new = _small()
    b.seq_lens[1] = 2
    (gk, gv), (wk, wv) = run_both(b, k_new, v_new, seed=13, expect_status=pa.PA_DEV_BAD_QLEN)
    assert np.array_equal(gk, wk) and np.array_equal(gv, wv)


def test_bad_query_start_loc_writes_nothing():
    b, k_new, v_new = _small()
    b.query_start_loc[1], b.query_start_loc[2] = 5, 2  # decreasing
    (gk, gv), (wk, wv) = run_both(b, k_new, v_new, seed=14, expect_status=pa.PA_DEV_BAD_QSL)
    assert np.array_equal(gk, wk) and np.array_equal(gv, wv)
