"""pa_forward on the GPU against the fp64 oracle (element by element, same
seeded inputs), at small sizes that still span several tiles and pages with a
ragged tail, at the full workload sizes on sampled rows, and on the edge
cases: empty and zero-length requests, single-key contexts, forced splits,
bad metadata, request permutations and CUDA-graph replay."""
import math

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


# --------------------------------------------------------------------------
# the workloads
# --------------------------------------------------------------------------

def test_tiny_decode_f32_full():
    b = inputs.tiny_decode_f32()
    got = parity.gpu_forward(b)
    parity.compare(got, parity.oracle_forward(b), "f32", what="tiny fp32 decode")


def test_llama_decode_b1_full():
    b = inputs.llama_decode(1)
    got = parity.gpu_forward(b)
    parity.compare(got, parity.oracle_forward(b), "bf16", what="llama b1")


def test_llama_decode_b64_full():
    b = inputs.llama_decode(64)
    got = parity.gpu_forward(b)
    parity.compare(got, parity.oracle_forward(b), "bf16", what="llama b64")


def test_mixed_qwen3_sampled():
    """Every decode row, 1536 random extend / prefill rows, and the first and
    last row of every 128-row tile of the longest prefill and extend."""
    b = inputs.mixed_qwen3()
    edges = parity.tile_edge_rows(b, [parity.longest_requests(b, "prefill"),
                                      parity.longest_requests(b, "extend")])
    rows = np.unique(np.concatenate([parity.sample_rows(b, 1536, seed=1), edges]))
    got = parity.gpu_forward(b)
    parity.compare(got, parity.oracle_forward(b, rows=rows), "bf16", rows=rows, what="mixed")


def test_long_chunked_sampled():
    """Every decode row, 96 random extend rows, and the first and last row of
    every 128-row tile of one 2048-token extend on its 96K prefix."""
    b = inputs.long_chunked()
    edges = parity.tile_edge_rows(b, [parity.longest_requests(b, "extend")])
    rows = np.unique(np.concatenate([parity.sample_rows(b, 96, seed=2), edges]))
    got = parity.gpu_forward(b)
    parity.compare(got, parity.oracle_forward(b, rows=rows), "bf16", rows=rows, what="long")


# --------------------------------------------------------------------------
# shapes: every group size and head_dim, both dtypes, ragged small batches
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("group", [1, 2, 4, 8, 16])
def test_small_mixed_all_shapes(dtype, head_dim, group):
    Hk = 2
    q_lens = [1, 1, 37, 5, 1, 130, 0, 3]
    ctx = [1, 300, 37, 261, 17, 200, 9, 3]
    b = inputs.paged_batch(q_lens, ctx, Hk * group, Hk, head_dim, 16, dtype=dtype,
                           seed=group * 10 + head_dim)
    got = parity.gpu_forward(b)
    parity.compare(got, parity.oracle_forward(b), dtype, what=f"{dtype} D{head_dim} G{group}")


@pytest.mark.parametrize("block_size", [16, 32, 64, 256])
def test_block_sizes(block_size):
    b = inputs.paged_batch([1, 9, 1, 70], [1000, 333, 64, 70], 16, 4, 128, block_size,
                           dtype="bf16", seed=block_size)
    got = parity.gpu_forward(b)
    parity.compare(got, parity.oracle_forward(b), "bf16", what=f"bs{block_size}")


@pytest.mark.parametrize("kvs", [16, 48, 256, 32768])
def test_forced_splits_match_oracle(kvs):
    b = inputs.paged_batch([1, 1, 40, 1], [2000, 70, 300, 16], 8, 2, 128, 16, dtype="bf16",
                           seed=kvs)
    got = parity.gpu_forward(b, kv_split_tokens=kvs)
    parity.compare(got, parity.oracle_forward(b), "bf16", what=f"kvs {kvs}")


@pytest.mark.parametrize("kvs", [0, 64])
def test_more_requests_than_one_planner_block(kvs):
    """1500 requests (the planner and the merge kernel keep up to 1024
    requests in shared memory; beyond that they read the lists from global
    memory): mostly decodes, some extends, a few long contexts whose rows
    have more than 32 splits at kv_split_tokens = 64."""
    rng = np.random.default_rng(1500 + kvs)
    n = 1500
    q_lens = [1] * n
    ctx = [int(x) for x in rng.integers(1, 300, n)]
    for i in range(0, n, 97):  # extends
        q_lens[i] = int(rng.integers(2, 40))
        ctx[i] = q_lens[i] + int(rng.integers(0, 200))
    for i in (5, 700, 1499):  # long rows
        q_lens[i], ctx[i] = 1, 3000
    b = inputs.paged_batch(q_lens, ctx, 16, 4, 128, 16, dtype="bf16", seed=1500 + kvs)
    got = parity.gpu_forward(b, kv_split_tokens=kvs)
    parity.compare(got, parity.oracle_forward(b), "bf16", what=f"1500 requests kvs {kvs}")


# --------------------------------------------------------------------------
# edge cases
# --------------------------------------------------------------------------

def test_empty_batch():
    q = torch.empty((0, 8, 128), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((1, 16, 2, 128), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((0, 1), dtype=torch.int32, device="cuda")
    sl = torch.zeros((0,), dtype=torch.int32, device="cuda")
    qsl = torch.zeros((1,), dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    pa.pa_forward(q, kc, kc, bt, sl, qsl, 8, 2, 128, 16, 0.1, out, max_seq_len=16)
    torch.cuda.synchronize()
    assert pa.pa_get_device_status() == 0


def test_zero_length_requests_and_single_keys():
    b = inputs.paged_batch([0, 1, 0, 1, 2, 0], [5, 1, 0, 1, 2, 33], 8, 8, 64, 16, dtype="f32",
                           seed=3)
    got = parity.gpu_forward(b)
    parity.compare(got, parity.oracle_forward(b), "f32", what="zero-length")


def test_bad_block_id_zeroes_affected_rows():
    b = inputs.paged_batch([1, 1, 4], [100, 50, 40], 8, 2, 128, 16, dtype="bf16", seed=5)
    want = parity.oracle_forward(b)
    b.block_table[1, 2] = b.num_blocks + 5  # page 2 of request 1 (positions 32..47)
    got = parity.gpu_forward(b, expect_status=pa.PA_DEV_BAD_BLOCK)
    H = b.num_heads
    assert np.all(got[1] == 0.0)
    parity.compare(got[[0, 2, 3, 4, 5]], want[[0, 2, 3, 4, 5]], "bf16", what="healthy rows")


def test_q_len_above_context_is_flagged():
    b = inputs.paged_batch([1, 3, 2], [30, 20, 2], 8, 2, 64, 16, dtype="f32", seed=6)
    want = parity.oracle_forward(b)
    b.seq_lens[1] = 2  # q_len 3 > seq_len 2
    got = parity.gpu_forward(b, expect_status=pa.PA_DEV_BAD_QLEN)
    assert np.all(got[1:4] == 0.0)
    parity.compare(got[[0, 4, 5]], want[[0, 4, 5]], "f32", what="healthy rows")


def test_seq_len_above_bound_is_flagged():
    b = inputs.paged_batch([1, 1], [30, 20], 8, 2, 64, 16, dtype="f32", seed=7)
    want = parity.oracle_forward(b)
    b.max_seq_len = 25
    got = parity.gpu_forward(b, expect_status=pa.PA_DEV_BAD_SEQLEN)
    assert np.all(got[0] == 0.0)
    parity.compare(got[1:], want[1:], "f32", what="healthy rows")


def test_bad_query_start_loc_zeroes_everything():
    b = inputs.paged_batch([1, 2], [30, 20], 8, 2, 64, 16, dtype="f32", seed=8)
    b.query_start_loc[2] = 2  # != num_tokens (3)
    got = parity.gpu_forward(b, expect_status=pa.PA_DEV_BAD_QSL)
    assert np.all(got == 0.0)


def test_request_permutation_is_bit_exact():
    q_lens = [1, 7, 1, 20, 1]
    ctx = [900, 50, 33, 20, 4000]
    b = inputs.paged_batch(q_lens, ctx, 16, 4, 128, 16, dtype="bf16", seed=9)
    base = parity.gpu_forward(b)
    perm = [4, 1, 3, 0, 2]
    qsl = b.query_start_loc.numpy()
    rows = np.concatenate([np.arange(qsl[s], qsl[s + 1]) for s in perm])
    pq_lens = [q_lens[s] for s in perm]
    pb = inputs.PagedBatch(
        q=b.q[torch.from_numpy(rows)], k_cache=b.k_cache, v_cache=b.v_cache,
        block_table=b.block_table[torch.tensor(perm)], seq_lens=b.seq_lens[torch.tensor(perm)],
        query_start_loc=torch.tensor(np.concatenate([[0], np.cumsum(pq_lens)]), dtype=torch.int32),
        num_heads=16, num_kv_heads=4, head_dim=128, block_size=16, scale=b.scale, dtype="bf16",
        max_seq_len=b.max_seq_len)
    got = parity.gpu_forward(pb)
    np.testing.assert_array_equal(got, base[rows])


def test_debug_gather_is_bit_exact():
    from oracle import oracle as orc
    b = inputs.paged_batch([1, 1, 1], [77, 16, 300], 8, 2, 64, 16, dtype="bf16", seed=10)
    d = pa.to_device(b)
    msl = 300
    dense = torch.zeros((3, msl, 2 * 64), dtype=torch.bfloat16, device="cuda")
    pa.pa_debug_gather(d.k_cache, d.block_table, d.seq_lens, 16, msl, dense)
    torch.cuda.synchronize()
    want = orc.gather_rows(inputs.storage_array(b.k_cache), b.block_table.numpy(),
                           b.seq_lens.numpy(), 16, msl)
    got = dense.cpu().view(torch.int16).numpy().view(np.uint16)
    for s, c in enumerate([77, 16, 300]):
        np.testing.assert_array_equal(got[s, :c], want[s, :c])


def test_cuda_graph_replay_with_new_metadata():
    """Capture once; change seq_lens / block_table / q contents within the
    captured capacities; replay; re-check parity."""
    H, Hk, D, bs = 32, 8, 128, 16
    b1 = inputs.paged_batch([1] * 6, [500, 1200, 64, 3000, 17, 800], H, Hk, D, bs, seed=11,
                            max_seq_len=4096, pool_pages=700)
    b2 = inputs.paged_batch([1] * 6, [4000, 20, 2222, 1, 999, 3500], H, Hk, D, bs, seed=12,
                            max_seq_len=4096, pool_pages=700)
    mb = max(b1.max_blocks_per_seq, b2.max_blocks_per_seq)

    def pad(t):
        o = torch.full((6, mb), -1, dtype=torch.int32)
        o[:, :t.shape[1]] = t
        return o

    b1.block_table, b2.block_table = pad(b1.block_table), pad(b2.block_table)
    d = pa.to_device(b1)
    out = torch.empty_like(d.q)
    need = pa.pa_forward_workspace_bytes(pa.PA_BF16, 6, 6, H, Hk, D, 4096)
    pa.pa_reserve(need)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pa.forward(d, out=out, stream=s)  # warm-up outside capture
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            pa.forward(d, out=out, stream=s)
    torch.cuda.synchronize()
    for b in (b1, b2):
        d.q.copy_(b.q.cuda())
        d.k_cache.copy_(b.k_cache.cuda())
        d.v_cache.copy_(b.v_cache.cuda())
        d.block_table.copy_(b.block_table.cuda())
        d.seq_lens.copy_(b.seq_lens.cuda())
        g.replay()
        torch.cuda.synchronize()
        assert pa.pa_get_device_status() == 0
        got = out.float().cpu().numpy().astype(np.float64)
        parity.compare(got, parity.oracle_forward(b), "bf16", what="graph replay")


def test_capture_without_workspace_is_refused():
    """During capture the library never allocates: a call that needs more
    workspace than reserved returns PA_ERR_WORKSPACE."""
    b = pa.to_device(inputs.paged_batch([1], [64], 8, 2, 64, 16, dtype="f32", seed=13))
    out = torch.empty_like(b.q)
    s = torch.cuda.Stream()
    huge = 2**31 - 1  # a max_seq_len far beyond anything reserved so far
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        g.capture_begin()
        try:
            st = pa.pa_forward(b.q, b.k_cache, b.v_cache, b.block_table, b.seq_lens,
                               b.query_start_loc, 8, 2, 64, 16, b.scale, out, s,
                               max_seq_len=huge, check=False)
        finally:
            g.capture_end()
    assert st == pa.PA_ERR_WORKSPACE


# --------------------------------------------------------------------------
# tensor-core tile path (bf16 extend / prefill)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("group", [1, 4, 16])
def test_tile_prefill_and_extend_full(group):
    Hk = 2
    b = inputs.paged_batch([600, 1, 300, 77], [600, 1500, 1300, 77], Hk * group, Hk, 128, 16,
                           dtype="bf16", seed=100 + group)
    got = parity.gpu_forward(b)
    parity.compare(got, parity.oracle_forward(b), "bf16", what=f"tile G{group}")


def test_tile_chunked_extend_matches_unchunked():
    b = inputs.paged_batch([200, 1], [3000, 2500], 16, 2, 128, 64, dtype="bf16", seed=7)
    want = parity.oracle_forward(b)
    for kvs in (0, 1024, 2048):
        got = parity.gpu_forward(b, kv_split_tokens=kvs)
        parity.compare(got, want, "bf16", what=f"chunk {kvs}")


@pytest.mark.parametrize("kvs", [64, 96])
def test_tile_equal_splits_on_a_large_extend(kvs):
    """Tile rows under kv_split_tokens are cut into equal splits of whole
    64-position tiles (doubled in count only when the batch's tile work is
    small against the tile grid, which depends on the SM count): with two
    extends of 300 and 200 tokens on 8000 and 6000 positions the 8000-position
    request has over 80 splits, so its rows also take the merge's block pass."""
    b = inputs.paged_batch([300, 1, 200], [8000, 3000, 6000], 16, 4, 128, 16, dtype="bf16",
                           seed=500 + kvs)
    got = parity.gpu_forward(b, kv_split_tokens=kvs)
    parity.compare(got, parity.oracle_forward(b), "bf16", what=f"equal splits kvs {kvs}")


def test_bad_block_in_extend_zeroes_its_rows():
    b = inputs.paged_batch([1, 40, 30], [100, 540, 30], 16, 2, 128, 16, dtype="bf16", seed=21)
    want = parity.oracle_forward(b)
    b.block_table[1, 3] = -7  # positions 48..63 of the extend request (prefix 500)
    got = parity.gpu_forward(b, expect_status=pa.PA_DEV_BAD_BLOCK)
    assert np.all(got[1:41] == 0.0)
    parity.compare(got[[0] + list(range(41, 71))], want[[0] + list(range(41, 71))], "bf16",
                   what="healthy rows")
