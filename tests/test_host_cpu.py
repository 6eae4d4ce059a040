"""Host-side logic, CPU only: the bench's algorithmic byte and FLOP counts
(which the roofline fractions divide by) against brute-force counts over the
visible (row, key) pairs, with and without a sliding window; and the seeded
input generators (deterministic, the documented shapes, HND a permutation of
NHD, poison only where no kernel may read)."""
import numpy as np
import torch

import bench
from paged_kv_attention_16_gb300 import inputs


def _visible_pairs(b, window=0):
    qsl, ctx = b.query_start_loc.tolist(), b.seq_lens.tolist()
    pairs, seen = 0, 0
    for s in range(b.num_seqs):
        ql = qsl[s + 1] - qsl[s]
        keys = set()
        for i in range(ql):
            p = ctx[s] - ql + i
            lo = max(0, p - window + 1) if window else 0
            pairs += p - lo + 1
            keys.update(range(lo, p + 1))
        seen += len(keys)
    return pairs, seen


def test_flops_and_bytes_match_brute_force():
    b = inputs.paged_batch([1, 5, 9, 0, 33], [20, 22, 9, 4, 40], 8, 2, 64, 16, dtype="f32",
                           seed=1, poison=False)
    for window in (0, 1, 4, 16, 1000):
        pairs, seen = _visible_pairs(b, window)
        assert bench.attn_flops(b, window) == 4 * 64 * 8 * pairs
        if window:
            assert bench.kv_bytes(b, window) == seen * 2 * 64 * 4 * 2
    assert bench.kv_bytes(b) == _visible_pairs(b, 10**9)[1] * 2 * 64 * 4 * 2


def test_generators_are_seeded_and_shaped():
    a = inputs.mixed_qwen3(poison=False)
    b = inputs.mixed_qwen3(poison=False)
    assert torch.equal(a.q.view(torch.int16), b.q.view(torch.int16))
    assert torch.equal(a.block_table, b.block_table)
    assert a.num_seqs == 64 and a.num_heads == 64 and a.num_kv_heads == 4
    q_lens = (a.query_start_loc[1:] - a.query_start_loc[:-1]).tolist()
    assert sorted(q_lens).count(1) == 48
    m = inputs.mla_prefill_deepseek(poison=False)
    assert m.q.shape[1:] == (128, 192) and m.kv_cache.shape[1:] == (64, 576)
    assert m.w_kv.shape == (128, 256, 512)
    assert m.max_total_kv == int(m.seq_lens.sum())
    w = m.w_kv.float()
    assert abs(float(w.std()) * np.sqrt(512) - 1.0) < 0.02  # N(0, 1/512)


def test_hnd_is_a_permutation_of_nhd():
    b = inputs.paged_batch([1, 3], [40, 17], 8, 2, 64, 16, dtype="bf16", seed=3)
    h = inputs.as_hnd(b)
    assert h.kv_layout == "hnd" and h.k_cache.shape == (b.k_cache.shape[0], 2, 16, 64)
    assert torch.equal(h.k_cache.permute(0, 2, 1, 3).view(torch.int16),
                       b.k_cache.view(torch.int16))
    assert torch.equal(h.block_table, b.block_table)


def test_poison_only_where_nothing_may_read():
    """NaN only in unused pages and past each context; block-table entries
    past each context's pages are never valid page ids."""
    b = inputs.paged_batch([1, 2, 7], [33, 16, 70], 4, 1, 64, 16, dtype="f32", seed=4)
    ctx, bs = b.seq_lens.tolist(), b.block_size
    nb = b.k_cache.shape[0]
    used = set()
    for s, c in enumerate(ctx):
        for lp in range(-(-c // bs)):
            page = int(b.block_table[s, lp])
            assert 0 <= page < nb
            used.add(page)
            n = min(bs, c - lp * bs)
            assert torch.isfinite(b.k_cache[page, :n]).all()
            assert torch.isnan(b.k_cache[page, n:]).all()
        for lp in range(-(-c // bs), b.block_table.shape[1]):
            assert not 0 <= int(b.block_table[s, lp]) < nb
    for page in set(range(nb)) - used:
        assert torch.isnan(b.k_cache[page]).all()
