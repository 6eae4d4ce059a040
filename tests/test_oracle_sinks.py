"""Pins for the oracle's sink tokens (CPU only): a brute-force softmax with
the sink as one more column that carries no value, and two closed forms (a
sink at -inf changes nothing; a sink equal to the row's key log-sum-exp
halves the output)."""
import math

import numpy as np

from oracle import oracle as orc
from tests import oracle_pins


def _problem(seed):
    q_lens, ctx = [1, 3, 2], [5, 7, 2]
    H, Hk, D, bs = 4, 2, 8, 4
    qs, ks, vs = oracle_pins.make_dense(q_lens, ctx, H, Hk, D, seed)
    kc, vc, bt = oracle_pins.scatter_pages(ks, vs, bs, seed)
    q = np.concatenate(qs).astype(np.float32)
    qsl = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    return dict(q=q, k_cache=kc, v_cache=vc, block_table=bt, seq_lens=np.array(ctx, np.int32),
                query_start_loc=qsl, num_heads=H, num_kv_heads=Hk, head_dim=D, block_size=bs,
                scale=0.7), (qs, ks, vs, q_lens, ctx)


def test_sinks_match_brute_force():
    p, (qs, ks, vs, q_lens, ctx) = _problem(3)
    sinks = np.array([0.5, -1.0, 2.0, 0.0])
    got = orc.paged_attention(**p, sinks=sinks)
    H, G = p["num_heads"], p["num_heads"] // p["num_kv_heads"]
    t = 0
    for s, (ql, c) in enumerate(zip(q_lens, ctx)):
        for i in range(ql):
            for h in range(H):
                k = ks[s][: c - ql + i + 1, h // G].astype(np.float64)
                v = vs[s][: c - ql + i + 1, h // G].astype(np.float64)
                sc = p["scale"] * (k @ qs[s][i, h].astype(np.float64))
                cols = np.concatenate([sc, [sinks[h]]])
                w = np.exp(cols - cols.max())
                w /= w.sum()
                want = w[:-1] @ v
                np.testing.assert_allclose(got[t, h], want, rtol=1e-12, atol=1e-14)
            t += 1


def test_sink_at_minus_infinity_changes_nothing():
    p, _ = _problem(4)
    plain = orc.paged_attention(**p)
    got = orc.paged_attention(**p, sinks=np.full(p["num_heads"], -np.inf))
    np.testing.assert_array_equal(got, plain)


def test_sink_equal_to_key_lse_halves_the_output():
    p, _ = _problem(5)
    plain, lse = orc.paged_attention(**p, with_lse=True)
    # one token's lse per head as the sinks: that token's rows halve exactly
    t = 2
    got = orc.paged_attention(**p, sinks=lse[t])
    np.testing.assert_allclose(got[t], 0.5 * plain[t], rtol=1e-14, atol=0)
    assert math.isfinite(float(lse[t].sum()))
