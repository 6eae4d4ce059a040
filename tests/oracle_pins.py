"""Pins for the fp64 oracle: each check compares it with something other than
itself -- torch's own scaled_dot_product_attention in fp64 (a library routine
for the prefix-free special case, and with an explicit mask for extend), closed
forms (single key, identical keys, zero scale, rows of p summing to one), a
hand-worked example, and invariants (page placement, request order, split-KV
merged by log-sum-exp).

Every pin takes the oracle library handle so that the mutation tests can run
the same pins against deliberately broken copies of the oracle.
"""
import math
import os

import numpy as np
import torch

from oracle import oracle as orc
from paged_kv_attention_16_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------------------
# helpers: build paged problems from dense per-request K/V by scattering rows
# into a permuted page pool (the inverse of the oracle's gather)
# ---------------------------------------------------------------------------

def scatter_pages(dense_k, dense_v, block_size, seed, extra_pages=3):
    """dense_k[s]: [ctx_s, Hk, D] float32 arrays.  Returns caches, table."""
    rng = np.random.default_rng(seed)
    pages = [math.ceil(k.shape[0] / block_size) for k in dense_k]
    pool = sum(pages) + extra_pages
    Hk, D = dense_k[0].shape[1:]
    kc = np.full((pool, block_size, Hk, D), np.nan, dtype=np.float32)
    vc = np.full_like(kc, np.nan)
    perm = rng.permutation(pool)
    table = np.full((len(dense_k), max(pages)), -1, dtype=np.int32)
    off = 0
    for s, (k, v) in enumerate(zip(dense_k, dense_v)):
        for p in range(pages[s]):
            page = perm[off + p]
            table[s, p] = page
            rows = slice(p * block_size, min((p + 1) * block_size, k.shape[0]))
            n = rows.stop - rows.start
            kc[page, :n] = k[rows]
            vc[page, :n] = v[rows]
        off += pages[s]
    return kc, vc, table


def make_dense(q_lens, ctx_lens, H, Hk, D, seed):
    rng = np.random.default_rng(seed)
    qs = [rng.standard_normal((ql, H, D)).astype(np.float32) for ql in q_lens]
    ks = [rng.standard_normal((c, Hk, D)).astype(np.float32) for c in ctx_lens]
    vs = [rng.standard_normal((c, Hk, D)).astype(np.float32) for c in ctx_lens]
    return qs, ks, vs


def run_oracle(lib, qs, ks, vs, q_lens, ctx_lens, H, Hk, D, bs, scale, seed=0, **kw):
    kc, vc, table = scatter_pages(ks, vs, bs, seed)
    q = np.concatenate(qs, 0) if qs else np.zeros((0, H, D), np.float32)
    qsl = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    return orc.paged_attention(q, kc, vc, table, np.array(ctx_lens, np.int32), qsl, H, Hk, D,
                               bs, scale, lib=lib, **kw)


def sdpa_request(q, k, v, ctx, scale):
    """torch SDPA in fp64 for one request: q [ql, H, D], k/v [ctx, Hk, D];
    bottom-right causal mask given explicitly."""
    ql, H, D = q.shape
    Hk = k.shape[1]
    G = H // Hk
    qt = torch.from_numpy(q.astype(np.float64)).permute(1, 0, 2)[None]
    kt = torch.from_numpy(k.astype(np.float64)).repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    vt = torch.from_numpy(v.astype(np.float64)).repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    prefix = ctx - ql
    mask = torch.arange(ctx)[None, :] <= (prefix + torch.arange(ql))[:, None]
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask,
                                                           scale=scale)
    return out[0].permute(1, 0, 2).numpy()


# ---------------------------------------------------------------------------
# pins
# ---------------------------------------------------------------------------

def pin_sdpa_prefill_causal(lib):
    """Prefix-free prefill equals SDPA(is_causal=True) with K/V repeated per
    GQA group (textbook special case)."""
    H, Hk, D, bs = 8, 2, 16, 4
    ql = 37
    qs, ks, vs = make_dense([ql], [ql], H, Hk, D, seed=11)
    scale = 0.3
    out = run_oracle(lib, qs, ks, vs, [ql], [ql], H, Hk, D, bs, scale, seed=5)
    G = H // Hk
    qt = torch.from_numpy(qs[0].astype(np.float64)).permute(1, 0, 2)[None]
    kt = torch.from_numpy(ks[0].astype(np.float64)).repeat_interleave(G, 1).permute(1, 0, 2)[None]
    vt = torch.from_numpy(vs[0].astype(np.float64)).repeat_interleave(G, 1).permute(1, 0, 2)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True,
                                                           scale=scale)[0].permute(1, 0, 2)
    np.testing.assert_allclose(out, ref.numpy(), rtol=0, atol=1e-12)


def pin_sdpa_mixed_batch(lib):
    """decode + extend + prefill in one batch, random page placement: each
    request equals SDPA with the bottom-right causal mask."""
    H, Hk, D, bs = 6, 3, 8, 4
    q_lens = [1, 5, 9, 1, 3]
    ctx = [13, 22, 9, 1, 3]
    qs, ks, vs = make_dense(q_lens, ctx, H, Hk, D, seed=12)
    scale = 1 / math.sqrt(D)
    out = run_oracle(lib, qs, ks, vs, q_lens, ctx, H, Hk, D, bs, scale, seed=6)
    off = 0
    for s in range(len(q_lens)):
        ref = sdpa_request(qs[s], ks[s], vs[s], ctx[s], scale)
        np.testing.assert_allclose(out[off:off + q_lens[s]], ref, rtol=0, atol=1e-12)
        off += q_lens[s]


def pin_extend_is_tail_of_prefill(lib):
    """Rows of an extend request equal the last q_len rows of a prefill over
    the same ctx tokens; a decode equals the last row."""
    H, Hk, D, bs = 4, 1, 8, 8
    ctx = 29
    qs, ks, vs = make_dense([ctx], [ctx], H, Hk, D, seed=13)
    scale = 0.25
    full = run_oracle(lib, qs, ks, vs, [ctx], [ctx], H, Hk, D, bs, scale, seed=7)
    for ql in (1, 4, 11):
        part = run_oracle(lib, [qs[0][ctx - ql:]], ks, vs, [ql], [ctx], H, Hk, D, bs, scale,
                          seed=8)
        np.testing.assert_array_equal(part, full[ctx - ql:])


def pin_single_key(lib):
    """One visible key: the output is that key's value, exactly."""
    H, Hk, D, bs = 4, 2, 8, 16
    qs, ks, vs = make_dense([1], [1], H, Hk, D, seed=14)
    out = run_oracle(lib, qs, ks, vs, [1], [1], H, Hk, D, bs, 0.7)
    for h in range(H):
        np.testing.assert_array_equal(out[0, h], vs[0][0, h // 2].astype(np.float64))


def pin_identical_keys_mean(lib):
    """Identical keys (or zero scale): uniform weights, output = mean of the
    visible values."""
    H, Hk, D, bs = 4, 2, 8, 4
    q_lens, ctx = [3, 1], [10, 7]
    qs, ks, vs = make_dense(q_lens, ctx, H, Hk, D, seed=15)
    ks = [np.broadcast_to(k[:1], k.shape).copy() for k in ks]
    for scale, keys in ((0.9, ks), (0.0, make_dense(q_lens, ctx, H, Hk, D, 16)[1])):
        out = run_oracle(lib, qs, keys, vs, q_lens, ctx, H, Hk, D, bs, scale)
        off = 0
        for s in range(2):
            pre = ctx[s] - q_lens[s]
            for i in range(q_lens[s]):
                vis = vs[s][:pre + i + 1].astype(np.float64)
                for h in range(H):
                    np.testing.assert_allclose(out[off + i, h], vis[:, h // 2].mean(0),
                                               rtol=0, atol=1e-12)
            off += q_lens[s]


def pin_rows_sum_to_one(lib):
    """With every value row equal to 1 the output is sum_j p_j = 1."""
    H, Hk, D, bs = 4, 4, 8, 4
    q_lens, ctx = [1, 6], [40, 6]
    qs, ks, vs = make_dense(q_lens, ctx, H, Hk, D, seed=17)
    ones = [np.ones_like(v) for v in vs]
    qs = [q * 3 for q in qs]
    out = run_oracle(lib, qs, ks, ones, q_lens, ctx, H, Hk, D, bs, 1.0)
    np.testing.assert_allclose(out, 1.0, rtol=0, atol=1e-12)


def pin_page_placement_invariance(lib):
    """Any page permutation, and a single contiguous page, give the same
    result bit for bit."""
    H, Hk, D = 4, 2, 8
    q_lens, ctx = [1, 4, 7], [33, 20, 7]
    qs, ks, vs = make_dense(q_lens, ctx, H, Hk, D, seed=18)
    base = run_oracle(lib, qs, ks, vs, q_lens, ctx, H, Hk, D, 4, 0.4, seed=1)
    for bs, seed in ((4, 2), (4, 3), (8, 4), (64, 5)):
        other = run_oracle(lib, qs, ks, vs, q_lens, ctx, H, Hk, D, bs, 0.4, seed=seed)
        np.testing.assert_array_equal(other, base)


def pin_request_order_invariance(lib):
    """Permuting the requests (with their rows) permutes the outputs."""
    H, Hk, D, bs = 4, 2, 8, 4
    q_lens, ctx = [1, 4, 7, 2], [33, 20, 7, 9]
    qs, ks, vs = make_dense(q_lens, ctx, H, Hk, D, seed=19)
    base = run_oracle(lib, qs, ks, vs, q_lens, ctx, H, Hk, D, bs, 0.4)
    perm = [2, 0, 3, 1]
    out = run_oracle(lib, [qs[i] for i in perm], [ks[i] for i in perm], [vs[i] for i in perm],
                     [q_lens[i] for i in perm], [ctx[i] for i in perm], H, Hk, D, bs, 0.4,
                     seed=9)
    offs = np.concatenate([[0], np.cumsum(q_lens)])
    want = np.concatenate([base[offs[i]:offs[i + 1]] for i in perm])
    np.testing.assert_array_equal(out, want)


def pin_split_merge(lib):
    """Split-KV partials (the oracle restricted to KV windows) merged by LSE
    equal the unsplit result, for split sizes 1, block_size, 7 and 32768."""
    H, Hk, D, bs = 4, 2, 8, 4
    q_lens, ctx = [1, 5, 3], [45, 17, 3]
    qs, ks, vs = make_dense(q_lens, ctx, H, Hk, D, seed=20)
    kc, vc, table = scatter_pages(ks, vs, bs, 3)
    q = np.concatenate(qs)
    qsl = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    sl = np.array(ctx, np.int32)
    full = orc.paged_attention(q, kc, vc, table, sl, qsl, H, Hk, D, bs, 0.5, lib=lib)
    for split in (1, bs, 7, 32768):
        n = math.ceil(max(ctx) / split)
        parts, lses = [], []
        for p in range(n):
            o, l = orc.paged_attention(q, kc, vc, table, sl, qsl, H, Hk, D, bs, 0.5, lib=lib,
                                       kv_window=(p * split, (p + 1) * split), with_lse=True)
            parts.append(o)
            lses.append(l)
        parts = np.stack(parts, 2)  # [T, H, P, D]
        lses = np.stack(lses, 2)    # [T, H, P]
        for t in range(q.shape[0]):
            for h in range(H):
                merged, _ = orc.lse_merge(parts[t, h], lses[t, h], lib=lib)
                np.testing.assert_allclose(merged, full[t, h], rtol=0, atol=1e-12)


def pin_merge_closed_form(lib):
    """Two partials with lse a and b: weights are the logistic function of
    a - b; an empty partial (lse = -inf) gets weight 0; all empty gives 0."""
    o = np.array([[1.0, 2.0], [5.0, -3.0]])
    a, b = 0.3, -1.2
    out, lse = orc.lse_merge(o, np.array([a, b]), lib=lib)
    wa = 1.0 / (1.0 + math.exp(b - a))
    np.testing.assert_allclose(out, wa * o[0] + (1 - wa) * o[1], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, math.log(math.exp(a) + math.exp(b)), rtol=1e-15)
    out, lse = orc.lse_merge(o, np.array([a, -np.inf]), lib=lib)
    np.testing.assert_array_equal(out, o[0])
    out, lse = orc.lse_merge(o, np.array([-np.inf, -np.inf]), lib=lib)
    np.testing.assert_array_equal(out, 0.0)
    assert lse == -np.inf


def pin_mla_vs_sdpa(lib):
    """Absorbed MLA decode equals SDPA in fp64 with one shared KV head,
    d_k = latent + rope, values = the latent slice of the same rows."""
    L, R, H, bs = 32, 8, 8, 4
    ctx = [9, 1, 23]
    rng = np.random.default_rng(21)
    lat = [rng.standard_normal((c, 1, L + R)).astype(np.float32) for c in ctx]
    kc, _, table = scatter_pages(lat, lat, bs, 4)
    kc = kc[:, :, 0, :]
    q = rng.standard_normal((len(ctx), H, L + R)).astype(np.float32)
    scale = 1 / math.sqrt(12.0)
    out = orc.mla_decode(q, kc, table, np.array(ctx, np.int32), L, R, bs, scale, lib=lib)
    for s, c in enumerate(ctx):
        qt = torch.from_numpy(q[s].astype(np.float64))[:, None, :][None]      # [1,H,1,L+R]
        kt = torch.from_numpy(lat[s][:, 0].astype(np.float64))[None, None].expand(1, H, c, L + R)
        vt = kt[..., :L]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
        np.testing.assert_allclose(out[s], ref[0, :, 0].numpy(), rtol=0, atol=1e-12)


def pin_bf16_widening(lib):
    """bf16 storage is read as the exact binary32 value it encodes: the result
    equals the fp32 run on the same (bf16-representable) values, bit for bit."""
    b = inputs.paged_batch([1, 3], [19, 8], 4, 2, 16, 4, dtype="bf16", seed=3)
    as32 = dict(q=b.q.float(), k=b.k_cache.float(), v=b.v_cache.float())
    args = (b.block_table.numpy(), b.seq_lens.numpy(), b.query_start_loc.numpy(), 4, 2, 16, 4,
            b.scale)
    o16 = orc.paged_attention(inputs.storage_array(b.q), inputs.storage_array(b.k_cache),
                              inputs.storage_array(b.v_cache), *args, lib=lib)
    o32 = orc.paged_attention(as32["q"].numpy(), as32["k"].numpy(), as32["v"].numpy(), *args,
                              lib=lib)
    np.testing.assert_array_equal(o16, o32)
    assert np.isfinite(o16).all()


def pin_golden_two_key(lib):
    """Hand-worked two-key decode (tests/golden/two_key_decode.txt)."""
    vals = {}
    with open(os.path.join(GOLDEN, "two_key_decode.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, *rest = line.split()
            vals[key] = [float(x) for x in rest]
    q = np.array([[vals["q"]]], np.float32)              # [T=1, H=1, D=2]
    kc = np.array([[[vals["k0"]], [vals["k1"]]]], np.float32)  # [1 page, bs=2, Hk=1, D=2]
    vc = np.array([[[vals["v0"]], [vals["v1"]]]], np.float32)
    out = orc.paged_attention(q, kc, vc, np.array([[0]], np.int32), np.array([2], np.int32),
                              np.array([0, 1], np.int32), 1, 1, 2, 2, vals["scale"][0], lib=lib)
    np.testing.assert_allclose(out[0, 0], vals["expected"], rtol=0, atol=1e-14)


def sdpa_request_masked(q, k, v, ctx, scale, window=0, slopes=None, use_sqrt=False):
    """torch SDPA in fp64 for one request with an additive float mask written
    from the definitions: -inf outside p - window < j <= p (p the query's
    position; no lower bound without a window), plus the ALiBi term
    -m_h (p - j) or -m_h sqrt(p - j) per head."""
    ql, H, D = q.shape
    G = H // k.shape[1]
    qt = torch.from_numpy(q.astype(np.float64)).permute(1, 0, 2)[None]
    kt = torch.from_numpy(k.astype(np.float64)).repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    vt = torch.from_numpy(v.astype(np.float64)).repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    pos = (ctx - ql + torch.arange(ql, dtype=torch.float64))[:, None]   # [ql, 1]
    j = torch.arange(ctx, dtype=torch.float64)[None, :]                 # [1, ctx]
    visible = j <= pos
    if window:
        visible &= j > pos - window
    dist = (pos - j).clamp(min=0)
    bias = torch.zeros((H, ql, ctx), dtype=torch.float64)
    if slopes is not None:
        m = torch.as_tensor(np.asarray(slopes, np.float64))[:, None, None]
        bias = -m * (dist.sqrt() if use_sqrt else dist)[None]
    mask = torch.where(visible[None], bias, torch.tensor(-math.inf, dtype=torch.float64))
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask[None],
                                                           scale=scale)
    return out[0].permute(1, 0, 2).numpy()


def alibi_slopes(H):
    """The geometric ALiBi slopes 2^(-8 h / H), h = 1..H."""
    return np.array([2.0 ** (-8.0 * (h + 1) / H) for h in range(H)])


def pin_window_alibi_vs_sdpa(lib):
    """Sliding windows, linear and sqrt ALiBi, alone and together, on a
    decode + extend + prefill batch: each request equals SDPA with the mask
    and bias written out densely."""
    H, Hk, D, bs = 6, 2, 8, 4
    q_lens = [1, 5, 9, 1, 4]
    ctx = [23, 22, 9, 1, 4]
    qs, ks, vs = make_dense(q_lens, ctx, H, Hk, D, seed=21)
    scale = 1 / math.sqrt(D)
    sl = alibi_slopes(H)
    for window, slopes, use_sqrt in ((3, None, False), (7, None, False), (0, sl, False),
                                     (0, sl, True), (5, sl, False), (4, sl * 3, True)):
        out = run_oracle(lib, qs, ks, vs, q_lens, ctx, H, Hk, D, bs, scale, seed=9,
                         sliding_window=window, alibi_slopes=slopes, alibi_sqrt=use_sqrt)
        off = 0
        for s in range(len(q_lens)):
            ref = sdpa_request_masked(qs[s], ks[s], vs[s], ctx[s], scale, window, slopes,
                                      use_sqrt)
            np.testing.assert_allclose(out[off:off + q_lens[s]], ref, rtol=0, atol=1e-12)
            off += q_lens[s]


def pin_window_of_one_is_own_value(lib):
    """A window of one position: every query sees only its own key, so the
    output is exactly its own value row (whatever the ALiBi slopes)."""
    H, Hk, D, bs = 4, 2, 8, 4
    q_lens, ctx = [1, 6, 3], [10, 6, 11]
    qs, ks, vs = make_dense(q_lens, ctx, H, Hk, D, seed=22)
    for slopes in (None, alibi_slopes(H)):
        out = run_oracle(lib, qs, ks, vs, q_lens, ctx, H, Hk, D, bs, 0.5, seed=3,
                         sliding_window=1, alibi_slopes=slopes)
        off = 0
        for s in range(len(q_lens)):
            own = vs[s][ctx[s] - q_lens[s]:].astype(np.float64)   # [ql, Hk, D]
            want = np.repeat(own, H // Hk, axis=1)
            np.testing.assert_array_equal(out[off:off + q_lens[s]], want)
            off += q_lens[s]


def pin_wide_window_and_zero_slopes_are_plain(lib):
    """A window covering every context, and ALiBi slopes of zero, change
    nothing: bit-identical to plain attention."""
    H, Hk, D, bs = 4, 1, 8, 4
    q_lens, ctx = [1, 7, 5], [19, 12, 5]
    qs, ks, vs = make_dense(q_lens, ctx, H, Hk, D, seed=23)
    plain = run_oracle(lib, qs, ks, vs, q_lens, ctx, H, Hk, D, bs, 0.4, seed=4)
    for kw in (dict(sliding_window=19), dict(sliding_window=1000),
               dict(alibi_slopes=np.zeros(H)), dict(alibi_slopes=np.zeros(H), alibi_sqrt=True)):
        got = run_oracle(lib, qs, ks, vs, q_lens, ctx, H, Hk, D, bs, 0.4, seed=4, **kw)
        np.testing.assert_array_equal(got, plain)


def pin_alibi_geometric_closed_form(lib):
    """q = 0 makes every dot product 0, so with linear ALiBi the decode
    query at position p weighs key j by r^(p - j) / Z, r = e^(-m).  With
    values V_j = (1, j): out = (1, p - S1 / S0), S0 = sum_k r^k and
    S1 = sum_k k r^k over k = 0..p, in closed form."""
    p, m = 12, 0.3
    ctx = p + 1
    q = np.zeros((1, 1, 2), np.float32)
    k = np.random.default_rng(24).standard_normal((ctx, 1, 2)).astype(np.float32)
    v = np.stack([np.ones(ctx), np.arange(ctx)], axis=1)[:, None, :].astype(np.float32)
    out = run_oracle(lib, [q], [k], [v], [1], [ctx], 1, 1, 2, 4, 1.0, seed=2,
                     alibi_slopes=np.array([m]))
    r = math.exp(-m)
    s0 = (1 - r ** (p + 1)) / (1 - r)
    s1 = r * (1 - (p + 1) * r ** p + p * r ** (p + 1)) / (1 - r) ** 2
    np.testing.assert_allclose(out[0, 0], [1.0, p - s1 / s0], rtol=0, atol=1e-12)


ALL_PINS = [pin_sdpa_prefill_causal, pin_sdpa_mixed_batch, pin_extend_is_tail_of_prefill,
            pin_single_key, pin_identical_keys_mean, pin_rows_sum_to_one,
            pin_page_placement_invariance, pin_request_order_invariance, pin_split_merge,
            pin_merge_closed_form, pin_mla_vs_sdpa, pin_bf16_widening, pin_golden_two_key,
            pin_window_alibi_vs_sdpa, pin_window_of_one_is_own_value,
            pin_wide_window_and_zero_slopes_are_plain, pin_alibi_geometric_closed_form]
