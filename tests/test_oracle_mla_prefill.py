"""Pins for the oracle's non-absorbed MLA prefill / extend (CPU only).

Each pin checks the oracle against something other than itself:
  * the absorption identity -- q_nope . (W_K c) = (W_K^T q_nope) . c and
    sum_j p_j W_V c_j = W_V sum_j p_j c_j -- so every row must equal W_V
    applied to the C oracle's absorbed MLA decode over the same latents with
    the absorbed query [W_K^T q_nope ; q_rope] and the row's visible prefix
    (small integer inputs keep every product exact, so the absorbed query is
    exactly representable);
  * torch's scaled_dot_product_attention in fp64 on keys and values
    decompressed by torch.einsum, with the bottom-right causal mask;
  * invariants: extend rows are the tail of the prefill over the same
    context, and the page placement changes nothing.
Textual mutations of the oracle (key and value projections swapped, the rope
part dropped, the causal bound off by one, the scale dropped) must each fail
a pin.
"""
import inspect
import math
import textwrap

import numpy as np
import pytest
import torch

from oracle import oracle as orc

L, R, NOPE, DV = 16, 8, 8, 8


def _problem(seed, q_lens, ctx, H=4, bs=4, integer=False, perm=True):
    rng = np.random.default_rng(seed)
    S = len(q_lens)
    npages = [-(-c // bs) for c in ctx]
    nb = sum(npages) + 2
    order = rng.permutation(nb) if perm else np.arange(nb)
    bt = np.full((S, max(npages)), -1, np.int32)
    k = 0
    for s in range(S):
        bt[s, :npages[s]] = order[k:k + npages[s]]
        k += npages[s]
    T = sum(q_lens)
    if integer:
        draw = lambda *sh: rng.integers(-2, 3, sh).astype(np.float32)  # noqa: E731
    else:
        draw = lambda *sh: rng.standard_normal(sh).astype(np.float32)  # noqa: E731
    w = draw(H, NOPE + DV, L)
    if not integer:
        w /= np.float32(math.sqrt(L))
    return dict(q=draw(T, H, NOPE + R), kv_cache=draw(nb, bs, L + R), w_kv=w,
                block_table=bt, seq_lens=np.array(ctx, np.int32),
                query_start_loc=np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32),
                kv_lora_rank=L, qk_nope_dim=NOPE, rope_dim=R, v_head_dim=DV, block_size=bs,
                scale=0.05 if integer else 1 / math.sqrt(NOPE + R))


def pin_absorbed_identity(fn):
    p = _problem(1, [1, 3, 5], [6, 9, 5], integer=True)
    out = fn(**p)
    q, w = p["q"], p["w_kv"]
    H = q.shape[1]
    qsl, ctx = p["query_start_loc"], p["seq_lens"]
    for s in range(len(ctx)):
        for i in range(qsl[s + 1] - qsl[s]):
            t = qsl[s] + i
            vis = int(ctx[s]) - (qsl[s + 1] - qsl[s]) + i + 1
            # absorbed query per head: [W_K,h^T q_nope ; q_rope], exact in fp32
            q_abs = np.concatenate([np.einsum("dl,d->l", w[h, :NOPE].astype(np.float64),
                                              q[t, h, :NOPE].astype(np.float64))[None]
                                    for h in range(H)], 0)
            q_abs = np.concatenate([q_abs, q[t, :, NOPE:].astype(np.float64)], 1)
            assert np.array_equal(q_abs.astype(np.float32).astype(np.float64), q_abs)
            lat = orc.mla_decode(q_abs.astype(np.float32)[None], p["kv_cache"],
                                 p["block_table"][s:s + 1], np.array([vis], np.int32), L, R,
                                 p["block_size"], p["scale"])[0]          # [H, L]
            want = np.einsum("hdl,hl->hd", w[:, NOPE:].astype(np.float64), lat)
            np.testing.assert_allclose(out[t], want, rtol=0, atol=1e-12)


def pin_sdpa(fn):
    p = _problem(2, [1, 4, 7, 1], [11, 10, 7, 1])
    out = fn(**p)
    H = p["q"].shape[1]
    qsl, ctx, bs = p["query_start_loc"], p["seq_lens"], p["block_size"]
    w = torch.from_numpy(p["w_kv"].astype(np.float64))
    for s in range(len(ctx)):
        c_len, ql = int(ctx[s]), int(qsl[s + 1] - qsl[s])
        pos = torch.arange(c_len)
        pages = torch.from_numpy(p["block_table"][s].astype(np.int64))[pos // bs]
        lat = torch.from_numpy(p["kv_cache"].astype(np.float64))[pages, pos % bs]
        k = torch.cat([torch.einsum("hdl,jl->hjd", w[:, :NOPE], lat[:, :L]),
                       lat[:, L:][None].expand(H, -1, -1)], dim=2)      # [H, ctx, 16]
        v = torch.einsum("hdl,jl->hjd", w[:, NOPE:], lat[:, :L])        # [H, ctx, DV]
        qq = torch.from_numpy(p["q"][qsl[s]:qsl[s + 1]].astype(np.float64)).permute(1, 0, 2)
        mask = pos[None, :] <= (c_len - ql + torch.arange(ql))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qq[None], k[None], v[None], attn_mask=mask, scale=p["scale"])[0].permute(1, 0, 2)
        np.testing.assert_allclose(out[qsl[s]:qsl[s + 1]], ref.numpy(), rtol=0, atol=1e-12)


def pin_extend_is_tail_of_prefill(fn):
    p = _problem(3, [12], [12])
    full = fn(**p)
    for ql in (1, 5):
        e = dict(p, q=p["q"][12 - ql:], query_start_loc=np.array([0, ql], np.int32))
        np.testing.assert_allclose(fn(**e), full[12 - ql:], rtol=0, atol=1e-13)


def pin_page_placement(fn):
    a = _problem(4, [3, 6], [9, 6], perm=False)
    b = _problem(4, [3, 6], [9, 6], perm=True)
    # same values, pages moved: rebuild b's cache from a's by its table
    cache = np.full_like(a["kv_cache"], np.nan)
    for s in range(2):
        for lp in range(-(-int(a["seq_lens"][s]) // 4)):
            cache[b["block_table"][s, lp]] = a["kv_cache"][a["block_table"][s, lp]]
    b = dict(a, kv_cache=cache, block_table=b["block_table"])
    np.testing.assert_allclose(fn(**b), fn(**a), rtol=0, atol=1e-13)


PINS = [pin_absorbed_identity, pin_sdpa, pin_extend_is_tail_of_prefill, pin_page_placement]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(orc.mla_prefill)


def test_sampled_rows_match_full():
    p = _problem(5, [2, 6], [8, 6])
    full = orc.mla_prefill(**p)
    rows = np.array([1, 5, 17, 30])
    part = orc.mla_prefill(**p, rows=rows)
    H = p["q"].shape[1]
    np.testing.assert_array_equal(part.reshape(-1, DV)[rows], full.reshape(-1, DV)[rows])
    others = np.setdiff1d(np.arange(p["q"].shape[0] * H), rows)
    assert np.isnan(part.reshape(-1, DV)[others]).all()


MUTATIONS = {
    "key_value_swapped": ("w_k, w_v = w[:, :qk_nope_dim, :], w[:, qk_nope_dim:, :]",
                          "w_v, w_k = w[:, :qk_nope_dim, :], w[:, qk_nope_dim:, :]"),
    "rope_dropped": ("+ np.einsum(\"ihd,jd->hij\", qb[:, :, qk_nope_dim:], k_rope)) * scale",
                     "+ 0.0) * scale"),
    "causal_off_by_one": ("visible = j[None, :] <= (prefix + ii)[:, None]",
                          "visible = j[None, :] < (prefix + ii)[:, None]"),
    "scale_dropped": (") * scale\n", ") * 1.0\n"),
}


def _mutated(name):
    old, new = MUTATIONS[name]
    src = textwrap.dedent(inspect.getsource(orc.mla_prefill))
    assert src.count(old) == 1, name
    ns = dict(vars(orc))
    exec(compile(src.replace(old, new), f"<mutated {name}>", "exec"), ns)
    return ns["mla_prefill"]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name):
    broken = _mutated(name)
    failures = 0
    for pin in PINS:
        try:
            pin(broken)
        except (AssertionError, IndexError, ValueError, FloatingPointError):
            failures += 1
    assert failures > 0, f"no pin caught the mutation {name}"
