"""Pins for the oracle's head-major (HND) cache layout (CPU only).

The HND storage is written here element by element from its offset formula
-- element (page, slot, head, d) at ((page * Hk + head) * block_size + slot)
* D + d -- with plain Python loops, independently of the oracle's view.
Attention over that storage must equal attention over the NHD cache bit for
bit (the layout moves bytes, it changes no value), and the cache write must
put each new row at its formula offset.  A plausible mistake in the view (a
reshape where a transpose belongs) must fail a pin.
"""
import inspect
import textwrap

import numpy as np
import pytest

from oracle import oracle as orc


def _to_hnd_by_offsets(nhd):
    nb, bs, hk, d = nhd.shape
    flat = np.empty(nhd.size, nhd.dtype)
    for page in range(nb):
        for slot in range(bs):
            for head in range(hk):
                for x in range(d):
                    flat[((page * hk + head) * bs + slot) * d + x] = nhd[page, slot, head, x]
    return flat.reshape(nb, hk, bs, d)


def _batch(seed, bs=4, Hk=2, G=2, D=8, q_lens=(1, 3, 1), ctx=(7, 9, 1)):
    rng = np.random.default_rng(seed)
    S = len(q_lens)
    npages = [-(-c // bs) for c in ctx]
    nb = sum(npages) + 2
    perm = rng.permutation(nb)
    bt = np.full((S, max(npages)), -1, np.int32)
    k = 0
    for s in range(S):
        bt[s, :npages[s]] = perm[k:k + npages[s]]
        k += npages[s]
    T = sum(q_lens)
    return dict(q=rng.standard_normal((T, Hk * G, D)).astype(np.float32),
                k=rng.standard_normal((nb, bs, Hk, D)).astype(np.float32),
                v=rng.standard_normal((nb, bs, Hk, D)).astype(np.float32),
                bt=bt, sl=np.array(ctx, np.int32),
                qsl=np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32),
                H=Hk * G, Hk=Hk, D=D, bs=bs)


def pin_view_matches_offsets(view):
    b = _batch(1)
    hnd = _to_hnd_by_offsets(b["k"])
    assert np.array_equal(view(hnd, "hnd"), b["k"])
    assert view(b["k"], "nhd") is b["k"]


def pin_attention_is_layout_invariant(view):
    for seed in (2, 3):
        b = _batch(seed)
        args = (b["bt"], b["sl"], b["qsl"], b["H"], b["Hk"], b["D"], b["bs"], 0.3)
        want = orc.paged_attention(b["q"], b["k"], b["v"], *args)
        kh, vh = _to_hnd_by_offsets(b["k"]), _to_hnd_by_offsets(b["v"])
        got = orc.paged_attention(b["q"], np.ascontiguousarray(view(kh, "hnd")),
                                  np.ascontiguousarray(view(vh, "hnd")), *args)
        assert np.array_equal(got, want)


def pin_cache_write_lands_at_offsets(write):
    b = _batch(4)
    hk, d, bs = b["Hk"], b["D"], b["bs"]
    rng = np.random.default_rng(5)
    T = b["q"].shape[0]
    k_new = rng.standard_normal((T, hk, d)).astype(np.float32)
    kh, vh = _to_hnd_by_offsets(b["k"]), _to_hnd_by_offsets(b["v"])
    k_out, v_out, st = write(k_new, k_new, kh, vh, b["bt"], b["sl"], b["qsl"], bs,
                             kv_layout="hnd")
    assert st == 0 and k_out.shape == kh.shape
    flat_in, flat_out = kh.reshape(-1), k_out.reshape(-1)
    touched = np.zeros(flat_in.size, bool)
    qsl = b["qsl"]
    for s in range(len(b["sl"])):
        q_len = int(qsl[s + 1] - qsl[s])
        for i in range(q_len):
            pos = int(b["sl"][s]) - q_len + i
            page = int(b["bt"][s][pos // bs])
            for head in range(hk):
                off = ((page * hk + head) * bs + pos % bs) * d
                assert np.array_equal(flat_out[off:off + d], k_new[qsl[s] + i, head])
                touched[off:off + d] = True
    assert np.array_equal(flat_out[~touched], flat_in[~touched])


def _pins(view, write):
    return [lambda: pin_view_matches_offsets(view), lambda: pin_attention_is_layout_invariant(view),
            lambda: pin_cache_write_lands_at_offsets(write)]


@pytest.mark.parametrize("i", range(3))
def test_pin(i):
    _pins(orc.nhd_view, orc.cache_write)[i]()


MUTATIONS = {
    "reshape_for_transpose": ("return cache.transpose(0, 2, 1, 3)",
                              "return cache.reshape(cache.shape[0], cache.shape[2], "
                              "cache.shape[1], cache.shape[3])"),
    "heads_and_dims_swapped": ("return cache.transpose(0, 2, 1, 3)",
                               "return cache.transpose(0, 3, 1, 2)"),
}


def _mutated(name):
    old, new = MUTATIONS[name]
    src = textwrap.dedent(inspect.getsource(orc.nhd_view))
    assert src.count(old) == 1, name
    ns = dict(vars(orc))
    exec(compile(src.replace(old, new), f"<mutated {name}>", "exec"), ns)
    view = ns["nhd_view"]
    # the cache write reads the layout through the same view
    wsrc = textwrap.dedent(inspect.getsource(orc.cache_write))
    exec(compile(wsrc, "<cache_write over the mutated view>", "exec"), ns)
    return view, ns["cache_write"]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name):
    view, write = _mutated(name)
    failures = 0
    for pin in _pins(view, write):
        try:
            pin()
        except (AssertionError, IndexError, ValueError):
            failures += 1
    assert failures > 0, f"no pin caught the mutation {name}"


def test_paged_attention_reads_hnd_storage():
    """paged_attention(kv_layout="hnd") on the offset-built storage equals
    the NHD result bit for bit, sinks and split windows included."""
    b = _batch(6, bs=8, Hk=4, G=1, D=16, q_lens=(5, 1, 2), ctx=(21, 3, 17))
    args = (b["bt"], b["sl"], b["qsl"], b["H"], b["Hk"], b["D"], b["bs"], 0.25)
    sk = np.linspace(-1.0, 2.0, b["H"])
    kh, vh = _to_hnd_by_offsets(b["k"]), _to_hnd_by_offsets(b["v"])
    for kw in (dict(), dict(sinks=sk), dict(kv_window=(4, 12), with_lse=True)):
        want = orc.paged_attention(b["q"], b["k"], b["v"], *args, **kw)
        got = orc.paged_attention(b["q"], kh, vh, *args, kv_layout="hnd", **kw)
        for g, w in zip(got if isinstance(got, tuple) else (got,),
                        want if isinstance(want, tuple) else (want,)):
            assert np.array_equal(g, w, equal_nan=True)
