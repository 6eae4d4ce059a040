"""Pins for the oracle's paged KV-cache write (CPU only).

Each pin checks the oracle against something other than itself: a flat
slot-mapping formulation of the same write (slot = page * block_size +
position % block_size on the cache viewed as [num_blocks * block_size, ...]),
the C oracle's gather through the block table (the write's inverse), the
bytes it must leave alone, and the metadata errors.  Textual mutations of the
oracle (a swapped page/slot, an off-by-one position, K and V swapped) must
each fail at least one pin.
"""
import inspect
import textwrap

import numpy as np
import pytest

from oracle import oracle as orc


def _problem(seed, q_lens, ctx, Hk=2, D=8, bs=4, dtype=np.float32, extra_pages=3):
    """Random caches (stale values everywhere), new K/V rows and a permuted
    block table covering every request's context."""
    rng = np.random.default_rng(seed)
    S = len(q_lens)
    npages = [max(1, -(-c // bs)) for c in ctx]
    nb = sum(npages) + extra_pages
    perm = rng.permutation(nb)
    maxb = max(npages) + 1
    bt = np.full((S, maxb), -1, np.int32)
    k = 0
    for s in range(S):
        bt[s, :npages[s]] = perm[k:k + npages[s]]
        k += npages[s]
    T = sum(q_lens)
    qsl = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)

    def arr(*shape):
        a = rng.standard_normal(shape).astype(np.float32)
        return a if dtype == np.float32 else a.view(np.uint32).astype(np.uint16)

    return dict(k_new=arr(T, Hk, D), v_new=arr(T, Hk, D), k_cache=arr(nb, bs, Hk, D),
                v_cache=arr(nb, bs, Hk, D), block_table=bt,
                seq_lens=np.array(ctx, np.int32), query_start_loc=qsl, block_size=bs)


def _flat_slot_write(p):
    """The same write, written as a slot mapping over the flattened pool
    (tokens with no valid slot, and requests with q_len > seq_len, are
    skipped)."""
    bs, nb = p["block_size"], p["k_cache"].shape[0]
    kc = p["k_cache"].copy().reshape(-1, *p["k_cache"].shape[2:])
    vc = p["v_cache"].copy().reshape(-1, *p["v_cache"].shape[2:])
    qsl = p["query_start_loc"]
    for s in range(len(p["seq_lens"])):
        q_len = int(qsl[s + 1] - qsl[s])
        if int(p["seq_lens"][s]) < q_len:
            continue
        for t in range(int(qsl[s]), int(qsl[s + 1])):
            pos = int(p["seq_lens"][s]) - q_len + (t - int(qsl[s]))
            page = int(p["block_table"][s][pos // bs])
            if not 0 <= page < nb:
                continue
            kc[page * bs + pos % bs] = p["k_new"][t]
            vc[page * bs + pos % bs] = p["v_new"][t]
    return kc.reshape(p["k_cache"].shape), vc.reshape(p["v_cache"].shape)


CASES = [
    (1, [1, 1, 1], [5, 17, 1]),                 # decodes, one single-key context
    (2, [3, 0, 9, 1], [10, 4, 9, 40]),          # extend, empty request, prefill, decode
    (3, [16, 5], [16, 21]),                     # prefill filling pages exactly, page crossing
]


def pin_cache_write_matches_slot_mapping(write):
    for seed, q_lens, ctx in CASES:
        for dtype in (np.float32, np.uint16):
            p = _problem(seed, q_lens, ctx, dtype=dtype)
            k, v, st = write(**p)
            kw, vw = _flat_slot_write(p)
            assert st == 0
            assert np.array_equal(k, kw) and np.array_equal(v, vw)


def pin_cache_write_read_back_by_gather(write):
    """The C oracle's gather of each request's new positions returns the new
    rows; positions before them return what was there."""
    for seed, q_lens, ctx in CASES:
        p = _problem(seed, q_lens, ctx)
        k, v, _ = write(**p)
        maxlen = max(ctx)
        for cache, new, old in ((k, p["k_new"], p["k_cache"]), (v, p["v_new"], p["v_cache"])):
            after = orc.gather_rows(cache, p["block_table"], p["seq_lens"], p["block_size"], maxlen)
            before = orc.gather_rows(old, p["block_table"], p["seq_lens"], p["block_size"], maxlen)
            qsl = p["query_start_loc"]
            for s, (ql, c) in enumerate(zip(q_lens, ctx)):
                row = new.shape[1] * new.shape[2]
                got = after[s, c - ql:c].reshape(ql, row)
                assert np.array_equal(got, new[qsl[s]:qsl[s + 1]].reshape(ql, row))
                assert np.array_equal(after[s, :c - ql], before[s, :c - ql])


def pin_cache_write_leaves_other_slots(write):
    for seed, q_lens, ctx in CASES:
        p = _problem(seed, q_lens, ctx)
        k, _, _ = write(**p)
        touched = np.zeros(p["k_cache"].shape[:2], bool)
        bs = p["block_size"]
        for s, (ql, c) in enumerate(zip(q_lens, ctx)):
            for pos in range(c - ql, c):
                touched[p["block_table"][s][pos // bs], pos % bs] = True
        assert np.array_equal(k[~touched], p["k_cache"][~touched])
        assert touched.sum() == sum(q_lens)


def pin_cache_write_bad_metadata(write):
    # a block id outside the pool on the second request's last page: only
    # its tokens there are skipped
    p = _problem(4, [2, 3], [6, 7])
    p["block_table"][1, 1] = p["k_cache"].shape[0] + 5
    k, v, st = write(**p)
    kw, vw = _flat_slot_write(p)
    assert st == orc.DEV_BAD_BLOCK and np.array_equal(k, kw) and np.array_equal(v, vw)
    assert not np.array_equal(k, p["k_cache"])  # the rest was written
    # q_len above the context: that request is skipped
    p = _problem(5, [2, 3], [6, 7])
    p["seq_lens"][1] = 2
    k, _, st = write(**p)
    kw, _ = _flat_slot_write(p)
    assert st == orc.DEV_BAD_QLEN and np.array_equal(k, kw)
    # a bad query_start_loc: nothing is written
    p = _problem(6, [2, 3], [6, 7])
    p["query_start_loc"] = np.array([0, 3, 2], np.int32)
    k, _, st = write(**p)
    assert st == orc.DEV_BAD_QSL and np.array_equal(k, p["k_cache"])


PINS = [pin_cache_write_matches_slot_mapping, pin_cache_write_read_back_by_gather,
        pin_cache_write_leaves_other_slots, pin_cache_write_bad_metadata]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(orc.cache_write)


# plausible mistakes in the oracle, each of which a pin must catch
MUTATIONS = {
    "page_slot_swapped": ("k_out[page, pos % block_size] = k_new[qsl[s] + i]",
                          "k_out[page, pos // block_size % block_size] = k_new[qsl[s] + i]"),
    "position_off_by_one": ("prefix = int(seq_lens[s]) - q_len",
                            "prefix = int(seq_lens[s]) - q_len + 1"),
    "k_and_v_swapped": ("v_out[page, pos % block_size] = v_new[qsl[s] + i]",
                        "v_out[page, pos % block_size] = k_new[qsl[s] + i]"),
    "wrong_token_row": ("k_out[page, pos % block_size] = k_new[qsl[s] + i]",
                        "k_out[page, pos % block_size] = k_new[i]"),
}


def _mutated(name):
    old, new = MUTATIONS[name]
    src = textwrap.dedent(inspect.getsource(orc.cache_write))
    assert src.count(old) == 1, name
    ns = dict(vars(orc))
    exec(compile(src.replace(old, new), f"<mutated {name}>", "exec"), ns)
    return ns["cache_write"]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name):
    broken = _mutated(name)
    failures = 0
    for pin in PINS:
        try:
            pin(broken)
        except (AssertionError, IndexError, ValueError):
            failures += 1
    assert failures > 0, f"no pin caught the mutation {name}"
