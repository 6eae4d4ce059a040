"""ctypes front end of the fp64 CPU oracle (test infrastructure only).

Only the test-suite, the smoke check and the benchmark's CPU-baseline leg may
import this module.  It takes numpy arrays holding the *stored* input values:
float32 arrays for fp32 inputs, uint16 arrays of bf16 bit patterns for bf16
inputs.  Everything is computed in double precision by oracle.c.
"""
import ctypes
import os

import numpy as np

from . import build as _build

F32, BF16 = 0, 1

_I32P = ctypes.POINTER(ctypes.c_int32)
_I64P = ctypes.POINTER(ctypes.c_int64)
_F64P = ctypes.POINTER(ctypes.c_double)
_VP = ctypes.c_void_p

_ERR = {1: "bad arguments", 2: "bad metadata", 3: "out of memory"}


class OracleError(RuntimeError):
    pass


def load(path=None):
    """Load (building first if needed) an oracle shared library."""
    path = path or _build.build()
    lib = ctypes.CDLL(path)
    lib.oracle_paged_attention_window.argtypes = [
        _VP, _VP, _VP, ctypes.c_int, _I32P, _I32P, _I32P, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_double, ctypes.c_longlong, ctypes.c_longlong, _I64P, ctypes.c_longlong,
        _F64P, _F64P]
    lib.oracle_paged_attention_window.restype = ctypes.c_int
    lib.oracle_paged_attention_ex.argtypes = [
        _VP, _VP, _VP, ctypes.c_int, _I32P, _I32P, _I32P, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_double, ctypes.c_longlong, ctypes.c_longlong, ctypes.c_longlong, _F64P,
        ctypes.c_int, _I64P, ctypes.c_longlong, _F64P, _F64P]
    lib.oracle_paged_attention_ex.restype = ctypes.c_int
    lib.oracle_lse_merge.argtypes = [ctypes.c_int, ctypes.c_int, _F64P, _F64P, _F64P, _F64P]
    lib.oracle_lse_merge.restype = ctypes.c_int
    lib.oracle_mla_decode.argtypes = [
        _VP, _VP, ctypes.c_int, _I32P, _I32P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, _I64P,
        ctypes.c_longlong, _F64P]
    lib.oracle_mla_decode.restype = ctypes.c_int
    lib.oracle_gather_rows.argtypes = [
        _VP, ctypes.c_int, ctypes.c_int, _I32P, _I32P, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_int, ctypes.c_longlong, _VP]
    lib.oracle_gather_rows.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    return lib


_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        _LIB = load()
    return _LIB


def _dtype_code(arr):
    if arr.dtype == np.float32:
        return F32
    if arr.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle inputs must be float32 or uint16 (bf16 bits), got {arr.dtype}")


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(a, typ):
    return a.ctypes.data_as(typ)


def _check(rc):
    if rc != 0:
        raise OracleError(_ERR.get(rc, f"oracle error {rc}"))


def nhd_view(cache, kv_layout):
    """A paged cache seen as [num_blocks, block_size, Hk, D] (a numpy view,
    writes go through).  kv_layout "nhd" stores it that way; "hnd" stores
    [num_blocks, Hk, block_size, D], i.e. element (page, slot, head, d) at
    flat offset ((page * Hk + head) * block_size + slot) * D + d ("vLLM AMD
    ROCm attention backend optimisation", section "ROCM_AITER_FA": a KV cache
    laid out for the hardware's access pattern)."""
    if kv_layout == "nhd":
        return cache
    if kv_layout == "hnd":
        return cache.transpose(0, 2, 1, 3)
    raise ValueError(kv_layout)


def paged_attention(q, k_cache, v_cache, block_table, seq_lens, query_start_loc,
                    num_heads, num_kv_heads, head_dim, block_size, scale,
                    rows=None, kv_window=None, lib=None, with_lse=False, sinks=None,
                    kv_layout="nhd", sliding_window=0, alibi_slopes=None, alibi_sqrt=False):
    """fp64 unified paged attention.  Shapes:
    q [T, H, D]; k_cache, v_cache [num_blocks, block_size, Hk, D];
    block_table [S, max_blocks]; seq_lens [S]; query_start_loc [S+1].
    rows: optional int64 array of flat (token * H + head) indices to compute;
    rows not listed come back as NaN.  kv_window=(lo, hi) restricts every
    request to KV positions in [lo, hi) (used to form split-KV partials).
    sinks: optional [H] sink logits ("vLLM Triton attention backend deep
    dive", section "Usage scenarios": sink tokens are one of the model
    features the unified backend supports): head h's softmax denominator
    gains exp(sinks[h]) while the sink contributes no value, so
      out = sum_j exp(s_j) v_j / (sum_j exp(s_j) + exp(sinks[h]))
          = out_keys / (1 + exp(sinks[h] - lse)),
    lse = log sum_j exp(s_j) over the row's visible keys (s_j = scale q.k_j).
    The returned lse stays that of the keys alone.
    kv_layout: "nhd" or "hnd" storage of the caches (see nhd_view).
    sliding_window W > 0: the query at position p sees p - W < j <= p only.
    alibi_slopes: optional [H] slopes m_h (natural-log units per position):
    every score of head h gains -m_h * (p - j), or -m_h * sqrt(p - j) with
    alibi_sqrt.  (The pages name ALiBi sqrt and GPT-OSS behaviour among the
    unified backend's model features without defining them; these are the
    readings.)
    Returns out [T, H, D] float64 (and lse [T, H] when with_lse)."""
    lib = lib or _lib()
    q = np.ascontiguousarray(q)
    k_cache = np.ascontiguousarray(nhd_view(k_cache, kv_layout))
    v_cache = np.ascontiguousarray(nhd_view(v_cache, kv_layout))
    dt = _dtype_code(q)
    assert _dtype_code(k_cache) == dt and _dtype_code(v_cache) == dt
    bt = _i32(block_table)
    sl = _i32(seq_lens)
    qsl = _i32(query_start_loc)
    S = int(sl.shape[0])
    T = int(q.shape[0])
    out = np.full((T, num_heads, head_dim), np.nan, dtype=np.float64)
    lse = np.full((T, num_heads), np.nan, dtype=np.float64)
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        rows_p, nrows = _ptr(rows, _I64P), int(rows.shape[0])
    else:
        rows_p, nrows = None, 0
    lo, hi = (0, 2**62) if kv_window is None else kv_window
    max_blocks = int(bt.shape[1]) if bt.ndim == 2 else 0
    slopes = None
    if alibi_slopes is not None:
        slopes = np.ascontiguousarray(np.asarray(alibi_slopes, dtype=np.float64).reshape(-1))
        assert slopes.shape[0] == num_heads
    rc = lib.oracle_paged_attention_ex(
        q.ctypes.data, k_cache.ctypes.data, v_cache.ctypes.data, dt,
        _ptr(bt, _I32P), _ptr(sl, _I32P), _ptr(qsl, _I32P), S, T, num_heads,
        num_kv_heads, head_dim, block_size, max_blocks, int(k_cache.shape[0]),
        float(scale), int(lo), int(hi), int(sliding_window),
        None if slopes is None else _ptr(slopes, _F64P), int(bool(alibi_sqrt)), rows_p, nrows,
        _ptr(out, _F64P), _ptr(lse, _F64P))
    _check(rc)
    if sinks is not None:
        sk = np.asarray(sinks, dtype=np.float64).reshape(1, num_heads)
        out = out / (1.0 + np.exp(sk - lse))[:, :, None]
    return (out, lse) if with_lse else out


def lse_merge(partial_out, partial_lse, lib=None):
    """Merge P partial results of one row: partial_out [P, D], partial_lse [P]."""
    lib = lib or _lib()
    po = np.ascontiguousarray(partial_out, dtype=np.float64)
    pl = np.ascontiguousarray(partial_lse, dtype=np.float64)
    P, D = po.shape
    out = np.zeros(D, dtype=np.float64)
    lse = np.zeros(1, dtype=np.float64)
    _check(lib.oracle_lse_merge(P, D, _ptr(po, _F64P), _ptr(pl, _F64P), _ptr(out, _F64P),
                                _ptr(lse, _F64P)))
    return out, float(lse[0])


def mla_decode(q, kv_cache, block_table, seq_lens, kv_lora_rank, rope_dim, block_size,
               scale, rows=None, lib=None):
    """fp64 absorbed-MLA decode.  q [S, H, L+R]; kv_cache [num_blocks, bs, L+R];
    returns out [S, H, L] float64 (rows not listed come back NaN)."""
    lib = lib or _lib()
    q = np.ascontiguousarray(q)
    kv_cache = np.ascontiguousarray(kv_cache)
    dt = _dtype_code(q)
    assert _dtype_code(kv_cache) == dt
    bt = _i32(block_table)
    sl = _i32(seq_lens)
    S, H, _ = q.shape
    out = np.full((S, H, kv_lora_rank), np.nan, dtype=np.float64)
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        rows_p, nrows = _ptr(rows, _I64P), int(rows.shape[0])
    else:
        rows_p, nrows = None, 0
    rc = lib.oracle_mla_decode(q.ctypes.data, kv_cache.ctypes.data, dt, _ptr(bt, _I32P),
                               _ptr(sl, _I32P), S, H, kv_lora_rank, rope_dim, block_size,
                               int(bt.shape[1]), int(kv_cache.shape[0]), float(scale),
                               rows_p, nrows, _ptr(out, _F64P))
    _check(rc)
    return out


def gather_rows(k_cache, block_table, seq_lens, block_size, max_seq_len):
    """Dense gather of K rows through the block table: returns
    [S, max_seq_len, row_elems] with untouched positions zero."""
    lib = _lib()
    kc = np.ascontiguousarray(k_cache)
    nb = kc.shape[0]
    row_elems = int(np.prod(kc.shape[2:]))
    bt = _i32(block_table)
    sl = _i32(seq_lens)
    S = int(sl.shape[0])
    dense = np.zeros((S, max_seq_len, row_elems), dtype=kc.dtype)
    _check(lib.oracle_gather_rows(kc.ctypes.data, kc.dtype.itemsize, row_elems,
                                  _ptr(bt, _I32P), _ptr(sl, _I32P), S, int(bt.shape[1]), nb,
                                  block_size, int(max_seq_len), dense.ctypes.data))
    return dense


# Status bits, as the library's device status word defines them.
DEV_BAD_BLOCK, DEV_BAD_QLEN, DEV_BAD_QSL = 0x1, 0x2, 0x8


def cache_write(k_new, v_new, k_cache, v_cache, block_table, seq_lens, query_start_loc,
                block_size, kv_layout="nhd"):
    """The paged KV-cache write that precedes attention ("vLLM Triton attention
    backend deep dive", section "Technical implementation of paged
    attention": the cache is a pool of fixed-size blocks, and a sequence's
    block table maps its logical block j to a physical block).

    For request s with q_len = qsl[s+1] - qsl[s] new tokens on a context of
    seq_lens[s] positions (the new tokens included), new token i sits at
    position pos = seq_lens[s] - q_len + i, in physical block
    block_table[s][pos // block_size] at slot pos % block_size; its K and V
    rows ([num_kv_heads, head_dim] each) are copied there.

    k_new, v_new: [T, Hk, D]; k_cache, v_cache: [num_blocks, block_size, Hk, D]
    (any one dtype: values are copied, not converted).  Returns the two new
    caches (copies) and the status bits: a request with q_len > seq_len is
    skipped (DEV_BAD_QLEN); a token whose block id is outside the pool is
    skipped (DEV_BAD_BLOCK); a query_start_loc that does not start at 0,
    decreases, or does not end at T writes nothing (DEV_BAD_QSL).
    kv_layout "hnd": the caches are stored [num_blocks, Hk, block_size, D]
    (see nhd_view); the same rows land in that storage."""
    k_store, v_store = k_cache.copy(), v_cache.copy()
    k_out, v_out = nhd_view(k_store, kv_layout), nhd_view(v_store, kv_layout)
    qsl = [int(x) for x in query_start_loc]
    S, T = len(seq_lens), k_new.shape[0]
    nb = k_out.shape[0]
    if qsl[0] != 0 or qsl[S] != T or any(qsl[s + 1] < qsl[s] for s in range(S)):
        return k_store, v_store, DEV_BAD_QSL
    status = 0
    for s in range(S):
        q_len = qsl[s + 1] - qsl[s]
        prefix = int(seq_lens[s]) - q_len
        if prefix < 0:
            status |= DEV_BAD_QLEN
            continue
        for i in range(q_len):
            pos = prefix + i
            lp = pos // block_size
            page = int(block_table[s][lp]) if lp < block_table.shape[1] else -1
            if page < 0 or page >= nb:
                status |= DEV_BAD_BLOCK
                continue
            k_out[page, pos % block_size] = k_new[qsl[s] + i]
            v_out[page, pos % block_size] = v_new[qsl[s] + i]
    return k_store, v_store, status


def widen(a):
    """Stored values as float64: float32 as is, uint16 bf16 bit patterns as
    the exact binary32 they encode."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if a.dtype == np.float32:
        return a.astype(np.float64)
    raise TypeError(f"oracle inputs must be float32 or uint16 (bf16 bits), got {a.dtype}")


def mla_prefill(q, kv_cache, w_kv, block_table, seq_lens, query_start_loc, kv_lora_rank,
                qk_nope_dim, rope_dim, v_head_dim, block_size, scale, rows=None, q_block=64):
    """fp64 non-absorbed MLA prefill / extend ("vLLM AMD ROCm attention backend
    optimisation", section "AITER MLA backend: optimised for DeepSeek": prefill
    and extend run a standard multi-head attention on the uncompressed
    representation; decode works on the 576-wide compressed latent).

    q        [T, H, qk_nope_dim + rope_dim]: each head's no-position part,
             then its rotary part
    kv_cache [num_blocks, block_size, kv_lora_rank + rope_dim]: per position
             the latent c_j, then the rotary key k^R_j shared by all heads
    w_kv     [H, qk_nope_dim + v_head_dim, kv_lora_rank]: head h's
             up-projection; its first qk_nope_dim rows make the key, the
             rest the value

    The cache is decompressed position by position (a matrix product is the
    step): for every visible position j of a request,
        k_{j,h} = [ W_K,h c_j ; k^R_j ],   v_{j,h} = W_V,h c_j,
    and query i of request s, at position p = seq_len - q_len + i, attends to
    j <= p with the causal softmax of scale * q_{i,h} . k_{j,h}:
        out_{i,h} = sum_j softmax_j(scale q_{i,h} . k_{j,h}) v_{j,h}.
    rows: optional flat (token * H + head) indices; other rows are NaN.
    Returns out [T, H, v_head_dim] float64."""
    q = widen(q)
    cache = widen(kv_cache)
    w = widen(w_kv)
    T, H, dqk = q.shape
    assert dqk == qk_nope_dim + rope_dim
    assert cache.shape[2] == kv_lora_rank + rope_dim
    assert w.shape == (H, qk_nope_dim + v_head_dim, kv_lora_rank)
    w_k, w_v = w[:, :qk_nope_dim, :], w[:, qk_nope_dim:, :]
    qsl = [int(x) for x in query_start_loc]
    S = len(seq_lens)
    nb = cache.shape[0]
    out = np.full((T, H, v_head_dim), np.nan)
    want_tok = None
    if rows is not None:
        want_tok = np.zeros(T, bool)
        want_tok[np.asarray(rows, np.int64) // H] = True
    for s in range(S):
        q_len, ctx = qsl[s + 1] - qsl[s], int(seq_lens[s])
        if q_len <= 0:
            continue
        if q_len > ctx:
            raise OracleError("q_len above the context")
        toks = np.arange(qsl[s], qsl[s + 1])
        if want_tok is not None and not want_tok[toks].any():
            continue
        # the request's latent rows through its block table
        j = np.arange(ctx)
        pages = np.asarray(block_table)[s, j // block_size].astype(np.int64)
        if (pages < 0).any() or (pages >= nb).any():
            raise OracleError("block id outside the pool")
        lat = cache[pages, j % block_size]                    # [ctx, L + R]
        c, k_rope = lat[:, :kv_lora_rank], lat[:, kv_lora_rank:]
        k_nope = np.einsum("jl,hdl->jhd", c, w_k)              # [ctx, H, nope]
        v = np.einsum("jl,hdl->jhd", c, w_v)                   # [ctx, H, dv]
        prefix = ctx - q_len
        for b0 in range(0, q_len, q_block):
            ii = np.arange(b0, min(b0 + q_block, q_len))
            if want_tok is not None and not want_tok[qsl[s] + ii].any():
                continue
            qb = q[qsl[s] + ii]                                # [n, H, dqk]
            sc = (np.einsum("ihd,jhd->hij", qb[:, :, :qk_nope_dim], k_nope)
                  + np.einsum("ihd,jd->hij", qb[:, :, qk_nope_dim:], k_rope)) * scale
            visible = j[None, :] <= (prefix + ii)[:, None]      # [n, ctx]
            sc = np.where(visible[None], sc, -np.inf)
            mx = sc.max(axis=2, keepdims=True)
            p = np.exp(sc - mx)
            p /= p.sum(axis=2, keepdims=True)
            out[qsl[s] + ii] = np.einsum("hij,jhd->ihd", p, v)
    if rows is not None:
        keep = np.zeros(T * H, bool)
        keep[np.asarray(rows, np.int64)] = True
        out.reshape(T * H, v_head_dim)[~keep] = np.nan
    return out


def num_threads(lib=None):
    """Threads the oracle's OpenMP regions run with (its host cores)."""
    return int((lib or _lib()).oracle_num_threads())
