"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and the fp64 oracle on the same seeded inputs, compare element by element."""
import numpy as np
import torch

from oracle import oracle as orc
from paged_kv_attention_16_gb300 import inputs, pa

# Tolerances fixed for this method: fp32 inputs within max-abs 1e-4; bf16
# storage with fp32 accumulation within max-abs 2e-2 and mean-abs 2e-3.
TOL = {"f32": dict(max_abs=1e-4, mean_abs=1e-4), "bf16": dict(max_abs=2e-2, mean_abs=2e-3)}


def oracle_forward(b, rows=None, sinks=None, **variant):
    """The oracle on batch b; variant: sliding_window, alibi_slopes,
    alibi_sqrt (see oracle.paged_attention)."""
    return orc.paged_attention(
        inputs.storage_array(b.q), inputs.storage_array(b.k_cache),
        inputs.storage_array(b.v_cache), b.block_table.numpy(), b.seq_lens.numpy(),
        b.query_start_loc.numpy(), b.num_heads, b.num_kv_heads, b.head_dim, b.block_size,
        b.scale, rows=rows, sinks=None if sinks is None else np.asarray(sinks, np.float64),
        kv_layout=b.kv_layout, **variant)


def oracle_mla(b, rows=None):
    return orc.mla_decode(inputs.storage_array(b.q), inputs.storage_array(b.kv_cache),
                          b.block_table.numpy(), b.seq_lens.numpy(), b.kv_lora_rank, b.rope_dim,
                          b.block_size, b.scale, rows=rows)


def gpu_forward(b, kv_split_tokens=None, out=None, expect_status=0, sinks=None,
                sliding_window=0, alibi_slopes=None, alibi_sqrt=False, max_query_len=0):
    d = pa.to_device(b)
    if sinks is not None:
        sinks = torch.as_tensor(sinks, dtype=torch.float32).cuda()
    if alibi_slopes is not None:
        alibi_slopes = torch.as_tensor(alibi_slopes, dtype=torch.float32).cuda()
    got = pa.forward(d, out=out, kv_split_tokens=kv_split_tokens, sinks=sinks,
                     sliding_window=sliding_window, alibi_slopes=alibi_slopes,
                     alibi_sqrt=alibi_sqrt, max_query_len=max_query_len)
    status = pa.pa_get_device_status()
    assert status == expect_status, f"device status {status:#x}, expected {expect_status:#x}"
    return got.float().cpu().numpy().astype(np.float64)


def compare(got, want, dtype, rows=None, what=""):
    """Element-wise comparison on the listed flat (token*H + head) rows."""
    g = got.reshape(-1, got.shape[-1])
    w = want.reshape(-1, want.shape[-1])
    if rows is not None:
        g, w = g[rows], w[rows]
    assert np.isfinite(w).all(), "oracle produced non-finite values"
    assert np.isfinite(g).all(), f"{what}: GPU produced non-finite values"
    err = np.abs(g - w)
    tol = TOL[dtype]
    max_abs, mean_abs = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    assert max_abs <= tol["max_abs"], f"{what}: max-abs {max_abs:.3e} > {tol['max_abs']}"
    assert mean_abs <= tol["mean_abs"], f"{what}: mean-abs {mean_abs:.3e} > {tol['mean_abs']}"
    return max_abs, mean_abs


def sample_rows(b, n_other, seed=0, all_decode=True):
    """All rows of decode requests plus n_other random rows of the rest."""
    H = b.num_heads
    qsl = b.query_start_loc.numpy()
    dec, other = [], []
    for s in range(b.num_seqs):
        toks = np.arange(qsl[s], qsl[s + 1])
        rows = (toks[:, None] * H + np.arange(H)[None, :]).ravel()
        (dec if qsl[s + 1] - qsl[s] == 1 else other).append(rows)
    dec = np.concatenate(dec) if dec else np.zeros(0, np.int64)
    other = np.concatenate(other) if other else np.zeros(0, np.int64)
    rng = np.random.default_rng(seed)
    if len(other) > n_other:
        other = rng.choice(other, n_other, replace=False)
    rows = np.concatenate([dec if all_decode else dec[:0], other]).astype(np.int64)
    return np.sort(rows)


def cuda_ok():
    return torch.cuda.is_available()


def oracle_mla_prefill(b, rows=None):
    return orc.mla_prefill(inputs.storage_array(b.q), inputs.storage_array(b.kv_cache),
                           inputs.storage_array(b.w_kv), b.block_table.numpy(),
                           b.seq_lens.numpy(), b.query_start_loc.numpy(), b.kv_lora_rank,
                           b.qk_nope_dim, b.rope_dim, b.v_head_dim, b.block_size, b.scale,
                           rows=rows)


def tile_edge_rows(b, requests, tile_rows=128):
    """Flat (token * H + head) rows at the first and the last row of every
    tensor-core tile of the listed requests: a tile packs tile_rows / G
    tokens x the G query heads of one KV head, so its first row is (first
    token, first head of the group) and its last (last token, last head)."""
    H, Hk = b.num_heads, b.num_kv_heads
    G = H // Hk
    TQ = tile_rows // G
    qsl = b.query_start_loc.numpy()
    rows = []
    for s in requests:
        q0, q1 = int(qsl[s]), int(qsl[s + 1])
        for t0 in range(0, q1 - q0, TQ):
            t_last = min(t0 + TQ, q1 - q0) - 1
            for k in range(Hk):
                rows.append((q0 + t0) * H + k * G)
                rows.append((q0 + t_last) * H + k * G + G - 1)
    return np.asarray(rows, dtype=np.int64)


def longest_requests(b, kind):
    """Index of the longest prefill ("prefill": no cached prefix) or extend
    ("extend") request of a batch, by new tokens."""
    qsl = b.query_start_loc.numpy()
    ctx = b.seq_lens.numpy()
    best, best_len = None, 0
    for s in range(b.num_seqs):
        ql = int(qsl[s + 1] - qsl[s])
        is_prefill = ql == int(ctx[s]) and ql > 1
        is_extend = 1 < ql < int(ctx[s])
        if ((kind == "prefill" and is_prefill) or (kind == "extend" and is_extend)) and ql > best_len:
            best, best_len = s, ql
    return best

