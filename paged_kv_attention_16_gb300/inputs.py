"""Seeded synthetic inputs for unified paged attention and absorbed-MLA decode.

This module only draws numbers and lays them out; it holds none of the
attention arithmetic, so both the CUDA path and the fp64 oracle can be fed
from it.  Every tensor is created on the CPU with a seeded torch.Generator,
rounded to the storage dtype, and handed over as is.

Layouts (the library's, see include/pa.h):
  q                [num_tokens, num_heads, head_dim]
  k_cache, v_cache [num_blocks, block_size, num_kv_heads, head_dim]
  block_table      [num_seqs, max_blocks_per_seq] int32
  seq_lens         [num_seqs] int32   (context length including new tokens)
  query_start_loc  [num_seqs + 1] int32
MLA:
  q                [num_seqs, num_heads, kv_lora_rank + rope_dim]
  kv_cache         [num_blocks, block_size, kv_lora_rank + rope_dim]

Page placement is a seeded random permutation of a pool sized to the pages
in use plus slack.  With poison=True, unused pool pages, tail slots of each
request's last page and unused block-table entries hold NaN / invalid ids, so
a kernel that reads outside the visible range shows it.
"""
import dataclasses
from dataclasses import dataclass, field
import math

import numpy as np
import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclass
class PagedBatch:
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    block_table: torch.Tensor
    seq_lens: torch.Tensor
    query_start_loc: torch.Tensor
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    scale: float
    dtype: str
    max_seq_len: int
    kv_split_tokens: int = 0
    kinds: list = field(default_factory=list)
    kv_layout: str = "nhd"  # "nhd": caches [nb, bs, Hk, D]; "hnd": [nb, Hk, bs, D]

    @property
    def num_seqs(self):
        return int(self.seq_lens.shape[0])

    @property
    def num_tokens(self):
        return int(self.q.shape[0])

    @property
    def num_blocks(self):
        return int(self.k_cache.shape[0])

    @property
    def max_blocks_per_seq(self):
        return int(self.block_table.shape[1])


@dataclass
class MlaBatch:
    q: torch.Tensor
    kv_cache: torch.Tensor
    block_table: torch.Tensor
    seq_lens: torch.Tensor
    num_heads: int
    kv_lora_rank: int
    rope_dim: int
    block_size: int
    scale: float
    dtype: str
    max_seq_len: int
    kv_split_tokens: int = 0

    @property
    def num_seqs(self):
        return int(self.seq_lens.shape[0])

    @property
    def num_blocks(self):
        return int(self.kv_cache.shape[0])

    @property
    def max_blocks_per_seq(self):
        return int(self.block_table.shape[1])


def _gen(seed):
    return torch.Generator().manual_seed(int(seed))


def _normal(shape, gen, dtype):
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(DTYPES[dtype])


def _place_pages(ctx_lens, block_size, gen, slack, pool_pages, poison):
    pages = [max(1, math.ceil(c / block_size)) if c > 0 else 0 for c in ctx_lens]
    used = sum(pages)
    pool = pool_pages if pool_pages is not None else used + max(1, math.ceil(slack * used))
    if pool < used:
        raise ValueError("page pool smaller than the pages in use")
    perm = torch.randperm(pool, generator=gen).to(torch.int32)
    max_blocks = max(pages) if pages else 1
    max_blocks = max(max_blocks, 1)
    # Unused entries hold ids the kernel must never follow.
    bad = -1 if poison else 0
    table = torch.full((len(ctx_lens), max_blocks), bad, dtype=torch.int32)
    if poison and max_blocks > 1:
        table[:, 1::2] = pool + 1000  # out of range as well
    off = 0
    for s, n in enumerate(pages):
        table[s, :n] = perm[off:off + n]
        off += n
    return table, pool, perm[:used]


def paged_batch(q_lens, ctx_lens, num_heads, num_kv_heads, head_dim, block_size,
                dtype="bf16", seed=0, poison=True, slack=0.1, pool_pages=None,
                scale=None, kv_split_tokens=0, max_seq_len=None, order_seed=None):
    """Build a mixed batch.  q_lens[s] new tokens on a context of ctx_lens[s]
    positions (the new tokens included).  order_seed, if given, shuffles the
    request order (the library is expected to reorder the work itself)."""
    q_lens = [int(x) for x in q_lens]
    ctx_lens = [int(x) for x in ctx_lens]
    if order_seed is not None:
        perm = torch.randperm(len(q_lens), generator=_gen(order_seed)).tolist()
        q_lens = [q_lens[i] for i in perm]
        ctx_lens = [ctx_lens[i] for i in perm]
    for ql, c in zip(q_lens, ctx_lens):
        if ql > c or ql < 0:
            raise ValueError("q_len must lie in [0, ctx]")
    g_layout = _gen(seed * 7919 + 1)
    g_vals = _gen(seed * 104729 + 2)
    table, pool, _ = _place_pages(ctx_lens, block_size, g_layout, slack, pool_pages, poison)
    T = sum(q_lens)
    q = _normal((T, num_heads, head_dim), g_vals, dtype)
    k = _normal((pool, block_size, num_kv_heads, head_dim), g_vals, dtype)
    v = _normal((pool, block_size, num_kv_heads, head_dim), g_vals, dtype)
    if poison:
        _poison_cache([k, v], table, ctx_lens, block_size, pool)
    qsl = torch.zeros(len(q_lens) + 1, dtype=torch.int32)
    if q_lens:
        qsl[1:] = torch.cumsum(torch.tensor(q_lens, dtype=torch.int64), 0).to(torch.int32)
    kinds = []
    for ql, c in zip(q_lens, ctx_lens):
        kinds.append("decode" if ql == 1 else ("prefill" if c == ql else "extend"))
    return PagedBatch(
        q=q, k_cache=k, v_cache=v, block_table=table,
        seq_lens=torch.tensor(ctx_lens, dtype=torch.int32), query_start_loc=qsl,
        num_heads=num_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
        block_size=block_size,
        scale=scale if scale is not None else 1.0 / math.sqrt(head_dim),
        dtype=dtype, max_seq_len=max_seq_len or max(ctx_lens + [1]),
        kv_split_tokens=kv_split_tokens, kinds=kinds)


def _poison_cache(caches, table, ctx_lens, block_size, pool):
    used = torch.zeros(pool, dtype=torch.bool)
    for s, c in enumerate(ctx_lens):
        n = math.ceil(c / block_size) if c > 0 else 0
        ids = table[s, :n].long()
        used[ids] = True
        tail = c - (n - 1) * block_size if n else 0
        if n and tail < block_size:
            for cache in caches:
                cache[ids[n - 1], tail:] = float("nan")
    for cache in caches:
        cache[~used] = float("nan")


def mla_batch(ctx_lens, num_heads=128, kv_lora_rank=512, rope_dim=64, block_size=64,
              dtype="bf16", seed=0, poison=True, slack=0.1, scale=None, kv_split_tokens=0,
              max_seq_len=None):
    ctx_lens = [int(x) for x in ctx_lens]
    g_layout = _gen(seed * 7919 + 3)
    g_vals = _gen(seed * 104729 + 4)
    table, pool, _ = _place_pages(ctx_lens, block_size, g_layout, slack, None, poison)
    width = kv_lora_rank + rope_dim
    q = _normal((len(ctx_lens), num_heads, width), g_vals, dtype)
    kv = _normal((pool, block_size, width), g_vals, dtype)
    if poison:
        _poison_cache([kv], table, ctx_lens, block_size, pool)
    return MlaBatch(q=q, kv_cache=kv, block_table=table,
                    seq_lens=torch.tensor(ctx_lens, dtype=torch.int32), num_heads=num_heads,
                    kv_lora_rank=kv_lora_rank, rope_dim=rope_dim, block_size=block_size,
                    scale=scale if scale is not None else 1.0 / math.sqrt(192.0),
                    dtype=dtype, max_seq_len=max_seq_len or max(ctx_lens + [1]),
                    kv_split_tokens=kv_split_tokens)


@dataclass
class MlaPrefillBatch:
    q: torch.Tensor          # [T, H, qk_nope_dim + rope_dim]
    kv_cache: torch.Tensor   # [num_blocks, block_size, kv_lora_rank + rope_dim]
    w_kv: torch.Tensor       # [H, qk_nope_dim + v_head_dim, kv_lora_rank]
    block_table: torch.Tensor
    seq_lens: torch.Tensor
    query_start_loc: torch.Tensor
    num_heads: int
    kv_lora_rank: int
    qk_nope_dim: int
    rope_dim: int
    v_head_dim: int
    block_size: int
    scale: float
    dtype: str
    max_seq_len: int
    max_total_kv: int
    kv_split_tokens: int = 0

    @property
    def num_seqs(self):
        return int(self.seq_lens.shape[0])

    @property
    def num_tokens(self):
        return int(self.q.shape[0])


def mla_prefill_batch(q_lens, ctx_lens, num_heads=128, kv_lora_rank=512, qk_nope_dim=128,
                      rope_dim=64, v_head_dim=128, block_size=64, seed=0, poison=True,
                      slack=0.1, kv_split_tokens=0):
    """Non-absorbed MLA prefill / extend inputs: queries of qk_nope_dim +
    rope_dim per head, the latent cache of pa_mla_decode, and a synthetic
    up-projection w_kv drawn N(0, 1 / kv_lora_rank) (so decompressed keys
    and values have unit variance); scale 1/sqrt(qk_nope_dim + rope_dim)."""
    q_lens = [int(x) for x in q_lens]
    ctx_lens = [int(x) for x in ctx_lens]
    g_layout = _gen(seed * 7919 + 5)
    g_vals = _gen(seed * 104729 + 6)
    table, pool, _ = _place_pages(ctx_lens, block_size, g_layout, slack, None, poison)
    dqk = qk_nope_dim + rope_dim
    q = _normal((sum(q_lens), num_heads, dqk), g_vals, "bf16")
    kv = _normal((pool, block_size, kv_lora_rank + rope_dim), g_vals, "bf16")
    w = (torch.randn((num_heads, qk_nope_dim + v_head_dim, kv_lora_rank), generator=g_vals)
         / math.sqrt(kv_lora_rank)).to(torch.bfloat16)
    if poison:
        _poison_cache([kv], table, ctx_lens, block_size, pool)
    qsl = torch.tensor([0] + list(np.cumsum(q_lens)), dtype=torch.int32)
    return MlaPrefillBatch(q=q, kv_cache=kv, w_kv=w, block_table=table,
                           seq_lens=torch.tensor(ctx_lens, dtype=torch.int32),
                           query_start_loc=qsl, num_heads=num_heads, kv_lora_rank=kv_lora_rank,
                           qk_nope_dim=qk_nope_dim, rope_dim=rope_dim, v_head_dim=v_head_dim,
                           block_size=block_size, scale=1.0 / math.sqrt(dqk), dtype="bf16",
                           max_seq_len=max(ctx_lens + [1]), max_total_kv=sum(ctx_lens),
                           kv_split_tokens=kv_split_tokens)


def _uniform_ints(gen, n, lo, hi):
    """n integers uniform on [lo, hi] (both ends included)."""
    if n == 0:
        return []
    return torch.randint(lo, hi + 1, (n,), generator=gen).tolist()


# ---------------------------------------------------------------------------
# The five workload shapes.  Lengths are drawn with seed 1234 + workload index.
# ---------------------------------------------------------------------------

def tiny_decode_f32(poison=True, seed=0):
    """4 decodes, contexts {17, 64, 129, 200}; 8 q heads, 2 KV heads, head_dim 64,
    block_size 16, fp32; a 64-page pool placed by a seeded permutation."""
    return paged_batch([1, 1, 1, 1], [17, 64, 129, 200], 8, 2, 64, 16, dtype="f32",
                       seed=seed, poison=poison, pool_pages=64)


def llama_decode(batch, poison=True, seed=1):
    """Llama-3.1-8B-shaped GQA decode: 32 q heads, 8 KV heads, head_dim 128,
    block_size 16, bf16.  batch 1 at context 500, otherwise contexts uniform on
    [500, 8192]."""
    if batch == 1:
        ctx = [500]
    else:
        ctx = _uniform_ints(_gen(1234 + 1), batch, 500, 8192)
    return paged_batch([1] * batch, ctx, 32, 8, 128, 16, dtype="bf16", seed=seed,
                       poison=poison)


def mixed_qwen3(poison=True, seed=2, n_decode=48, n_extend=12, n_prefill=4):
    """Qwen3-235B-shaped mixed continuous batch: 64 q heads, 4 KV heads,
    head_dim 128, block_size 16, bf16.  48 decodes on contexts 1K-16K, 12
    extends of 64-512 new tokens on 1K-8K cached, 4 prefills of 512-4096
    tokens; the request order is shuffled."""
    g = _gen(1234 + 2)
    dec_ctx = _uniform_ints(g, n_decode, 1024, 16384)
    ext_new = _uniform_ints(g, n_extend, 64, 512)
    ext_pre = _uniform_ints(g, n_extend, 1024, 8192)
    pre_len = _uniform_ints(g, n_prefill, 512, 4096)
    q_lens = [1] * n_decode + ext_new + pre_len
    ctx = dec_ctx + [a + b for a, b in zip(ext_new, ext_pre)] + pre_len
    return paged_batch(q_lens, ctx, 64, 4, 128, 16, dtype="bf16", seed=seed, poison=poison,
                       order_seed=1234 + 2)


def long_chunked(poison=True, seed=3, ctx_decode=131072, n_decode=4, n_extend=2,
                 ext_new=2048, ext_prefix=98304):
    """Long-context chunked extend/decode: 8 q heads, 1 KV head, head_dim 128,
    block_size 64, bf16.  4 decodes at 128K context plus 2 extends of 2048
    tokens on 96K cached; KV processed in 32K-token chunks."""
    q_lens = [1] * n_decode + [ext_new] * n_extend
    ctx = [ctx_decode] * n_decode + [ext_prefix + ext_new] * n_extend
    return paged_batch(q_lens, ctx, 8, 1, 128, 64, dtype="bf16", seed=seed, poison=poison,
                       kv_split_tokens=32768)


def mla_decode_batch(batch=64, poison=True, seed=4):
    """DeepSeek-style absorbed MLA decode: 128 q heads on one 576-wide latent
    (512 + 64 rope), value width 512, block_size 64, bf16; contexts uniform on
    [1K, 16K]; scale 1/sqrt(192)."""
    ctx = _uniform_ints(_gen(1234 + 4), batch, 1024, 16384)
    return mla_batch(ctx, 128, 512, 64, 64, dtype="bf16", seed=seed, poison=poison)


def mla_prefill_deepseek(poison=True, seed=5, n_prefill=4, n_extend=4):
    """DeepSeek-style non-absorbed MLA prefill / extend: 128 heads, latent 512
    + rope 64, key rows 128 + 64, value rows 128, block_size 64, bf16; 4
    prefills of 512-2048 tokens and 4 extends of 128-512 new tokens on 1K-4K
    cached."""
    g = _gen(1234 + 5)
    pre = _uniform_ints(g, n_prefill, 512, 2048)
    ext_new = _uniform_ints(g, n_extend, 128, 512)
    ext_pre = _uniform_ints(g, n_extend, 1024, 4096)
    q_lens = pre + ext_new
    ctx = pre + [a + b for a, b in zip(ext_new, ext_pre)]
    return mla_prefill_batch(q_lens, ctx, seed=seed, poison=poison)


WORKLOADS = {
    "tiny_decode_f32": tiny_decode_f32,
    "llama_decode_b1": lambda poison=True: llama_decode(1, poison),
    "llama_decode_b64": lambda poison=True: llama_decode(64, poison),
    "mixed_qwen3": mixed_qwen3,
    "long_chunked": long_chunked,
    "mla_decode": mla_decode_batch,
    "mla_prefill": mla_prefill_deepseek,
}


def storage_array(t):
    """The stored bits of a CPU tensor as numpy: float32 stays float32, bf16
    comes back as uint16 bit patterns (what the oracle reads)."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy()
    if t.dtype == torch.int32:
        return t.numpy()
    raise TypeError(t.dtype)


def as_hnd(b):
    """The same batch with its caches stored head-major, [nb, Hk, bs, D]
    (a copy; values and block table unchanged)."""
    fields = {f.name: getattr(b, f.name) for f in dataclasses.fields(b)}
    fields["k_cache"] = b.k_cache.permute(0, 2, 1, 3).contiguous()
    fields["v_cache"] = b.v_cache.permute(0, 2, 1, 3).contiguous()
    fields["kv_layout"] = "hnd"
    return type(b)(**fields)
