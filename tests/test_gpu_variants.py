"""Sliding-window and ALiBi attention through pa_forward_ex on the GPU
against the oracle ("vLLM Triton attention backend deep dive", section
"Usage scenarios": ALiBi sqrt, sink tokens and GPT-OSS behaviour are model
features of the unified backend).  Every path is covered: the bf16 row
kernel and the fp32 row kernel, the tensor-core tile, split partials with
both merge passes, page boundaries inside a window, pages wholly below every
window left unmapped (-1), and the variants combined with sinks."""
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


def slopes(H, scale=1.0):
    """Geometric ALiBi slopes 2^(-8 h / H), h = 1..H, times `scale`."""
    return (scale * 2.0 ** (-8.0 * np.arange(1, H + 1) / H)).astype(np.float32)


def check(b, dtype, what, rows=None, kvs=None, expect_status=0, **variant):
    got = parity.gpu_forward(b, kv_split_tokens=kvs, expect_status=expect_status, **variant)
    want = parity.oracle_forward(b, rows=rows, **variant)
    parity.compare(got, want, dtype, rows=rows, what=what)


def small(dtype, head_dim, group, seed):
    Hk = 2
    return inputs.paged_batch([1, 1, 37, 5, 1, 130, 0, 3], [1, 300, 37, 261, 17, 200, 9, 3],
                              Hk * group, Hk, head_dim, 16, dtype=dtype, seed=seed)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("group", [1, 4, 16])
@pytest.mark.parametrize("window", [1, 16, 37, 100])
def test_sliding_window_small(dtype, head_dim, group, window):
    b = small(dtype, head_dim, group, seed=window + group)
    check(b, dtype, f"window {window} {dtype} D{head_dim} G{group}", sliding_window=window)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("group", [1, 8])
@pytest.mark.parametrize("use_sqrt", [False, True])
def test_alibi_small(dtype, head_dim, group, use_sqrt):
    b = small(dtype, head_dim, group, seed=3 * group + head_dim)
    check(b, dtype, f"alibi sqrt={use_sqrt} {dtype} D{head_dim} G{group}",
          alibi_slopes=slopes(b.num_heads), alibi_sqrt=use_sqrt)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_window_alibi_and_sinks_together(dtype):
    b = small(dtype, 128, 4, seed=77)
    sk = np.random.default_rng(1).normal(0.5, 1.5, b.num_heads).astype(np.float32)
    for use_sqrt in (False, True):
        check(b, dtype, f"all variants sqrt={use_sqrt}", sliding_window=50, sinks=sk,
              alibi_slopes=slopes(b.num_heads, 0.5), alibi_sqrt=use_sqrt)


@pytest.mark.parametrize("kvs", [16, 48, 256])
@pytest.mark.parametrize("window", [100, 700])
def test_window_with_forced_splits(kvs, window):
    """At kvs = 16 a 700-position window spans 45 splits (the merge's block
    pass, whose long-row list also holds windowed rows it must skip); the
    others go through the warp pass."""
    b = inputs.paged_batch([1, 1, 40, 1, 300], [2000, 70, 300, 16, 1200], 8, 2, 128, 16,
                           dtype="bf16", seed=kvs + window)
    check(b, "bf16", f"window {window} kvs {kvs}", kvs=kvs, sliding_window=window)
    check(b, "bf16", f"window {window} kvs {kvs} alibi", kvs=kvs, sliding_window=window,
          alibi_slopes=slopes(8), alibi_sqrt=True)


@pytest.mark.parametrize("kvs", [0, 1024])
def test_window_tile_chunked_extend(kvs):
    b = inputs.paged_batch([200, 1, 333], [3000, 2500, 333], 16, 2, 128, 64, dtype="bf16",
                           seed=kvs + 5)
    for window in (128, 1500):
        check(b, "bf16", f"tile window {window} kvs {kvs}", kvs=kvs, sliding_window=window)
    check(b, "bf16", f"tile alibi kvs {kvs}", kvs=kvs, alibi_slopes=slopes(16))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_pages_below_every_window_are_never_read(dtype):
    """Block-table entries of pages that lie wholly below every window of
    their request are set to -1 (freed): no status bit, same result."""
    window = 40
    b = inputs.paged_batch([1, 20, 1, 64], [900, 400, 50, 300], 8, 2, 128, 16, dtype=dtype,
                           seed=31)
    want = parity.oracle_forward(b, sliding_window=window)
    qsl, ctx, bs = b.query_start_loc.tolist(), b.seq_lens.tolist(), b.block_size
    freed = 0
    for s in range(b.num_seqs):
        lo = max(0, ctx[s] - (qsl[s + 1] - qsl[s]) - window + 1)  # first row's window
        for lp in range(lo // bs):
            b.block_table[s, lp] = -1
            freed += 1
    assert freed > 0
    got = parity.gpu_forward(b, sliding_window=window)
    parity.compare(got, want, dtype, what="freed pages below the window")


def test_window_mixed_qwen3_sampled():
    """The mixed batch with a 128-position window (GPT-OSS-style local
    layers), sinks and the full-size shapes, on sampled rows."""
    b = inputs.mixed_qwen3()
    rows = parity.sample_rows(b, 768, seed=7)
    sk = np.random.default_rng(2).normal(0.0, 1.0, b.num_heads).astype(np.float32)
    check(b, "bf16", "mixed window 128", rows=rows, sliding_window=128, sinks=sk)


def test_window_llama_decode_b64_full():
    b = inputs.llama_decode(64)
    check(b, "bf16", "llama b64 window 1024", sliding_window=1024)


@pytest.mark.parametrize("scale", [0.0, -0.09])
def test_zero_and_negative_scale(scale):
    """Masks must win over the scale whatever its sign: scale 0 (uniform
    weights over the visible keys) and a negative scale, on rows and tiles."""
    b = inputs.paged_batch([1, 1, 150, 77], [500, 33, 800, 77], 16, 2, 128, 16, dtype="bf16",
                           seed=8)
    b.scale = scale
    check(b, "bf16", f"scale {scale}")
    check(b, "bf16", f"scale {scale} window", sliding_window=60)
