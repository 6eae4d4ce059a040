"""Attention sinks through pa_forward_ex on the GPU against the oracle's
sink-aware attention ("vLLM Triton attention backend deep dive", section
"Usage scenarios": sink tokens are a model feature of the unified backend):
every path that finishes a row -- the decode row kernels writing directly,
the tensor-core tile writing directly, and both passes of the split merge --
must fold exp(sink) into the softmax denominator exactly once."""
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


def head_sinks(num_heads, seed, loc=1.0, spread=2.0):
    """Per-head sink logits (learned scalars in the models that use them):
    normal around `loc`, natural-log units."""
    return np.random.default_rng(seed).normal(loc, spread, num_heads).astype(np.float32)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("group", [1, 8])
def test_sinks_small_mixed(dtype, head_dim, group):
    Hk = 2
    b = inputs.paged_batch([1, 1, 37, 5, 1, 130, 0, 3], [1, 300, 37, 261, 17, 200, 9, 3],
                           Hk * group, Hk, head_dim, 16, dtype=dtype, seed=group + head_dim)
    sk = head_sinks(b.num_heads, seed=group)
    got = parity.gpu_forward(b, sinks=sk)
    parity.compare(got, parity.oracle_forward(b, sinks=sk), dtype,
                   what=f"sinks {dtype} D{head_dim} G{group}")


@pytest.mark.parametrize("kvs", [16, 48, 256])
def test_sinks_through_split_merge(kvs):
    """Forced splits: at 16 the 2000-key decode row has 125 splits (the
    merge's block pass over long rows), at 48 and 256 the warp pass."""
    b = inputs.paged_batch([1, 1, 40, 1], [2000, 70, 300, 16], 8, 2, 128, 16, dtype="bf16",
                           seed=kvs)
    sk = head_sinks(b.num_heads, seed=kvs)
    got = parity.gpu_forward(b, kv_split_tokens=kvs, sinks=sk)
    parity.compare(got, parity.oracle_forward(b, sinks=sk), "bf16", what=f"sinks kvs {kvs}")


def test_sinks_tile_chunked_extend():
    b = inputs.paged_batch([200, 1], [3000, 2500], 16, 2, 128, 64, dtype="bf16", seed=7)
    sk = head_sinks(b.num_heads, seed=3)
    want = parity.oracle_forward(b, sinks=sk)
    for kvs in (0, 1024):
        got = parity.gpu_forward(b, kv_split_tokens=kvs, sinks=sk)
        parity.compare(got, want, "bf16", what=f"sinks chunk {kvs}")


def test_sinks_llama_decode_b64_full():
    b = inputs.llama_decode(64)
    sk = head_sinks(b.num_heads, seed=64)
    got = parity.gpu_forward(b, sinks=sk)
    parity.compare(got, parity.oracle_forward(b, sinks=sk), "bf16", what="sinks llama b64")


def test_sinks_mixed_qwen3_sampled():
    b = inputs.mixed_qwen3()
    rows = parity.sample_rows(b, 768, seed=5)
    sk = head_sinks(b.num_heads, seed=5)
    got = parity.gpu_forward(b, sinks=sk)
    parity.compare(got, parity.oracle_forward(b, rows=rows, sinks=sk), "bf16", rows=rows,
                   what="sinks mixed")


@pytest.mark.parametrize("kvs", [0, 16])
def test_extreme_sinks(kvs):
    """Sinks of +-60 beside ordinary ones: a sink far above every score
    drives its head's output to ~0, one far below leaves plain attention."""
    b = inputs.paged_batch([1, 1, 24, 1], [700, 5, 24, 64], 8, 2, 64, 16, dtype="f32", seed=9)
    sk = np.array([60.0, -60.0, 0.0, 3.0, -60.0, 60.0, 1.5, -2.0], np.float32)
    got = parity.gpu_forward(b, kv_split_tokens=kvs, sinks=sk)
    want = parity.oracle_forward(b, sinks=sk)
    parity.compare(got, want, "f32", what=f"extreme sinks kvs {kvs}")
    assert np.abs(got[:, [0, 5]]).max() < 1e-12
    plain = parity.oracle_forward(b)
    parity.compare(got[:, [1, 4]], plain[:, [1, 4]], "f32", what="sink -60 is plain attention")


@pytest.mark.parametrize("kvs", [0, 16])
def test_minus_inf_sinks_are_bit_exact_with_none(kvs):
    """A sink of -inf adds exp(-inf) = 0 to every denominator: the output of
    pa_forward_ex must equal pa_forward's bit for bit, split or not."""
    b = inputs.paged_batch([1, 9, 1, 70], [1000, 333, 64, 70], 16, 4, 128, 16, dtype="bf16",
                           seed=1)
    d = pa.to_device(b)
    plain = pa.forward(d, kv_split_tokens=kvs)
    sk = torch.full((b.num_heads,), float("-inf"), device="cuda")
    with_sinks = pa.forward(d, kv_split_tokens=kvs, sinks=sk)
    assert pa.pa_get_device_status() == 0
    assert torch.equal(plain.view(torch.int16), with_sinks.view(torch.int16))
