"""Non-absorbed MLA prefill / extend (pa_mla_prefill) on the GPU against the
oracle ("vLLM AMD ROCm attention backend optimisation", section "AITER MLA
backend: optimised for DeepSeek": prefill and extend run standard multi-head
attention on the decompressed keys and values): mixed prefill / extend /
one-token batches, page sizes, head counts, forced KV splits through the
merge, bad metadata and an undersized decompression bound."""
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


def run(b, kv_split_tokens=None, expect_status=0):
    d = pa.to_device(b)
    got = pa.mla_prefill(d, kv_split_tokens=kv_split_tokens)
    status = pa.pa_get_device_status()
    assert status == expect_status, f"device status {status:#x}, expected {expect_status:#x}"
    return got.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("heads", [1, 16, 128])
@pytest.mark.parametrize("block_size", [16, 64])
def test_mla_prefill_small(heads, block_size):
    b = inputs.mla_prefill_batch([1, 7, 37, 130, 0, 3], [50, 7, 300, 130, 9, 3],
                                 num_heads=heads, block_size=block_size, seed=heads + block_size)
    parity.compare(run(b), parity.oracle_mla_prefill(b), "bf16",
                   what=f"mla prefill H{heads} bs{block_size}")


@pytest.mark.parametrize("kvs", [16, 64, 256])
def test_mla_prefill_forced_splits(kvs):
    b = inputs.mla_prefill_batch([200, 1, 64], [900, 333, 64], num_heads=16, seed=kvs)
    parity.compare(run(b, kv_split_tokens=kvs), parity.oracle_mla_prefill(b), "bf16",
                   what=f"mla prefill kvs {kvs}")


def test_mla_prefill_deepseek_sampled():
    b = inputs.mla_prefill_deepseek()
    H = b.num_heads
    rng = np.random.default_rng(3)
    toks = np.sort(rng.choice(b.num_tokens, 24, replace=False))
    rows = (toks[:, None] * H + np.arange(H)[None, :]).ravel()
    got = run(b)
    parity.compare(got, parity.oracle_mla_prefill(b, rows=rows), "bf16", rows=rows,
                   what="mla prefill deepseek")


def test_mla_prefill_bad_block_is_flagged():
    b = inputs.mla_prefill_batch([5, 3], [40, 100], num_heads=16, block_size=16, seed=9)
    want = parity.oracle_mla_prefill(b)
    b.block_table[1, 2] = 10_000  # a page of the second request
    got = run(b, expect_status=pa.PA_DEV_BAD_BLOCK)
    parity.compare(got[:5], want[:5], "bf16", what="healthy request")
    assert np.all(got[5:] == 0.0)


def test_mla_prefill_decompression_bound_overflow():
    b = inputs.mla_prefill_batch([5, 3], [40, 100], num_heads=16, seed=10)
    b.max_total_kv = 20  # far below 140 positions
    got = run(b, expect_status=pa.PA_DEV_OVERFLOW | pa.PA_DEV_BAD_BLOCK)
    assert np.all(got == 0.0)
