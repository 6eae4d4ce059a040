"""pa_forward_static_scratch: the entry point for callers that cannot let the
library allocate device memory (graph capture in global mode, serving
runtimes that own every byte, latency-critical loops).  It must give the same
answer as pa_forward, call after call, while its scratch lives in one fixed
static region that every call reuses.

The file is named so that pytest collects it last: a run that stops at the
first failure has then already run every other test.  It also passes alone in
a fresh process."""
import ctypes

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
    pa.pa_get_device_status()


def static_call(d, out, status, kv_split_tokens=0, max_seq_len=None):
    """The new entry point, called directly through the C ABI."""
    L = pa.lib()
    return L.pa_forward_static_scratch(
        d.q.data_ptr(), d.k_cache.data_ptr(), d.v_cache.data_ptr(), d.block_table.data_ptr(),
        d.seq_lens.data_ptr(), d.query_start_loc.data_ptr(), d.num_heads, d.num_kv_heads,
        d.head_dim, d.block_size, ctypes.c_float(d.scale), out.data_ptr(),
        torch.cuda.current_stream().cuda_stream, pa.PA_BF16, d.num_seqs, d.num_tokens,
        d.max_blocks_per_seq, d.num_blocks, max_seq_len or d.max_seq_len, kv_split_tokens,
        status.data_ptr())


def test_static_scratch_matches_pa_forward_two_calls_in_a_row():
    batches = [
        # decode-heavy batch with long contexts (split partials + merge)
        inputs.paged_batch([1, 1, 1, 40, 1], [5000, 700, 1, 300, 2222], 32, 8, 128, 16,
                           dtype="bf16", seed=71),
        # different shapes of the same call kind: extend, prefill, GQA 16 decode
        inputs.paged_batch([1, 130, 64, 1], [3000, 900, 64, 17], 64, 4, 128, 16,
                           dtype="bf16", seed=72),
    ]
    for b in batches:
        d = pa.to_device(b)
        ref = pa.forward(d)  # the existing, allocating entry point
        torch.cuda.synchronize()
        assert pa.pa_get_device_status() == 0
        out = torch.full_like(d.q, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert static_call(d, out, status) == pa.PA_OK
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        got = out.float().cpu().numpy().astype(np.float64)
        want = ref.float().cpu().numpy().astype(np.float64)
        parity.compare(got, want, "bf16", what="static scratch vs pa_forward")


def test_static_scratch_reports_bad_metadata_in_the_callers_word():
    b = inputs.paged_batch([1, 1], [300, 40], 32, 8, 128, 16, dtype="bf16", seed=73)
    b.block_table[0, 3] = b.num_blocks + 9
    d = pa.to_device(b)
    out = torch.empty_like(d.q)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert static_call(d, out, status) == pa.PA_OK
    torch.cuda.synchronize()
    assert int(status.item()) & pa.PA_DEV_BAD_BLOCK
    assert torch.all(out[0] == 0)


def test_static_scratch_rejects_calls_beyond_its_size():
    b = inputs.paged_batch([1], [64], 32, 8, 128, 16, dtype="bf16", seed=74)
    d = pa.to_device(b)
    out = torch.empty_like(d.q)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # a max_seq_len whose split-partial bound exceeds the static region
    st = static_call(d, out, status, max_seq_len=1 << 22)
    assert st == pa.PA_ERR_SCRATCH_LIMIT
    assert "static scratch" in pa.status_string(st)
