"""pa_forward_static_scratch: the entry point for callers that cannot let the
library allocate device memory (graph capture in global mode, serving
runtimes that own every byte, latency-critical loops).  It runs the same
kernels as pa_forward on the same inputs, so its output must equal
pa_forward's bit for bit, call after call, while its scratch lives in one
fixed static region that every call reuses; and it must match the fp64
oracle within the bf16 tolerance.

The file is named so that pytest collects it last: a run that stops at the
first failure has then already run every other test.  It also passes alone in
a fresh process."""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from paged_kv_attention_16_gb300 import inputs, pa
from tests import parity

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_attention_16_gb300 import build
    build.build()
    pa.lib()
    pa.pa_get_device_status()


def static_call(d, out, status, kv_split_tokens=0, max_seq_len=None, stream=None):
    """The allocation-free entry point, called directly through the C ABI."""
    L = pa.lib()
    s = stream if stream is not None else torch.cuda.current_stream()
    return L.pa_forward_static_scratch(
        d.q.data_ptr(), d.k_cache.data_ptr(), d.v_cache.data_ptr(), d.block_table.data_ptr(),
        d.seq_lens.data_ptr(), d.query_start_loc.data_ptr(), d.num_heads, d.num_kv_heads,
        d.head_dim, d.block_size, ctypes.c_float(d.scale), out.data_ptr(), s.cuda_stream,
        pa.PA_BF16, d.num_seqs, d.num_tokens, d.max_blocks_per_seq, d.num_blocks,
        max_seq_len or d.max_seq_len, kv_split_tokens,
        None if status is None else status.data_ptr())


def bits(t):
    return t.view(torch.int16).cpu().numpy()


BATCHES = [
    # decode-heavy batch with long contexts (split partials + merge)
    lambda: inputs.paged_batch([1, 1, 1, 40, 1], [5000, 700, 1, 300, 2222], 32, 8, 128, 16,
                               dtype="bf16", seed=71),
    # extend, prefill and GQA-16 decode rows (tile kernel, row kernel, merge)
    lambda: inputs.paged_batch([1, 130, 64, 1], [3000, 900, 64, 17], 64, 4, 128, 16,
                               dtype="bf16", seed=72),
]


def test_static_scratch_equals_pa_forward_and_the_oracle_two_calls_in_a_row():
    for make in BATCHES:
        b = make()
        d = pa.to_device(b)
        ref = pa.forward(d)  # the allocating entry point, same kernels
        torch.cuda.synchronize()
        assert pa.pa_get_device_status() == 0
        want = parity.oracle_forward(b)
        for _ in range(2):  # the second call reuses the region the first left behind
            out = torch.full_like(d.q, float("nan"))
            status = torch.zeros(1, dtype=torch.int32, device="cuda")
            assert static_call(d, out, status) == pa.PA_OK
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            assert np.array_equal(bits(out), bits(ref)), "static scratch differs from pa_forward"
            got = out.float().cpu().numpy().astype(np.float64)
            parity.compare(got, want, "bf16", what="static scratch vs oracle")


def test_static_scratch_back_to_back_without_a_sync():
    """Two different calls queued on one stream with no synchronisation in
    between: stream order alone keeps the shared region consistent."""
    outs, refs = [], []
    devs = [pa.to_device(make()) for make in BATCHES]
    for d in devs:
        refs.append(pa.forward(d))
    torch.cuda.synchronize()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for d in devs:
        out = torch.full_like(d.q, float("nan"))
        assert static_call(d, out, status) == pa.PA_OK
        outs.append(out)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for out, ref in zip(outs, refs):
        assert np.array_equal(bits(out), bits(ref))


def test_static_scratch_graph_replay_with_new_metadata():
    """Captured once in global mode on a side stream; seq_lens, block_table
    and the cache contents change in place; every replay equals pa_forward on
    the new contents bit for bit and the oracle within tolerance."""
    H, Hk, D, bs = 32, 8, 128, 16
    b1 = inputs.paged_batch([1, 1, 1, 1, 1, 1], [500, 1200, 64, 3000, 17, 800], H, Hk, D, bs,
                            seed=81, max_seq_len=4096, pool_pages=700)
    b2 = inputs.paged_batch([1, 1, 1, 1, 1, 1], [4000, 20, 2222, 1, 999, 3500], H, Hk, D, bs,
                            seed=82, max_seq_len=4096, pool_pages=700)
    mb = max(b1.max_blocks_per_seq, b2.max_blocks_per_seq)

    def pad(t):
        o = torch.full((6, mb), -1, dtype=torch.int32)
        o[:, :t.shape[1]] = t
        return o

    b1.block_table, b2.block_table = pad(b1.block_table), pad(b2.block_table)
    d = pa.to_device(b1)
    out = torch.empty_like(d.q)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        assert static_call(d, out, status, stream=s) == pa.PA_OK  # warm-up, outside capture
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s, capture_error_mode="global"):
            st = static_call(d, out, status, stream=s)
    torch.cuda.synchronize()
    assert st == pa.PA_OK
    for b in (b2, b1):
        d.q.copy_(b.q.cuda())
        d.k_cache.copy_(b.k_cache.cuda())
        d.v_cache.copy_(b.v_cache.cuda())
        d.block_table.copy_(b.block_table.cuda())
        d.seq_lens.copy_(b.seq_lens.cuda())
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        ref = pa.forward(d)
        torch.cuda.synchronize()
        assert np.array_equal(bits(out), bits(ref)), "replay differs from pa_forward"
        got = out.float().cpu().numpy().astype(np.float64)
        parity.compare(got, parity.oracle_forward(b), "bf16", what="static scratch replay")


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


FIRST_CALL_IN_CAPTURE = r"""
import ctypes, sys, torch
sys.path.insert(0, sys.argv[1])
from paged_kv_attention_16_gb300 import inputs, pa
from tests.test_zz_no_alloc import static_call
d = pa.to_device(inputs.paged_batch([1, 1], [300, 40], 32, 8, 128, 16, dtype="bf16", seed=75))
out = torch.empty_like(d.q)
status = torch.zeros(1, dtype=torch.int32, device="cuda")
torch.cuda.synchronize()
s = torch.cuda.Stream()
with torch.cuda.stream(s):
    g = torch.cuda.CUDAGraph()
    g.capture_begin(capture_error_mode="global")
    try:
        st = static_call(d, out, status, stream=s)
    finally:
        g.capture_end()
assert st == pa.PA_ERR_WORKSPACE, st
with torch.cuda.stream(s):
    assert static_call(d, out, status, stream=s) == pa.PA_OK
torch.cuda.synchronize()
assert int(status.item()) == 0
print("FIRST_CALL_OK")
"""


def test_static_scratch_first_call_during_capture_is_refused_cleanly():
    """In a fresh process, where the region is not yet set up, a first call
    made while the stream captures returns PA_ERR_WORKSPACE, launches nothing
    and leaves the capture valid; the next call, outside capture, works."""
    r = subprocess.run([sys.executable, "-c", FIRST_CALL_IN_CAPTURE, ROOT], cwd=ROOT,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "FIRST_CALL_OK" in r.stdout, r.stdout + r.stderr
