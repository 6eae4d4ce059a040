"""The kernels' failure path on the GPU, made to happen without faulting
anything: a bounded mbarrier wait that nothing completes runs out after a
millisecond, sets PA_DEV_TIMEOUT and its kernel returns; the context stays
usable and the next attention call is parity-green with a clean status."""
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


def test_bounded_wait_runs_out_and_reports_timeout():
    done = torch.zeros(1, dtype=torch.int32, device="cuda")
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    pa.pa_debug_wait_timeout(1_000_000, done)  # 1 ms
    end.record()
    torch.cuda.synchronize()
    assert int(done.item()) == 2  # timed out, then the latched second wait returned at once
    assert pa.pa_get_device_status() == pa.PA_DEV_TIMEOUT
    ms = start.elapsed_time(end)
    assert 0.9 <= ms < 100.0, f"the wait gave up after {ms:.3f} ms"
    # the context is intact: a full attention call afterwards is correct
    b = inputs.paged_batch([1, 40, 1], [700, 300, 33], 32, 8, 128, 16, dtype="bf16", seed=5)
    got = parity.gpu_forward(b)  # asserts a clean status word
    parity.compare(got, parity.oracle_forward(b), "bf16", what="after a timeout")


def test_wait_timeout_rejects_bad_limits():
    done = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert pa.pa_debug_wait_timeout(0, done, check=False) == pa.PA_ERR_INVALID_ARG
    assert pa.pa_debug_wait_timeout(2_000_000_000, done, check=False) == pa.PA_ERR_INVALID_ARG
    assert pa.pa_debug_wait_timeout(1000, None, check=False) == pa.PA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert int(done.item()) == 0
    assert pa.pa_get_device_status() == 0
