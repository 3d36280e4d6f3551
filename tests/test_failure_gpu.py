"""The failure path of the library's bounded waits, exercised without faulting
or hanging the GPU: a kernel whose wait (on an mbarrier phase nothing
completes) gives up after 1 ms records the timeout in the device error word;
ssd_device_status reports SSD_ERR_TIMEOUT once and clears it; the context is
still usable afterwards (a forward pass matches the oracle)."""
import ctypes

import numpy as np
import pytest
import torch

from oracle import oracle as orc

pytestmark = pytest.mark.gpu

SSD_ERR_TIMEOUT = 6


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from state_space_model_gb300 import _native, build
    build.build()
    return _native.load()


def test_bounded_wait_reports_timeout_and_context_survives(lib):
    from state_space_model_gb300 import inputs as gen, ssd
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.ssd_device_status(stream) == 0
    assert lib.ssd_selftest_wait_timeout(1_000_000, stream) == 0   # launched
    assert lib.ssd_device_status(stream) == SSD_ERR_TIMEOUT
    assert "bounded wait" in lib.ssd_last_error_detail().decode()
    assert lib.ssd_device_status(stream) == 0                      # read once, then cleared
    # the context still runs the forward correctly
    w = gen.small_case("bf16", batch=1, seqlen=300, nheads=2, ngroups=1, chunk_size=128)
    inp = gen.make_inputs(w)
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    y, f = ssd.chunked_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"],
                           d["initial_states"], w.chunk_size, w.ngroups)
    torch.cuda.synchronize()
    assert lib.ssd_device_status(stream) == 0
    yr, fr = orc.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                            inp["initial_states"], ngroups=w.ngroups)
    rel = lambda a, b: float(np.max(np.abs(a - b)) / np.max(np.abs(b)))
    assert rel(y.double().cpu().numpy(), yr) <= 2e-2
    assert rel(f.double().cpu().numpy(), fr) <= 2e-2
