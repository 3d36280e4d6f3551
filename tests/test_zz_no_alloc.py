"""The allocation-free entry point, ssd_chunked_fwd_static_scratch.

It serves callers that cannot give the library device workspace (no
allocator reachable from where they run, or cudaMalloc's device-wide
synchronisation and unbounded latency are not acceptable there): its scratch
is a fixed device array inside the library.  Here it is called through the C
ABI and its outputs are compared with those of ssd_chunked_fwd (caller
workspace) on the same inputs, on two calls in a row, within the bf16 parity
bar the other tests use.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from state_space_model_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from state_space_model_gb300 import _native, build
    build.build()
    return _native.load()


def rel(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-30))


# Both plans that need scratch memory: the four-step path (chunk 64, which
# the single-kernel path does not take) and the single-kernel path's sequence
# split (a few (batch, head) slabs over a long sequence).
CASES = {
    "four_step": dict(batch=2, seqlen=600, nheads=4, ngroups=2, chunk_size=64),
    "sequence_split": dict(batch=1, seqlen=8000, nheads=4, ngroups=2, chunk_size=256),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_static_scratch_matches_workspace_entry_point(lib, case):
    from state_space_model_gb300 import ssd
    w = gen.small_case("bf16", **CASES[case])
    assert ssd.workspace_size(w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups,
                              w.chunk_size, torch.bfloat16) > 0
    plan = ssd.describe_plan(w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups,
                             w.chunk_size, torch.bfloat16)
    assert plan.startswith("staged" if case == "four_step" else "fused"), plan
    inp = {k: (None if v is None else v.cuda()) for k, v in gen.make_inputs(w).items()}
    y_ref, f_ref = ssd.chunked_fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                                   inp["initial_states"], w.chunk_size, w.ngroups)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        y = torch.full_like(y_ref, float("nan"))
        f = torch.full_like(f_ref, float("nan"))
        st = lib.ssd_chunked_fwd_static_scratch(
            ssd._desc(inp["x"]), ssd._desc(inp["dt"]), ssd._desc(inp["A"]), ssd._desc(inp["B"]),
            ssd._desc(inp["C"]), ssd._desc(inp["D"]), ssd._desc(inp["initial_states"]),
            w.chunk_size, w.ngroups, ssd._desc(y), ssd._desc(f), stream)
        assert st == 0, lib.ssd_last_error_detail().decode()
        torch.cuda.synchronize()
        assert torch.isfinite(y.float()).all() and torch.isfinite(f).all()
        assert rel(y, y_ref) < TOL_BF16
        assert rel(f, f_ref) < TOL_BF16


def test_static_scratch_rejects_problems_above_its_size(lib):
    from state_space_model_gb300 import ssd
    from state_space_model_gb300._native import SsdError
    B, L, H, P, N = 2, 8192, 32, 64, 128
    need = ssd.workspace_size(B, L, H, P, N, 1, 64, torch.bfloat16)
    assert need > (64 << 20)
    x = torch.zeros(B, L, H, P, dtype=torch.bfloat16, device="cuda")
    dt = torch.zeros(B, L, H, device="cuda")
    A = torch.zeros(H, device="cuda")
    Bm = torch.zeros(B, L, 1, N, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(SsdError) as ei:
        ssd.chunked_fwd_static_scratch(x, dt, A, Bm, Bm.clone(), chunk_size=64, ngroups=1)
    assert ei.value.status == 4 and "static scratch" in ei.value.detail
