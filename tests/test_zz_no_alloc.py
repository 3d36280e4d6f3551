"""The allocation-free entry point, ssd_chunked_fwd_static_scratch.

It serves callers that cannot give the library device workspace (no
allocator reachable from where they run, or cudaMalloc's device-wide
synchronisation and unbounded latency are not acceptable there): its scratch
is a fixed device array inside the library.  Here it is called through the C
ABI and its outputs are compared with those of ssd_chunked_fwd (caller
workspace) on the same inputs, bit for bit, on two calls in a row on
different inputs, and against the fp64 oracle within the bf16 parity bar the
other tests use.  This file is collected last on purpose.
"""
import ctypes
import os

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
# split (a few slabs over a long sequence).  Each family has a first, larger
# call that fills the scratch and a second call on different inputs (another
# seed, a sequence length that leaves a different partial last chunk): if a
# call read scratch bytes an earlier call left behind, the second call would
# not reproduce the workspace entry point bit for bit.
CASES = {
    "four_step": (dict(batch=2, seqlen=1500, nheads=4, ngroups=2, chunk_size=64, seed=71),
                  dict(batch=2, seqlen=1337, nheads=4, ngroups=2, chunk_size=64, seed=72)),
    "sequence_split": (dict(batch=1, seqlen=9000, nheads=4, ngroups=2, chunk_size=256, seed=73),
                       dict(batch=1, seqlen=7777, nheads=4, ngroups=2, chunk_size=256, seed=74)),
}


def _call_static(lib, ssd, inp, w, like_y, like_f):
    y = torch.full_like(like_y, float("nan"))
    f = torch.full_like(like_f, float("nan"))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.ssd_chunked_fwd_static_scratch(
        ssd._desc(inp["x"]), ssd._desc(inp["dt"]), ssd._desc(inp["A"]), ssd._desc(inp["B"]),
        ssd._desc(inp["C"]), ssd._desc(inp["D"]), ssd._desc(inp["initial_states"]),
        w.chunk_size, w.ngroups, ssd._desc(y), ssd._desc(f), stream)
    assert st == 0, lib.ssd_last_error_detail().decode()
    torch.cuda.synchronize()
    return y, f


@pytest.mark.parametrize("case", sorted(CASES))
def test_static_scratch_matches_oracle_and_workspace_entry_point(lib, case):
    from oracle import oracle as orc
    from state_space_model_gb300 import ssd
    if case == "sequence_split" and os.environ.get("SSD_NO_SPLIT") == "1":
        pytest.skip("SSD_NO_SPLIT=1 turns the sequence split off")
    for n, kw in enumerate(CASES[case]):
        w = gen.small_case("bf16", **kw)
        assert ssd.workspace_size(w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups,
                                  w.chunk_size, torch.bfloat16) > 0
        plan = ssd.describe_plan(w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups,
                                 w.chunk_size, torch.bfloat16)
        if case == "four_step":
            assert plan.startswith("staged"), plan
        else:
            assert plan.startswith("fused") and "segments" in plan, plan
        host = gen.make_inputs(w)
        inp = {k: (None if v is None else v.cuda()) for k, v in host.items()}
        y_ws, f_ws = ssd.chunked_fwd(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"],
                                     inp["D"], inp["initial_states"], w.chunk_size, w.ngroups)
        y, f = _call_static(lib, ssd, inp, w, y_ws, f_ws)
        assert torch.isfinite(y.float()).all() and torch.isfinite(f).all()
        # against the definition: the fp64 recurrence, the bf16 parity bar
        yr, fr = orc.recurrence(host["x"], host["dt"], host["A"], host["B"], host["C"],
                                host["D"], host["initial_states"], ngroups=w.ngroups)
        assert rel(y, torch.from_numpy(yr)) < TOL_BF16, (case, n)
        assert rel(f, torch.from_numpy(fr)) < TOL_BF16, (case, n)
        # the same kernels on the same inputs: bit for bit the workspace entry
        # point's result, whatever the earlier call left in the scratch
        assert torch.equal(y, y_ws) and torch.equal(f, f_ws), (case, n)


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
