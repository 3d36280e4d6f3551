"""The bounds-checked debug build (libssd_gb300_debug.so, -DSSD_DEBUG_BOUNDS).

compute-sanitizer is not available on the GPU pool these tests run on, so
the kernels carry their own checks in a debug build: every global index,
and every range of state or workspace elements a kernel computes itself, is
tested before use; a failure sets a bit in the device error word, records
the file and line, and the access is skipped (nothing traps).  These tests
build that library and, in a child process that loads it (SSD_DEBUG_BOUNDS=1),
run every plan the forward takes on small ragged cases, check parity with the
fp64 oracle, and require that no check fired.  A self-test hook shows that a
failing check is reported, with its file, and cleared.
"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (dtype, B, L, H, G, Q, initial states, environment): every plan of the forward
CASES = [
    ("bf16", 2, 640, 152, 2, 256, True, {}),                        # pair kernel, whole slabs
    ("bf16", 1, 3000, 308, 2, 256, True, {}),                       # pair kernel, sequence split
    ("bf16", 2, 1000, 3, 1, 256, True, {}),                         # single-head kernel, split
    ("bf16", 3, 389, 6, 6, 128, False, {}),                         # single-head kernel, whole
    ("bf16", 2, 700, 4, 2, 128, True, {"SSD_FORCE_STAGED": "1"}),   # staged tcgen05 steps
    ("bf16", 1, 1000, 4, 4, 64, True, {}),                          # staged: tc state, simt scan
    ("f32", 2, 333, 6, 3, 128, True, {}),                           # staged fp32 tensor-core steps
    ("f32", 2, 333, 6, 3, 128, True, {"SSD_FORCE_SIMT": "1"}),      # staged CUDA-core steps
]

CHILD = r"""
import ctypes, json, sys
import numpy as np, torch
sys.path.insert(0, sys.argv[1])
from oracle import oracle as orc
from state_space_model_gb300 import _native, inputs as gen, ssd
case = json.loads(sys.argv[2])
assert _native.LIB_PATH.endswith("libssd_gb300_debug.so"), _native.LIB_PATH
dtype, B, L, H, G, Q, h0 = case[:7]
w = gen.small_case(dtype, batch=B, seqlen=L, nheads=H, ngroups=G, chunk_size=Q,
                   init_states=h0, seed=606 + L)
plan = ssd.describe_plan(B, L, H, w.headdim, w.dstate, G, Q, w.torch_dtype)
inp = gen.make_inputs(w)
d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
y, f = ssd.chunked_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["initial_states"], Q, G)
lib = _native.load()
st = lib.ssd_device_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
detail = lib.ssd_last_error_detail().decode()
yr, fr = orc.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                        inp["initial_states"], ngroups=G)
rel = lambda a, b: float(np.max(np.abs(a - b)) / np.max(np.abs(b)))
print(json.dumps({"status": st, "detail": detail, "plan": plan,
                  "y": rel(y.float().cpu().double().numpy(), yr),
                  "f": rel(f.cpu().double().numpy(), fr)}))
"""

SELFTEST = r"""
import ctypes, json, sys
import torch
sys.path.insert(0, sys.argv[1])
from state_space_model_gb300 import _native
lib = _native.load()
stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
a = lib.ssd_selftest_bounds_check(stream)
b = lib.ssd_device_status(stream)
detail = lib.ssd_last_error_detail().decode()
c = lib.ssd_device_status(stream)
print(json.dumps({"launch": a, "status": b, "detail": detail, "after": c}))
"""


@pytest.fixture(scope="module")
def debug_lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from state_space_model_gb300 import build
    return build.build(debug_bounds=True)


def _child(code, *args, extra_env=None):
    env = dict(os.environ, SSD_DEBUG_BOUNDS="1", **(extra_env or {}))
    r = subprocess.run([sys.executable, "-c", code, ROOT, *args], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    return json.loads(r.stdout.strip().splitlines()[-1])


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c[:6])))
def test_debug_build_runs_every_plan_without_a_bounds_failure(debug_lib, case):
    out = _child(CHILD, json.dumps(list(case)), extra_env=case[7])
    assert out["status"] == 0, out["detail"]
    tol = 1e-4 if case[0] == "f32" else 2e-2
    assert out["y"] < tol and out["f"] < tol, out
    if case[7].get("SSD_FORCE_STAGED") == "1":
        assert out["plan"].startswith("staged") and "tcgen05" in out["plan"], out["plan"]


FULL = r"""
import ctypes, json, sys
import torch
sys.path.insert(0, sys.argv[1])
from state_space_model_gb300 import _native, inputs as gen, ssd
assert _native.LIB_PATH.endswith("libssd_gb300_debug.so"), _native.LIB_PATH
lib = _native.load()
w = gen.WORKLOADS[sys.argv[2]]
inp = gen.make_inputs(w)
d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
y, f = ssd.chunked_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["initial_states"],
                       w.chunk_size, w.ngroups)
torch.cuda.synchronize()
st = lib.ssd_device_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
print(json.dumps({"status": st, "detail": lib.ssd_last_error_detail().decode(),
                  "finite": bool(torch.isfinite(y.float()).all() and torch.isfinite(f).all())}))
"""


@pytest.mark.parametrize("name", ["tiny_f32", "mamba2_130m", "mamba2_2p7b", "hybrid_g8",
                                  "long_64k"])
def test_debug_build_at_full_size(debug_lib, name):
    """Every workload at its full size, in the plan the benchmark times,
    through the bounds-checked build: no check fires (parity at full size is
    tested on the normal build)."""
    out = _child(FULL, name)
    assert out["status"] == 0, out["detail"]
    assert out["finite"]


def test_debug_build_reports_a_failed_check(debug_lib):
    out = _child(SELFTEST)
    assert out["launch"] == 0
    assert out["status"] == 7 and "ssd_selftest.cu" in out["detail"], out   # SSD_ERR_DEVICE_BOUNDS
    assert out["after"] == 0, out   # reported once, then cleared


def test_normal_build_has_no_bounds_checks():
    import ctypes
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from state_space_model_gb300 import _native, build
    build.build()
    if _native.LIB_PATH.endswith("_debug.so"):
        pytest.skip("this process loads the debug build")
    lib = _native.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.ssd_selftest_bounds_check(stream) == 2   # SSD_ERR_UNSUPPORTED, nothing launched
