"""Sequence sharding over ranks through the library's kernels, the ranks
emulated one after another on one GPU (nothing waits on another kernel: the
exchange is a host-side stack of every rank's pair).  Each rank's segment is
run from a zero state, the pairs are gathered, and every rank is finished
with the combine and the correction; the reassembled y and the final states
are compared with the fp64 oracle over the whole sequence, at the parity
bars of the forward (1e-4 fp32, 2e-2 bf16).
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from state_space_model_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from state_space_model_gb300 import build
    build.build()


def _rel(a, b):
    return float(np.max(np.abs(a - b)) / np.max(np.abs(b)))


def _device_ok():
    from state_space_model_gb300 import _native
    lib = _native.load()
    st = lib.ssd_device_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.ssd_last_error_detail().decode()


CASES = [
    # dtype, ranks, B, L, H, G, Q, initial states
    ("bf16", 2, 2, 3000, 4, 2, 256, True),
    ("bf16", 4, 1, 5000, 8, 1, 128, False),
    ("bf16", 3, 2, 1000, 6, 6, 256, True),
    ("f32", 3, 2, 700, 4, 2, 64, True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_ranks_emulated_on_one_gpu_match_the_oracle(case):
    from state_space_model_gb300 import seqshard
    dtype, R, B, L, H, G, Q, h0 = case
    P, N = (16, 32) if dtype == "f32" else (64, 128)
    w = gen.small_case(dtype, batch=B, seqlen=L, nheads=H, headdim=P, dstate=N, ngroups=G,
                       chunk_size=Q, init_states=h0, dt_mu=-3.0, seed=313 + L)
    inp = gen.make_inputs(w)
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    cuts = [0] + [int(L * (r + 1) / R) - 5 * r for r in range(R - 1)] + [L]
    segs = [{k: d[k][:, cuts[r]:cuts[r + 1]] for k in ("x", "dt", "B", "C")} for r in range(R)]
    local = [seqshard.local_pass(s["x"], s["dt"], d["A"], s["B"], s["C"], d["D"], Q, G)
             for s in segs]
    ld_all = torch.stack([p[2] for p in local])
    st_all = torch.stack([p[1] for p in local])
    finals = [seqshard.finish(r, local[r][0], local[r][1], local[r][2], ld_all, st_all,
                              segs[r]["dt"], d["A"], segs[r]["C"], d["initial_states"], G)
              for r in range(R)]
    torch.cuda.synchronize()
    _device_ok()
    y = torch.cat([p[0] for p in local], dim=1).float().cpu().double().numpy()
    yr, fr = orc.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                            inp["initial_states"], ngroups=G)
    assert _rel(y, yr) < TOL[dtype]
    for r in range(R):
        end = cuts[r + 1]
        _, fe = orc.recurrence(inp["x"][:, :end], inp["dt"][:, :end], inp["A"],
                               inp["B"][:, :end], inp["C"][:, :end], inp["D"],
                               inp["initial_states"], ngroups=G)
        assert _rel(finals[r].cpu().double().numpy(), fe) < TOL[dtype], r
    assert _rel(finals[-1].cpu().double().numpy(), fr) < TOL[dtype]


def test_segment_logdecay_is_the_sum_of_a_dt():
    from state_space_model_gb300 import seqshard
    w = gen.small_case("bf16", batch=3, seqlen=1111, nheads=40, ngroups=1, seed=9)
    inp = gen.make_inputs(w)
    ld = seqshard.LibraryOps().logdecay(inp["dt"].cuda(), inp["A"].cuda())
    want = inp["A"].double()[None, :] * inp["dt"].double().sum(dim=1)
    assert torch.allclose(ld.cpu().double(), want, rtol=1e-6, atol=0)
