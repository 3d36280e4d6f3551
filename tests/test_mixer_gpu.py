"""GPU parity of the mixer prologue (ssd_mixer_prologue: causal conv1d + SiLU,
x / B / C split, dt bias + softplus, conv state and windows) against the fp64
oracle, and of the prologue followed by the scan against the recurrence.

Bars: x, B, C within 2e-2 (bf16 outputs) or 1e-4 (fp32) as max|gpu - ref| /
max|ref|; dt' within 1e-5 (fp32 softplus of fp32 inputs); the conv state and
windows are copies of inputs, so they match exactly.
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle as orc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ssd():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from state_space_model_gb300 import build, ssd as mod
    build.build()
    return mod


def rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-30))


def make_mixer(B, L, H, P, G, N, W, dtype, seed, state=True, bias=True):
    g = torch.Generator().manual_seed(seed)
    r = lambda *s: torch.randn(s, generator=g)
    Dc = H * P + 2 * G * N
    return dict(xBC=r(B, L, Dc).to(dtype), conv_weight=r(Dc, W) / math.sqrt(W),
                conv_bias=0.1 * r(Dc) if bias else None,
                conv_state=r(B, Dc, W).to(dtype) if state else None,
                dt=r(B, L, H) * 0.5 - 2.0, dt_bias=0.1 * r(H) if bias else None)


CASES = [
    # (B, L, H, P, G, N, W, dtype, state, windows, bias, softplus)
    (2, 300, 4, 64, 2, 128, 4, torch.bfloat16, True, False, True, True),    # several runs
    (1, 50, 8, 64, 1, 128, 4, torch.bfloat16, True, True, True, True),      # one run, windows
    (3, 130, 2, 32, 1, 16, 3, torch.float32, False, False, False, False),
    (2, 2, 4, 16, 2, 16, 4, torch.bfloat16, True, True, True, True),        # L < W
    (1, 64, 4, 64, 1, 128, 1, torch.float32, True, True, True, True),       # W = 1, one run
    (2, 65, 4, 64, 1, 64, 2, torch.bfloat16, True, False, True, False),     # just past a run
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}L{c[1]}H{c[2]}P{c[3]}G{c[4]}"
                         f"N{c[5]}W{c[6]}-{str(c[7])[6:]}-st{int(c[8])}win{int(c[9])}")
def test_mixer_prologue_matches_oracle(ssd, case):
    B, L, H, P, G, N, W, dtype, state, windows, bias, sp = case
    inp = make_mixer(B, L, H, P, G, N, W, dtype, seed=L * 7 + W, state=state, bias=bias)
    out_ref, st_ref, win_ref = orc.causal_conv1d(inp["xBC"], inp["conv_weight"],
                                                 inp["conv_bias"], inp["conv_state"])
    x_ref, b_ref, c_ref = orc.split_xbc(out_ref, H, P, G, N)
    dt_ref = orc.dt_prologue(inp["dt"], inp["dt_bias"], sp)
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    Dc = H * P + 2 * G * N
    win = torch.empty((B, L, Dc, W), dtype=dtype, device="cuda") if windows else None
    x, Bm, Cm, dt = ssd.mixer_prologue(d["xBC"], d["conv_weight"], d["dt"], H, P, G, N,
                                       conv_bias=d["conv_bias"], conv_state=d["conv_state"],
                                       conv_windows=win, dt_bias=d["dt_bias"], dt_softplus=sp)
    torch.cuda.synchronize()
    bar = 2e-2 if dtype == torch.bfloat16 else 1e-4
    for got, ref in ((x, x_ref), (Bm, b_ref), (Cm, c_ref)):
        assert got.dtype == dtype
        assert rel(got.double().cpu().numpy(), ref) <= bar
    assert rel(dt.double().cpu().numpy(), dt_ref) <= 1e-5
    cast = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dtype)
    if state:
        assert torch.equal(d["conv_state"].cpu(), cast(st_ref))
    if windows:
        assert torch.equal(win.cpu(), cast(win_ref))


def test_conv_state_carries_across_calls(ssd):
    """Two calls over the halves of a sequence, the state carried in place,
    equal one call over the whole sequence bit for bit."""
    H, P, G, N, W = 4, 64, 1, 128, 4
    inp = make_mixer(2, 200, H, P, G, N, W, torch.bfloat16, seed=3)
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    st_one = d["conv_state"].clone()
    whole = ssd.mixer_prologue(d["xBC"], d["conv_weight"], d["dt"], H, P, G, N,
                               conv_bias=d["conv_bias"], conv_state=st_one, dt_bias=d["dt_bias"])
    st_two = d["conv_state"].clone()
    parts = []
    for lo, hi in ((0, 77), (77, 200)):
        parts.append(ssd.mixer_prologue(d["xBC"][:, lo:hi].contiguous(), d["conv_weight"],
                                        d["dt"][:, lo:hi].contiguous(), H, P, G, N,
                                        conv_bias=d["conv_bias"], conv_state=st_two,
                                        dt_bias=d["dt_bias"]))
    torch.cuda.synchronize()
    for i in range(4):
        assert torch.equal(whole[i], torch.cat([parts[0][i], parts[1][i]], dim=1))
    assert torch.equal(st_one, st_two)


def test_prologue_then_scan_matches_the_recurrence(ssd):
    """The mixer's prologue feeding the fused scan: y against the recurrence run on
    the oracle's own prologue outputs."""
    B, L, H, P, G, N, W = 2, 512, 8, 64, 2, 128, 4
    inp = make_mixer(B, L, H, P, G, N, W, torch.bfloat16, seed=9)
    g = torch.Generator().manual_seed(10)
    A = -torch.exp(torch.rand(H, generator=g) * math.log(16.0))
    D = torch.randn(H, generator=g)
    out_ref, _, _ = orc.causal_conv1d(inp["xBC"], inp["conv_weight"], inp["conv_bias"],
                                      inp["conv_state"])
    x_ref, b_ref, c_ref = (torch.from_numpy(np.ascontiguousarray(a))
                           for a in orc.split_xbc(out_ref, H, P, G, N))
    dt_ref = torch.from_numpy(orc.dt_prologue(inp["dt"], inp["dt_bias"]))
    y_ref, fin_ref = orc.recurrence(x_ref, dt_ref, A, b_ref, c_ref, D, None, ngroups=G)
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    x, Bm, Cm, dt = ssd.mixer_prologue(d["xBC"], d["conv_weight"], d["dt"], H, P, G, N,
                                       conv_bias=d["conv_bias"], conv_state=d["conv_state"],
                                       dt_bias=d["dt_bias"])
    y, fin = ssd.chunked_fwd(x, dt, A.cuda(), Bm, Cm, D.cuda(), None, 256, G)
    torch.cuda.synchronize()
    assert rel(y.double().cpu().numpy(), y_ref) <= 2e-2
    assert rel(fin.double().cpu().numpy(), fin_ref) <= 2e-2


GATED = [
    # (B, L, H, P, N, G, Q, dtype, h0): fused plan (bf16, P 64, N 128) incl. a ragged
    # end and a sequence split; four-step plan (fp32, other P / N)
    (2, 512, 8, 64, 128, 2, 256, torch.bfloat16, False),
    (1, 300, 4, 64, 128, 1, 128, torch.bfloat16, True),
    (1, 8000, 4, 64, 128, 2, 256, torch.bfloat16, True),
    (2, 200, 4, 32, 64, 2, 64, torch.bfloat16, False),
    (1, 130, 3, 16, 16, 1, 64, torch.float32, True),
]


@pytest.mark.parametrize("case", GATED, ids=lambda c: f"B{c[0]}L{c[1]}H{c[2]}P{c[3]}N{c[4]}"
                         f"G{c[5]}Q{c[6]}-{str(c[7])[6:]}-h0{int(c[8])}")
def test_gated_forward_matches_oracle(ssd, case):
    from state_space_model_gb300 import inputs as gen
    B, L, H, P, N, G, Q, dtype, h0 = case
    w = gen.small_case("bf16" if dtype == torch.bfloat16 else "f32", batch=B, seqlen=L,
                       nheads=H, headdim=P, dstate=N, ngroups=G, chunk_size=Q, init_states=h0)
    inp = gen.make_inputs(w)
    z = torch.randn((B, L, H, P), generator=torch.Generator().manual_seed(L)).to(dtype)
    y_ref, fin_ref = orc.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                                    inp["initial_states"], ngroups=G)
    yg_ref = orc.gate(y_ref, z)
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    y, fin = ssd.chunked_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"],
                             d["initial_states"], Q, G, z=z.cuda())
    torch.cuda.synchronize()
    bar = 2e-2 if dtype == torch.bfloat16 else 1e-4
    assert rel(y.double().cpu().numpy(), yg_ref) <= bar
    assert rel(fin.double().cpu().numpy(), fin_ref) <= bar


SLOT_CASES = [
    # (B, S, L, H, P, G, N, W, dtype, windows)
    (5, 8, 300, 4, 64, 2, 128, 4, torch.bfloat16, False),   # several runs: the tail kernel
    (4, 6, 3, 4, 64, 1, 128, 4, torch.bfloat16, True),      # decode-sized calls, windows
    (3, 5, 40, 2, 32, 1, 16, 3, torch.float32, True),
]


@pytest.mark.parametrize("case", SLOT_CASES, ids=lambda c: f"B{c[0]}S{c[1]}L{c[2]}W{c[7]}"
                         f"-{str(c[8])[6:]}-win{int(c[9])}")
def test_mixer_prologue_slots_match_oracle(ssd, case):
    """Conv-state slots: real rows match the oracle on their slots, padding rows
    leave every output untouched, other slots and their windows are unchanged."""
    B, S, L, H, P, G, N, W, dtype, windows = case
    inp = make_mixer(B, L, H, P, G, N, W, dtype, seed=S * 11 + L, state=False)
    Dc = H * P + 2 * G * N
    g = torch.Generator().manual_seed(S + L)
    pool = torch.randn((S, Dc, W), generator=g).to(dtype)
    idx = torch.randperm(S, generator=g)[:B].to(torch.int32)
    idx[0], idx[-1] = S + 1, -1                 # two padding rows
    out_ref, st_ref, win_ref = orc.causal_conv1d(inp["xBC"], inp["conv_weight"],
                                                 inp["conv_bias"], pool, state_indices=idx)
    x_ref, b_ref, c_ref = orc.split_xbc(out_ref, H, P, G, N)
    dt_ref = orc.dt_prologue(inp["dt"], inp["dt_bias"], True)
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    state = pool.cuda()
    win = torch.full((S, L, Dc, W), 5.0, dtype=dtype, device="cuda") if windows else None
    outs = (torch.full((B, L, H, P), 9.0, dtype=dtype, device="cuda"),
            torch.full((B, L, G, N), 9.0, dtype=dtype, device="cuda"),
            torch.full((B, L, G, N), 9.0, dtype=dtype, device="cuda"),
            torch.full((B, L, H), 9.0, dtype=torch.float32, device="cuda"))
    x, Bm, Cm, dt = ssd.mixer_prologue(d["xBC"], d["conv_weight"], d["dt"], H, P, G, N,
                                       conv_bias=d["conv_bias"], conv_state=state,
                                       conv_windows=win, conv_state_indices=idx.cuda(),
                                       dt_bias=d["dt_bias"], out=outs)
    torch.cuda.synchronize()
    real = [b for b in range(B) if 0 <= int(idx[b]) < S]
    used = [int(idx[b]) for b in real]
    bar = 2e-2 if dtype == torch.bfloat16 else 1e-4
    for got, ref in ((x, x_ref), (Bm, b_ref), (Cm, c_ref)):
        got = got.double().cpu().numpy()
        assert rel(got[real], ref[real]) <= bar
        assert np.all(got[[0, B - 1]] == 9.0)
    dtg = dt.double().cpu().numpy()
    assert rel(dtg[real], dt_ref[real]) <= 1e-5 and np.all(dtg[[0, B - 1]] == 9.0)
    cast = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dtype)
    assert torch.equal(state.cpu(), cast(st_ref))           # used slots replaced, others kept
    if windows:
        wg = win.cpu()
        assert torch.equal(wg[used], cast(win_ref[real]))
        unused = sorted(set(range(S)) - set(used))
        assert torch.all(wg[unused] == 5.0)


def test_prologue_benchmark_shape_sampled(ssd):
    """The prologue benchmark's call (Mamba-2 2.7B mixer shape: batch 8, 4096
    tokens, 5376 channels, width 4, conv state in place, bias, softplus) with
    its seeded inputs; every output of two sampled sequences checked against
    the oracle (the convolution is independent per sequence)."""
    from state_space_model_gb300 import inputs as gen
    w = gen.WORKLOADS["mamba2_2p7b"]
    Bn, L, H, P, G, N, W = w.batch, w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate, 4
    cpu = gen.make_prologue_inputs(Bn, L, H, P, G, N, W, seed=20280)
    d = {k: v.cuda() for k, v in cpu.items()}
    x, Bm, Cm, dt = ssd.mixer_prologue(d["xBC"], d["conv_weight"], d["dt"], H, P, G, N,
                                       conv_bias=d["conv_bias"], conv_state=d["conv_state"],
                                       dt_bias=d["dt_bias"], dt_softplus=True)
    torch.cuda.synchronize()
    rows = [2, 7]
    out_ref, st_ref, _ = orc.causal_conv1d(cpu["xBC"][rows], cpu["conv_weight"],
                                           cpu["conv_bias"], cpu["conv_state"][rows])
    x_ref, b_ref, c_ref = orc.split_xbc(out_ref, H, P, G, N)
    for got, ref in ((x, x_ref), (Bm, b_ref), (Cm, c_ref)):
        assert rel(got[rows].double().cpu().numpy(), ref) <= 2e-2
    dt_ref = orc.dt_prologue(cpu["dt"][rows], cpu["dt_bias"], True)
    assert rel(dt[rows].double().cpu().numpy(), dt_ref) <= 1e-5
    cast = torch.from_numpy(np.ascontiguousarray(st_ref)).to(torch.bfloat16)
    assert torch.equal(d["conv_state"][rows].cpu(), cast)
