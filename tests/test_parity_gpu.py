"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Error metric, per output tensor: max|gpu - ref| / max|ref| with ref the fp64
oracle on the same stored inputs.  Bar: 1e-4 for fp32 inputs, 2e-2 for bf16
inputs (fp32 accumulation), for y and final_states alike.  Stage tests feed
each step the oracle's own inputs for that step, rounded to the storage
precision the library uses, so errors do not compound.

The fp32 cumulative sum G gets its own bar: an in-chunk prefix sum of Q fp32
products carries at most about (Q + 2) * 2^-24 * max|G| of rounding, so
3e-5 relative covers Q <= 256.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from state_space_model_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}
G_TOL = 3e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from state_space_model_gb300 import build
    build.build()


def ssd():
    from state_space_model_gb300 import ssd as m
    return m


def rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.max(np.abs(b))
    return float(np.max(np.abs(a - b)) / den) if den > 0 else float(np.max(np.abs(a)))


def to_dev(inp):
    return {k: (None if v is None else v.cuda()) for k, v in inp.items()}


def device_ok():
    """No kernel gave up a bounded wait since the last check."""
    import ctypes
    from state_space_model_gb300 import _native
    lib = _native.load()
    st = lib.ssd_device_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.ssd_last_error_detail().decode()


def run(w, inp, **kw):
    d = to_dev(inp)
    y, f = ssd().chunked_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"],
                             d["initial_states"], w.chunk_size, w.ngroups, **kw)
    torch.cuda.synchronize()
    device_ok()
    return y.float().cpu().double().numpy(), (None if f is None else f.cpu().double().numpy())


def oracle_full(w, inp):
    return orc.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                          inp["initial_states"], ngroups=w.ngroups)


def oracle_chunked(w, inp):
    out = orc.chunked(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                      inp["initial_states"], ngroups=w.ngroups, chunk_size=w.chunk_size)
    B, H = w.batch, w.nheads
    nc = -(-w.seqlen // w.chunk_size)
    res = {}
    res["G"] = out["G"].reshape(B, H, -1)
    res["S"] = out["S"].reshape(B, H, nc, w.headdim, w.dstate).transpose(0, 2, 1, 3, 4)
    res["h_prev"] = out["h_prev"].reshape(B, H, nc, w.headdim, w.dstate).transpose(0, 2, 1, 3, 4)
    res["final"] = out["final"].reshape(B, H, w.headdim, w.dstate)
    res["y"] = out["y"].reshape(B, H, w.seqlen, w.headdim).transpose(0, 2, 1, 3)
    return res


def padded_G(w, G):
    """Oracle G [B,H,L] -> the library's [B,H,nc*Q] (padding repeats the
    chunk's last real value, as zero dt leaves the sum unchanged)."""
    B, H, L = G.shape
    Q = w.chunk_size
    nc = -(-L // Q)
    out = np.empty((B, H, nc * Q))
    out[:, :, :L] = G
    if nc * Q > L:
        out[:, :, L:] = G[:, :, L - 1:L]
    return out


STAGE_CASES = [
    gen.small_case("bf16", batch=2, seqlen=600, nheads=4, ngroups=2, chunk_size=128),
    gen.small_case("bf16", batch=1, seqlen=520, nheads=3, ngroups=1, chunk_size=256,
                   init_states=False),
    gen.small_case("f32", batch=2, seqlen=200, nheads=4, headdim=16, dstate=16, ngroups=4,
                   chunk_size=64),
    gen.small_case("f32", batch=1, seqlen=300, nheads=2, headdim=32, dstate=64, ngroups=1,
                   chunk_size=128),
]


@pytest.mark.parametrize("w", STAGE_CASES, ids=lambda w: f"{w.dtype}-L{w.seqlen}-Q{w.chunk_size}")
def test_stage_parity(w):
    inp = gen.make_inputs(w)
    ref = oracle_chunked(w, inp)
    d = to_dev(inp)
    m = ssd()
    tol = TOL[w.dtype]
    Q = w.chunk_size
    # step 1
    G = m.chunk_cumsum(d["dt"], d["A"], Q)
    Gref = padded_G(w, ref["G"])
    assert rel(G.cpu().numpy(), Gref) < G_TOL
    # step 2, from the oracle's G
    Gin = torch.from_numpy(Gref).float().cuda()
    S = m.chunk_state(d["x"], d["B"], d["dt"], Gin, Q, w.ngroups)
    assert rel(S.cpu().numpy(), ref["S"]) < tol
    # step 3, from the oracle's S
    Sin = torch.from_numpy(np.ascontiguousarray(ref["S"])).float().cuda()
    hp, fin = m.state_passing(Sin, Gin, d["initial_states"], Q, state_dtype=w.torch_dtype)
    assert rel(hp.float().cpu().numpy(), ref["h_prev"]) < tol
    assert rel(fin.cpu().numpy(), ref["final"]) < TOL["f32"]
    # step 4, from the oracle's entering states
    hpin = torch.from_numpy(np.ascontiguousarray(ref["h_prev"])).to(w.torch_dtype).cuda()
    y = m.chunk_scan(d["x"], d["dt"], Gin, d["B"], d["C"], d["D"], hpin, Q, w.ngroups)
    assert rel(y.float().cpu().numpy(), ref["y"]) < tol


E2E_CASES = [
    # (dtype, B, L, H, P, N, G, Q, h0)
    ("f32", 1, 256, 4, 16, 16, 1, 64, False),
    ("f32", 1, 130, 2, 128, 32, 2, 64, True),
    # fp32 on the tensor cores (P = 64, N = 128, Q of 128 or 256: bf16 hi / lo
    # pairs, three products each), two or one head per chunk_state CTA
    ("f32", 2, 333, 6, 64, 128, 3, 128, True),
    ("f32", 1, 700, 4, 64, 128, 2, 256, True),
    ("f32", 2, 1000, 3, 64, 128, 1, 128, False),
    ("f32", 1, 129, 2, 64, 128, 2, 256, True),
    ("f32", 2, 1, 2, 64, 128, 1, 128, True),      # one token: a single partial block
    ("f32", 1, 255, 4, 64, 128, 4, 256, False),   # one token short of a chunk
    ("bf16", 2, 700, 4, 64, 128, 1, 256, True),
    ("bf16", 3, 389, 8, 64, 128, 2, 128, False),
    ("bf16", 1, 1000, 4, 64, 128, 4, 64, True),
    ("bf16", 2, 256, 4, 32, 64, 2, 128, True),
    ("bf16", 1, 300, 2, 128, 128, 1, 128, True),
    ("bf16", 1, 77, 2, 16, 32, 1, 256, True),
    # fused bf16 path with one head per group (ngroups = nheads: the single-head
    # kernel) and two heads per group (the pair kernel: a full wave of pair
    # slabs), ragged L
    ("bf16", 2, 1000, 6, 64, 128, 6, 256, True),
    ("bf16", 2, 777, 152, 64, 128, 76, 128, True),
]


@pytest.mark.parametrize("case", E2E_CASES, ids=lambda c: "-".join(map(str, c)))
def test_end_to_end_parity(case):
    dtype, B, L, H, P, N, G, Q, h0 = case
    w = gen.small_case(dtype, batch=B, seqlen=L, nheads=H, headdim=P, dstate=N, ngroups=G,
                       chunk_size=Q, init_states=h0, seed=1000 + E2E_CASES.index(case))
    inp = gen.make_inputs(w)
    y, f = run(w, inp)
    yr, fr = oracle_full(w, inp)
    assert rel(y, yr) < TOL[dtype]
    assert rel(f, fr) < TOL[dtype]


@pytest.mark.parametrize("name", ["tiny_f32", "mamba2_130m", "mamba2_2p7b", "hybrid_g8",
                                  "long_64k"])
def test_workload_parity(name):
    """The five workloads at full size through ssd_chunked_fwd (as the
    benchmark calls it), in the plan the benchmark times; y and final_states
    of every (b, h) slab checked against the fp64 recurrence.  The oracle runs
    in batches of slabs so its fp64 output stays within a few hundred MB."""
    w = gen.WORKLOADS[name]
    inp = gen.make_inputs(w)
    d = to_dev(inp)
    yd, fd = ssd().chunked_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"],
                               d["initial_states"], w.chunk_size, w.ngroups)
    torch.cuda.synchronize()
    device_ok()
    y, f = yd.cpu(), fd.cpu()
    del yd, fd, d
    assert torch.isfinite(y.float()).all() and torch.isfinite(f).all()
    slabs = [(b, h) for b in range(w.batch) for h in range(w.nheads)]
    per = max(1, (256 << 20) // (w.seqlen * w.headdim * 8))
    for i in range(0, len(slabs), per):
        part = slabs[i:i + per]
        yr, fr = orc.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                                inp["initial_states"], ngroups=w.ngroups, slabs=part)
        # the bar is per tensor; apply it per slab (stricter)
        for k, (b, h) in enumerate(part):
            assert rel(y[b, :, h, :].double().numpy(), yr[k]) < TOL[w.dtype], f"y slab {(b, h)}"
            assert rel(f[b, h].double().numpy(), fr[k]) < TOL[w.dtype], f"final slab {(b, h)}"


@pytest.mark.parametrize("Q", [128, 256])
def test_staged_path_composed_on_device(Q):
    """The four step entry points chained on the GPU (the path ssd_chunked_fwd
    takes where the fused kernel does not apply) against the recurrence."""
    w = gen.small_case("bf16", batch=2, seqlen=700, nheads=4, ngroups=2, chunk_size=Q)
    inp = gen.make_inputs(w)
    d = to_dev(inp)
    m = ssd()
    G = m.chunk_cumsum(d["dt"], d["A"], Q)
    S = m.chunk_state(d["x"], d["B"], d["dt"], G, Q, w.ngroups)
    hp, fin = m.state_passing(S, G, d["initial_states"], Q, state_dtype=torch.bfloat16)
    y = m.chunk_scan(d["x"], d["dt"], G, d["B"], d["C"], d["D"], hp, Q, w.ngroups)
    torch.cuda.synchronize()
    device_ok()
    yr, fr = oracle_full(w, inp)
    assert rel(y.float().cpu().numpy(), yr) < TOL["bf16"]
    assert rel(fin.cpu().numpy(), fr) < TOL["bf16"]


def test_plan_names_the_kernel():
    """Two heads per CTA where the heads per group are even, one otherwise."""
    m = ssd()
    assert "k_ssd_pair" in m.describe_plan(8, 4096, 80, 64, 128, 1, 256)
    assert "k_ssd_pair" in m.describe_plan(2, 777, 152, 64, 128, 76, 128)
    assert "k_ssd_fused" in m.describe_plan(2, 1000, 6, 64, 128, 6, 256)
    assert "k_ssd_fused" in m.describe_plan(2, 1000, 3, 64, 128, 1, 256)
    assert "k_ssd_fused" in m.describe_plan(1, 16384, 128, 64, 128, 8, 128)   # 64 pair slabs


def test_plan_choice():
    m = ssd()
    assert m.describe_plan(8, 4096, 80, 64, 128, 1, 256).startswith("fused")
    assert m.describe_plan(1, 256, 4, 16, 16, 1, 64, torch.float32).startswith("staged")


# ---------------------------------------------------------------------------
# edge cases


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_empty_sequence_returns_initial_state(dtype):
    w = gen.small_case(dtype, batch=2, seqlen=0, nheads=4, ngroups=2, chunk_size=128)
    inp = gen.make_inputs(w)
    y, f = run(w, inp)
    assert y.shape == (2, 0, 4, 64)
    np.testing.assert_array_equal(f, inp["initial_states"].double().numpy())
    inp["initial_states"] = None
    y, f = run(w, inp)
    np.testing.assert_array_equal(f, 0.0)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_empty_batch(dtype):
    w = gen.small_case(dtype, batch=0, seqlen=100, nheads=4, ngroups=2, chunk_size=128)
    inp = gen.make_inputs(w)
    y, f = run(w, inp)
    assert y.shape[0] == 0 and f.shape[0] == 0


@pytest.mark.parametrize("L", [1, 63, 64, 65, 255])
def test_short_and_ragged_sequences(L):
    w = gen.small_case("bf16", batch=1, seqlen=L, nheads=2, ngroups=1, chunk_size=64)
    inp = gen.make_inputs(w)
    y, f = run(w, inp)
    yr, fr = oracle_full(w, inp)
    assert rel(y, yr) < TOL["bf16"] and rel(f, fr) < TOL["bf16"]


@pytest.mark.parametrize("L", [1, 127, 128, 129])
def test_short_and_ragged_sequences_f32_tensor_cores(L):
    """fp32 at P = 64, N = 128, Q = 128 (the tensor-core steps with bf16 hi / lo
    copies) around one chunk."""
    w = gen.small_case("f32", batch=1, seqlen=L, nheads=2, ngroups=1, chunk_size=128)
    inp = gen.make_inputs(w)
    y, f = run(w, inp)
    yr, fr = oracle_full(w, inp)
    assert rel(y, yr) < TOL["f32"] and rel(f, fr) < TOL["f32"]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_dt_zero_keeps_initial_state(dtype):
    w = gen.small_case(dtype, batch=1, seqlen=300, nheads=2, ngroups=1, chunk_size=128)
    inp = gen.make_inputs(w)
    inp["dt"] = torch.zeros_like(inp["dt"])
    y, f = run(w, inp)
    np.testing.assert_array_equal(f, inp["initial_states"].double().numpy())
    yr, fr = oracle_full(w, inp)
    assert rel(y, yr) < TOL[dtype]


def test_decay_free_and_strong_decay():
    w = gen.small_case("bf16", batch=1, seqlen=400, nheads=4, ngroups=2, chunk_size=128)
    inp = gen.make_inputs(w)
    inp["A"] = torch.zeros_like(inp["A"])                  # no decay at all
    y, f = run(w, inp)
    yr, fr = oracle_full(w, inp)
    assert rel(y, yr) < TOL["bf16"] and rel(f, fr) < TOL["bf16"]
    inp = gen.make_inputs(w)
    inp["A"] = torch.full_like(inp["A"], -200.0)          # exp(A dt) underflows
    inp["dt"] = inp["dt"] + 1.0
    y, f = run(w, inp)
    yr, fr = oracle_full(w, inp)
    assert np.isfinite(y).all() and np.isfinite(f).all()
    assert rel(y, yr) < TOL["bf16"] and rel(f, fr) < TOL["bf16"]


def test_optional_arguments_absent():
    w = gen.small_case("bf16", batch=2, seqlen=300, nheads=4, ngroups=2, chunk_size=128,
                       init_states=False)
    inp = gen.make_inputs(w)
    inp["D"] = None
    y, f = run(w, inp, return_final_states=False)
    assert f is None
    yr, _ = oracle_full(w, inp)
    assert rel(y, yr) < TOL["bf16"]


def test_strided_inputs():
    """x, B, C, y as views into wider buffers (16-byte-multiple strides)."""
    w = gen.small_case("bf16", batch=2, seqlen=300, nheads=4, ngroups=2, chunk_size=128)
    inp = gen.make_inputs(w)
    d = to_dev(inp)
    wide = torch.zeros(2, 300, 4, 64 + 8, dtype=torch.bfloat16, device="cuda")
    wide[..., :64] = d["x"]
    xv = wide[..., :64]
    bw = torch.zeros(2, 300, 2, 128 + 8, dtype=torch.bfloat16, device="cuda")
    bw[..., :128] = d["B"]
    cw = torch.zeros(2, 300, 2, 128 + 8, dtype=torch.bfloat16, device="cuda")
    cw[..., :128] = d["C"]
    yw = torch.zeros(2, 300, 4, 64 + 8, dtype=torch.bfloat16, device="cuda")
    _, f = ssd().chunked_fwd(xv, d["dt"], d["A"], bw[..., :128], cw[..., :128], d["D"],
                             d["initial_states"], 128, 2, y=yw[..., :64])
    torch.cuda.synchronize()
    yr, fr = oracle_full(w, inp)
    assert rel(yw[..., :64].float().cpu().numpy(), yr) < TOL["bf16"]
    assert rel(f.cpu().numpy(), fr) < TOL["bf16"]
    assert (yw[..., 64:] == 0).all()


def test_deterministic():
    w = gen.small_case("bf16", batch=2, seqlen=700, nheads=4, ngroups=2, chunk_size=256)
    inp = gen.make_inputs(w)
    y1, f1 = run(w, inp)
    y2, f2 = run(w, inp)
    np.testing.assert_array_equal(y1, y2)
    np.testing.assert_array_equal(f1, f2)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_resume_at_chunk_boundary_is_exact(dtype):
    """Two calls with final_states fed back as initial_states equal one call,
    bit for bit, when the split falls on a chunk boundary."""
    Q = 128
    w = gen.small_case(dtype, batch=2, seqlen=640, nheads=4, ngroups=2, chunk_size=Q)
    inp = gen.make_inputs(w)
    y, f = run(w, inp)
    t = 3 * Q
    first = dict(inp, x=inp["x"][:, :t].contiguous(), dt=inp["dt"][:, :t].contiguous(),
                 B=inp["B"][:, :t].contiguous(), C=inp["C"][:, :t].contiguous())
    y1, f1 = run(w.with_(seqlen=t), first)
    second = dict(inp, x=inp["x"][:, t:].contiguous(), dt=inp["dt"][:, t:].contiguous(),
                  B=inp["B"][:, t:].contiguous(), C=inp["C"][:, t:].contiguous(),
                  initial_states=torch.from_numpy(f1).float())
    y2, f2 = run(w.with_(seqlen=640 - t), second)
    np.testing.assert_array_equal(np.concatenate([y1, y2], axis=1), y)
    np.testing.assert_array_equal(f2, f)


@pytest.mark.parametrize("B,H,L,G", [(1, 4, 8000, 2), (2, 3, 5000, 1), (1, 308, 4000, 2)])
def test_fused_split_matches_oracle(B, H, L, G):
    """Few slabs over a long sequence: each slab runs as sequence segments on
    separate SMs, started from the combined states of a states-only pass.
    Ragged L; initial states and D given."""
    w = gen.small_case("bf16", batch=B, seqlen=L, nheads=H, ngroups=G, chunk_size=256,
                       init_states=True, seed=4242 + L)
    plan = ssd().describe_plan(w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups,
                               w.chunk_size, w.torch_dtype)
    assert "segments" in plan, plan
    inp = gen.make_inputs(w)
    y, fin = run(w, inp)
    yr, fr = oracle_full(w, inp)
    assert rel(y, yr) <= TOL["bf16"]
    assert rel(fin, fr) <= TOL["bf16"]
    for b in range(B):
        for h in range(H):
            assert rel(y[b, :, h], yr[b, :, h]) <= TOL["bf16"]
            assert rel(fin[b, h], fr[b, h]) <= TOL["bf16"]


@pytest.mark.parametrize("B,H,L,G", [(2, 96, 640, 2), (3, 102, 300, 1)])
def test_fused_many_slabs_match_oracle(B, H, L, G):
    """More (batch, head) slabs than SMs (several waves of CTAs, heads and
    batches mixed within a wave).  Every slab checked; ragged L; initial states
    and D given."""
    w = gen.small_case("bf16", batch=B, seqlen=L, nheads=H, ngroups=G, chunk_size=256,
                       init_states=True, seed=977 + L)
    plan = ssd().describe_plan(w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups,
                               w.chunk_size, w.torch_dtype)
    assert plan.startswith("fused") and "segments" not in plan, plan
    inp = gen.make_inputs(w)
    y, fin = run(w, inp)
    yr, fr = oracle_full(w, inp)
    for b in range(B):
        for h in range(H):
            assert rel(y[b, :, h], yr[b, :, h]) <= TOL["bf16"], (b, h)
            assert rel(fin[b, h], fr[b, h]) <= TOL["bf16"], (b, h)


def test_f32_tensor_core_plan_and_per_slab_parity():
    """fp32 inputs at P = 64, N = 128 run chunk_state and chunk_scan on the
    tensor cores (bf16 hi / lo copies, three products per MMA); the plan names
    the kernels, and every (b, h) slab meets the fp32 bar against the fp64
    recurrence."""
    import os
    if os.environ.get("SSD_FORCE_SIMT") == "1":
        pytest.skip("SSD_FORCE_SIMT=1 selects the CUDA-core steps")
    w = gen.small_case("f32", batch=2, seqlen=900, nheads=4, headdim=64, dstate=128, ngroups=2,
                       chunk_size=256, init_states=True, seed=4711)
    plan = ssd().describe_plan(w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups,
                               w.chunk_size, w.torch_dtype)
    assert "k_chunk_state_tc_f32" in plan and "k_chunk_scan_tc_f32" in plan, plan
    inp = gen.make_inputs(w)
    y, f = run(w, inp)
    yr, fr = oracle_full(w, inp)
    for b in range(w.batch):
        for h in range(w.nheads):
            assert rel(y[b, :, h], yr[b, :, h]) < TOL["f32"], (b, h)
            assert rel(f[b, h], fr[b, h]) < TOL["f32"], (b, h)
