"""GPU parity of the decode step (ssd_state_update) against the fp64 oracle.

Bars: out within 2e-2 (bf16 inputs and output) or 1e-4 (fp32) of the oracle,
as max|gpu - ref| / max|ref|; the fp32 state within 1e-4 in both cases (it is
computed in fp32 from the stored inputs, so only fp32 rounding separates it
from the oracle).  Also: prefill with ssd_chunked_fwd followed by decode steps
continues the same recurrence, and repeated calls are bitwise identical.

A bf16 state is checked against the oracle's model of a bf16-kept state (the
update from the stored values in float64, rounded to nearest even when kept):
the kernel's fp32 update can land on the other side of a rounding boundary,
so a kept element equals the oracle's or is one bf16 step (2^-7 of its
magnitude at most, plus fp32 rounding where the update cancels) away, and
almost all are equal.
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


def make_step(B, H, P, N, G, dtype, seed, D=True, z=False, bias=False, softplus=False):
    g = torch.Generator().manual_seed(seed)
    r = lambda *s: torch.randn(s, generator=g)
    dt_raw = r(B, H) * 0.5 - 2.0
    inp = dict(
        state=0.5 * r(B, H, P, N),
        x=r(B, H, P).to(dtype),
        dt=dt_raw if softplus else torch.nn.functional.softplus(dt_raw),
        A=-torch.exp(torch.rand(H, generator=g) * math.log(16.0)),
        Bm=(r(B, G, N) / math.sqrt(N)).to(dtype),
        Cm=(r(B, G, N) / math.sqrt(N)).to(dtype),
        D=r(H) if D else None,
        z=r(B, H, P).to(dtype) if z else None,
        dt_bias=0.3 * r(H) if bias else None,
        dt_softplus=softplus,
        ngroups=G,
    )
    return inp


CASES = [
    # (B, H, P, N, G, dtype, D, z, bias, softplus)
    (3, 8, 64, 128, 2, torch.bfloat16, True, True, True, True),
    (2, 4, 16, 16, 1, torch.float32, False, False, False, False),
    (1, 128, 64, 128, 8, torch.bfloat16, True, True, False, False),
    (5, 3, 32, 64, 3, torch.float32, True, False, True, False),
    (4, 6, 128, 32, 2, torch.bfloat16, False, True, True, True),
    (40, 16, 32, 128, 2, torch.float32, True, True, True, True),     # many 16 KB heads
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}H{c[1]}P{c[2]}N{c[3]}G{c[4]}"
                         f"-{str(c[5])[6:]}-D{int(c[6])}z{int(c[7])}b{int(c[8])}sp{int(c[9])}")
def test_state_update_matches_oracle(ssd, case):
    B, H, P, N, G, dtype, D, z, bias, sp = case
    inp = make_step(B, H, P, N, G, dtype, seed=B * 1000 + H, D=D, z=z, bias=bias, softplus=sp)
    out_ref, st_ref = orc.ssu_step(**inp)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    state = dev.pop("state").clone()
    out = ssd.state_update(state, dev["x"], dev["dt"], dev["A"], dev["Bm"], dev["Cm"],
                           D=dev["D"], z=dev["z"], dt_bias=dev["dt_bias"],
                           dt_softplus=dev["dt_softplus"], ngroups=G)
    torch.cuda.synchronize()
    assert out.dtype == dtype and out.shape == (B, H, P)
    bar = 2e-2 if dtype == torch.bfloat16 else 1e-4
    assert rel(out.double().cpu().numpy(), out_ref) <= bar
    assert rel(state.double().cpu().numpy(), st_ref) <= 1e-4


def test_prefill_then_decode_continues_the_recurrence(ssd):
    from state_space_model_gb300 import inputs as gen
    L, T = 384, 5
    w = gen.small_case("bf16", batch=2, seqlen=L + T, nheads=4, ngroups=2, chunk_size=128,
                       init_states=True)
    inp = gen.make_inputs(w)
    y_ref, fin_ref = orc.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                                    inp["initial_states"], ngroups=2)
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    # prefill over the first L tokens
    y, state = ssd.chunked_fwd(d["x"][:, :L], d["dt"][:, :L], d["A"], d["B"][:, :L],
                               d["C"][:, :L], d["D"], d["initial_states"], 128, 2)
    outs = []
    for t in range(L, L + T):
        outs.append(ssd.state_update(state, d["x"][:, t], d["dt"][:, t], d["A"], d["B"][:, t],
                                     d["C"][:, t], D=d["D"], ngroups=2))
    torch.cuda.synchronize()
    dec = torch.stack(outs, dim=1).double().cpu().numpy()
    assert rel(y.double().cpu().numpy(), y_ref[:, :L]) <= 2e-2
    assert rel(dec, y_ref[:, L:]) <= 2e-2
    assert rel(state.double().cpu().numpy(), fin_ref) <= 2e-2


def test_state_update_is_deterministic(ssd):
    inp = make_step(4, 16, 64, 128, 4, torch.bfloat16, seed=11, z=True, bias=True, softplus=True)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    runs = []
    for _ in range(2):
        st = dev["state"].clone()
        o = ssd.state_update(st, dev["x"], dev["dt"], dev["A"], dev["Bm"], dev["Cm"],
                             D=dev["D"], z=dev["z"], dt_bias=dev["dt_bias"], dt_softplus=True,
                             ngroups=4)
        runs.append((o.clone(), st))
    torch.cuda.synchronize()
    assert torch.equal(runs[0][0], runs[1][0]) and torch.equal(runs[0][1], runs[1][1])


# ---- several tokens per call -------------------------------------------------

def make_tokens(B, T, H, P, N, G, dtype, seed, z=True, bias=True, softplus=True):
    g = torch.Generator().manual_seed(seed)
    r = lambda *s: torch.randn(s, generator=g)
    dt_raw = r(B, T, H) * 0.5 - 2.0
    return dict(
        state=0.5 * r(B, H, P, N),
        x=r(B, T, H, P).to(dtype),
        dt=dt_raw if softplus else torch.nn.functional.softplus(dt_raw),
        A=-torch.exp(torch.rand(H, generator=g) * math.log(16.0)),
        Bm=(r(B, T, G, N) / math.sqrt(N)).to(dtype),
        Cm=(r(B, T, G, N) / math.sqrt(N)).to(dtype),
        D=r(H),
        z=r(B, T, H, P).to(dtype) if z else None,
        dt_bias=0.3 * r(H) if bias else None,
        dt_softplus=softplus,
        ngroups=G,
    )


def random_tree(B, T, seed):
    """parent[b, t] in [-1, t): a random draft tree per sequence (-1 = previous token)."""
    g = torch.Generator().manual_seed(seed)
    par = torch.full((B, T), -1, dtype=torch.int32)
    for t in range(1, T):
        par[:, t] = torch.randint(-1, t, (B,), generator=g, dtype=torch.int32)
    return par


TOKEN_CASES = [
    # (B, T, H, P, N, G, dtype, cache, tree, update)
    (4, 4, 16, 64, 128, 2, torch.bfloat16, True, True, True),
    (3, 6, 8, 64, 128, 8, torch.bfloat16, True, False, False),
    (2, 3, 6, 32, 64, 3, torch.float32, False, False, True),
    (64, 2, 32, 64, 128, 8, torch.bfloat16, False, False, True),    # a full grid: whole heads
    (1, 5, 4, 128, 128, 1, torch.float32, True, True, True),        # few heads: rows split
    (2, 3, 4, 16, 16, 2, torch.bfloat16, True, True, False),        # P below a pass of rows
    (5, 1, 3, 128, 32, 1, torch.float32, True, False, True),
    (48, 3, 16, 64, 64, 4, torch.bfloat16, True, True, True),       # many 16 KB heads
]


@pytest.mark.parametrize("case", TOKEN_CASES, ids=lambda c: f"B{c[0]}T{c[1]}H{c[2]}P{c[3]}N{c[4]}"
                         f"G{c[5]}-{str(c[6])[6:]}-cache{int(c[7])}tree{int(c[8])}up{int(c[9])}")
def test_state_update_tokens_matches_oracle(ssd, case):
    B, T, H, P, N, G, dtype, cache, tree, update = case
    inp = make_tokens(B, T, H, P, N, G, dtype, seed=B * 100 + T * 10 + N)
    parent = random_tree(B, T, seed=T) if tree else None
    out_ref, fin_ref, cache_ref = orc.ssu_tokens(**inp, parent=parent, update_state=update)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    state = dev.pop("state").clone()
    inter = torch.empty((B, T, H, P, N), dtype=torch.float32, device="cuda") if cache else None
    out = ssd.state_update_tokens(state, dev["x"], dev["dt"], dev["A"], dev["Bm"], dev["Cm"],
                                  D=dev["D"], z=dev["z"], dt_bias=dev["dt_bias"],
                                  dt_softplus=dev["dt_softplus"], ngroups=G,
                                  intermediate_states=inter,
                                  parent=None if parent is None else parent.cuda(),
                                  update_state=update)
    torch.cuda.synchronize()
    assert out.dtype == dtype and out.shape == (B, T, H, P)
    bar = 2e-2 if dtype == torch.bfloat16 else 1e-4
    assert rel(out.double().cpu().numpy(), out_ref) <= bar
    if update:
        assert rel(state.double().cpu().numpy(), fin_ref) <= 1e-4
    else:   # untouched, bit for bit
        assert torch.equal(state.cpu(), inp["state"])
    if cache:
        assert rel(inter.double().cpu().numpy(), cache_ref) <= 1e-4


def test_one_token_call_equals_the_single_step(ssd):
    inp = make_step(6, 24, 64, 128, 4, torch.bfloat16, seed=21, z=True, bias=True, softplus=True)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    st1, st2 = dev["state"].clone(), dev["state"].clone()
    o1 = ssd.state_update(st1, dev["x"], dev["dt"], dev["A"], dev["Bm"], dev["Cm"], D=dev["D"],
                          z=dev["z"], dt_bias=dev["dt_bias"], dt_softplus=True, ngroups=4)
    u = lambda t: None if t is None else t.unsqueeze(1)
    o2 = ssd.state_update_tokens(st2, u(dev["x"]), u(dev["dt"]), dev["A"], u(dev["Bm"]),
                                 u(dev["Cm"]), D=dev["D"], z=u(dev["z"]), dt_bias=dev["dt_bias"],
                                 dt_softplus=True, ngroups=4)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2[:, 0]) and torch.equal(st1, st2)


def test_state_update_tokens_zero_tokens_is_a_no_op(ssd):
    inp = make_tokens(2, 0, 4, 64, 128, 2, torch.bfloat16, seed=1)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    state = dev["state"].clone()
    out = ssd.state_update_tokens(state, dev["x"], dev["dt"], dev["A"], dev["Bm"], dev["Cm"],
                                  D=dev["D"], z=dev["z"], dt_bias=dev["dt_bias"],
                                  dt_softplus=True, ngroups=2)
    torch.cuda.synchronize()
    assert out.shape == (2, 0, 4, 64) and torch.equal(state, dev["state"])


# ---- a state kept in bf16 ----------------------------------------------------

def bf16_step_check(got, ref, min_equal):
    """got within one bf16 step of ref everywhere, and equal on at least
    min_equal of the elements.  Where the update cancels (decayed state and
    input term nearly opposite) the kept value is small and its bf16 step
    smaller than the fp32 rounding of the two terms: 1e-5 max|ref| of slack
    covers that (the terms are at most a few times max|ref|, fp32 keeps 2^-24
    of them)."""
    d = np.abs(got - ref)
    assert np.all(d <= np.abs(ref) * 2.0 ** -7 + 1e-5 * np.max(np.abs(ref)))
    assert np.mean(d == 0) >= min_equal


BF16_STATE_CASES = [
    # (B, H, P, N, G, dtype, z, bias, softplus)
    (3, 8, 64, 128, 2, torch.bfloat16, True, True, True),
    (2, 4, 16, 16, 1, torch.float32, False, False, False),
    (64, 32, 64, 128, 8, torch.bfloat16, True, False, False),   # a full grid
    (1, 6, 128, 32, 2, torch.float32, True, True, True),       # few heads: rows split
]


@pytest.mark.parametrize("case", BF16_STATE_CASES, ids=lambda c: f"B{c[0]}H{c[1]}P{c[2]}N{c[3]}"
                         f"G{c[4]}-{str(c[5])[6:]}")
def test_bf16_state_update_matches_oracle(ssd, case):
    B, H, P, N, G, dtype, z, bias, sp = case
    inp = make_step(B, H, P, N, G, dtype, seed=B * 31 + N, z=z, bias=bias, softplus=sp)
    inp["state"] = inp["state"].to(torch.bfloat16)
    u = lambda t: None if t is None else t.unsqueeze(1)
    out_ref, fin_ref, _ = orc.ssu_tokens(**{**inp, "x": u(inp["x"]), "dt": u(inp["dt"]),
                                            "Bm": u(inp["Bm"]), "Cm": u(inp["Cm"]),
                                            "z": u(inp["z"])}, state_dtype="bf16")
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    state = dev.pop("state").clone()
    out = ssd.state_update(state, dev["x"], dev["dt"], dev["A"], dev["Bm"], dev["Cm"],
                           D=dev["D"], z=dev["z"], dt_bias=dev["dt_bias"],
                           dt_softplus=dev["dt_softplus"], ngroups=G)
    torch.cuda.synchronize()
    assert state.dtype == torch.bfloat16
    # out comes from the unrounded fp32 update: the fp32 bar when out is fp32
    bar = 2e-2 if dtype == torch.bfloat16 else 1e-4
    assert rel(out.double().cpu().numpy(), out_ref[:, 0]) <= bar
    bf16_step_check(state.double().cpu().numpy(), fin_ref, 0.99)


BF16_TOKEN_CASES = [
    # (B, T, H, P, N, G, dtype, cache, tree, update)
    (4, 4, 16, 64, 128, 2, torch.bfloat16, True, True, True),
    (3, 6, 8, 64, 128, 8, torch.float32, True, False, True),
    (2, 3, 4, 16, 16, 2, torch.bfloat16, True, True, False),
    (32, 2, 32, 64, 128, 8, torch.bfloat16, False, False, True),    # a full grid
    (40, 3, 16, 64, 128, 2, torch.bfloat16, True, True, True),      # a full grid, cache, tree
    (40, 2, 16, 32, 64, 2, torch.float32, True, True, False),       # small heads
]


@pytest.mark.parametrize("case", BF16_TOKEN_CASES, ids=lambda c: f"B{c[0]}T{c[1]}H{c[2]}P{c[3]}"
                         f"N{c[4]}G{c[5]}-{str(c[6])[6:]}-cache{int(c[7])}tree{int(c[8])}"
                         f"up{int(c[9])}")
def test_bf16_state_tokens_match_oracle(ssd, case):
    B, T, H, P, N, G, dtype, cache, tree, update = case
    inp = make_tokens(B, T, H, P, N, G, dtype, seed=B * 7 + T)
    inp["state"] = inp["state"].to(torch.bfloat16)
    parent = random_tree(B, T, seed=T + 1) if tree else None
    out_ref, fin_ref, cache_ref = orc.ssu_tokens(**inp, parent=parent, update_state=update,
                                                 state_dtype="bf16")
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    state = dev.pop("state").clone()
    inter = torch.empty((B, T, H, P, N), dtype=torch.bfloat16, device="cuda") if cache else None
    out = ssd.state_update_tokens(state, dev["x"], dev["dt"], dev["A"], dev["Bm"], dev["Cm"],
                                  D=dev["D"], z=dev["z"], dt_bias=dev["dt_bias"],
                                  dt_softplus=dev["dt_softplus"], ngroups=G,
                                  intermediate_states=inter,
                                  parent=None if parent is None else parent.cuda(),
                                  update_state=update)
    torch.cuda.synchronize()
    # a rounding that went the other way at one token moves the later ones by
    # about one bf16 step of that element: bars in units of max|ref|
    bar = 2e-2 if dtype == torch.bfloat16 else 2e-3
    assert rel(out.double().cpu().numpy(), out_ref) <= bar
    if update:
        assert rel(state.double().cpu().numpy(), fin_ref) <= 1e-2
        assert np.mean(state.double().cpu().numpy() == fin_ref) >= 0.95
    else:
        assert torch.equal(state.cpu(), inp["state"])
    if cache:
        got = inter.double().cpu().numpy()
        bf16_step_check(got[:, 0], cache_ref[:, 0], 0.99)   # the first token: one rounding
        assert rel(got, cache_ref) <= 1e-2
        assert np.mean(got == cache_ref) >= 0.95


@pytest.mark.parametrize("B", [8, 64])
def test_bf16_state_is_the_f32_update_rounded(ssd, B):
    """One token: the bf16 state's update equals the f32 state's update (same
    inputs, the state's values bf16) rounded to nearest even, bit for bit, and
    the outputs are identical."""
    inp = make_step(B, 16, 64, 128, 4, torch.bfloat16, seed=5, z=True, bias=True, softplus=True)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    sb = dev["state"].to(torch.bfloat16)
    sf = sb.float()
    kw = dict(D=dev["D"], z=dev["z"], dt_bias=dev["dt_bias"], dt_softplus=True, ngroups=4)
    ob = ssd.state_update(sb, dev["x"], dev["dt"], dev["A"], dev["Bm"], dev["Cm"], **kw)
    of = ssd.state_update(sf, dev["x"], dev["dt"], dev["A"], dev["Bm"], dev["Cm"], **kw)
    torch.cuda.synchronize()
    assert torch.equal(ob, of)
    assert torch.equal(sb, sf.to(torch.bfloat16))


# ---- slot indirection: a state pool and padding rows --------------------------

SLOT_CASES = [
    # (B, S, T, H, P, N, G, dtype, state dtype, cache, tree)
    (6, 9, 3, 8, 64, 128, 2, torch.bfloat16, torch.float32, True, True),
    (5, 7, 1, 4, 32, 64, 1, torch.float32, torch.bfloat16, True, False),
    (64, 80, 2, 32, 64, 128, 8, torch.bfloat16, torch.float32, False, False),   # a full grid
]


@pytest.mark.parametrize("case", SLOT_CASES, ids=lambda c: f"B{c[0]}S{c[1]}T{c[2]}H{c[3]}P{c[4]}"
                         f"N{c[5]}-{str(c[7])[6:]}-state{str(c[8])[6:]}-cache{int(c[9])}"
                         f"tree{int(c[10])}")
def test_state_slots_match_oracle(ssd, case):
    B, S, T, H, P, N, G, dtype, sdt, cache, tree = case
    inp = make_tokens(B, T, H, P, N, G, dtype, seed=B + S + T)
    g = torch.Generator().manual_seed(S)
    pool = (0.5 * torch.randn((S, H, P, N), generator=g)).to(sdt)
    idx = torch.randperm(S, generator=g)[:B].to(torch.int32)
    idx[1], idx[-1] = -1, S + 3                 # two padding rows: a pad id and one past the pool
    parent = random_tree(B, T, seed=T + 2) if tree else None
    bf = sdt == torch.bfloat16
    out_ref, fin_ref, cache_ref = orc.ssu_tokens(**{**inp, "state": pool}, parent=parent,
                                                 state_dtype="bf16" if bf else None,
                                                 state_indices=idx)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    state = pool.cuda()
    inter = torch.full((S, T, H, P, N), 3.0, dtype=sdt, device="cuda") if cache else None
    out = torch.full((B, T, H, P), 7.0, dtype=dtype, device="cuda")
    ssd.state_update_tokens(state, dev["x"], dev["dt"], dev["A"], dev["Bm"], dev["Cm"],
                            D=dev["D"], z=dev["z"], dt_bias=dev["dt_bias"],
                            dt_softplus=dev["dt_softplus"], ngroups=G, intermediate_states=inter,
                            parent=None if parent is None else parent.cuda(),
                            state_indices=idx.cuda(), out=out)
    torch.cuda.synchronize()
    real = [b for b in range(B) if 0 <= int(idx[b]) < S]
    used = [int(idx[b]) for b in real]
    o = out.double().cpu().numpy()
    bar = 2e-2 if dtype == torch.bfloat16 else (2e-3 if bf else 1e-4)
    assert rel(o[real], out_ref[real]) <= bar
    assert np.all(o[[1, B - 1]] == 7.0)         # padding rows: out not written
    st = state.double().cpu().numpy()
    if bf and T == 1:
        bf16_step_check(st[used], fin_ref[used], 0.99)
    elif bf:
        assert rel(st[used], fin_ref[used]) <= 1e-2
    else:
        assert rel(st[used], fin_ref[used]) <= 1e-4
    unused = sorted(set(range(S)) - set(used))
    assert torch.equal(state[unused].cpu(), pool[unused])      # other slots untouched
    if cache:
        ic = inter.double().cpu().numpy()
        assert rel(ic[used], cache_ref[real]) <= (1e-2 if bf else 1e-4)
        assert np.all(ic[unused] == 3.0)


# ---- the benchmark's shape and launch, sampled --------------------------------

@pytest.mark.parametrize("T,sdt", [(1, torch.float32), (1, torch.bfloat16), (4, torch.float32),
                                   (4, torch.bfloat16)], ids=["T1-f32", "T1-bf16", "T4-f32",
                                                              "T4-bf16"])
def test_decode_benchmark_shape_sampled(ssd, T, sdt):
    """The decode benchmark's inputs (batch 64, 128 heads, P 64, N 128, 8 groups,
    gated, dt bias + softplus; four tokens keep the cache) through the same
    calls; outputs, states and cache checked on sampled sequences against the
    oracle."""
    from state_space_model_gb300 import inputs as gen
    sh = gen.SSU_SHAPE
    Bn, H, P, N, G = sh["batch"], sh["nheads"], sh["headdim"], sh["dstate"], sh["ngroups"]
    cpu = gen.make_ssu_inputs(Bn, H, P, N, G, seed=20270, tokens=T if T > 1 else None)
    cpu["state"] = cpu["state"].to(sdt)
    d = {k: (None if v is None else v.cuda()) for k, v in cpu.items()}
    state = d["state"].clone()
    kw = dict(D=d["D"], z=d["z"], dt_bias=d["dt_bias"], dt_softplus=True, ngroups=G)
    if T > 1:
        inter = torch.empty((Bn, T, H, P, N), dtype=sdt, device="cuda")
        out = ssd.state_update_tokens(state, d["x"], d["dt"], d["A"], d["B"], d["C"],
                                      intermediate_states=inter, **kw)
    else:
        inter = None
        out = ssd.state_update(state, d["x"], d["dt"], d["A"], d["B"], d["C"], **kw)
    torch.cuda.synchronize()
    rows = [0, 29, 63]
    sel = lambda t: None if t is None else t[rows]
    tk = (lambda t: t) if T > 1 else (lambda t: None if t is None else t.unsqueeze(1))
    bf = sdt == torch.bfloat16
    out_ref, fin_ref, cache_ref = orc.ssu_tokens(
        sel(cpu["state"]), tk(sel(cpu["x"])), tk(sel(cpu["dt"])), cpu["A"], tk(sel(cpu["B"])),
        tk(sel(cpu["C"])), D=cpu["D"], z=tk(sel(cpu["z"])), dt_bias=cpu["dt_bias"],
        dt_softplus=True, ngroups=G, state_dtype="bf16" if bf else None)
    got = out[rows].double().cpu().numpy()
    assert rel(got if T > 1 else got[:, None], out_ref) <= 2e-2
    st = state[rows].double().cpu().numpy()
    if bf and T == 1:
        bf16_step_check(st, fin_ref, 0.99)
    else:
        assert rel(st, fin_ref) <= (1e-2 if bf else 1e-4)
    if inter is not None:
        assert rel(inter[rows].double().cpu().numpy(), cache_ref) <= (1e-2 if bf else 1e-4)
