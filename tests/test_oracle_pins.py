"""Pins of the fp64 oracle to facts outside itself (CPU only).

Each check ties one part of the oracle to something the pages or the
mathematics fix: hand-derived worked examples (tests/golden/), the decay-free
closed form (causal linear attention), the geometric-series closed form
for inputs held constant, scipy's first-order filter when the decay is
constant, the dt = 0 invariant, the scalar
first-order recurrence, chunk-size invariance of the chunked form, the state
hand-off (resumability) and linearity.  ``test_pins_reject_planted_mistakes``
shows that a plausible mistake (an index, a sign, a dropped term, a transposed
operand, a wrong head-to-group map) fails at least one of them.
"""
import glob
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
f64 = torch.float64


def _num(v):
    if isinstance(v, str):
        return float(eval(v, {"__builtins__": {}},
                          {"sqrt2": math.sqrt(2.0), "ln2": math.log(2.0)}))
    return float(v)


def _arr(v):
    if isinstance(v, list):
        return [_arr(e) for e in v]
    return _num(v)


def load_golden(path):
    with open(path) as f:
        g = json.load(f)
    s = g["shape"]
    Bn, L, H, P, N, G = s["B"], s["L"], s["H"], s["P"], s["N"], s["G"]
    t = lambda v, shape: torch.tensor(_arr(v), dtype=f64).reshape(shape)
    inp = dict(
        x=t(g["x"], (Bn, L, H, P)), dt=t(g["dt"], (Bn, L, H)), A=t(g["A"], (H,)),
        Bm=t(g["B"], (Bn, L, G, N)), Cm=t(g["C"], (Bn, L, G, N)),
        D=t(g["D"], (H,)),
        h0=None if g["h0"] is None else t(g["h0"], (Bn, H, P, N)),
        ngroups=G,
    )
    y = np.array(_arr(g["y"]), dtype=np.float64).reshape(Bn, L, H, P)
    fin = np.array(_arr(g["final"]), dtype=np.float64).reshape(Bn, H, P, N)
    return g, inp, y, fin


GOLDENS = sorted(glob.glob(os.path.join(GOLDEN, "*.json")))


def rand_inputs(B=2, L=24, H=4, P=3, N=5, G=2, dtype=f64, seed=0, h0=True,
                D=True, A_zero=False, dt_zero=False):
    g = torch.Generator().manual_seed(seed)
    r = lambda *s: torch.randn(s, generator=g, dtype=torch.float64)
    dt = torch.nn.functional.softplus(r(B, L, H) - 1.0)
    if dt_zero:
        dt = torch.zeros_like(dt)
    A = -torch.exp(torch.rand(H, generator=g, dtype=torch.float64) * math.log(4.0))
    if A_zero:
        A = torch.zeros_like(A)
    return dict(
        x=r(B, L, H, P).to(dtype), dt=dt.to(torch.float32 if dtype != f64 else f64),
        A=A.to(torch.float32 if dtype != f64 else f64),
        Bm=r(B, L, G, N).to(dtype), Cm=r(B, L, G, N).to(dtype),
        D=r(H).to(torch.float32 if dtype != f64 else f64) if D else None,
        h0=(0.3 * r(B, H, P, N)).to(torch.float32 if dtype != f64 else f64) if h0 else None,
        ngroups=G,
    )


def rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# ----------------------------------------------------------------------------
# worked examples derived by hand


@pytest.mark.parametrize("path", GOLDENS, ids=[os.path.basename(p) for p in GOLDENS])
def test_golden_recurrence(path):
    _, inp, y, fin = load_golden(path)
    yo, fo = orc.recurrence(**inp)
    np.testing.assert_allclose(yo, y, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(fo, fin, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("path", GOLDENS, ids=[os.path.basename(p) for p in GOLDENS])
@pytest.mark.parametrize("Q", [1, 2, 3])
def test_golden_chunked(path, Q):
    _, inp, y, fin = load_golden(path)
    out = orc.chunked(**inp, chunk_size=Q)
    Bn, L, H, P = y.shape
    yo = out["y"].reshape(Bn, H, L, P).transpose(0, 2, 1, 3)
    np.testing.assert_allclose(yo, y, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out["final"].reshape(fin.shape), fin, rtol=1e-12,
                               atol=1e-12)


@pytest.mark.parametrize("path", GOLDENS, ids=[os.path.basename(p) for p in GOLDENS])
def test_golden_quadratic(path):
    _, inp, y, fin = load_golden(path)
    yq, fq = orc.quadratic(**inp)
    Bn, L, H, P = y.shape
    np.testing.assert_allclose(yq.reshape(Bn, H, L, P).transpose(0, 2, 1, 3), y,
                               rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(fq.reshape(fin.shape), fin, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------
# two forms of the page against each other


@pytest.mark.parametrize("dtype", [f64, torch.float32, torch.bfloat16])
@pytest.mark.parametrize("G", [1, 2, 4])
def test_recurrence_equals_quadratic(dtype, G):
    inp = rand_inputs(B=2, L=20, H=4, P=3, N=5, G=G, dtype=dtype, seed=G)
    y, f = orc.recurrence(**inp)
    yq, fq = orc.quadratic(**inp)
    B, L, H, P = y.shape
    assert rel(yq.reshape(B, H, L, P).transpose(0, 2, 1, 3), y) < 1e-12
    assert rel(fq.reshape(f.shape), f) < 1e-12


def test_decay_free_closed_form():
    """A = 0: causal linear attention with queries C, keys B, values dt*x,
    inclusive of the diagonal, plus the initial-state and skip terms."""
    inp = rand_inputs(B=2, L=17, H=4, P=3, N=6, G=2, A_zero=True, seed=7)
    y, f = orc.recurrence(**inp)
    x, dt, Bm, Cm, D, h0 = (inp[k].numpy() for k in ("x", "dt", "Bm", "Cm", "D", "h0"))
    Bn, L, H, P = x.shape
    hpg = H // inp["ngroups"]
    for b in range(Bn):
        for h in range(H):
            g = h // hpg
            Cg, Bg = Cm[b, :, g, :], Bm[b, :, g, :]
            att = np.tril(Cg @ Bg.T)                      # M: inclusive causal mask
            Y = Cg @ h0[b, h].T + att @ (dt[b, :, h][:, None] * x[b, :, h, :]) \
                + D[h] * x[b, :, h, :]
            assert rel(y[b, :, h, :], Y) < 1e-12
            F = h0[b, h] + (dt[b, :, h][:, None] * x[b, :, h, :]).T @ Bg
            assert rel(f[b, h], F) < 1e-12


@pytest.mark.parametrize("form", ["recurrence", "chunked"])
def test_constant_inputs_geometric_series(form):
    """Inputs held constant over the sequence (x per (b, h); B, C per
    (b, g); dt per head): the recurrence is a geometric series, so after
    token t (counting from 0), with alpha = exp(A dt),
        S_t = alpha^(t+1) H0 + dt x b^T (1 - alpha^(t+1)) / (1 - alpha),
        y_t = S_t c + D x.
    Long sequences with decays from 0.37 to 0.9995 per token exercise the
    decay far beyond the hand-derived examples, on both oracle forms (the
    chunked one with a partial last chunk)."""
    Bn, L, H, P, N, G = 2, 300, 4, 3, 5, 2
    g = torch.Generator().manual_seed(31)
    r = lambda *s: torch.randn(s, generator=g, dtype=f64)
    xc, bc, cc, h0, D = r(Bn, H, P), r(Bn, G, N), r(Bn, G, N), r(Bn, H, P, N), r(H)
    dtc = torch.tensor([0.05, 0.5, 0.01, 0.25], dtype=f64)
    A = torch.tensor([-0.01, -2.0, -0.05, -1.0], dtype=f64)
    inp = dict(x=xc[:, None].expand(Bn, L, H, P).contiguous(),
               dt=dtc.expand(Bn, L, H).contiguous(), A=A,
               Bm=bc[:, None].expand(Bn, L, G, N).contiguous(),
               Cm=cc[:, None].expand(Bn, L, G, N).contiguous(), D=D, h0=h0, ngroups=G)
    if form == "recurrence":
        y, f = orc.recurrence(**inp)
    else:
        out = orc.chunked(**inp, chunk_size=64)
        y = out["y"].reshape(Bn, H, L, P).transpose(0, 2, 1, 3)
        f = out["final"].reshape(Bn, H, P, N)
    t1 = np.arange(1, L + 1, dtype=np.float64)
    for b in range(Bn):
        for h in range(H):
            gi = h // (H // G)
            alpha = math.exp(float(A[h] * dtc[h]))
            pw = alpha ** t1                                              # alpha^(t+1)
            geo = (1.0 - pw) / (1.0 - alpha)
            inj = float(dtc[h]) * np.outer(xc[b, h].numpy(), bc[b, gi].numpy())
            S = pw[:, None, None] * h0[b, h].numpy() + geo[:, None, None] * inj
            Y = S @ cc[b, gi].numpy() + float(D[h]) * xc[b, h].numpy()
            assert rel(y[b, :, h, :], Y) < 1e-11
            assert rel(f[b, h], S[-1]) < 1e-11


def test_constant_decay_equals_scipy_lfilter():
    """dt held constant per head (x, B and C still vary per token): every state
    element follows the first-order filter s_t = alpha s_(t-1) + dt x_t[p] B_t[n]
    with alpha = exp(A dt) and s_(-1) = H0[p, n], which scipy.signal.lfilter
    computes ([1], [1, -alpha], with the initial condition alpha H0); then
    y_t[p] = sum_n C_t[n] s_t[p, n] + D x_t[p].  Checks the outer-product
    orientation, the head-to-group map and the contraction over n against a
    library routine."""
    signal = pytest.importorskip("scipy.signal")
    Bn, L, H, P, N, G = 2, 200, 4, 3, 5, 2
    inp = rand_inputs(B=Bn, L=L, H=H, P=P, N=N, G=G, seed=41)
    dtc = torch.tensor([0.02, 0.3, 0.7, 0.1], dtype=f64)
    inp["dt"] = dtc.expand(Bn, L, H).contiguous()
    y, f = orc.recurrence(**inp)
    x, Bm, Cm, D, h0, A = (inp[k].numpy() for k in ("x", "Bm", "Cm", "D", "h0", "A"))
    for b in range(Bn):
        for h in range(H):
            g = h // (H // G)
            alpha = math.exp(A[h] * float(dtc[h]))
            u = float(dtc[h]) * x[b, :, h, :, None] * Bm[b, :, g, None, :]   # [L, P, N]
            S, _ = signal.lfilter([1.0], [1.0, -alpha], u, axis=0,
                                  zi=(alpha * h0[b, h])[None])
            Y = np.einsum("tpn,tn->tp", S, Cm[b, :, g, :]) + D[h] * x[b, :, h, :]
            assert rel(y[b, :, h, :], Y) < 1e-12
            assert rel(f[b, h], S[-1]) < 1e-12


def test_dt_zero_keeps_state():
    inp = rand_inputs(B=1, L=9, H=2, P=2, N=3, G=1, dt_zero=True, seed=3)
    y, f = orc.recurrence(**inp)
    h0, Cm, x, D = inp["h0"].numpy(), inp["Cm"].numpy(), inp["x"].numpy(), inp["D"].numpy()
    np.testing.assert_array_equal(f, h0)
    for h in range(2):
        Y = Cm[0, :, 0, :] @ h0[0, h].T + D[h] * x[0, :, h, :]
        assert rel(y[0, :, h, :], Y) < 1e-14


def test_dt_zero_steps_leave_state_unchanged():
    inp = rand_inputs(B=1, L=12, H=2, P=2, N=3, G=1, seed=5)
    zero_steps = [2, 3, 7]
    for t in zero_steps:
        inp["dt"][0, t, :] = 0.0
    sl = lambda k, t: inp[k][:, :t] if k in ("x", "dt", "Bm", "Cm") else inp[k]
    for t in zero_steps:
        _, f_before = orc.recurrence(**{k: sl(k, t) for k in inp if k != "ngroups"}, ngroups=1)
        _, f_after = orc.recurrence(**{k: sl(k, t + 1) for k in inp if k != "ngroups"}, ngroups=1)
        np.testing.assert_array_equal(f_before, f_after)


def test_scalar_case_is_first_order_iir():
    g = torch.Generator().manual_seed(11)
    L = 50
    x, b, c = (torch.randn(L, generator=g, dtype=f64) for _ in range(3))
    dt = torch.rand(L, generator=g, dtype=f64)
    a, d, s0 = -1.7, 0.4, 0.9
    ys, s = orc.scalar_iir(x.tolist(), dt.tolist(), a, b.tolist(), c.tolist(), d, s0)
    y, f = orc.recurrence(x.view(1, L, 1, 1), dt.view(1, L, 1), torch.tensor([a], dtype=f64),
                          b.view(1, L, 1, 1), c.view(1, L, 1, 1), torch.tensor([d], dtype=f64),
                          torch.tensor([[[[s0]]]], dtype=f64), ngroups=1)
    np.testing.assert_allclose(y.ravel(), ys, rtol=1e-14, atol=1e-14)
    assert abs(f.item() - s) < 1e-13


# ----------------------------------------------------------------------------
# the chunked decomposition and its intermediates


@pytest.mark.parametrize("Q", [1, 3, 16, 64, 100])
def test_chunk_size_invariance(Q):
    inp = rand_inputs(B=2, L=100, H=4, P=4, N=6, G=2, seed=21)
    y, f = orc.recurrence(**inp)
    out = orc.chunked(**inp, chunk_size=Q)
    B, L, H, P = y.shape
    assert rel(out["y"].reshape(B, H, L, P).transpose(0, 2, 1, 3), y) < 1e-12
    assert rel(out["final"].reshape(f.shape), f) < 1e-12


def test_chunked_intermediates_have_their_meaning():
    """h_prev[c] is the recurrence's state after the first c*Q tokens;
    S[c] is the state one chunk leaves behind when it starts from zero;
    2^(G at a chunk's end) is the product of that chunk's exp(A dt_t)."""
    Q = 8
    inp = rand_inputs(B=1, L=29, H=2, P=3, N=4, G=1, seed=9)
    out = orc.chunked(**inp, chunk_size=Q)
    L = 29
    nc = -(-L // Q)
    for c in range(nc):
        pre = {k: (inp[k][:, : c * Q] if k in ("x", "dt", "Bm", "Cm") else inp[k])
               for k in inp}
        _, f_pre = orc.recurrence(**pre)
        assert rel(out["h_prev"][:, c], f_pre.reshape(2, 3, 4)) < 1e-12
        chunk = {k: (inp[k][:, c * Q: (c + 1) * Q] if k in ("x", "dt", "Bm", "Cm") else inp[k])
                 for k in inp}
        chunk["h0"] = None
        _, f_chunk = orc.recurrence(**chunk)
        assert rel(out["S"][:, c], f_chunk.reshape(2, 3, 4)) < 1e-12
        for h in range(2):
            last = min((c + 1) * Q, L) - 1
            prod = 1.0
            for t in range(c * Q, last + 1):
                prod *= math.exp(float(inp["A"][h]) * float(inp["dt"][0, t, h]))
            assert abs(2.0 ** out["G"][h, last] - prod) <= 1e-13 * max(prod, 1e-300)


def test_resumability():
    inp = rand_inputs(B=2, L=40, H=2, P=3, N=4, G=1, seed=13)
    y, f = orc.recurrence(**inp)
    t = 17
    first = {k: (inp[k][:, :t] if k in ("x", "dt", "Bm", "Cm") else inp[k]) for k in inp}
    y1, f1 = orc.recurrence(**first)
    second = {k: (inp[k][:, t:] if k in ("x", "dt", "Bm", "Cm") else inp[k]) for k in inp}
    second["h0"] = torch.from_numpy(f1)
    y2, f2 = orc.recurrence(**second)
    assert rel(np.concatenate([y1, y2], axis=1), y) < 1e-13
    assert rel(f2, f) < 1e-13


def test_linearity():
    inp = rand_inputs(B=1, L=15, H=2, P=3, N=4, G=1, seed=17, h0=False)
    y, f = orc.recurrence(**inp)
    inp2 = dict(inp, x=2.5 * inp["x"])
    y2, f2 = orc.recurrence(**inp2)
    assert rel(y2, 2.5 * y) < 1e-13 and rel(f2, 2.5 * f) < 1e-13
    z = rand_inputs(B=1, L=15, H=2, P=3, N=4, G=1, seed=17)
    z["x"] = torch.zeros_like(z["x"])
    y3, f3 = orc.recurrence(**z)
    z["h0"] = -3.0 * z["h0"]
    y4, f4 = orc.recurrence(**z)
    assert rel(y4, -3.0 * y3) < 1e-13 and rel(f4, -3.0 * f3) < 1e-13


def test_slab_subset_matches_full():
    inp = rand_inputs(B=3, L=10, H=4, P=2, N=3, G=2, seed=19)
    y, f = orc.recurrence(**inp)
    pairs = [(2, 3), (0, 1), (1, 0)]
    ys, fs = orc.recurrence(**inp, slabs=pairs)
    for k, (b, h) in enumerate(pairs):
        np.testing.assert_array_equal(ys[k], y[b, :, h, :])
        np.testing.assert_array_equal(fs[k], f[b, h])


# ----------------------------------------------------------------------------
# the pins have power: planted mistakes in a copy of the recurrence fail them


def _mutant_recurrence(inp, mistake):
    """A pure-Python copy of the recurrence with one planted mistake."""
    x, dt, A, Bm, Cm = (inp[k].numpy() for k in ("x", "dt", "A", "Bm", "Cm"))
    D = inp["D"].numpy() if inp["D"] is not None else np.zeros(A.shape)
    Bn, L, H, P = x.shape
    G, N = Bm.shape[2], Bm.shape[3]
    y = np.zeros_like(x)
    fin = np.zeros((Bn, H, P, N))
    for b in range(Bn):
        for h in range(H):
            g = h % G if mistake == "group_interleaved" else h // (H // G)
            S = np.zeros((P, N)) if inp["h0"] is None else inp["h0"].numpy()[b, h].copy()
            for t in range(L):
                sgn = -1.0 if mistake == "decay_sign" else 1.0
                alpha = math.exp(sgn * A[h] * dt[b, t, h])
                prev = S.copy()
                u = 1.0 if mistake == "drop_dt_input" else dt[b, t, h]
                if mistake == "transposed_state" and P == N:
                    S = alpha * S + u * np.outer(Bm[b, t, g], x[b, t, h])
                else:
                    S = alpha * S + u * np.outer(x[b, t, h], Bm[b, t, g])
                Sy = prev if mistake == "previous_state" else S
                dterm = 0.0 if mistake == "drop_D" else D[h]
                y[b, t, h] = Sy @ Cm[b, t, g] + dterm * x[b, t, h]
            fin[b, h] = S
    return y, fin


@pytest.mark.parametrize("mistake", ["previous_state", "decay_sign", "drop_D",
                                     "drop_dt_input", "transposed_state",
                                     "group_interleaved"])
def test_pins_reject_planted_mistakes(mistake):
    caught = []
    for path in GOLDENS:
        _, inp, y, fin = load_golden(path)
        ym, fm = _mutant_recurrence(inp, mistake)
        ok = np.allclose(ym, y, rtol=1e-12, atol=1e-12) and np.allclose(fm, fin, rtol=1e-12,
                                                                        atol=1e-12)
        caught.append(not ok)
    assert any(caught), f"no golden example distinguishes the mistake {mistake!r}"
    # and the unmutated copy passes them all
    for path in GOLDENS:
        _, inp, y, fin = load_golden(path)
        ym, fm = _mutant_recurrence(inp, None)
        np.testing.assert_allclose(ym, y, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(fm, fin, rtol=1e-12, atol=1e-12)
