"""Pins of the oracle's decode step (selective state update) to facts outside it.

The step is one token of the layer recurrence (section 6.1 "The SSU Math" of
"Optimizing Nemotron v3 Super in TensorRT-LLM"), plus the dt bias, softplus
and z gate of the reference in section 6.2.  Pinned by: a hand-derived worked
example (tests/golden/ssu/), agreement of repeated steps with the C
recurrence (an independent implementation, itself pinned in
test_oracle_pins.py), the limits of softplus and silu, and planted mistakes
that each fail one of these.
"""
import glob
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ssu")
f64 = torch.float64


def _num(v):
    if isinstance(v, str):
        return float(eval(v, {"__builtins__": {}},
                          {"ln2": math.log(2.0), "ln3": math.log(3.0), "ln": math.log,
                           "e": math.e}))
    return float(v)


def _arr(v):
    return [_arr(e) for e in v] if isinstance(v, list) else _num(v)


def load_ssu(path):
    with open(path) as f:
        g = json.load(f)
    s = g["shape"]
    Bn, H, P, N, G = s["B"], s["H"], s["P"], s["N"], s["G"]
    t = lambda key, shape: torch.tensor(_arr(g[key]), dtype=f64).reshape(shape)
    inp = dict(state=t("state", (Bn, H, P, N)), x=t("x", (Bn, H, P)), dt=t("dt", (Bn, H)),
               A=t("A", (H,)), Bm=t("B", (Bn, G, N)), Cm=t("C", (Bn, G, N)), D=t("D", (H,)),
               z=t("z", (Bn, H, P)), dt_bias=t("dt_bias", (H,)), dt_softplus=g["softplus"],
               ngroups=G)
    out = np.array(_arr(g["out"])).reshape(Bn, H, P)
    new = np.array(_arr(g["new_state"])).reshape(Bn, H, P, N)
    return inp, out, new


SSU_GOLDENS = sorted(glob.glob(os.path.join(GOLDEN, "*.json")))


def rand_step_inputs(B=2, H=4, P=3, N=5, G=2, T=6, seed=0):
    g = torch.Generator().manual_seed(seed)
    r = lambda *s: torch.randn(s, generator=g, dtype=f64)
    return dict(
        x=r(B, T, H, P), dt=torch.nn.functional.softplus(r(B, T, H) - 1.0),
        A=-torch.exp(torch.rand(H, generator=g, dtype=f64) * math.log(4.0)),
        Bm=r(B, T, G, N), Cm=r(B, T, G, N), D=r(H), h0=0.3 * r(B, H, P, N), ngroups=G)


def run_steps(step, inp):
    """Applies `step` token by token; returns (y [B,T,H,P], final state)."""
    state = inp["h0"].clone()
    T = inp["x"].shape[1]
    ys = []
    for t in range(T):
        o, new = step(state, inp["x"][:, t], inp["dt"][:, t], inp["A"], inp["Bm"][:, t],
                      inp["Cm"][:, t], D=inp["D"], ngroups=inp["ngroups"])
        ys.append(o)
        state = torch.from_numpy(new)
    return np.stack(ys, axis=1), state.numpy()


@pytest.mark.parametrize("path", SSU_GOLDENS, ids=[os.path.basename(p) for p in SSU_GOLDENS])
def test_ssu_golden(path):
    inp, out, new = load_ssu(path)
    o, n = orc.ssu_step(**inp)
    np.testing.assert_allclose(o, out, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(n, new, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("G", [1, 2, 4])
def test_ssu_steps_equal_the_recurrence(G):
    inp = rand_step_inputs(G=G, seed=G)
    y_steps, fin_steps = run_steps(orc.ssu_step, inp)
    y_ref, fin_ref = orc.recurrence(inp["x"], inp["dt"], inp["A"], inp["Bm"], inp["Cm"],
                                    inp["D"], inp["h0"], ngroups=G)
    np.testing.assert_allclose(y_steps, y_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(fin_steps, fin_ref, rtol=1e-12, atol=1e-12)


def test_softplus_tends_to_identity():
    inp, _, _ = load_ssu(SSU_GOLDENS[0])
    inp["dt"] = torch.full_like(inp["dt"], 30.0)
    inp["dt_bias"] = None
    o_sp, n_sp = orc.ssu_step(**inp)
    o_id, n_id = orc.ssu_step(**dict(inp, dt_softplus=False))
    np.testing.assert_allclose(o_sp, o_id, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(n_sp, n_id, rtol=1e-11, atol=1e-12)


def test_gate_limits():
    inp, _, _ = load_ssu(SSU_GOLDENS[0])
    o_free, _ = orc.ssu_step(**dict(inp, z=None))
    o_zero, _ = orc.ssu_step(**dict(inp, z=torch.zeros_like(inp["z"])))
    np.testing.assert_array_equal(o_zero, 0.0)                       # silu(0) = 0
    o_big, _ = orc.ssu_step(**dict(inp, z=torch.full_like(inp["z"], 40.0)))
    np.testing.assert_allclose(o_big, 40.0 * o_free, rtol=1e-14)      # silu(z) -> z


def _mutant_step(mistake):
    def step(state, x, dt, A, Bm, Cm, D=None, z=None, dt_bias=None, dt_softplus=False,
             ngroups=1):
        st = state.numpy().astype(np.float64)
        xv, dtv, Av = x.numpy(), dt.numpy(), A.numpy()
        Bv, Cv = Bm.numpy(), Cm.numpy()
        Dv = None if D is None else D.numpy()
        zv = None if z is None else z.numpy()
        bv = None if dt_bias is None else dt_bias.numpy()
        Bn, H, P, N = st.shape
        hpg = H // ngroups
        out = np.empty((Bn, H, P))
        new = np.empty_like(st)
        for b in range(Bn):
            for h in range(H):
                g = h % ngroups if mistake == "group_interleaved" else h // hpg
                d = dtv[b, h]
                if mistake == "bias_after_softplus":
                    d = (np.logaddexp(0.0, d) if dt_softplus else d) + (bv[h] if bv is not None else 0)
                else:
                    d = d + (bv[h] if bv is not None else 0.0)
                    d = np.logaddexp(0.0, d) if dt_softplus else d
                dA = math.exp(A.numpy()[h] * d)
                u = 1.0 if mistake == "drop_dt_input" else d
                new[b, h] = st[b, h] * dA + u * np.outer(xv[b, h], Bv[b, g])
                src = st[b, h] if mistake == "old_state_output" else new[b, h]
                o = src @ Cv[b, g] + (Dv[h] * xv[b, h] if Dv is not None else 0.0)
                if zv is not None:
                    gate = 1.0 / (1.0 + np.exp(-zv[b, h]))
                    if mistake != "sigmoid_gate":
                        gate = zv[b, h] * gate
                    o = o * gate
                out[b, h] = o
        return out, new
    return step


@pytest.mark.parametrize("mistake", ["old_state_output", "drop_dt_input", "sigmoid_gate",
                                     "bias_after_softplus", "group_interleaved"])
def test_ssu_pins_reject_planted_mistakes(mistake):
    step = _mutant_step(mistake)
    caught = False
    for path in SSU_GOLDENS:
        inp, out, new = load_ssu(path)
        o, n = step(**inp)
        caught |= not (np.allclose(o, out, rtol=1e-12, atol=1e-12) and
                       np.allclose(n, new, rtol=1e-12, atol=1e-12))
    inp = rand_step_inputs(G=2, seed=7)
    y, fin = run_steps(step, inp)
    y_ref, fin_ref = orc.recurrence(inp["x"], inp["dt"], inp["A"], inp["Bm"], inp["Cm"],
                                    inp["D"], inp["h0"], ngroups=2)
    caught |= not (np.allclose(y, y_ref, rtol=1e-10) and np.allclose(fin, fin_ref, rtol=1e-10))
    assert caught, f"no pin distinguishes the mistake {mistake!r}"
    # the unmutated copy passes them all
    clean = _mutant_step(None)
    for path in SSU_GOLDENS:
        inp, out, new = load_ssu(path)
        o, n = clean(**inp)
        np.testing.assert_allclose(o, out, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(n, new, rtol=1e-12, atol=1e-12)
