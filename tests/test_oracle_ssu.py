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


# ---- several tokens per call (section 10.4 of the same page) ----------------

def rand_token_inputs(B=2, T=6, H=4, P=3, N=5, G=2, seed=0):
    g = torch.Generator().manual_seed(seed)
    r = lambda *s: torch.randn(s, generator=g, dtype=f64)
    return dict(state=0.3 * r(B, H, P, N), x=r(B, T, H, P),
                dt=torch.nn.functional.softplus(r(B, T, H) - 1.0),
                A=-torch.exp(torch.rand(H, generator=g, dtype=f64) * math.log(4.0)),
                Bm=r(B, T, G, N), Cm=r(B, T, G, N), D=r(H), ngroups=G)


def _pred(parent_row, t):
    """The token whose state token t starts from (-1: the call's initial state)."""
    if t == 0:
        return -1
    p = int(parent_row[t])
    return p if 0 <= p < t else t - 1


def _path(parent_row, t):
    path = []
    while t >= 0:
        path.append(t)
        t = _pred(parent_row, t)
    return path[::-1]


def _recurrence_on_path(inp, b, path):
    """The C recurrence over the tokens of `path` of sequence b: (y of the last
    token [H,P], state after it [H,P,N])."""
    idx = torch.tensor(path)
    y, fin = orc.recurrence(inp["x"][b:b + 1, idx], inp["dt"][b:b + 1, idx], inp["A"],
                            inp["Bm"][b:b + 1, idx], inp["Cm"][b:b + 1, idx], inp["D"],
                            inp["state"][b:b + 1], ngroups=inp["ngroups"])
    return y[0, -1], fin[0]


def test_tokens_chain_equals_the_recurrence():
    inp = rand_token_inputs(seed=3)
    out, final, cache = orc.ssu_tokens(**inp)
    y, fin = orc.recurrence(inp["x"], inp["dt"], inp["A"], inp["Bm"], inp["Cm"], inp["D"],
                            inp["state"], ngroups=inp["ngroups"])
    np.testing.assert_allclose(out, y, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(final, fin, rtol=1e-12, atol=1e-12)
    T = inp["x"].shape[1]
    for t in range(T):   # the cache holds the state after each prefix
        _, fin_t = orc.recurrence(inp["x"][:, :t + 1], inp["dt"][:, :t + 1], inp["A"],
                                  inp["Bm"][:, :t + 1], inp["Cm"][:, :t + 1], inp["D"],
                                  inp["state"], ngroups=inp["ngroups"])
        np.testing.assert_allclose(cache[:, t], fin_t, rtol=1e-12, atol=1e-12)


TREES = [
    [[-1, 0, 0, 1, 1, 2], [-1, -1, 0, 2, 2, 0]],     # two sequences, branching drafts
    [[-1, 0, 1, 2, 3, 4], [-1, 0, 0, 0, 0, 0]],      # a chain and a star
]


@pytest.mark.parametrize("tree", TREES, ids=["branching", "chain_star"])
def test_tokens_tree_follows_each_tokens_path(tree):
    inp = rand_token_inputs(seed=5)
    parent = torch.tensor(tree, dtype=torch.int32)
    out, final, cache = orc.ssu_tokens(**inp, parent=parent)
    B, T = parent.shape
    for b in range(B):
        for t in range(T):
            y_t, st_t = _recurrence_on_path(inp, b, _path(tree[b], t))
            np.testing.assert_allclose(out[b, t], y_t, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(cache[b, t], st_t, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(final[b], cache[b, T - 1], rtol=0, atol=0)


def test_tokens_parent_values_outside_the_earlier_tokens_keep_the_chain():
    inp = rand_token_inputs(seed=6)
    chain = orc.ssu_tokens(**inp)
    odd = torch.tensor([[5, 1, 2, 9, -3, 5], [0, 7, -1, 3, 100, -2]], dtype=torch.int32)
    got = orc.ssu_tokens(**inp, parent=odd)
    for a, b in zip(chain, got):
        np.testing.assert_array_equal(a, b)


def test_tokens_without_state_update_leave_the_state():
    inp = rand_token_inputs(seed=8)
    out, final, cache = orc.ssu_tokens(**inp, update_state=False)
    out2, final2, cache2 = orc.ssu_tokens(**inp)
    np.testing.assert_array_equal(final, inp["state"].numpy())
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(cache, cache2)
    assert not np.array_equal(final2, final)


def _mutant_tokens(mistake):
    """A copy of the token loop with one plausible mistake planted."""
    def run(state, x, dt, A, Bm, Cm, D=None, ngroups=1, parent=None, update_state=True):
        Bn, T = x.shape[0], x.shape[1]
        out = np.empty(tuple(x.shape))
        cache = np.empty((Bn, T) + tuple(state.shape[1:]))
        final = state.numpy().copy()
        for b in range(Bn):
            run_st = state[b:b + 1]
            for t in range(T):
                if parent is not None and t > 0:
                    p = int(parent[b, t])
                    if mistake == "parent_off_by_one":
                        p = p - 1
                    if mistake != "parent_ignored" and 0 <= p < t:
                        run_st = torch.from_numpy(cache[b:b + 1, p].copy())
                o, new = orc.ssu_step(run_st, x[b:b + 1, t], dt[b:b + 1, t], A, Bm[b:b + 1, t],
                                      Cm[b:b + 1, t], D=D, ngroups=ngroups)
                out[b, t] = o[0]
                cache[b, t] = run_st[0].numpy() if mistake == "cache_before_update" else new[0]
                if mistake != "state_not_carried":
                    run_st = torch.from_numpy(new)
            if update_state:
                final[b] = run_st[0].numpy()
        return out, final, cache
    return run


@pytest.mark.parametrize("mistake", ["parent_off_by_one", "parent_ignored", "cache_before_update",
                                     "state_not_carried"])
def test_tokens_pins_reject_planted_mistakes(mistake):
    inp = rand_token_inputs(seed=5)
    parent = torch.tensor(TREES[0], dtype=torch.int32)
    mut = _mutant_tokens(mistake)
    caught = False
    for par in (None, parent):
        o, f, c = mut(**inp, parent=par)
        ref = orc.ssu_tokens(**inp, parent=par)
        # the pins above compare against the recurrence on each token's path
        B, T = inp["x"].shape[:2]
        for b in range(B):
            for t in range(T):
                row = TREES[0][b] if par is not None else [-1] * T
                y_t, st_t = _recurrence_on_path(inp, b, _path(row, t))
                caught |= not (np.allclose(o[b, t], y_t, rtol=1e-10) and
                               np.allclose(c[b, t], st_t, rtol=1e-10))
        del ref
    assert caught, f"no pin distinguishes the mistake {mistake!r}"
    clean = _mutant_tokens(None)
    for par in (None, parent):
        for a, b in zip(clean(**inp, parent=par), orc.ssu_tokens(**inp, parent=par)):
            np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-13)


# ---- a state kept in bf16 (the pages' fp16 / bf16 state caches) -------------

def test_bf16_state_rounds_only_what_is_kept():
    inp = rand_token_inputs(seed=12)
    # a kept state is bf16: start from bf16-representable values
    inp["state"] = inp["state"].to(torch.bfloat16).to(f64)
    out1, fin1, cache1 = orc.ssu_tokens(**{**inp, "x": inp["x"][:, :1], "dt": inp["dt"][:, :1],
                                           "Bm": inp["Bm"][:, :1], "Cm": inp["Cm"][:, :1]},
                                        state_dtype="bf16")
    out0, fin0, _ = orc.ssu_tokens(**{**inp, "x": inp["x"][:, :1], "dt": inp["dt"][:, :1],
                                      "Bm": inp["Bm"][:, :1], "Cm": inp["Cm"][:, :1]})
    # one token: the output comes from the unrounded update; the kept state is
    # that update rounded to bf16, nothing else changes
    np.testing.assert_array_equal(out1, out0)
    np.testing.assert_array_equal(fin1, torch.from_numpy(fin0).to(torch.bfloat16).to(f64).numpy())
    np.testing.assert_array_equal(cache1[:, 0], fin1)
    assert not np.array_equal(fin1, fin0)


def test_bf16_state_tokens_equal_rounded_single_steps():
    inp = rand_token_inputs(seed=13)
    inp["state"] = inp["state"].to(torch.bfloat16).to(f64)
    out, fin, cache = orc.ssu_tokens(**inp, state_dtype="bf16")
    st = inp["state"]
    T = inp["x"].shape[1]
    for t in range(T):
        o, new = orc.ssu_step(st, inp["x"][:, t], inp["dt"][:, t], inp["A"], inp["Bm"][:, t],
                              inp["Cm"][:, t], D=inp["D"], ngroups=inp["ngroups"])
        np.testing.assert_array_equal(out[:, t], o)
        st = torch.from_numpy(new).to(torch.bfloat16).to(f64)
        np.testing.assert_array_equal(cache[:, t], st.numpy())
    np.testing.assert_array_equal(fin, st.numpy())
    # and it stays within bf16 rounding of the float64 run
    out64, fin64, _ = orc.ssu_tokens(**inp)
    assert np.max(np.abs(out - out64)) / np.max(np.abs(out64)) < 2e-2


# ---- slot indirection (a state pool and padding rows) ------------------------

@pytest.mark.parametrize("indices", [[3, -1, 0], [4, 7, 1]], ids=["pad_negative", "pad_past_end"])
def test_slots_run_each_row_on_its_slot(indices):
    B, S = 3, 5
    inp = rand_token_inputs(B=B, seed=14)
    g = torch.Generator().manual_seed(15)
    pool = 0.3 * torch.randn((S,) + tuple(inp["state"].shape[1:]), generator=g, dtype=f64)
    idx = torch.tensor(indices, dtype=torch.int32)
    out, final, cache = orc.ssu_tokens(**{**inp, "state": pool}, state_indices=idx)
    used = set()
    for b, slot in enumerate(indices):
        if not 0 <= slot < S:               # padding: nothing computed for the row
            assert np.all(np.isnan(out[b])) and np.all(np.isnan(cache[b]))
            continue
        used.add(slot)
        # the C recurrence of row b's tokens from the slot's state
        y, fin = orc.recurrence(inp["x"][b:b + 1], inp["dt"][b:b + 1], inp["A"],
                                inp["Bm"][b:b + 1], inp["Cm"][b:b + 1], inp["D"],
                                pool[slot:slot + 1], ngroups=inp["ngroups"])
        np.testing.assert_allclose(out[b], y[0], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(final[slot], fin[0], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(cache[b, -1], fin[0], rtol=1e-12, atol=1e-12)
    for slot in set(range(S)) - used:       # other slots untouched, bit for bit
        np.testing.assert_array_equal(final[slot], pool[slot].numpy())


def test_identity_slots_equal_the_plain_call():
    inp = rand_token_inputs(seed=16)
    a = orc.ssu_tokens(**inp)
    b = orc.ssu_tokens(**inp, state_indices=torch.arange(inp["x"].shape[0], dtype=torch.int32))
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)
