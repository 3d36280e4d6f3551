"""Pins of the oracle's mixer prologue and epilogue (causal conv1d + SiLU, the
x / B / C split, dt bias + softplus, the z gate) to facts outside it.

The convolution is the causal depthwise one of "Optimizing Nemotron v3 Super in
TensorRT-LLM", sections 8 and 10.5, with the conv state laid out as the page's
cache holds it ([batch, conv_dim, d_conv], oldest input first).  Pinned by:
numpy's own convolution (an independent library routine), causality, carrying
the state across a split sequence, token-by-token calls against one call, the
width-1 and identity-activation special cases, the limits of softplus and silu,
and planted mistakes that each fail one of these.
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle as orc

f64 = torch.float64


def rand_conv(B=2, L=9, Dc=6, W=4, seed=0, state=True):
    g = torch.Generator().manual_seed(seed)
    r = lambda *s: torch.randn(s, generator=g, dtype=f64)
    return dict(xBC=r(B, L, Dc), weight=r(Dc, W), bias=r(Dc),
                conv_state=r(B, Dc, W) if state else None)


def silu(v):
    return v / (1.0 + np.exp(-v))


@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("with_state", [False, True])
def test_conv_equals_numpy_convolve(W, with_state):
    inp = rand_conv(W=W, seed=W, state=with_state)
    out, new, _ = orc.causal_conv1d(**inp, silu=False)
    x, w, b = inp["xBC"].numpy(), inp["weight"].numpy(), inp["bias"].numpy()
    B, L, Dc = x.shape
    st = inp["conv_state"].numpy() if with_state else np.zeros((B, Dc, W))
    for bb in range(B):
        for c in range(Dc):
            u = np.concatenate([st[bb, c], x[bb, :, c]])
            # 'valid' entry i is sum_k u[i + k] w[c, k] taken in reverse: the window ending at u[i + W - 1]
            ref = np.convolve(u, w[c][::-1], mode="valid")[1:] + b[c]
            np.testing.assert_allclose(out[bb, :, c], ref, rtol=1e-13, atol=1e-13)
            np.testing.assert_array_equal(new[bb, c], u[-W:])
    out_s, _, _ = orc.causal_conv1d(**inp, silu=True)
    np.testing.assert_allclose(out_s, silu(out), rtol=1e-14, atol=1e-15)


def test_conv_is_causal():
    inp = rand_conv(L=12, seed=3)
    out, _, _ = orc.causal_conv1d(**inp)
    x2 = inp["xBC"].clone()
    x2[:, 7:] += 5.0
    out2, _, _ = orc.causal_conv1d(**dict(inp, xBC=x2))
    np.testing.assert_array_equal(out[:, :7], out2[:, :7])
    assert not np.allclose(out[:, 7:], out2[:, 7:])


@pytest.mark.parametrize("split", [1, 2, 5, 8])
def test_conv_state_carries_across_a_split_sequence(split):
    inp = rand_conv(L=9, seed=4)
    out, new, win = orc.causal_conv1d(**inp)
    a, s1, wa = orc.causal_conv1d(**dict(inp, xBC=inp["xBC"][:, :split]))
    bo, s2, wb = orc.causal_conv1d(**dict(inp, xBC=inp["xBC"][:, split:],
                                          conv_state=torch.from_numpy(s1)))
    np.testing.assert_allclose(np.concatenate([a, bo], axis=1), out, rtol=1e-14, atol=1e-14)
    np.testing.assert_array_equal(s2, new)
    np.testing.assert_array_equal(np.concatenate([wa, wb], axis=1), win)


def test_token_by_token_equals_one_call_and_windows_are_the_states():
    inp = rand_conv(L=6, seed=5)
    out, new, win = orc.causal_conv1d(**inp)
    st = inp["conv_state"]
    for t in range(6):
        o, st_np, _ = orc.causal_conv1d(**dict(inp, xBC=inp["xBC"][:, t:t + 1], conv_state=st))
        np.testing.assert_allclose(o[:, 0], out[:, t], rtol=1e-14, atol=1e-14)
        np.testing.assert_array_equal(win[:, t], st_np)
        st = torch.from_numpy(st_np)
    np.testing.assert_array_equal(st.numpy(), new)


def test_width_one_is_pointwise_and_short_sequences_keep_old_inputs():
    inp = rand_conv(W=1, seed=6)
    out, _, _ = orc.causal_conv1d(**inp, silu=False)
    ref = inp["xBC"].numpy() * inp["weight"].numpy()[:, 0] + inp["bias"].numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-14)
    inp = rand_conv(L=2, W=4, seed=7)
    _, new, _ = orc.causal_conv1d(**inp)
    np.testing.assert_array_equal(new[:, :, :2], inp["conv_state"].numpy()[:, :, 2:])
    np.testing.assert_array_equal(new[:, :, 2:], inp["xBC"].numpy().transpose(0, 2, 1))


def test_dt_prologue_limits():
    dt = torch.tensor([[0.0, 40.0, -40.0]], dtype=f64)
    bias = torch.tensor([0.0, 0.0, 0.0], dtype=f64)
    d = orc.dt_prologue(dt, bias)
    assert d[0, 0] == pytest.approx(math.log(2.0), rel=1e-15)
    assert d[0, 1] == pytest.approx(40.0, rel=1e-15)
    assert d[0, 2] == pytest.approx(math.exp(-40.0), rel=1e-12)
    # the bias is added before softplus
    d2 = orc.dt_prologue(torch.tensor([[-1.0]], dtype=f64), torch.tensor([1.0], dtype=f64))
    assert d2[0, 0] == pytest.approx(math.log(2.0), rel=1e-15)
    np.testing.assert_array_equal(orc.dt_prologue(dt, bias, dt_softplus=False), dt.numpy())


def test_split_order_is_x_then_b_then_c():
    H, P, G, N = 2, 3, 1, 2
    Dc = H * P + 2 * G * N
    xbc = np.arange(Dc, dtype=np.float64).reshape(1, 1, Dc)
    x, b, c = orc.split_xbc(xbc, H, P, G, N)
    np.testing.assert_array_equal(x[0, 0], [[0, 1, 2], [3, 4, 5]])
    np.testing.assert_array_equal(b[0, 0], [[6, 7]])
    np.testing.assert_array_equal(c[0, 0], [[8, 9]])


def test_gate_limits():
    y = torch.tensor([1.5, -2.0, 3.0], dtype=f64)
    z = torch.tensor([0.0, 50.0, -50.0], dtype=f64)
    g = orc.gate(y, z)
    assert g[0] == 0.0
    assert g[1] == pytest.approx(-100.0, rel=1e-15)
    assert abs(g[2]) < 1e-18


def _mutant_conv(mistake):
    def run(xBC, weight, bias=None, conv_state=None, silu=True):
        x, w = xBC.numpy(), weight.numpy()
        B, L, Dc = x.shape
        W = w.shape[1]
        b = bias.numpy() if bias is not None else np.zeros(Dc)
        st = conv_state.numpy() if conv_state is not None else np.zeros((B, Dc, W))
        if mistake == "state_newest_first":
            st = st[:, :, ::-1]
        if mistake == "taps_flipped":
            w = w[:, ::-1]
        u = np.concatenate([st.transpose(0, 2, 1), x], axis=1)
        out = np.empty((B, L, Dc))
        for t in range(L):
            lo = t if mistake == "window_one_early" else t + 1
            win = u[:, lo:lo + W, :]
            pre = np.einsum("bkc,ck->bc", win, w)
            if mistake == "bias_after_silu":
                out[:, t] = pre / (1.0 + np.exp(-pre)) + b if silu else pre + b
            else:
                pre = pre + b
                out[:, t] = pre / (1.0 + np.exp(-pre)) if silu else pre
        new = u[:, L:L + W, :].transpose(0, 2, 1)
        return out, new, None
    return run


@pytest.mark.parametrize("mistake", ["taps_flipped", "window_one_early", "state_newest_first",
                                     "bias_after_silu"])
def test_conv_pins_reject_planted_mistakes(mistake):
    mut = _mutant_conv(mistake)
    inp = rand_conv(seed=11)
    x, w, b, st = (inp[k].numpy() for k in ("xBC", "weight", "bias", "conv_state"))
    B, L, Dc = x.shape
    W = w.shape[1]
    o, _, _ = mut(**inp, silu=True)
    o_lin, _, _ = mut(**inp, silu=False)
    ref_lin = np.empty_like(o_lin)
    for bb in range(B):
        for c in range(Dc):
            u = np.concatenate([st[bb, c], x[bb, :, c]])
            ref_lin[bb, :, c] = np.convolve(u, w[c][::-1], mode="valid")[1:] + b[c]
    caught = not (np.allclose(o_lin, ref_lin, rtol=1e-12) and
                  np.allclose(o, silu(ref_lin), rtol=1e-12))
    assert caught, f"no pin distinguishes the mistake {mistake!r}"
    clean = _mutant_conv(None)
    o2, n2, _ = clean(**inp)
    o_ref, n_ref, _ = orc.causal_conv1d(**inp)
    np.testing.assert_allclose(o2, o_ref, rtol=1e-14, atol=1e-14)
    np.testing.assert_array_equal(n2, n_ref)


@pytest.mark.parametrize("indices", [[4, -1, 1], [0, 2, 9]], ids=["pad_negative", "pad_past_end"])
def test_conv_slots_run_each_row_on_its_slot(indices):
    """A conv-state pool: each real row equals numpy's convolution of that row
    preceded by its slot's inputs, its slot is replaced by the row's last W
    inputs, other slots are unchanged and padding rows are not computed."""
    S, W = 5, 4
    inp = rand_conv(B=3, L=7, W=W, seed=21)
    g = torch.Generator().manual_seed(22)
    pool = torch.randn((S, 6, W), generator=g, dtype=f64)
    out, new, win = orc.causal_conv1d(**dict(inp, conv_state=pool), silu=False,
                                      state_indices=torch.tensor(indices, dtype=torch.int32))
    x, w, b = inp["xBC"].numpy(), inp["weight"].numpy(), inp["bias"].numpy()
    used = set()
    for bb, slot in enumerate(indices):
        if not 0 <= slot < S:
            assert np.all(np.isnan(out[bb])) and np.all(np.isnan(win[bb]))
            continue
        used.add(slot)
        for c in range(x.shape[2]):
            u = np.concatenate([pool[slot, c].numpy(), x[bb, :, c]])
            ref = np.convolve(u, w[c][::-1], mode="valid")[1:] + b[c]
            np.testing.assert_allclose(out[bb, :, c], ref, rtol=1e-13, atol=1e-13)
            np.testing.assert_array_equal(new[slot, c], u[-W:])
    for slot in set(range(S)) - used:
        np.testing.assert_array_equal(new[slot], pool[slot].numpy())
