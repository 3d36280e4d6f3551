"""TEST INFRASTRUCTURE ONLY -- fp64 CPU oracle for the Mamba-2 SSD chunked forward.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  It shares no code with the CUDA path
(``state_space_model_gb300``) and neither imports the other.

Four independent evaluations of the same layer, all in float64 on the stored
input values (bf16 and fp32 upcast exactly):

* :func:`recurrence` -- the definition: the token-by-token recurrence of
  "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in NVIDIA
  CUDA Tile", section "Mamba-2 architecture", evaluated in plain C
  (``ssd_recurrence.c``), OpenMP over (batch, head) slabs.
* :func:`quadratic` -- the masked-decay "attention" form of the same page
  (the output equation with exp(G - G^T) and the causal mask M, taken with a
  single chunk spanning the whole sequence), written with explicit sums.
* :func:`chunked` -- the chunkwise algorithm in the page's order: kernel 1
  (in-chunk cumulative sum of A*dt, scaled by log2(e)), kernel 2
  (fwd_pass_state: hidden state at each chunk start via the jump formula
  h_{t+T} = exp(G_last) h_t + (exp(G_last - G) * B)^T X, split here into the
  per-chunk state and the sequential state passing), kernel 3 (compute_out:
  Y = exp(G) C h + (exp(G - G^T) * (C B^T) * M) X + D X).  Its intermediates
  are the references for the four GPU stages.
* :func:`scalar_iir` -- the H = G = P = N = 1 special case, a first-order
  linear recurrence, in pure Python.
* :func:`ssu_step` -- one decode step (the selective state update) of
  "Optimizing Nemotron v3 Super in TensorRT-LLM", section 6.1 "The SSU Math",
  with the dt bias, softplus and z gate of section 6.2's reference, in numpy.

Readings of the pages taken here (where they are silent or contradict):
the output uses the updated state h_t (inclusive causal mask i >= j);
head h reads group h // (H // G); D and initial_states absent mean zero;
a sequence length that is not a multiple of the chunk size is zero-padded
(dt = 0, x = B = C = 0) and the padded outputs are dropped.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_recurrence.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()

_DT_CODE = {torch.float32: 0, torch.bfloat16: 1, torch.float64: 2}
LOG2E = 1.4426950408889634  # log2(e), the scale of the stored cumulative sum


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` with gcc (plain C, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    ):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", _SRC,
             "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_ssd_recurrence.restype = ctypes.c_int
            vp, ci, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
            lib.oracle_ssd_recurrence.argtypes = [
                vp, ci, vp, ci, vp, ci, vp, vp, ci, vp, ci, vp, ci,
                i64, i64, i64, i64, i64, i64, vp, i64, vp, vp, ci,
            ]
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _as_cpu(t):
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        t = torch.from_numpy(t)
    t = t.detach().to("cpu").contiguous()
    if t.dtype not in _DT_CODE:
        raise TypeError(f"oracle: unsupported dtype {t.dtype}")
    return t


def _shapes(x, dt, A, Bm, Cm, ngroups):
    B, L, H, P = x.shape
    N = Bm.shape[-1]
    if tuple(dt.shape) != (B, L, H) or tuple(A.shape) != (H,):
        raise ValueError("oracle: dt must be [B,L,H] and A [H]")
    if tuple(Bm.shape) != (B, L, ngroups, N) or tuple(Cm.shape) != (B, L, ngroups, N):
        raise ValueError("oracle: B and C must be [B,L,G,N]")
    if H % ngroups:
        raise ValueError("oracle: nheads must be a multiple of ngroups")
    return B, L, H, P, N


def _slab_list(slabs, B, H):
    if slabs is None:
        return [(b, h) for b in range(B) for h in range(H)]
    return [(int(b), int(h)) for b, h in slabs]


def recurrence(x, dt, A, Bm, Cm, D=None, h0=None, ngroups=1, slabs=None,
               threads=0):
    """The definition: per-token recurrence in fp64 (C, OpenMP over slabs).

    Returns ``(y, final)`` as float64 numpy arrays.  With ``slabs=None`` they
    are ``[B,L,H,P]`` and ``[B,H,P,N]``; with a list of ``(b, h)`` pairs they
    are ``[nslab, L, P]`` and ``[nslab, P, N]`` in that order.
    """
    x, dt, A, Bm, Cm, D, h0 = (_as_cpu(t) for t in (x, dt, A, Bm, Cm, D, h0))
    B, L, H, P, N = _shapes(x, dt, A, Bm, Cm, ngroups)
    if Bm.dtype != Cm.dtype:
        raise TypeError("oracle: B and C must share a dtype")
    pairs = _slab_list(slabs, B, H)
    flat = np.array([b * H + h for b, h in pairs], dtype=np.int64)
    y = np.empty((len(pairs), L, P), dtype=np.float64)
    fin = np.empty((len(pairs), P, N), dtype=np.float64)
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    code = lambda t: 0 if t is None else _DT_CODE[t.dtype]
    rc = _load().oracle_ssd_recurrence(
        ptr(x), code(x), ptr(dt), code(dt), ptr(A), code(A),
        ptr(Bm), ptr(Cm), code(Bm), ptr(D), code(D), ptr(h0), code(h0),
        B, L, H, P, N, ngroups,
        flat.ctypes.data_as(ctypes.c_void_p), len(pairs),
        y.ctypes.data_as(ctypes.c_void_p), fin.ctypes.data_as(ctypes.c_void_p),
        int(threads),
    )
    if rc != 0:
        raise RuntimeError(f"oracle_ssd_recurrence failed ({rc})")
    if slabs is None:
        y = y.reshape(B, H, L, P).transpose(0, 2, 1, 3).copy()
        fin = fin.reshape(B, H, P, N)
    return y, fin


def _slab64(x, dt, A, Bm, Cm, D, h0, b, h, g):
    """fp64 numpy views of one (batch, head) slab's inputs."""
    f = lambda t: t.to(torch.float64).numpy()
    xs = f(x[b, :, h, :])                 # [L, P]
    dts = f(dt[b, :, h])                  # [L]
    bs = f(Bm[b, :, g, :])                # [L, N]
    cs = f(Cm[b, :, g, :])                # [L, N]
    a = float(A[h].to(torch.float64))
    d = 0.0 if D is None else float(D[h].to(torch.float64))
    P, N = xs.shape[1], bs.shape[1]
    hs = np.zeros((P, N)) if h0 is None else f(h0[b, h])
    return xs, dts, bs, cs, a, d, hs


def quadratic(x, dt, A, Bm, Cm, D=None, h0=None, ngroups=1, slabs=None):
    """Masked-decay "attention" form, one chunk spanning the whole sequence.

    y_i = sum_{j<=i} exp(sum_{k=j+1..i} a_k) dt_j (C_i . B_j) x_j
          + exp(sum_{k=0..i} a_k) (h0 C_i) + D x_i,       a_k = A dt_k
    final = exp(sum_k a_k) h0 + sum_j exp(sum_{k=j+1..L-1} a_k) dt_j x_j B_j^T

    O(L^2) explicit sums: for tiny inputs only.  Returns per-slab arrays
    ``[nslab, L, P]`` and ``[nslab, P, N]``.
    """
    x, dt, A, Bm, Cm, D, h0 = (_as_cpu(t) for t in (x, dt, A, Bm, Cm, D, h0))
    B, L, H, P, N = _shapes(x, dt, A, Bm, Cm, ngroups)
    pairs = _slab_list(slabs, B, H)
    ys, fs = [], []
    for b, h in pairs:
        xs, dts, bs, cs, a, d, hs = _slab64(x, dt, A, Bm, Cm, D, h0, b, h,
                                            h // (H // ngroups))
        ak = a * dts
        y = np.zeros((L, P))
        for i in range(L):
            y[i] += math.exp(float(np.sum(ak[: i + 1]))) * (hs @ cs[i])
            for j in range(i + 1):
                w = math.exp(float(np.sum(ak[j + 1: i + 1]))) * dts[j]
                y[i] += w * float(cs[i] @ bs[j]) * xs[j]
            y[i] += d * xs[i]
        fin = math.exp(float(np.sum(ak))) * hs
        for j in range(L):
            w = math.exp(float(np.sum(ak[j + 1:]))) * dts[j]
            fin = fin + w * np.outer(xs[j], bs[j])
        ys.append(y)
        fs.append(fin)
    return np.stack(ys), np.stack(fs)


def chunked(x, dt, A, Bm, Cm, D=None, h0=None, ngroups=1, chunk_size=64,
            slabs=None):
    """Chunkwise evaluation in the order of the page's three kernels.

    Returns a dict of per-slab float64 arrays (slab order as given):
      ``G``      [nslab, L]        in-chunk inclusive cumsum of A*dt, times log2(e)
      ``S``      [nslab, nc, P, N] per-chunk state  sum_j 2^(G_last-G_j) dt_j x_j B_j^T
      ``h_prev`` [nslab, nc, P, N] state entering each chunk (h_prev[0] = h0)
      ``final``  [nslab, P, N]     state after the last token
      ``y``      [nslab, L, P]
    """
    x, dt, A, Bm, Cm, D, h0 = (_as_cpu(t) for t in (x, dt, A, Bm, Cm, D, h0))
    B, L, H, P, N = _shapes(x, dt, A, Bm, Cm, ngroups)
    Q = int(chunk_size)
    if Q <= 0:
        raise ValueError("oracle: chunk_size must be positive")
    nc = -(-L // Q)
    Lp = nc * Q
    pairs = _slab_list(slabs, B, H)
    res = {k: [] for k in ("G", "S", "h_prev", "final", "y")}
    for b, h in pairs:
        xs, dts, bs, cs, a, d, hs = _slab64(x, dt, A, Bm, Cm, D, h0, b, h,
                                            h // (H // ngroups))
        # zero padding of the last chunk (padded tokens have dt = x = B = C = 0)
        pad = Lp - L
        xs = np.pad(xs, ((0, pad), (0, 0)))
        dts = np.pad(dts, (0, pad))
        bs = np.pad(bs, ((0, pad), (0, 0)))
        cs = np.pad(cs, ((0, pad), (0, 0)))

        # kernel 1: in-chunk cumulative sum of a*dt, scaled by log2(e)
        G = np.empty(Lp)
        for c in range(nc):
            sl = slice(c * Q, (c + 1) * Q)
            G[sl] = np.cumsum(a * dts[sl]) * LOG2E

        # kernel 2: per-chunk state, then the sequential pass over chunks
        S = np.empty((nc, P, N))
        h_prev = np.empty((nc, P, N))
        hid = hs.copy()
        for c in range(nc):
            sl = slice(c * Q, (c + 1) * Q)
            g = G[sl]
            g_last = g[-1]
            b_dt_d = bs[sl] * (dts[sl] * np.exp2(g_last - g))[:, None]  # [Q, N]
            S[c] = xs[sl].T @ b_dt_d                                      # [P, N]
            h_prev[c] = hid
            hid = np.exp2(g_last) * hid + S[c]

        # kernel 3: outputs of each chunk from its entering state
        y = np.empty((Lp, P))
        idx = np.arange(Q)
        causal = idx[:, None] >= idx[None, :]
        for c in range(nc):
            sl = slice(c * Q, (c + 1) * Q)
            g = G[sl]
            cb = cs[sl] @ bs[sl].T                                   # [Q, Q]
            # select before exponentiating: masked entries never see a positive exponent
            expo = np.where(causal, g[:, None] - g[None, :], -np.inf)
            cb = cb * np.exp2(expo)
            yc = (cs[sl] @ h_prev[c].T) * np.exp2(g)[:, None]        # [Q, P]
            yc = yc + cb @ (dts[sl][:, None] * xs[sl])
            y[sl] = yc + d * xs[sl]

        res["G"].append(G[:L])
        res["S"].append(S)
        res["h_prev"].append(h_prev)
        res["final"].append(hid)
        res["y"].append(y[:L])
    return {k: np.stack(v) for k, v in res.items()}


def scalar_iir(x, dt, a, b, c, d=0.0, s0=0.0):
    """First-order linear recurrence s_t = exp(a dt_t) s_{t-1} + dt_t b_t x_t,
    y_t = c_t s_t + d x_t (the one-head, one-channel, one-state case), in
    pure Python floats.  Returns (list of y, final s)."""
    s = float(s0)
    ys = []
    for xt, dtt, bt, ct in zip(x, dt, b, c):
        s = math.exp(a * dtt) * s + dtt * bt * xt
        ys.append(ct * s + d * xt)
    return ys, s


def ssu_step(state, x, dt, A, Bm, Cm, D=None, z=None, dt_bias=None, dt_softplus=False,
             ngroups=1):
    """One decode step of the recurrence for every (batch, head), in float64.

    Shapes: state [B,H,P,N], x [B,H,P], dt [B,H], A [H], Bm and Cm [B,G,N],
    D [H], z [B,H,P], dt_bias [H].  Following the SSU math: dt' = dt (+ dt_bias),
    softplus(dt') = log(1 + exp(dt')) when ``dt_softplus``; dA = exp(A dt');
    new_state = state dA + dt' x (outer) B; out = new_state C + D x; out is
    multiplied by silu(z) = z / (1 + exp(-z)) when z is given.  Head h reads
    group h // (H // G).  Returns ``(out [B,H,P], new_state [B,H,P,N])``.
    """
    f = lambda t: None if t is None else np.asarray(_as_cpu(t).to(torch.float64).numpy(),
                                                   dtype=np.float64)
    st, xv, dtv, Av, Bv, Cv, Dv, zv, bv = (f(t) for t in (state, x, dt, A, Bm, Cm, D, z,
                                                         dt_bias))
    Bn, H, P, N = st.shape
    if H % ngroups:
        raise ValueError("oracle: nheads must be a multiple of ngroups")
    hpg = H // ngroups
    out = np.empty((Bn, H, P), dtype=np.float64)
    new = np.empty_like(st)
    for b in range(Bn):
        for h in range(H):
            g = h // hpg
            d = dtv[b, h] + (bv[h] if bv is not None else 0.0)
            if dt_softplus:
                d = np.logaddexp(0.0, d)          # log(1 + e^d)
            dA = math.exp(Av[h] * d)
            new[b, h] = st[b, h] * dA + d * np.outer(xv[b, h], Bv[b, g])
            o = new[b, h] @ Cv[b, g]
            if Dv is not None:
                o = o + Dv[h] * xv[b, h]
            if zv is not None:
                o = o * (zv[b, h] / (1.0 + np.exp(-zv[b, h])))
            out[b, h] = o
    return out, new


def _round_state(a, state_dtype):
    """A state as kept in memory: float64 values rounded to the state's storage
    dtype ("f32" or "bf16", round to nearest even) and widened back."""
    t = torch.from_numpy(np.asarray(a, dtype=np.float64))
    if state_dtype == "bf16":
        return t.to(torch.bfloat16).to(torch.float64).numpy()
    if state_dtype == "f32":
        return t.to(torch.float32).to(torch.float64).numpy()
    raise ValueError(f"oracle: state dtype {state_dtype!r}")


def ssu_tokens(state, x, dt, A, Bm, Cm, D=None, z=None, dt_bias=None, dt_softplus=False,
               ngroups=1, parent=None, update_state=True, state_dtype=None, state_indices=None):
    """T decode steps per sequence, in float64, as one would apply them one
    token at a time -- the multi-token state update of "Optimizing Nemotron
    v3 Super in TensorRT-LLM", section 10.4, with the intermediate-state cache
    of section 10.3.

    Shapes: x, z [B,T,H,P]; dt [B,T,H]; Bm, Cm [B,T,G,N]; parent [B,T]
    integers or None.  Each sequence's running state starts at state[b]; token
    t applies ``ssu_step`` to it, except that for t > 0 with
    0 <= parent[b,t] < t it first restarts from the state cached after token
    parent[b,t] (a tree of draft tokens; other values keep the chain).
    Returns ``(out [B,T,H,P], final [B,H,P,N], cache [B,T,H,P,N])``: cache[:, t]
    is the state after token t; final is the running state after the last
    token, or the input state unchanged when ``update_state`` is false.

    ``state_dtype`` ("f32" or "bf16") models a state kept in that dtype: each
    token's update is computed from the kept state in float64 and its output
    from the unrounded result, and the state is then kept rounded (the running
    state, the cache and the final state alike).  None keeps float64 throughout.

    ``state_indices`` [B] integers (the slot indirection of the page's serving
    kernel, section 10.4: state_batch_idx, with pad_slot_id for padding rows)
    makes ``state`` a pool [S,H,P,N] of S slots: sequence b runs on
    state[state_indices[b]], and a row whose index is outside [0, S) is padding:
    it is not computed (its out and cache rows are NaN) and no slot changes for
    it.  ``final`` is then the whole pool, the slots of real rows updated.
    """
    f = lambda t: None if t is None else _as_cpu(t).to(torch.float64)
    st0 = f(state)
    xv, dtv, Bv, Cv, zv = (f(t) for t in (x, dt, Bm, Cm, z))
    Bn, T = xv.shape[0], xv.shape[1]
    H, P, N = st0.shape[1], st0.shape[2], st0.shape[3]
    par = None if parent is None else np.asarray(torch.as_tensor(parent).detach().cpu().numpy(),
                                                 dtype=np.int64)
    slots = np.arange(Bn) if state_indices is None else np.asarray(
        torch.as_tensor(state_indices).detach().cpu().numpy(), dtype=np.int64)
    out = np.full((Bn, T, H, P), np.nan, dtype=np.float64)
    cache = np.full((Bn, T, H, P, N), np.nan, dtype=np.float64)
    final = st0.numpy().copy()
    for b in range(Bn):
        slot = int(slots[b])
        if not 0 <= slot < st0.shape[0]:
            continue                                    # a padding row
        run = st0[slot:slot + 1]
        for t in range(T):
            if par is not None and t > 0 and 0 <= par[b, t] < t:
                run = torch.from_numpy(cache[b:b + 1, par[b, t]].copy())
            o, new = ssu_step(run, xv[b:b + 1, t], dtv[b:b + 1, t], A, Bv[b:b + 1, t],
                              Cv[b:b + 1, t], D=D, z=None if zv is None else zv[b:b + 1, t],
                              dt_bias=dt_bias, dt_softplus=dt_softplus, ngroups=ngroups)
            if state_dtype is not None:
                new = _round_state(new, state_dtype)
            out[b, t] = o[0]
            cache[b, t] = new[0]
            run = torch.from_numpy(new)
        if update_state and T > 0:
            final[slot] = run[0].numpy()
    return out, final, cache


def causal_conv1d(xBC, weight, bias=None, conv_state=None, silu=True, state_indices=None):
    """Causal depthwise convolution over the token axis, then SiLU -- the
    convolution that prepares x, B and C in the Mamba-2 mixer ("Optimizing
    Nemotron v3 Super in TensorRT-LLM", sections 8 "CausalConv1d Optimization"
    and 10.5), in float64.

    xBC [B, L, Dc]; weight [Dc, W]; bias [Dc] or None; conv_state [B, Dc, W]
    or None: the last W inputs before this call, oldest first (zeros when
    None).  With u the inputs preceded by that state,

        out[b, t, c] = silu(bias[c] + sum_k weight[c, k] u[b, t - (W - 1) + k, c])

    so weight[:, W - 1] multiplies the current token.  Returns
    ``(out [B, L, Dc], new_state [B, Dc, W], windows [B, L, Dc, W])``:
    new_state holds the last W inputs of the concatenation, windows[:, t] the
    last W inputs up to and including token t (the state after token t).

    ``state_indices`` [B] integers (the conv_state_indices of the page's
    section 10.5) makes ``conv_state`` a pool [S, Dc, W]: row b reads and
    replaces slot state_indices[b]; a row whose index is outside [0, S) is
    padding, not computed (its out and windows rows are NaN), and
    ``new_state`` is the whole pool with the slots of real rows replaced.
    """
    if state_indices is not None:
        pool = _as_cpu(conv_state).to(torch.float64).numpy()
        slots = np.asarray(torch.as_tensor(state_indices).cpu().numpy(), dtype=np.int64)
        real = (slots >= 0) & (slots < pool.shape[0])
        rows = np.where(real[:, None, None], pool[np.where(real, slots, 0)], 0.0)
        out, new_rows, windows = causal_conv1d(xBC, weight, bias, torch.from_numpy(rows), silu)
        out[~real] = np.nan
        windows[~real] = np.nan
        new_pool = pool.copy()
        new_pool[slots[real]] = new_rows[real]
        return out, new_pool, windows
    xv = _as_cpu(xBC).to(torch.float64).numpy()
    w = _as_cpu(weight).to(torch.float64).numpy()
    Bn, L, Dc = xv.shape
    W = w.shape[1]
    if w.shape[0] != Dc:
        raise ValueError("oracle: weight must be [Dc, W]")
    bv = np.zeros(Dc) if bias is None else _as_cpu(bias).to(torch.float64).numpy()
    st = (np.zeros((Bn, Dc, W)) if conv_state is None
          else _as_cpu(conv_state).to(torch.float64).numpy())
    u = np.concatenate([st.transpose(0, 2, 1), xv], axis=1)      # [B, W + L, Dc]
    out = np.empty((Bn, L, Dc))
    windows = np.empty((Bn, L, Dc, W))
    for t in range(L):
        win = u[:, t + 1:t + 1 + W, :]                            # inputs t-W+1 .. t
        pre = bv[None, :] + np.einsum("bkc,ck->bc", win, w)
        out[:, t] = pre / (1.0 + np.exp(-pre)) if silu else pre
        windows[:, t] = win.transpose(0, 2, 1)
    new_state = u[:, L:L + W, :].transpose(0, 2, 1).copy()
    return out, new_state, windows


def dt_prologue(dt, dt_bias=None, dt_softplus=True):
    """dt' = dt + dt_bias, then softplus(dt') = log(1 + exp(dt')) when asked
    (the dt preparation of the SSU reference, "Optimizing Nemotron v3 Super in
    TensorRT-LLM", section 6.2), in float64.  dt [..., H], dt_bias [H]."""
    d = _as_cpu(dt).to(torch.float64).numpy()
    if dt_bias is not None:
        d = d + _as_cpu(dt_bias).to(torch.float64).numpy()
    return np.logaddexp(0.0, d) if dt_softplus else d


def split_xbc(xbc, nheads, headdim, ngroups, dstate):
    """The channel order of the mixer's convolution output: x (H P channels),
    then B (G N), then C (G N).  [B, L, Dc] -> x [B, L, H, P], B and C
    [B, L, G, N] (numpy views)."""
    Bn, L, Dc = xbc.shape
    hp, gn = nheads * headdim, ngroups * dstate
    if Dc != hp + 2 * gn:
        raise ValueError("oracle: Dc must be H P + 2 G N")
    return (xbc[..., :hp].reshape(Bn, L, nheads, headdim),
            xbc[..., hp:hp + gn].reshape(Bn, L, ngroups, dstate),
            xbc[..., hp + gn:].reshape(Bn, L, ngroups, dstate))


def gate(y, z):
    """y silu(z) = y z / (1 + exp(-z)), the output gate of the mixer, in float64."""
    yv = np.asarray(y, dtype=np.float64) if not isinstance(y, torch.Tensor) else \
        _as_cpu(y).to(torch.float64).numpy()
    zv = _as_cpu(z).to(torch.float64).numpy()
    return yv * (zv / (1.0 + np.exp(-zv)))
