"""Python binding of the C ABI (include/ssd.h): argument marshalling only.

Every step of the computation runs in the CUDA kernels of
``libssd_gb300.so``; this module turns torch tensors into ``ssd_tensor``
descriptors, allocates outputs and workspace with torch on the inputs'
device, and passes the current torch stream.

Layouts: x [B,L,H,P], dt [B,L,H], A [H], B/C [B,L,G,N], D [H],
initial_states / final_states [B,H,P,N]; the decode step takes one token
per (batch, head): x, z [B,H,P], dt [B,H], B/C [B,G,N].
"""
from __future__ import annotations

import ctypes

import torch

from . import _native
from ._native import SsdError, SsdTensor  # noqa: F401  (re-exported)

_DTYPES = {torch.float32: _native.SSD_F32, torch.bfloat16: _native.SSD_BF16,
           torch.int32: _native.SSD_I32}


def _desc(t: torch.Tensor | None):
    """ctypes pointer to an ssd_tensor describing ``t`` (None -> NULL)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"expected a torch.Tensor, got {type(t).__name__}")
    if t.dim() > 5:
        raise ValueError("tensors of more than 5 dimensions are not supported")
    d = SsdTensor()
    d.data = t.data_ptr() if t.numel() > 0 else None
    d.dtype = _DTYPES.get(t.dtype, 99)
    d.ndim = t.dim()
    for i in range(t.dim()):
        d.shape[i] = t.shape[i]
        d.stride[i] = t.stride(i)
    return ctypes.pointer(d)


def _device_of(*ts):
    dev = None
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors (the library takes device pointers)")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"tensors on different devices: {dev} and {t.device}")
    return dev


def _stream(dev):
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def workspace_size(batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size,
                   dtype=torch.bfloat16) -> int:
    out = ctypes.c_size_t(0)
    st = _native.load().ssd_workspace_size(batch, seqlen, nheads, headdim, dstate, ngroups,
                                           chunk_size, _DTYPES.get(dtype, 99),
                                           ctypes.byref(out))
    _native.check(st, "ssd_workspace_size")
    return int(out.value)


def describe_plan(batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size,
                  dtype=torch.bfloat16) -> str:
    """Which kernels ssd_chunked_fwd launches for this problem ("fused: ..." or
    "staged: ..."), or why it would be rejected."""
    return _native.load().ssd_describe_plan(batch, seqlen, nheads, headdim, dstate, ngroups,
                                            chunk_size, _DTYPES.get(dtype, 99)).decode()


def chunked_fwd(x, dt, A, B, C, D=None, initial_states=None, chunk_size=256, ngroups=1, *,
                return_final_states=True, y=None, final_states=None, workspace=None, z=None):
    """SSD chunked forward.  Returns ``(y, final_states)`` (the latter None when
    ``return_final_states`` is False and no buffer was given).  With ``z``
    [B,L,H,P] (dtype of x) the output is gated, y * silu(z)
    (``ssd_chunked_fwd_gated``)."""
    dev = _device_of(x, dt, A, B, C, D, initial_states, y, final_states, workspace, z)
    lib = _native.load()
    Bn, L, H, P = x.shape
    N = B.shape[-1]
    if y is None:
        y = torch.empty((Bn, L, H, P), dtype=x.dtype, device=dev)
    if final_states is None and return_final_states:
        final_states = torch.empty((Bn, H, P, N), dtype=torch.float32, device=dev)
    need = workspace_size(Bn, L, H, P, N, ngroups, chunk_size, x.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    ws = (ctypes.c_void_p(workspace.data_ptr()), workspace.numel() * workspace.element_size())
    if z is None:
        st = lib.ssd_chunked_fwd(_desc(x), _desc(dt), _desc(A), _desc(B), _desc(C), _desc(D),
                                 _desc(initial_states), chunk_size, ngroups, _desc(y),
                                 _desc(final_states), *ws, _stream(dev))
        _native.check(st, "ssd_chunked_fwd")
    else:
        st = lib.ssd_chunked_fwd_gated(_desc(x), _desc(dt), _desc(A), _desc(B), _desc(C),
                                       _desc(D), _desc(z), _desc(initial_states), chunk_size,
                                       ngroups, _desc(y), _desc(final_states), *ws,
                                       _stream(dev))
        _native.check(st, "ssd_chunked_fwd_gated")
    return y, final_states


def chunked_fwd_static_scratch(x, dt, A, B, C, D=None, initial_states=None, chunk_size=256,
                               ngroups=1, *, return_final_states=True, y=None,
                               final_states=None):
    """The SSD forward without any workspace argument: the library takes its
    scratch from a fixed device array of SSD_STATIC_SCRATCH_BYTES (for callers
    that cannot allocate device memory).  Problems needing more scratch than
    that raise SsdError(SSD_ERR_WORKSPACE).  Calls that overlap on the GPU
    share that array and race; order them on one stream."""
    dev = _device_of(x, dt, A, B, C, D, initial_states, y, final_states)
    Bn, L, H, P = x.shape
    N = B.shape[-1]
    if y is None:
        y = torch.empty((Bn, L, H, P), dtype=x.dtype, device=dev)
    if final_states is None and return_final_states:
        final_states = torch.empty((Bn, H, P, N), dtype=torch.float32, device=dev)
    st = _native.load().ssd_chunked_fwd_static_scratch(
        _desc(x), _desc(dt), _desc(A), _desc(B), _desc(C), _desc(D), _desc(initial_states),
        chunk_size, ngroups, _desc(y), _desc(final_states), _stream(dev))
    _native.check(st, "ssd_chunked_fwd_static_scratch")
    return y, final_states


# ---- the four steps, one call each -----------------------------------------

def state_update(state, x, dt, A, B, C, D=None, z=None, dt_bias=None, dt_softplus=False,
                 ngroups=1, *, out=None):
    """One decode token (``ssd_state_update``): updates ``state`` [B,H,P,N]
    (fp32, or bf16: computed in fp32, kept rounded) in place and returns
    ``out`` [B,H,P] (dtype of x).  x, z
    [B,H,P]; dt [B,H]; A, D, dt_bias [H]; B, C [B,G,N]."""
    dev = _device_of(state, x, dt, A, B, C, D, z, dt_bias, out)
    if out is None:
        out = torch.empty(x.shape, dtype=x.dtype, device=dev)
    lib = _native.load()
    _native.check(lib.ssd_state_update(_desc(state), _desc(x), _desc(dt), _desc(A), _desc(B),
                                       _desc(C), _desc(D), _desc(z), _desc(dt_bias),
                                       1 if dt_softplus else 0, ngroups, _desc(out),
                                       _stream(dev)),
                  "ssd_state_update")
    return out


def state_update_tokens(state, x, dt, A, B, C, D=None, z=None, dt_bias=None, dt_softplus=False,
                        ngroups=1, *, intermediate_states=None, parent=None, update_state=True,
                        state_indices=None, out=None):
    """T decode tokens per sequence (``ssd_state_update_tokens``): x, z, out
    [B,T,H,P]; dt [B,T,H]; B, C [B,T,G,N]; optional intermediate_states
    [B,T,H,P,N] in the state's dtype (the state after every token) and parent
    [B,T] int32
    (token t starts from the state after token parent[b,t] when that is an
    earlier token).  Updates ``state`` in place unless ``update_state`` is
    false; returns ``out``.  ``state_indices`` [B] int32 makes ``state`` and
    ``intermediate_states`` pools of S slots ([S,H,P,N], [S,T,H,P,N]): row b
    uses slot state_indices[b]; rows with an index outside [0, S) are skipped
    (their out rows are not written)."""
    dev = _device_of(state, x, dt, A, B, C, D, z, dt_bias, intermediate_states, parent,
                     state_indices, out)
    if out is None:
        out = torch.empty(x.shape, dtype=x.dtype, device=dev)
    lib = _native.load()
    _native.check(lib.ssd_state_update_tokens(_desc(state), _desc(x), _desc(dt), _desc(A),
                                              _desc(B), _desc(C), _desc(D), _desc(z),
                                              _desc(dt_bias), 1 if dt_softplus else 0, ngroups,
                                              _desc(out), _desc(intermediate_states),
                                              _desc(parent), _desc(state_indices),
                                              1 if update_state else 0,
                                              _stream(dev)),
                  "ssd_state_update_tokens")
    return out


def mixer_prologue(xBC, conv_weight, dt, nheads, headdim, ngroups, dstate, *, conv_bias=None,
                   conv_state=None, conv_windows=None, conv_state_indices=None, dt_bias=None,
                   dt_softplus=True, out=None):
    """Causal conv1d + SiLU over xBC [B,L,Dc], split into x [B,L,H,P], B and C
    [B,L,G,N], and dt' = softplus(dt + dt_bias) [B,L,H] f32
    (``ssd_mixer_prologue``).  ``conv_state`` [B,Dc,W] is read as the left
    context and updated in place; ``conv_windows`` [B,L,Dc,W] receives the
    window after every token.  ``conv_state_indices`` [B] int32 makes both
    pools of S slots ([S,Dc,W], [S,L,Dc,W]), row b on slot
    conv_state_indices[b]; rows with an index outside [0, S) are skipped.
    Returns ``(x, B, C, dt')``; ``out`` may give those four buffers."""
    dev = _device_of(xBC, conv_weight, dt, conv_bias, conv_state, conv_windows,
                     conv_state_indices, dt_bias)
    Bn, L, _ = xBC.shape
    if out is None:
        out = (torch.empty((Bn, L, nheads, headdim), dtype=xBC.dtype, device=dev),
               torch.empty((Bn, L, ngroups, dstate), dtype=xBC.dtype, device=dev),
               torch.empty((Bn, L, ngroups, dstate), dtype=xBC.dtype, device=dev),
               torch.empty((Bn, L, nheads), dtype=torch.float32, device=dev))
    x, Bm, Cm, dt_out = out
    _device_of(x, Bm, Cm, dt_out)
    st = _native.load().ssd_mixer_prologue(_desc(xBC), _desc(conv_weight), _desc(conv_bias),
                                           _desc(conv_state), _desc(conv_windows),
                                           _desc(conv_state_indices), _desc(dt),
                                           _desc(dt_bias), 1 if dt_softplus else 0, ngroups,
                                           _desc(x), _desc(Bm), _desc(Cm), _desc(dt_out),
                                           _stream(dev))
    _native.check(st, "ssd_mixer_prologue")
    return x, Bm, Cm, dt_out


def chunk_cumsum(dt, A, chunk_size, out=None):
    """G [B, H, nc*Q] f32: log2(e) times the in-chunk inclusive cumsum of A*dt."""
    dev = _device_of(dt, A, out)
    Bn, L, H = dt.shape
    nc = -(-L // chunk_size)
    G = out if out is not None else torch.empty((Bn, H, nc * chunk_size), dtype=torch.float32,
                                                device=dev)
    st = _native.load().ssd_stage_chunk_cumsum(_desc(dt), _desc(A), chunk_size, _desc(G),
                                               _stream(dev))
    _native.check(st, "ssd_stage_chunk_cumsum")
    return G


def chunk_state(x, B, dt, G, chunk_size, ngroups, out=None):
    """S [B, nc, H, P, N] f32: each chunk's state when it starts from zero."""
    dev = _device_of(x, B, dt, G, out)
    Bn, L, H, P = x.shape
    N = B.shape[-1]
    nc = -(-L // chunk_size)
    S = out if out is not None else torch.empty((Bn, nc, H, P, N), dtype=torch.float32,
                                                device=dev)
    st = _native.load().ssd_stage_chunk_state(_desc(x), _desc(B), _desc(dt), _desc(G),
                                              chunk_size, ngroups, _desc(S), _stream(dev))
    _native.check(st, "ssd_stage_chunk_state")
    return S


def state_passing(S, G, initial_states, chunk_size, state_dtype=torch.float32,
                  return_final_states=True, out=None):
    """(h_prev [B, nc, H, P, N] in state_dtype, final_states [B, H, P, N] f32).
    ``out`` may give both buffers as a pair (final may be None)."""
    dev = _device_of(S, G, initial_states)
    Bn, nc, H, P, N = S.shape
    if out is not None:
        h_prev, final = out
    else:
        h_prev = torch.empty((Bn, nc, H, P, N), dtype=state_dtype, device=dev)
        final = (torch.empty((Bn, H, P, N), dtype=torch.float32, device=dev)
                 if return_final_states else None)
    _device_of(S, h_prev, final)
    st = _native.load().ssd_stage_state_passing(_desc(S), _desc(G), _desc(initial_states),
                                                chunk_size, _desc(h_prev), _desc(final),
                                                _stream(dev))
    _native.check(st, "ssd_stage_state_passing")
    return h_prev, final


def chunk_scan(x, dt, G, B, C, D, h_prev, chunk_size, ngroups, out=None):
    """y [B, L, H, P] in the dtype of x."""
    dev = _device_of(x, dt, G, B, C, D, h_prev, out)
    y = out if out is not None else torch.empty(x.shape, dtype=x.dtype, device=dev)
    st = _native.load().ssd_stage_chunk_scan(_desc(x), _desc(dt), _desc(G), _desc(B), _desc(C),
                                             _desc(D), _desc(h_prev), chunk_size, ngroups,
                                             _desc(y), _stream(dev))
    _native.check(st, "ssd_stage_chunk_scan")
    return y
