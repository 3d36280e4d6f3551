"""C-ABI checks that need no GPU: the library loads, exports every function
include/*.h declares, and its host-side argument checks return the right
status (and a detail naming the failed check) before any CUDA call.

The descriptors here point at fake, aligned addresses: each case fails a
pure-host check first, so nothing ever dereferences them.
"""
import ctypes
import glob
import os
import re
import subprocess

import pytest

from state_space_model_gb300 import _native
from state_space_model_gb300._native import SsdTensor

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
F32, BF16 = 0, 1
FAKE = 0x7F0000000000  # 256-byte aligned, never dereferenced


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        names |= set(re.findall(r"\b(ssd_[A-Za-z0-9_]+)\s*\(", src))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from state_space_model_gb300 import build
    build.build()
    return _native.load()


def test_exports_every_declared_function(lib):
    names = declared_functions()
    assert "ssd_chunked_fwd" in names and len(names) >= 8
    out = subprocess.run(["nm", "-D", "--defined-only", _native.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(\w+)", out))
    for n in names:
        assert n in exported, f"{n} declared in include/ but not exported"
        assert hasattr(lib, n)


def test_status_strings(lib):
    for code, name in _native.STATUS.items():
        assert lib.ssd_status_string(code).decode() == name


def tens(shape, dtype=BF16, strides=None, ptr=FAKE):
    d = SsdTensor()
    d.data = ptr
    d.dtype = dtype
    d.ndim = len(shape)
    if strides is None:
        strides, acc = [], 1
        for s in reversed(shape):
            strides.insert(0, acc)
            acc *= s
    for i, (s, st) in enumerate(zip(shape, strides)):
        d.shape[i] = s
        d.stride[i] = st
    return d


class Case:
    """A valid bf16 problem of fake device tensors at distinct addresses."""

    def __init__(self, B=2, L=300, H=4, P=64, N=128, G=2, Q=64, xdt=BF16):
        self.B, self.L, self.H, self.P, self.N, self.G, self.Q = B, L, H, P, N, G, Q
        base = [FAKE]

        def nxt(nbytes):
            p = base[0]
            base[0] += (nbytes + 4095) // 4096 * 4096 + 4096
            return p

        es = 2 if xdt == BF16 else 4
        self.x = tens((B, L, H, P), xdt, ptr=nxt(B * L * H * P * es))
        self.dt = tens((B, L, H), F32, ptr=nxt(B * L * H * 4))
        self.A = tens((H,), F32, ptr=nxt(H * 4))
        self.Bm = tens((B, L, G, N), xdt, ptr=nxt(B * L * G * N * es))
        self.Cm = tens((B, L, G, N), xdt, ptr=nxt(B * L * G * N * es))
        self.D = tens((H,), F32, ptr=nxt(H * 4))
        self.h0 = tens((B, H, P, N), F32, ptr=nxt(B * H * P * N * 4))
        self.y = tens((B, L, H, P), xdt, ptr=nxt(B * L * H * P * es))
        self.fin = tens((B, H, P, N), F32, ptr=nxt(B * H * P * N * 4))
        self.ws_bytes = 1 << 40
        self.ws = nxt(1 << 20) + (1 << 41)

    def call(self, lib, **over):
        a = dict(x=self.x, dt=self.dt, A=self.A, Bm=self.Bm, Cm=self.Cm, D=self.D,
                 h0=self.h0, y=self.y, fin=self.fin, Q=self.Q, G=self.G,
                 ws=self.ws, ws_bytes=self.ws_bytes)
        a.update(over)
        p = lambda t: None if t is None else ctypes.pointer(t)
        return lib.ssd_chunked_fwd(p(a["x"]), p(a["dt"]), p(a["A"]), p(a["Bm"]), p(a["Cm"]),
                                   p(a["D"]), p(a["h0"]), a["Q"], a["G"], p(a["y"]),
                                   p(a["fin"]), a["ws"], a["ws_bytes"], None)


def detail(lib):
    return lib.ssd_last_error_detail().decode()


def test_workspace_size(lib):
    out = ctypes.c_size_t()
    # the fused path needs no workspace for whole waves of slabs (its split of
    # the last partial wave is covered by test_fused_split_plan)
    assert lib.ssd_workspace_size(2, 4096, 152, 64, 128, 1, 256, BF16, ctypes.byref(out)) == 0
    assert out.value == 0
    # the four-step path keeps G, S and h_prev there
    assert lib.ssd_workspace_size(8, 4096, 80, 64, 128, 1, 64, BF16, ctypes.byref(out)) == 0
    B, L, H, P, N, Q = 8, 4096, 80, 64, 128, 64
    nc = L // Q
    need = B * H * nc * Q * 4 + B * nc * H * P * N * 4 + B * nc * H * P * N * 2
    assert need <= out.value < need + 3 * 256
    assert lib.ssd_workspace_size(1, 10, 3, 64, 128, 2, 256, BF16, ctypes.byref(out)) == 1
    assert "multiple of ngroups" in detail(lib)
    assert lib.ssd_workspace_size(1, 10, 4, 64, 128, 2, 100, BF16, ctypes.byref(out)) == 2
    assert lib.ssd_workspace_size(1, 10, 4, 48, 128, 2, 128, BF16, ctypes.byref(out)) == 2
    assert lib.ssd_workspace_size(1, 10, 4, 64, 128, 2, 128, 7, ctypes.byref(out)) == 1


def test_describe_plan(lib):
    d = lambda *a: lib.ssd_describe_plan(*a).decode()
    assert d(8, 4096, 80, 64, 128, 1, 256, BF16).startswith("fused")
    assert d(1, 256, 4, 16, 16, 1, 64, F32).startswith("staged")
    assert "tcgen05" in d(2, 300, 4, 64, 128, 1, 64, BF16)
    f32 = d(2, 300, 4, 64, 128, 1, 128, F32)   # fp32 on the tensor cores as bf16 hi / lo
    assert "k_chunk_state_tc_f32" in f32 and "k_chunk_scan_tc_f32" in f32, f32
    assert "tcgen05" not in d(2, 300, 4, 64, 128, 1, 64, F32)   # Q = 64: CUDA-core steps
    assert d(1, 10, 4, 64, 128, 1, 100, BF16).startswith("rejected")
    assert d(1, 10, 4, 64, 128, 1, 64, 9).startswith("rejected")


def test_fused_split_plan(lib):
    """The pair slabs (or, for odd heads per group, the slabs) left over after
    the last full wave of SMs are split by sequence.

    The plan names the segments; the workspace holds the tail segments' local
    states and decays and their entering states, each region 256-byte aligned.
    A whole number of waves, or one 128-token block per slab, is never split
    and needs no workspace.
    """
    import re
    d = lambda *a: lib.ssd_describe_plan(*a).decode()
    out = ctypes.c_size_t()
    a256 = lambda v: (v + 255) // 256 * 256
    PN = 64 * 128
    M = 152   # SM count assumed without a device
    # (B, L, H, G): two heads per CTA (heads per group even)
    for B, L, H, G in [(8, 4096, 80, 1), (3, 4096, 102, 1), (1, 20000, 308, 2)]:
        plan = d(B, L, H, 64, 128, G, 256, BF16)
        assert "k_ssd_pair" in plan, plan
        m = re.search(r"(\d+) whole \(batch, head pair\) slabs \+ the last (\d+) pair slabs in "
                      r"(\d+) segments of (\d+) tokens", plan)
        assert m, plan
        whole, tail, nseg, seg_len = map(int, m.groups())
        assert whole + tail == B * H // 2 and whole % M == 0 and 0 < tail < M
        assert nseg >= 2 and seg_len % 128 == 0
        assert (nseg - 1) * seg_len < L <= nseg * seg_len
        ws = a256(a256(a256(tail * (nseg - 1) * 2 * PN * 4) + tail * (nseg - 1) * 8) +
                  tail * nseg * 2 * PN * 4)
        assert lib.ssd_workspace_size(B, L, H, 64, 128, G, 256, BF16, ctypes.byref(out)) == 0
        assert out.value == ws, (plan, out.value, ws)
        assert f"workspace {ws} bytes" in plan
    # one head per CTA: odd heads per group, or fewer pair slabs than SMs
    for B, L, H in [(1, 65536, 3), (2, 8000, 3), (1, 32768, 25), (1, 65536, 8), (1, 16384, 4),
                    (1, 32768, 24)]:
        plan = d(B, L, H, 64, 128, 1, 256, BF16)
        assert "k_ssd_fused" in plan, plan
        m = re.search(r"the last (\d+) slabs in (\d+) segments of (\d+) tokens", plan)
        assert m, plan
        tail, nseg, seg_len = map(int, m.groups())
        assert tail == B * H and nseg >= 2 and seg_len % 128 == 0
        assert (nseg - 1) * seg_len < L <= nseg * seg_len
        ws = a256(a256(a256(tail * (nseg - 1) * PN * 4) + tail * (nseg - 1) * 4) + tail * nseg * PN * 4)
        assert lib.ssd_workspace_size(B, L, H, 64, 128, 1, 256, BF16, ctypes.byref(out)) == 0
        assert out.value == ws, (plan, out.value, ws)
        assert f"workspace {ws} bytes" in plan
    # whole waves of pair slabs, short pair slabs, or one block per slab: whole slabs only
    for B, L, H in [(2, 4096, 152), (2, 640, 96), (1, 128, 8)]:
        plan = d(B, L, H, 64, 128, 1, 256, BF16)
        assert "segments" not in plan, plan
        assert lib.ssd_workspace_size(B, L, H, 64, 128, 1, 256, BF16, ctypes.byref(out)) == 0
        assert out.value == 0
    assert "k_ssd_fused" in d(2, 4096, 153, 64, 128, 1, 256, BF16)   # odd heads per group
    assert "k_ssd_pair" in d(2, 4096, 152, 64, 128, 1, 256, BF16)
    assert "k_ssd_fused" in d(2, 4096, 150, 64, 128, 1, 256, BF16)   # 150 pair slabs < 152 SMs


def test_error_paths(lib):
    c = Case()
    # null required descriptor
    assert c.call(lib, x=None) == 1 and "x" in detail(lib)
    assert c.call(lib, dt=None) == 1 and "dt" in detail(lib)
    assert c.call(lib, y=None) == 1 and "y" in detail(lib)
    # wrong dtype
    assert c.call(lib, dt=tens((2, 300, 4), BF16, ptr=c.dt.data)) == 1
    assert "dt" in detail(lib) and "dtype" in detail(lib)
    assert c.call(lib, Bm=tens((2, 300, 2, 128), F32, ptr=c.Bm.data)) == 1
    assert c.call(lib, x=tens((2, 300, 4, 64), 5, ptr=c.x.data)) == 1
    # wrong shapes
    assert c.call(lib, dt=tens((2, 299, 4), F32, ptr=c.dt.data)) == 1
    assert "shape" in detail(lib)
    assert c.call(lib, y=tens((2, 300, 4, 32), BF16, ptr=c.y.data)) == 1
    assert c.call(lib, A=tens((5,), F32, ptr=c.A.data)) == 1
    # heads not a multiple of groups, unsupported geometry
    assert c.call(lib, G=3) == 1 and "ngroups" in detail(lib)
    assert c.call(lib, Q=96) == 2 and "chunk_size" in detail(lib)
    assert c.call(lib, Q=0) == 1
    c2 = Case(P=48)
    assert c2.call(lib) == 2 and "headdim" in detail(lib)
    c3 = Case(N=256)
    assert c3.call(lib) == 2 and "dstate" in detail(lib)
    # innermost stride
    assert c.call(lib, x=tens((2, 300, 4, 64), BF16, strides=(300 * 512, 512, 128, 2),
                              ptr=c.x.data)) == 1
    assert "innermost" in detail(lib)
    # alignment of base pointer and of outer strides
    assert c.call(lib, x=tens((2, 300, 4, 64), BF16, ptr=c.x.data + 2)) == 3
    assert c.call(lib, x=tens((2, 300, 4, 64), BF16, strides=(300 * 4 * 68, 4 * 68, 68, 1),
                              ptr=c.x.data)) == 3
    assert "16 bytes" in detail(lib)
    # non-contiguous states
    assert c.call(lib, h0=tens((2, 4, 64, 128), F32, strides=(4 * 64 * 256, 64 * 256, 256, 1),
                               ptr=c.h0.data)) == 1
    # workspace
    assert c.call(lib, ws_bytes=1000) == 4 and "workspace" in detail(lib)
    assert c.call(lib, ws=None) == 4
    assert c.call(lib, ws=c.ws + 16) == 3
    # aliasing: y on top of x, final on top of initial_states
    assert c.call(lib, y=tens((2, 300, 4, 64), BF16, ptr=c.x.data)) == 1
    assert "overlaps" in detail(lib)
    assert c.call(lib, fin=tens((2, 4, 64, 128), F32, ptr=c.h0.data)) == 1
    # an empty batch is valid and launches nothing
    e = Case(B=0)
    assert e.call(lib) == 0 and detail(lib) == ""


def test_stage_error_paths(lib):
    c = Case()
    p = ctypes.pointer
    nc = -(-c.L // c.Q)
    G = tens((2, 4, nc * c.Q), F32, ptr=c.ws)
    assert lib.ssd_stage_chunk_cumsum(p(c.dt), p(c.A), 100, p(G), None) == 2
    badG = tens((2, 4, c.L), F32, ptr=c.ws)
    assert lib.ssd_stage_chunk_cumsum(p(c.dt), p(c.A), c.Q, p(badG), None) == 1
    S = tens((2, nc, 4, 64, 128), F32, ptr=c.ws + (1 << 30))
    assert lib.ssd_stage_chunk_state(p(c.x), p(c.Bm), p(c.dt), p(G), c.Q, 3, p(S), None) == 1
    badS = tens((2, nc + 1, 4, 64, 128), F32, ptr=c.ws + (1 << 30))
    assert lib.ssd_stage_chunk_state(p(c.x), p(c.Bm), p(c.dt), p(G), c.Q, 2, p(badS), None) == 1
    hp = tens((2, nc, 4, 64, 128), BF16, ptr=c.ws + (1 << 31))
    assert lib.ssd_stage_state_passing(p(S), p(G), p(c.h0), c.Q, p(hp), p(c.h0), None) == 1
    assert "overlaps" in detail(lib)
    hp32 = tens((2, nc, 4, 64, 128), F32, ptr=c.ws + (1 << 31))
    assert lib.ssd_stage_chunk_scan(p(c.x), p(c.dt), p(G), p(c.Bm), p(c.Cm), p(c.D), p(hp32),
                                    c.Q, 2, p(c.y), None) == 1
    assert "h_prev" in detail(lib)


def test_python_binding_rejects_cpu_tensors(lib):
    import torch
    from state_space_model_gb300 import ssd
    x = torch.zeros(1, 64, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        ssd.chunked_fwd(x, torch.zeros(1, 64, 2), torch.zeros(2), torch.zeros(1, 64, 1, 128),
                        torch.zeros(1, 64, 1, 128), chunk_size=64)


def test_state_update_error_paths(lib):
    """ssd_state_update's host checks (fake pointers, never dereferenced)."""
    p = ctypes.pointer
    Bn, H, P, N, G = 2, 4, 64, 128, 2
    base = FAKE + (1 << 33)
    state = tens((Bn, H, P, N), F32, ptr=base)
    x = tens((Bn, H, P), BF16, ptr=base + (1 << 24))
    dt = tens((Bn, H), F32, ptr=base + (2 << 24))
    A = tens((H,), F32, ptr=base + (3 << 24))
    Bm = tens((Bn, G, N), BF16, ptr=base + (4 << 24))
    Cm = tens((Bn, G, N), BF16, ptr=base + (5 << 24))
    out = tens((Bn, H, P), BF16, ptr=base + (6 << 24))

    def call(**kw):
        a = dict(state=state, x=x, dt=dt, A=A, Bm=Bm, Cm=Cm, D=None, z=None, dt_bias=None,
                 softplus=0, G=G, out=out)
        a.update(kw)
        q = lambda t: None if t is None else p(t)
        return lib.ssd_state_update(q(a["state"]), q(a["x"]), q(a["dt"]), q(a["A"]),
                                    q(a["Bm"]), q(a["Cm"]), q(a["D"]), q(a["z"]),
                                    q(a["dt_bias"]), a["softplus"], a["G"], q(a["out"]), None)

    assert call(state=None) == 1 and "state" in detail(lib)
    assert call(x=None) == 1 and "x" in detail(lib)
    assert call(G=3) == 1 and "ngroups" in detail(lib)
    assert call(state=tens((Bn, H, 48, N), F32, ptr=base)) == 2 and "headdim" in detail(lib)
    assert call(state=tens((Bn, H, P, 256), F32, ptr=base)) == 2 and "dstate" in detail(lib)
    # f32 and bf16 states pass the host checks; int32 does not
    assert call(state=tens((Bn, H, P, N), 2, ptr=base)) == 1 and "dtype" in detail(lib)
    assert call(dt=tens((Bn, H + 1), F32, ptr=dt.data)) == 1 and "shape" in detail(lib)
    assert call(Cm=tens((Bn, G, N), F32, ptr=Cm.data)) == 1
    # non-contiguous state, misaligned B
    assert call(state=tens((Bn, H, P, N), F32, strides=(H * P * 256, P * 256, 256, 1),
                           ptr=base)) == 1 and "contiguous" in detail(lib)
    assert call(Bm=tens((Bn, G, N), BF16, ptr=Bm.data + 2)) == 3
    # B and C with different strides
    assert call(Cm=tens((Bn, G, N), BF16, strides=(G * N * 2, N * 2, 1), ptr=Cm.data)) == 1
    assert "same strides" in detail(lib)
    # aliasing: out over x, state over B
    assert call(out=tens((Bn, H, P), BF16, ptr=x.data)) == 1 and "overlaps" in detail(lib)
    assert call(Bm=tens((Bn, G, N), BF16, ptr=base)) == 1 and "overlaps" in detail(lib)
    # optional tensors are checked when given
    assert call(z=tens((Bn, H, P + 1), BF16, ptr=base + (7 << 24))) == 1 and "z" in detail(lib)
    assert call(dt_bias=tens((H,), BF16, ptr=base + (8 << 24))) == 1
    # an empty batch is valid and launches nothing
    e0 = tens((0, H, P, N), F32, ptr=base)
    assert call(state=e0, x=tens((0, H, P), BF16, ptr=x.data), dt=tens((0, H), F32, ptr=dt.data),
                Bm=tens((0, G, N), BF16, ptr=Bm.data), Cm=tens((0, G, N), BF16, ptr=Cm.data),
                out=tens((0, H, P), BF16, ptr=out.data)) == 0


def test_state_update_tokens_error_paths(lib):
    """ssd_state_update_tokens' host checks (fake pointers, never dereferenced)."""
    p = ctypes.pointer
    I32 = 2
    Bn, T, H, P, N, G = 2, 3, 4, 64, 128, 2
    base = FAKE + (1 << 34)
    state = tens((Bn, H, P, N), F32, ptr=base)
    x = tens((Bn, T, H, P), BF16, ptr=base + (1 << 24))
    dt = tens((Bn, T, H), F32, ptr=base + (2 << 24))
    A = tens((H,), F32, ptr=base + (3 << 24))
    Bm = tens((Bn, T, G, N), BF16, ptr=base + (4 << 24))
    Cm = tens((Bn, T, G, N), BF16, ptr=base + (5 << 24))
    out = tens((Bn, T, H, P), BF16, ptr=base + (6 << 24))
    inter = tens((Bn, T, H, P, N), F32, ptr=base + (8 << 24))
    parent = tens((Bn, T), I32, ptr=base + (7 << 24))

    def call(**kw):
        a = dict(state=state, x=x, dt=dt, A=A, Bm=Bm, Cm=Cm, out=out, inter=inter, parent=parent,
                 slots=None, upd=1)
        a.update(kw)
        q = lambda t: None if t is None else p(t)
        return lib.ssd_state_update_tokens(q(a["state"]), q(a["x"]), q(a["dt"]), q(a["A"]),
                                           q(a["Bm"]), q(a["Cm"]), None, None, None, 0, G,
                                           q(a["out"]), q(a["inter"]), q(a["parent"]),
                                           q(a["slots"]), a["upd"], None)

    assert call(inter=None) == 1 and "parent needs intermediate_states" in detail(lib)
    assert call(parent=tens((Bn, T), F32, ptr=parent.data)) == 1 and "dtype" in detail(lib)
    assert call(x=tens((Bn, H, P), BF16, ptr=x.data)) == 1 and "ndim" in detail(lib)
    assert call(dt=tens((Bn, T + 1, H), F32, ptr=dt.data)) == 1 and "shape" in detail(lib)
    assert call(inter=tens((Bn, T, H, P, N), BF16, ptr=inter.data)) == 1
    # a bf16 state keeps its cache in bf16 too
    sb = tens((Bn, H, P, N), BF16, ptr=base)
    assert call(state=sb) == 1 and "intermediate_states: dtype f32, expected bf16" in detail(lib)
    assert call(state=tens((Bn, H, P, N), I32, ptr=base)) == 1 and "dtype" in detail(lib)
    assert call(inter=tens((Bn, T + 1, H, P, N), F32, ptr=inter.data)) == 1
    assert call(inter=tens((Bn, T, H, P, N), F32, ptr=inter.data + 4)) == 3
    assert call(inter=tens((Bn, T, H, P, N), F32, ptr=base)) == 1 and "overlaps" in detail(lib)
    # int32 is accepted only where it is asked for
    assert call(x=tens((Bn, T, H, P), I32, ptr=x.data)) == 1 and "dtype" in detail(lib)
    # a state pool of S slots needs state_indices [B] int32, the cache a pool too
    S = 5
    pool = tens((S, H, P, N), F32, ptr=base + (9 << 24))
    ipool = tens((S, T, H, P, N), F32, ptr=base + (10 << 24))
    slots = tens((Bn,), I32, ptr=base + (11 << 24))
    assert call(state=pool) == 1 and "state_indices" in detail(lib)
    assert call(state=pool, slots=slots) == 1 and "intermediate_states: shape[0]" in detail(lib)
    assert call(state=pool, inter=ipool, slots=tens((Bn,), F32, ptr=slots.data)) == 1 and \
        "state_indices: dtype" in detail(lib)
    assert call(state=pool, inter=ipool, slots=tens((Bn + 1,), I32, ptr=slots.data)) == 1 and \
        "state_indices: shape" in detail(lib)
    assert call(state=pool, inter=ipool, slots=tens((Bn,), I32, ptr=pool.data)) == 1 and \
        "overlaps" in detail(lib)
    # no parent and no cache is valid as far as the host checks go; T = 0 launches nothing
    e = lambda shape, dtype, t: tens(shape, dtype, ptr=t.data)
    assert call(x=e((Bn, 0, H, P), BF16, x), dt=e((Bn, 0, H), F32, dt),
                Bm=e((Bn, 0, G, N), BF16, Bm), Cm=e((Bn, 0, G, N), BF16, Cm),
                out=e((Bn, 0, H, P), BF16, out), inter=e((Bn, 0, H, P, N), F32, inter),
                parent=e((Bn, 0), I32, parent)) == 0
    assert call(state=pool, slots=slots, x=e((Bn, 0, H, P), BF16, x), dt=e((Bn, 0, H), F32, dt),
                Bm=e((Bn, 0, G, N), BF16, Bm), Cm=e((Bn, 0, G, N), BF16, Cm),
                out=e((Bn, 0, H, P), BF16, out), inter=e((S, 0, H, P, N), F32, inter),
                parent=e((Bn, 0), I32, parent)) == 0
    assert call(state=sb, x=e((Bn, 0, H, P), BF16, x), dt=e((Bn, 0, H), F32, dt),
                Bm=e((Bn, 0, G, N), BF16, Bm), Cm=e((Bn, 0, G, N), BF16, Cm),
                out=e((Bn, 0, H, P), BF16, out), inter=e((Bn, 0, H, P, N), BF16, inter),
                parent=e((Bn, 0), I32, parent)) == 0


def test_selftest_wait_limit_is_checked_on_the_host(lib):
    assert lib.ssd_selftest_wait_timeout(200_000_000, None) == 1
    assert "100 ms" in detail(lib)


def test_mixer_prologue_slot_checks(lib):
    """ssd_mixer_prologue's host checks for conv-state slots (fake pointers)."""
    p = ctypes.pointer
    I32 = 2
    Bn, L, H, P, G, N, W, S = 2, 8, 2, 64, 1, 128, 4, 5
    Dc = H * P + 2 * G * N
    base = FAKE + (1 << 35)
    xbc = tens((Bn, L, Dc), BF16, ptr=base)
    w = tens((Dc, W), F32, ptr=base + (1 << 24))
    dt = tens((Bn, L, H), F32, ptr=base + (2 << 24))
    x = tens((Bn, L, H, P), BF16, ptr=base + (3 << 24))
    Bm = tens((Bn, L, G, N), BF16, ptr=base + (4 << 24))
    Cm = tens((Bn, L, G, N), BF16, ptr=base + (5 << 24))
    dto = tens((Bn, L, H), F32, ptr=base + (6 << 24))
    pool = tens((S, Dc, W), BF16, ptr=base + (7 << 24))
    slots = tens((Bn,), I32, ptr=base + (8 << 24))

    def call(state=pool, idx=slots, windows=None):
        q = lambda t: None if t is None else p(t)
        return lib.ssd_mixer_prologue(p(xbc), p(w), None, q(state), q(windows), q(idx), p(dt),
                                      None, 1, G, p(x), p(Bm), p(Cm), p(dto), None)

    assert call(state=None) == 1 and "needs conv_state" in detail(lib)
    assert call(idx=None) == 1 and "conv_state: shape[0]" in detail(lib)   # a pool needs slots
    assert call(idx=tens((Bn,), F32, ptr=slots.data)) == 1 and "dtype" in detail(lib)
    assert call(idx=tens((Bn + 1,), I32, ptr=slots.data)) == 1 and "shape" in detail(lib)
    assert call(windows=tens((Bn, L, Dc, W), BF16, ptr=base + (9 << 24))) == 1 and \
        "conv_windows: shape[0]" in detail(lib)                             # windows: a pool too
    assert call(idx=tens((Bn,), I32, ptr=pool.data)) == 1 and "overlaps" in detail(lib)
