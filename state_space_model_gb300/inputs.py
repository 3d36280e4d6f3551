"""Seeded synthetic inputs for the Mamba-2 SSD forward.

This module holds no arithmetic of the method: it only draws inputs.  Both
the CUDA path (benchmark, GPU tests) and the fp64 oracle (tests) read the
same tensors from here.

Recipe (one generator per workload, seed ``20260 + k`` for workload k):
draw order x, B, C, dt_raw, logA_u, D, h0; every draw in fp32 on the CPU
with ``torch.Generator``, then cast to the storage dtype.

* x, B, C ~ N(0, 1); for the bf16 workloads B and C are scaled by
  1/sqrt(N) in fp32 before the cast to bf16.
* dt = softplus(N(mu, 0.5)) with mu = -2 (mu = -3 for the long-context
  workload, so that the decay spans many chunks); dt stays fp32.
* A = -exp(U(log 1, log 16)), one value per head, fp32.
* D ~ N(0, 1), one value per head, fp32.
* initial_states ~ N(0, 0.1^2) fp32 where the workload has them, else None.

Layouts (contiguous): x [B,L,H,P], dt [B,L,H], A [H], B/C [B,L,G,N], D [H],
initial_states [B,H,P,N].
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int      # P
    dstate: int       # N
    ngroups: int      # G
    chunk_size: int   # Q
    dtype: str        # storage dtype of x, B, C and y: "f32" or "bf16"
    dt_mu: float = -2.0
    init_states: bool = False
    scale_bc: bool = True
    seed: int = 0

    @property
    def tokens(self) -> int:
        return self.batch * self.seqlen

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads: tiny fp32 case, Mamba-2 130M and 2.7B layer shapes, a
# hybrid-model grouped shape (16 heads per group) and a long-context shape.
WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", 1, 256, 4, 16, 16, 1, 64, "f32",
                         scale_bc=False, seed=20261),
    "mamba2_130m": Workload("mamba2_130m", 4, 2048, 24, 64, 128, 1, 256, "bf16",
                            seed=20262),
    "mamba2_2p7b": Workload("mamba2_2p7b", 8, 4096, 80, 64, 128, 1, 256, "bf16",
                            seed=20263),
    "hybrid_g8": Workload("hybrid_g8", 1, 16384, 128, 64, 128, 8, 128, "bf16",
                          init_states=True, seed=20264),
    "long_64k": Workload("long_64k", 2, 65536, 64, 64, 128, 1, 256, "bf16",
                         dt_mu=-3.0, init_states=True, seed=20265),
}
HEADLINE = "mamba2_2p7b"


def make_inputs(w: Workload, seed: int | None = None) -> dict:
    """Draw one workload's inputs on the CPU.  Returns a dict with keys
    x, dt, A, B, C, D, initial_states (the last may be None)."""
    g = torch.Generator().manual_seed(w.seed if seed is None else seed)
    Bn, L, H, P, N, G = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups
    f32 = torch.float32
    x = torch.randn((Bn, L, H, P), generator=g, dtype=f32)
    Bm = torch.randn((Bn, L, G, N), generator=g, dtype=f32)
    Cm = torch.randn((Bn, L, G, N), generator=g, dtype=f32)
    dt_raw = torch.randn((Bn, L, H), generator=g, dtype=f32) * 0.5 + w.dt_mu
    logA_u = torch.rand((H,), generator=g, dtype=f32) * math.log(16.0)
    D = torch.randn((H,), generator=g, dtype=f32)
    h0 = (torch.randn((Bn, H, P, N), generator=g, dtype=f32) * 0.1
          if w.init_states else None)
    if w.dtype == "bf16" and w.scale_bc:
        Bm = Bm * (1.0 / math.sqrt(N))
        Cm = Cm * (1.0 / math.sqrt(N))
    dt = torch.nn.functional.softplus(dt_raw)
    A = -torch.exp(logA_u)
    st = w.torch_dtype
    return {"x": x.to(st), "dt": dt, "A": A, "B": Bm.to(st), "C": Cm.to(st),
            "D": D, "initial_states": h0}


def small_case(dtype="bf16", batch=2, seqlen=600, nheads=4, headdim=64,
               dstate=128, ngroups=2, chunk_size=128, init_states=True,
               dt_mu=-2.0, seed=1234) -> Workload:
    """A parity-test workload that spans several chunks and tiles and ends in
    a ragged partial chunk (seqlen not a multiple of chunk_size)."""
    return Workload(f"small_{dtype}", batch, seqlen, nheads, headdim, dstate,
                    ngroups, chunk_size, dtype, dt_mu=dt_mu,
                    init_states=init_states, scale_bc=(dtype == "bf16"),
                    seed=seed)


# Decode-step (selective state update) workload: one token per sequence for
# a batch of sequences at the Nemotron hybrid layer shape (H = 128, P = 64,
# N = 128, G = 8), the carried state drawn like the prefill's initial state.
SSU_SHAPE = {"batch": 64, "nheads": 128, "headdim": 64, "dstate": 128, "ngroups": 8}


def make_ssu_inputs(batch, nheads, headdim, dstate, ngroups, seed=20270, gated=True,
                    tokens=None):
    """Draw decode-step inputs on the CPU: state [B,H,P,N] f32, x and z
    [B,H,P] bf16, raw dt [B,H] (softplus is applied by the step, after
    dt_bias), dt_bias, A, D [H] f32, B and C [B,G,N] bf16 scaled by 1/sqrt(N).
    With ``tokens`` = T the per-token tensors get a token axis after the batch
    ([B,T,H,P], [B,T,H], [B,T,G,N])."""
    g = torch.Generator().manual_seed(seed)
    f32 = torch.float32
    Bn, H, P, N, G = batch, nheads, headdim, dstate, ngroups
    tk = () if tokens is None else (tokens,)
    state = torch.randn((Bn, H, P, N), generator=g, dtype=f32) * 0.1
    x = torch.randn((Bn,) + tk + (H, P), generator=g, dtype=f32)
    Bm = torch.randn((Bn,) + tk + (G, N), generator=g, dtype=f32) * (1.0 / math.sqrt(N))
    Cm = torch.randn((Bn,) + tk + (G, N), generator=g, dtype=f32) * (1.0 / math.sqrt(N))
    dt_raw = torch.randn((Bn,) + tk + (H,), generator=g, dtype=f32) * 0.5 - 2.0
    dt_bias = torch.randn((H,), generator=g, dtype=f32) * 0.1
    A = -torch.exp(torch.rand((H,), generator=g, dtype=f32) * math.log(16.0))
    D = torch.randn((H,), generator=g, dtype=f32)
    z = torch.randn((Bn,) + tk + (H, P), generator=g, dtype=f32) if gated else None
    bf = torch.bfloat16
    return {"state": state, "x": x.to(bf), "dt": dt_raw, "dt_bias": dt_bias, "A": A,
            "B": Bm.to(bf), "C": Cm.to(bf), "D": D, "z": None if z is None else z.to(bf)}


def make_prologue_inputs(batch, seqlen, nheads, headdim, ngroups, dstate, width=4, seed=20280):
    """Draw the mixer prologue's inputs on the CPU: xBC [B, L, H P + 2 G N]
    ~ N(0, 1) bf16, conv weight [Dc, W] ~ N(0, 1/W) and bias [Dc] ~ N(0, 0.1^2)
    f32, conv state [B, Dc, W] ~ N(0, 1) bf16, raw dt [B, L, H] ~ N(-2, 0.5)
    and dt_bias [H] ~ N(0, 0.1^2) f32."""
    g = torch.Generator().manual_seed(seed)
    f32, bf = torch.float32, torch.bfloat16
    Dc = nheads * headdim + 2 * ngroups * dstate
    xBC = torch.randn((batch, seqlen, Dc), generator=g, dtype=f32).to(bf)
    w = torch.randn((Dc, width), generator=g, dtype=f32) / math.sqrt(width)
    b = torch.randn((Dc,), generator=g, dtype=f32) * 0.1
    st = torch.randn((batch, Dc, width), generator=g, dtype=f32).to(bf)
    dt = torch.randn((batch, seqlen, nheads), generator=g, dtype=f32) * 0.5 - 2.0
    dt_bias = torch.randn((nheads,), generator=g, dtype=f32) * 0.1
    return {"xBC": xBC, "conv_weight": w, "conv_bias": b, "conv_state": st, "dt": dt,
            "dt_bias": dt_bias}
