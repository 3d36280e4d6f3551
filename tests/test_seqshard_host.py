"""Sequence sharding over ranks: the host logic on CPU ranks with gloo.

``chunked_fwd_sequence_sharded`` runs each rank's segment from a zero state,
all-gathers the (log decay, state) pairs and finishes with the combine and
the correction.  On GPUs the compute steps are the library's kernels; here,
on CPU ranks, they are stand-ins built from the fp64 oracle, so what is
tested is the sequencing and the exchange: who sends what, in which order,
and that the pieces reassemble the whole sequence.  The stand-ins use the
oracle's recurrence only: a segment from zero for the local pass, and the
recurrence with zero input started from the entering state for the
correction (what the entering state contributes to y and to the final
state), so the arithmetic is the definition's.  The result is compared with
the oracle's recurrence over the whole sequence.
"""
from __future__ import annotations

import os
import socket
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


class OracleOps:
    """The four compute steps on CPU, from the oracle (fp64)."""

    def forward(self, x, dt, A, B, C, D, chunk_size, ngroups):
        from oracle import oracle as orc
        y, f = orc.recurrence(x, dt, A, B, C, D, None, ngroups=ngroups)
        return torch.from_numpy(y), torch.from_numpy(f)

    def logdecay(self, dt, A):
        return A.double()[None, :] * dt.double().sum(dim=1)

    def combine(self, logdecay_all, states_all, initial_states, rank):
        h = (initial_states.double().clone() if initial_states is not None
             else torch.zeros_like(states_all[0]))
        for q in range(rank):
            h = torch.exp(logdecay_all[q])[:, :, None, None] * h + states_all[q]
        return h

    def correct(self, dt, A, C, h_in, logdecay, ngroups, y, final_states):
        from oracle import oracle as orc
        Bn, L, H = dt.shape
        P = y.shape[-1]
        zero_x = torch.zeros(Bn, L, H, P, dtype=torch.float64)
        yc, fc = orc.recurrence(zero_x, dt, A, C, C, None, h_in, ngroups=ngroups)
        y += torch.from_numpy(yc)
        final_states += torch.from_numpy(fc)


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _case():
    from state_space_model_gb300 import inputs as gen
    w = gen.small_case("f32", batch=2, seqlen=700, nheads=4, headdim=16, dstate=32, ngroups=2,
                       chunk_size=64, init_states=True, seed=515)
    return w, gen.make_inputs(w)


def _bounds(L, world):
    # uneven segments, none a multiple of the chunk
    cuts = [0] + [int(L * (r + 1) / world) - 3 * r for r in range(world - 1)] + [L]
    return cuts


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    from state_space_model_gb300 import seqshard
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, inp = _case()
        cuts = _bounds(w.seqlen, world)
        lo, hi = cuts[rank], cuts[rank + 1]
        seg = {k: inp[k][:, lo:hi].contiguous() for k in ("x", "dt", "B", "C")}
        y, f = seqshard.chunked_fwd_sequence_sharded(
            seg["x"], seg["dt"], inp["A"], seg["B"], seg["C"], inp["D"],
            inp["initial_states"], w.chunk_size, w.ngroups, ops=OracleOps())
        q.put((rank, y.numpy(), f.numpy()))
    finally:
        dist.destroy_process_group()


def _run(world):
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    try:
        got = sorted((q.get(timeout=300) for _ in procs), key=lambda g: g[0])
    finally:
        for p in procs:
            p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    return got


def _check(got):
    from oracle import oracle as orc
    w, inp = _case()
    yr, fr = orc.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                            inp["initial_states"], ngroups=w.ngroups)
    y = np.concatenate([g[1] for g in got], axis=1)
    assert y.shape == yr.shape
    assert np.max(np.abs(y - yr)) / np.max(np.abs(yr)) < 1e-10
    # each rank ends with the state at the end of its segment
    cuts = _bounds(w.seqlen, len(got))
    for rank, _, f in got:
        end = cuts[rank + 1]
        _, fe = orc.recurrence(inp["x"][:, :end], inp["dt"][:, :end], inp["A"],
                               inp["B"][:, :end], inp["C"][:, :end], inp["D"],
                               inp["initial_states"], ngroups=w.ngroups)
        assert np.max(np.abs(f - fe)) / np.max(np.abs(fe)) < 1e-10, rank
    assert np.max(np.abs(got[-1][2] - fr)) / np.max(np.abs(fr)) < 1e-10


def test_two_ranks_reassemble_the_sequence_gloo():
    _check(_run(2))


def test_three_ranks_reassemble_the_sequence_gloo():
    _check(_run(3))


def test_first_rank_without_initial_state_needs_no_correction():
    from state_space_model_gb300 import seqshard

    class Counting(OracleOps):
        calls = 0

        def combine(self, *a):
            Counting.calls += 1
            return super().combine(*a)

    w, inp = _case()
    seg = {k: inp[k][:, :200].contiguous() for k in ("x", "dt", "B", "C")}
    ops = Counting()
    y, st, ld = seqshard.local_pass(seg["x"], seg["dt"], inp["A"], seg["B"], seg["C"], inp["D"],
                                    w.chunk_size, w.ngroups, ops)
    f = seqshard.finish(0, y, st, ld, ld[None], st[None], seg["dt"], inp["A"], seg["C"], None,
                        w.ngroups, ops)
    assert Counting.calls == 0 and f is st
