"""Sequence sharding of the SSD forward over ranks (one contiguous segment of
the sequence per rank, rank order = sequence order).

The recurrence over a run of tokens composes into one (decay, state) pair and
pairs compose associatively in sequence order ("mamba-metal", "The essence of
selective scan"), so the only exchange between ranks is one all-gather of
each rank's pair, B*H*P*N + B*H floats:

1. local pass: the forward on the rank's segment from a zero state
   (``ssd_chunked_fwd``) gives y from zero and the segment's state b;
   ``ssd_segment_logdecay`` gives log a = A * sum(dt);
2. exchange: every rank gathers all ranks' (log a, b);
3. finish: ``ssd_sequence_combine`` folds the pairs of the earlier ranks into
   the state entering this rank's segment (starting from the sequence's
   initial state), and ``ssd_shard_correct`` adds that state's contribution
   to y and makes b the rank's final state.

Every step of the arithmetic runs in the library's kernels; this module only
sequences the calls and the exchange (torch.distributed: NCCL between GPUs,
gloo on CPU).  The compute steps are taken from an ``ops`` object (the
library by default) so that the host logic can be exercised on CPU ranks.
"""
from __future__ import annotations

import torch

from . import _native
from . import ssd as _ssd


class LibraryOps:
    """The compute steps, through the C ABI (tensors on the current device)."""

    def forward(self, x, dt, A, B, C, D, chunk_size, ngroups):
        return _ssd.chunked_fwd(x, dt, A, B, C, D, None, chunk_size, ngroups)

    def logdecay(self, dt, A):
        out = torch.empty(dt.shape[0], dt.shape[2], dtype=torch.float32, device=dt.device)
        dev = _ssd._device_of(dt, A, out)
        _native.check(_native.load().ssd_segment_logdecay(_ssd._desc(dt), _ssd._desc(A),
                                                          _ssd._desc(out), _ssd._stream(dev)),
                      "ssd_segment_logdecay")
        return out

    def combine(self, logdecay_all, states_all, initial_states, rank):
        h_in = torch.empty(states_all.shape[1:], dtype=torch.float32, device=states_all.device)
        dev = _ssd._device_of(logdecay_all, states_all, initial_states, h_in)
        _native.check(_native.load().ssd_sequence_combine(
            _ssd._desc(logdecay_all), _ssd._desc(states_all), _ssd._desc(initial_states),
            int(rank), _ssd._desc(h_in), _ssd._stream(dev)), "ssd_sequence_combine")
        return h_in

    def correct(self, dt, A, C, h_in, logdecay, ngroups, y, final_states):
        dev = _ssd._device_of(dt, A, C, h_in, logdecay, y, final_states)
        _native.check(_native.load().ssd_shard_correct(
            _ssd._desc(dt), _ssd._desc(A), _ssd._desc(C), _ssd._desc(h_in), _ssd._desc(logdecay),
            int(ngroups), _ssd._desc(y), _ssd._desc(final_states), _ssd._stream(dev)),
            "ssd_shard_correct")


def local_pass(x, dt, A, B, C, D=None, chunk_size=256, ngroups=1, ops=None):
    """Step 1 on one rank: ``(y, state, logdecay)`` of its segment from a zero state."""
    ops = ops or LibraryOps()
    y, state = ops.forward(x, dt, A, B, C, D, chunk_size, ngroups)
    return y, state, ops.logdecay(dt, A)


def finish(rank, y, state, logdecay, logdecay_all, states_all, dt, A, C, initial_states=None,
           ngroups=1, ops=None):
    """Step 3 on one rank, given every rank's pair (stacked in rank order):
    corrects ``y`` in place and returns the rank's final state (``state``,
    updated in place)."""
    ops = ops or LibraryOps()
    if rank == 0 and initial_states is None:
        return state   # nothing enters the first segment
    h_in = ops.combine(logdecay_all, states_all, initial_states, rank)
    ops.correct(dt, A, C, h_in, logdecay, ngroups, y, state)
    return state


def chunked_fwd_sequence_sharded(x, dt, A, B, C, D=None, initial_states=None, chunk_size=256,
                                 ngroups=1, *, group=None, ops=None):
    """The forward of the whole sequence, this rank holding its segment of
    x, dt, B, C (the same batch and heads on every rank; initial_states, if
    any, is the state entering the whole sequence and is passed on every
    rank).  Returns this rank's ``(y, final_state)``: y of its segment, and
    the state at the end of its segment (the last rank's is the sequence's
    final state).  Collective over ``group``."""
    import torch.distributed as dist
    rank = dist.get_rank(group)
    world = dist.get_world_size(group)
    y, state, ld = local_pass(x, dt, A, B, C, D, chunk_size, ngroups, ops)
    ld_all = [torch.empty_like(ld) for _ in range(world)]
    st_all = [torch.empty_like(state) for _ in range(world)]
    dist.all_gather(ld_all, ld.contiguous(), group=group)
    dist.all_gather(st_all, state.contiguous(), group=group)
    state = finish(rank, y, state, ld, torch.stack(ld_all), torch.stack(st_all), dt, A, C,
                   initial_states, ngroups, ops)
    return y, state
