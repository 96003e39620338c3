"""One long sequence split over the ranks of a process group along time:
the forward pass, and its backward pass.

Rank r holds tokens [t_r, t_r + T_r) of every batch row, the ranks in
order.  The decay does not depend on the data, so a segment acts on the
carried state by decaying it by its length and adding its own sums
(``wkv_state_fold``).  Per rank, with every step in libwkv.so's kernels and
torch.distributed moving 3·B·C floats per rank once:

1. its segment's own state from the empty state (``forward_with_state``
   without outputs);
2. an all-gather of every segment's state and length;
3. the state its segment starts from: the fold of the segments before it,
   after the sequence's given state if any (``state_fold``);
4. its outputs from that state (``forward_with_state``).

Each rank reads its k, v twice.

The backward pass (``backward_tsplit``) needs, per rank, the gradient that
the tokens after its segment put on its end state.  Through tokens whose
outputs carry no gradient that gradient only decays (la <- e^{-w} la, lb
alike), so it is folded from the later segments' own start-state gradients
the way states are folded forwards, and the ranks' backward passes run at
the same time.  Per rank:

5. its segment's start-state gradient from its own gy alone (the summary
   pass of ``backward_with_state``: reads k, v, gy once, writes 3·B·C
   floats);
6. an all-gather of those gradients (3·B·C floats per rank);
7. its end gradient: the fold of the later segments' gradients, after the
   gradient given on the sequence's end state if any (``adjoint_fold``);
8. its full backward pass from its start state with that end gradient;
   gw and gu summed over the ranks by an all-reduce.

Each rank reads its k, v, gy twice in the backward pass too; nothing waits
on another rank's backward pass.
"""
from __future__ import annotations

import torch


def segment_state(w, u, k, v, *, ops=None):
    """Step 1: the state [3, B, C] after this segment, from the empty state."""
    ops = _ops(ops)
    return ops.forward_with_state(w, u, k, v, want_y=False)[1]


def start_state(w, states, lengths, rank: int, state_in=None, *, ops=None):
    """Step 3: the state segment ``rank`` starts from.  ``states`` [world, 3,
    B, C] and ``lengths`` [world] are every segment's own state and tokens;
    ``state_in`` [3, B, C] the state before the whole sequence (None: empty)."""
    ops = _ops(ops)
    lengths = [int(x) for x in lengths]
    if state_in is None:
        return ops.state_fold(w, states[:rank], lengths[:rank])
    head = torch.empty((rank + 1,) + tuple(states.shape[1:]), dtype=states.dtype, device=states.device)
    head[0].copy_(state_in)
    head[1:].copy_(states[:rank])
    return ops.state_fold(w, head, [0] + lengths[:rank])


def forward_tsplit(w, u, k, v, state_in=None, *, group=None, ops=None, want_start: bool = False):
    """wkv of this rank's segment k, v [B, T_r, C] of a sequence split over
    the ranks of ``group`` in rank order (``state_in``, the same on every
    rank: the state before the sequence).  Returns (y [B, T_r, C], the state
    after this rank's segment [3, B, C]): the last rank's is the state after
    the whole sequence; with ``want_start`` also the state the segment
    started from (what ``backward_tsplit`` takes).  ``ops``: the compute
    entry points (default: this package's CUDA binding)."""
    import torch.distributed as dist

    ops = _ops(ops)
    rank, world = dist.get_rank(group), dist.get_world_size(group)
    B, T, C = k.shape
    own = segment_state(w, u, k, v, ops=ops)
    states = torch.empty((world,) + tuple(own.shape), dtype=own.dtype, device=own.device)
    dist.all_gather(list(states.unbind(0)), own.contiguous(), group=group)
    lens = torch.empty((world, 1), dtype=torch.int64, device=own.device)
    dist.all_gather(list(lens.unbind(0)), torch.full((1,), T, dtype=torch.int64, device=own.device), group=group)
    start = start_state(w, states, lens.flatten().tolist(), rank, state_in, ops=ops)
    y, end = ops.forward_with_state(w, u, k, v, state_in=start)
    return (y, end, start) if want_start else (y, end)


def end_gradient(w, starts_grads, lengths, rank: int, gstate_end=None, *, ops=None):
    """Step 7: the gradient on segment ``rank``'s end state, [3, B, C] planes
    (g_num, g_den, pp), or None when there is none.  ``starts_grads`` [world,
    3, B, C] and ``lengths`` [world] are every segment's own start-state
    gradient and tokens; ``gstate_end`` the gradient given on the whole
    sequence's end state (None: none)."""
    ops = _ops(ops)
    lengths = [int(x) for x in lengths]
    later = starts_grads[rank + 1:]
    if later.shape[0] == 0:
        return gstate_end
    return ops.adjoint_fold(w, later.contiguous(), lengths[rank + 1:], gstate_end)


def backward_tsplit(w, u, k, v, gy, start, gstate_end=None, *, group=None, ops=None):
    """Gradients of sum(gy * wkv) over the whole split sequence for this
    rank's segment: ``start`` is the state the segment started from
    (``forward_tsplit(..., want_start=True)``), ``gstate_end`` (the same on
    every rank) the gradient on the state after the whole sequence, as
    (g_num, g_den, pp) planes (None: none).  Returns (gw, gu) summed over all
    ranks, and this segment's (gk, gv), and the gradient of the state before
    the whole sequence as (g_num, g_den, pp) on rank 0 (None elsewhere)."""
    import torch.distributed as dist

    ops = _ops(ops)
    rank, world = dist.get_rank(group), dist.get_world_size(group)
    B, T, C = k.shape
    own = ops.backward_with_state(w, u, k, v, gy, start, None, summary=True)[4]
    grads = torch.empty((world,) + tuple(own.shape), dtype=own.dtype, device=own.device)
    dist.all_gather(list(grads.unbind(0)), own.contiguous(), group=group)
    lens = torch.empty((world, 1), dtype=torch.int64, device=own.device)
    dist.all_gather(list(lens.unbind(0)), torch.full((1,), T, dtype=torch.int64, device=own.device), group=group)
    g_end = end_gradient(w, grads, lens.flatten().tolist(), rank, gstate_end, ops=ops)
    gw, gu, gk, gv, g_start = ops.backward_with_state(w, u, k, v, gy, start, g_end)
    dist.all_reduce(gw, group=group)
    dist.all_reduce(gu, group=group)
    return gw, gu, gk, gv, (g_start if rank == 0 else None)


def _ops(ops):
    if ops is None:
        from . import binding

        return binding
    return ops
