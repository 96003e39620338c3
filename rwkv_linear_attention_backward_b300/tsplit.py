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
the tokens after its segment put on its end state, so the ranks run in
turn, last first: a rank receives that gradient from the next rank, runs
``backward_with_state`` from its start state, and sends the gradient of its
start state (3·B·C floats) to the previous rank; gw and gu are summed over
the ranks by an all-reduce.  Its gk, gv are exact; the ranks' backward
passes do not overlap.
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


def backward_tsplit(w, u, k, v, gy, start, *, group=None, ops=None):
    """Gradients of sum(gy * wkv) over the whole split sequence for this
    rank's segment: ``start`` is the state the segment started from
    (``forward_tsplit(..., want_start=True)``).  Returns (gw, gu) summed over
    all ranks, and this segment's (gk, gv), and the gradient of the state
    before the whole sequence as (g_num, g_den, pp) on rank 0 (None
    elsewhere)."""
    import torch.distributed as dist

    ops = _ops(ops)
    rank, world = dist.get_rank(group), dist.get_world_size(group)
    B, T, C = k.shape
    g_end = None
    if rank + 1 < world:
        g_end = torch.empty((3, B, C), dtype=start.dtype, device=start.device)
        dist.recv(g_end, src=_global(group, rank + 1), group=group)
    gw, gu, gk, gv, g_start = ops.backward_with_state(w, u, k, v, gy, start, g_end)
    if rank > 0:
        dist.send(g_start.contiguous(), dst=_global(group, rank - 1), group=group)
    dist.all_reduce(gw, group=group)
    dist.all_reduce(gu, group=group)
    return gw, gu, gk, gv, (g_start if rank == 0 else None)


def _global(group, r: int) -> int:
    import torch.distributed as dist

    return r if group is None else dist.get_global_rank(group, r)


def _ops(ops):
    if ops is None:
        from . import binding

        return binding
    return ops
