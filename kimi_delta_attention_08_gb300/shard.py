"""Forward of sequences sharded along the token axis over ranks, with the
intracard segment scan nested inside each rank.

Kimi's context parallelism gives each rank one shard of a sequence, and the
intracard split assumes a whole sequence; nesting the two is named on the cuLA
FlashKDA pull request ("feat(kda): SM90 FlashKDA prefill, intracard CP, and
backend dispatch", review thread on Kimi CP) as something that should work but
was not built.  Here rank r of W holds tokens [t_r, t_{r+1}) of every sequence
of a batch (the same B, H and head layout on every rank, shards in rank order):

  1. piece    rank 0 runs its shard from the true initial state (outputs and its
              final state S_1, with the segment scan inside as kda_fwd plans it);
              its piece is (M_0, B_0) = (0, S_1).  Rank r > 0 computes the affine
              form of its shard, S_end = M_r S_start + B_r (kda_fwd_transition).
  2. exchange an all-gather of the pieces (2 x 64 KB fp32 per (sequence, head)
              per rank), ordered by rank.
  3. finish   rank r > 0 composes S_r = M_{r-1}(... (M_0 S_0 + B_0) ...) + B_{r-1}
              in rank order (kda_compose_states) and reruns its shard from S_r
              (kda_fwd, segment scan inside); the last rank's final state is the
              sequence's.

Every arithmetic step runs in the library's kernels; this module only moves
pieces between ranks (torch.distributed: NCCL between GPUs, gloo on CPU) and
orders the calls.  The phases are separate functions so that shards can also
be run one after another in one process with the pieces passed by hand.
States are fp32 on this path (the start states handed between ranks are).
"""
from __future__ import annotations

from . import kda_compose_states, kda_fwd, kda_fwd_transition, make_workspace


def _check_fp32_state(t, name):
    import torch
    if t is not None and t.dtype != torch.float32:
        raise TypeError(f"{name}: the sharded forward keeps fp32 states (got {t.dtype})")


def shard_piece(rank, q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound,
                initial_state=None, workspace=None, *, stream=None):
    """Phase 1 on rank `rank`: its piece, float32 [2, N, HV, 128, 128] = (M_r, B_r).
    Rank 0 also writes its outputs into `out`."""
    import torch
    _check_fp32_state(initial_state, "initial_state")
    B, T, HV = v.shape[0], v.shape[1], v.shape[2]
    dev = v.device
    if workspace is None:
        workspace = make_workspace(B * T, HV, dev)
    piece = torch.zeros((2, B, HV, 128, 128), dtype=torch.float32, device=dev)
    if rank == 0:
        kda_fwd(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state,
                piece[1], None, workspace, stream=stream)
    else:
        kda_fwd_transition(q, k, v, g, beta, A_log, dt_bias, lower_bound, piece[0], piece[1],
                           None, workspace, stream=stream)
    return piece


def exchange(piece, group=None):
    """Phase 2: every rank's piece, stacked in rank order [W, *piece.shape]."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    parts = [torch.empty_like(piece) for _ in range(world)]
    dist.all_gather(parts, piece.contiguous(), group=group)
    return torch.stack(parts)


def shard_finish(rank, pieces, q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound,
                 final_state=None, workspace=None, *, stream=None):
    """Phase 3 on rank `rank` > 0: compose its start state from the pieces of the
    ranks before it and rerun its shard, writing `out` and (if given) its final
    state.  On rank 0 only the final state is copied out of its piece."""
    import torch
    _check_fp32_state(final_state, "final_state")
    B, T, HV = v.shape[0], v.shape[1], v.shape[2]
    if rank == 0:
        if final_state is not None:
            final_state.copy_(pieces[0, 1])
        return
    dev = v.device
    start = torch.empty((B, HV, 128, 128), dtype=torch.float32, device=dev)
    M = pieces[:rank, 0].contiguous()
    Bo = pieces[:rank, 1].contiguous()
    kda_compose_states(M, Bo, start, None, stream=stream)
    if workspace is None:
        workspace = make_workspace(B * T, HV, dev)
    kda_fwd(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, start, final_state, None,
            workspace, stream=stream)


def fwd_sequence_shard(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound,
                       initial_state=None, final_state=None, group=None, *, stream=None):
    """The whole sharded forward on this rank (torch.distributed initialised):
    `initial_state` is read on rank 0 only, `final_state` is the sequence's final
    state on the last rank (the state at the end of this rank's shard elsewhere)."""
    import torch.distributed as dist
    rank = dist.get_rank(group)
    piece = shard_piece(rank, q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound,
                        initial_state if rank == 0 else None, stream=stream)
    pieces = exchange(piece, group)
    shard_finish(rank, pieces, q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound,
                 final_state, stream=stream)
