"""Vocabulary-parallel cross-entropy across processes (one GPU each).

"Distributed Training III: Model Parallelism" (CMU 11-868 Lecture 16 notes),
§5.5, and "LLM Internals" §7.3.4: card i holds the logits of its vocabulary
slice; it reduces them to three scalars per row (maximum, sum of exponentials,
target logit when it holds the target), the cards exchange those scalars, and
every card finishes the loss and computes its own slice's gradient locally.

Here each rank first folds its own shards' partials into one (max, sum exp)
pair per row, so the exchange is the pages' three scalars per token
whatever the number of local shards: one all-gather of the folded pairs (8
bytes per row and rank) and one all-reduce (sum) of the target logits (4
bytes per row, exact: one rank contributes per row).  The gathered pairs are
folded in rank order, so every rank computes the same logsumexp, loss and
n_valid; the backward then needs no communication.

The local steps run in the library's kernels (``vpce_partials``,
``vpce_fold_partials``, ``vpce_combine_partials``, ``vpce_backward``) through
:class:`CudaBackend`;
the collectives are ``torch.distributed`` (NCCL on GPUs).  A backend is any
object with the three methods below, which is how the orchestration is
exercised on CPU ranks.
"""
from __future__ import annotations

import ctypes

from . import vpce


class CudaBackend:
    """The library's kernels for the three local steps."""

    def partials(self, shards, vocab_start, targets, ignore_index, workspace, stream=None):
        import torch

        dtype, s, vs, ld = vpce._describe(shards, vocab_start)
        t = len(shards)
        part = torch.empty((t, s, 2), dtype=torch.float32, device=targets.device)
        tgt = torch.empty(s, dtype=torch.float32, device=targets.device)
        lib = vpce.load_library()
        code = int(lib.vpce_partials(ctypes.cast(vpce._ptr_array([sh.data_ptr() for sh in shards]), vpce._P),
                                     int(dtype), t, int(s), vpce._i64_array(vs), int(ld),
                                     ctypes.c_void_p(targets.data_ptr()), int(ignore_index),
                                     ctypes.c_void_p(part.data_ptr()), ctypes.c_void_p(tgt.data_ptr()),
                                     ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                                     vpce._stream_ptr(stream)))
        if code != vpce.VPCE_OK:
            raise vpce.VPCEError(code, "vpce_partials")
        return part, tgt

    def fold(self, part, stream=None):
        """[t, s, 2] partials -> [1, s, 2], shards folded in order."""
        import torch

        t, s = int(part.shape[0]), int(part.shape[1])
        out = torch.empty((1, s, 2), dtype=torch.float32, device=part.device)
        code = int(vpce.load_library().vpce_fold_partials(ctypes.c_void_p(part.data_ptr()), t, s,
                                                           ctypes.c_void_p(out.data_ptr()), vpce._stream_ptr(stream)))
        if code != vpce.VPCE_OK:
            raise vpce.VPCEError(code, "vpce_fold_partials")
        return out

    def combine(self, part, tgt, V, targets, ignore_index, reduction, t_local, workspace, stream=None):
        import torch

        s = tgt.numel()
        red = vpce.REDUCTIONS[reduction]
        loss = torch.empty((), dtype=torch.float32, device=tgt.device)
        row_loss = torch.empty(s, dtype=torch.float32, device=tgt.device)
        lib = vpce.load_library()
        code = int(lib.vpce_combine_partials(ctypes.c_void_p(part.data_ptr()), int(part.shape[0]),
                                             ctypes.c_void_p(tgt.data_ptr()), int(s), int(V),
                                             ctypes.c_void_p(targets.data_ptr()), int(ignore_index), int(red),
                                             ctypes.c_void_p(loss.data_ptr()), ctypes.c_void_p(row_loss.data_ptr()),
                                             int(t_local), ctypes.c_void_p(workspace.data_ptr()),
                                             workspace.numel(), vpce._stream_ptr(stream)))
        if code != vpce.VPCE_OK:
            raise vpce.VPCEError(code, "vpce_combine_partials")
        return (row_loss if reduction == "none" else loss), row_loss

    def backward(self, shards, vocab_start, targets, ignore_index, workspace, grad_output, stream=None):
        return vpce.vpce_backward(shards, targets, workspace, vocab_start, ignore_index=ignore_index,
                                  grad_output=grad_output, stream=stream)

    def new_workspace(self, t_local, s, device):
        return vpce.new_workspace(t_local, s, device)


def forward(shards, vocab_start, targets, V, *, group=None, ignore_index: int = -100, reduction: str = "mean",
            backend=None, workspace=None):
    """Loss of logits split over the ranks of ``group``.  ``shards`` are this
    rank's shards, ``vocab_start`` their t_local + 1 global column offsets,
    ``targets`` the whole batch's targets (replicated), ``V`` the whole
    vocabulary.  Every rank must hold the same number of shards and call this
    with the same ``targets``.  Returns ``(loss, row_loss, workspace)``;
    pass the workspace to :func:`backward`."""
    import torch
    import torch.distributed as dist

    be = backend or CudaBackend()
    t_local = len(shards)
    s = targets.numel()
    if workspace is None:
        workspace = be.new_workspace(t_local, s, targets.device)
    part, tgt = be.partials(shards, vocab_start, targets, ignore_index, workspace)
    # one (max, sum exp) pair per row for this rank's whole vocabulary slice
    mine = be.fold(part)
    world = dist.get_world_size(group)
    pieces = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(pieces, mine.contiguous(), group=group)
    # rank order: the combine folds rank 0's pair first, then rank 1's, ...
    gathered = torch.cat(pieces, dim=0)
    dist.all_reduce(tgt, op=dist.ReduceOp.SUM, group=group)
    loss, row_loss = be.combine(gathered, tgt, V, targets, ignore_index, reduction, t_local, workspace)
    return loss, row_loss, workspace


def backward(shards, vocab_start, targets, workspace, *, ignore_index: int = -100, grad_output: float = 1.0,
             backend=None):
    """dlogits of this rank's shards, in place (no communication: the
    workspace holds the global logsumexp and n_valid)."""
    be = backend or CudaBackend()
    return be.backward(shards, vocab_start, targets, ignore_index, workspace, grad_output)
