"""Row sharding of the cross-entropy across ranks (host-side logic).

Rows are independent (Liger-Kernel cross-entropy profile, §Tiling Strategy:
one program per row), so each rank runs ce_fwd on a contiguous block of
rows. Only the "mean" reduction couples the ranks, through its denominator
D = sum of w[t_i] over non-ignored rows:

* the loss: each rank reports its row-loss sum and its local D (the forward
  with reduction "sum" gives the first; `local_denominator` the second); one
  all-reduce of (loss sum, z-loss sum, correct count, D, valid count) gives
  the global mean;
* the gradient: a rank's forward with reduction "mean" scales its stored
  gradient by 1/D_local; calling ce_bwd with grad_output = D_local/D_global
  (times the upstream gradient) turns it into the global-mean gradient, so
  no collective is needed before the forward.

Or, with one exchange before the forward (`batch_counts`): every rank
counts its rows on the device (ce_count), one all-reduce of the two numbers
gives the batch's D and counted rows, and each rank's forward
(ce_fwd_shard) then scales its gradient by the batch's 1/D directly; the
ranks' loss outputs add up to the batch mean.
"""
from __future__ import annotations

import math


def shard_rows(rows: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous [start, stop) of `rows` for `rank` of `world`, sizes
    differing by at most one."""
    if world < 1 or not 0 <= rank < world or rows < 0:
        raise ValueError("bad shard request")
    base, extra = divmod(rows, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def local_denominator(target, ignore_index=-100, weight=None, V=None):
    """D_local and the valid-row count of one shard (host arrays or tensors;
    rows with an out-of-range target do not count)."""
    import numpy as np
    t = np.asarray(target).astype(np.int64).reshape(-1)
    valid = t != ignore_index
    if V is not None:
        valid &= (t >= 0) & (t < V)
    if weight is None:
        return float(valid.sum()), int(valid.sum())
    w = np.asarray(weight, dtype=np.float64)
    return float(w[t[valid]].sum()), int(valid.sum())


def reduce_mean(loss_sum, z_sum, n_correct, D_local, n_valid_local, group=None):
    """All-reduces the shard statistics and returns the global mean loss,
    mean z-loss, accuracy and D (NaN loss when no row counts anywhere)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([loss_sum, z_sum, n_correct, D_local, n_valid_local], dtype=torch.float64)
    if dist.is_available() and dist.is_initialized():
        if dist.get_backend(group) == "nccl":
            t = t.cuda()
        dist.all_reduce(t, group=group)
    L, Z, C, D, N = (float(v) for v in t.cpu())
    nan = float("nan")
    return {"loss": L / D if D else nan, "z_loss": Z / D if D else nan,
            "acc": C / N if N else nan, "D": D, "n_valid": N}


def mean_grad_factor(D_local: float, D_global: float) -> float:
    """grad_output for ce_bwd that turns a shard's local-mean gradient into
    the global-mean gradient (0 when the shard has no counted row: its
    gradient is all zeros anyway)."""
    if D_local == 0:
        return 0.0
    if D_global == 0 or math.isnan(D_global):
        raise ValueError("global denominator is zero while a shard has counted rows")
    return D_local / D_global


def batch_counts(target, V, weight=None, ignore_index=-100, group=None):
    """(D, counted rows) of the whole row-sharded batch on this rank's
    device: this rank's counts (ce_count) all-reduced over `group` (the
    rank's own counts when torch.distributed is not initialised). Pass the
    result to cross_entropy(..., batch_counts=...)."""
    import torch.distributed as dist

    from . import shard_counts
    counts = shard_counts(target, V, weight, ignore_index)
    if dist.is_available() and dist.is_initialized():
        if dist.get_backend(group) == "gloo":
            # a host-side exchange: the two doubles go through host memory
            host = counts.cpu()
            dist.all_reduce(host, group=group)
            counts.copy_(host)
        else:
            dist.all_reduce(counts, group=group)
    return counts
