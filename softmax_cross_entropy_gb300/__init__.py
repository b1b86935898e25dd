"""GB300-native fused softmax cross-entropy (forward + in-forward gradient).

    loss = cross_entropy(logits, target, weight=None, ignore_index=-100,
                         lse_square_scale=0.0, label_smoothing=0.0,
                         reduction="mean", softcap=None, return_z_loss=False,
                         return_token_accuracy=False,
                         return_predicted_tokens=False)

The arguments and outputs are those of the Liger-Kernel cross-entropy kernel
profile (§Forward Pass, §Module Parameters). ``logits`` is a 2-D (B*T, V)
CUDA tensor in float32, bfloat16 or float16, or an N-D (N, C, d1, ..., dk)
tensor with the class dimension at axis 1 (F.cross_entropy's N-D form; the
reductions then run over every non-class dimension); ``target`` holds int32
or int64 labels, shaped (B*T,) or (N, d1, ..., dk).
When ``logits.requires_grad`` the forward writes the gradient of the reduced
loss over ``logits`` itself (§Backward Pass: the gradient-in-forward trick),
so the logits' values are gone after the call and backward only scales that
buffer by grad_output. Every step runs in the CUDA kernels of libgbce.so
(see include/gbce.h); PyTorch supplies device memory, streams and autograd.
"""
from __future__ import annotations

import math
from collections import namedtuple

import torch

from . import _lib
from ._lib import (CEError, ce_bwd, ce_bwd_nd, ce_count, ce_device_status, ce_fwd,
                   ce_fwd_nd, ce_fwd_shard, ce_last_error, ce_status_string)

__all__ = ["cross_entropy", "CrossEntropyLoss", "CrossEntropyFunction", "CrossEntropyOutput",
           "CEError", "device_status", "shard_counts", "ce_fwd", "ce_fwd_shard", "ce_count",
           "ce_bwd", "ce_fwd_nd", "ce_bwd_nd", "ce_device_status", "ce_status_string",
           "ce_last_error"]

CrossEntropyOutput = namedtuple("CrossEntropyOutput",
                                ["loss", "z_loss", "token_accuracy", "predicted_tokens"])

_REDUCTIONS = {"none": _lib.CE_RED_NONE, "sum": _lib.CE_RED_SUM, "mean": _lib.CE_RED_MEAN}
_DTYPES = {torch.float32: _lib.CE_F32, torch.bfloat16: _lib.CE_BF16,
           torch.float16: _lib.CE_F16}


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(device):
    return torch.cuda.current_stream(device).cuda_stream


def _check_inputs(logits, target, weight):
    if not isinstance(logits, torch.Tensor) or logits.dim() < 2:
        raise ValueError("logits must be 2-D (B*T, V) or N-D (N, C, d1, ..., dk) with the "
                         "class dimension at axis 1")
    if not logits.is_cuda:
        raise ValueError("logits must be a CUDA tensor")
    if logits.dtype not in _DTYPES:
        raise TypeError(f"logits dtype {logits.dtype} is not supported "
                        "(float32, bfloat16, float16)")
    want = (logits.shape[0],) + tuple(logits.shape[2:])
    if tuple(target.shape) != want:
        raise ValueError(f"target must have shape {want}: one label per position of logits")
    if target.dtype not in (torch.int32, torch.int64):
        raise TypeError("target must be int32 or int64")
    if target.device != logits.device:
        raise ValueError("target must be on the logits' device")
    if weight is not None:
        if weight.dim() != 1 or weight.shape[0] != logits.shape[1]:
            raise ValueError("weight must have shape (V,)")
        if weight.device != logits.device:
            raise ValueError("weight must be on the logits' device")


def _forward(logits, target, weight, ignore_index, lse_square_scale, label_smoothing,
             reduction, softcap, want_grad, want_z, want_acc, want_pred, batch_counts=None):
    """Runs ce_fwd (ce_fwd_shard with batch_counts; ce_fwd_nd for N-D
    logits); returns (loss, z_loss, acc, pred). Writes dlogits over logits
    when want_grad."""
    nd = logits.dim() > 2
    dev = logits.device
    red = _REDUCTIONS[reduction]
    pos_shape = tuple(target.shape)  # (rows,) or (N, d1, ..., dk)
    out_shape = pos_shape if red == _lib.CE_RED_NONE else ()
    f32 = dict(dtype=torch.float32, device=dev)
    loss = torch.empty(out_shape, **f32)
    z_loss = torch.empty(out_shape, **f32) if want_z else None
    acc = torch.empty(out_shape, **f32) if want_acc else None
    pred = torch.empty(pos_shape, dtype=torch.int64, device=dev) if want_pred else None
    flags = ((_lib.CE_FLAG_GRAD if want_grad else 0) | (_lib.CE_FLAG_Z_LOSS if want_z else 0) |
             (_lib.CE_FLAG_ACC if want_acc else 0) | (_lib.CE_FLAG_PRED if want_pred else 0) |
             (_lib.CE_FLAG_TARGET_I64 if target.dtype == torch.int64 else 0))
    w = None if weight is None else weight.to(torch.float32).contiguous()
    opts = (_ptr(target), _ptr(w), int(ignore_index), float(label_smoothing),
            float(lse_square_scale), float(softcap) if softcap is not None else 0.0, red, flags,
            _ptr(loss), _ptr(z_loss), _ptr(acc), _ptr(pred))
    with torch.cuda.device(dev):
        if nd:
            if batch_counts is not None:
                raise ValueError("batch_counts applies to 2-D logits only")
            N, C = logits.shape[0], logits.shape[1]
            inner = math.prod(logits.shape[2:])
            rc, where = ce_fwd_nd(_ptr(logits), _DTYPES[logits.dtype], N, C, inner, *opts,
                                  _stream(dev)), "ce_fwd_nd"
        else:
            rows, V = logits.shape
            args = (_ptr(logits), _DTYPES[logits.dtype], rows, V, *opts)
            if batch_counts is None:
                rc, where = ce_fwd(*args, _stream(dev)), "ce_fwd"
            else:
                rc, where = (ce_fwd_shard(*args, _ptr(batch_counts), _stream(dev)),
                             "ce_fwd_shard")
    if rc != _lib.CE_OK:
        raise CEError(rc, where)
    return loss, z_loss, acc, pred


def shard_counts(target, V, weight=None, ignore_index=-100):
    """(D, counted rows) of these rows as a float64 CUDA tensor of 2 (ce_count):
    D = sum of weight[t] (the count without weights) over the rows whose
    target is neither ignore_index nor out of [0, V)."""
    if target.dim() != 1 or not target.is_cuda or target.dtype not in (torch.int32, torch.int64):
        raise ValueError("target must be a 1-D int32 or int64 CUDA tensor")
    target = target.contiguous()
    dev = target.device
    w = None if weight is None else weight.to(device=dev, dtype=torch.float32).contiguous()
    counts = torch.empty(2, dtype=torch.float64, device=dev)
    flags = _lib.CE_FLAG_TARGET_I64 if target.dtype == torch.int64 else 0
    with torch.cuda.device(dev):
        rc = ce_count(_ptr(target), _ptr(w), target.shape[0], int(V), int(ignore_index), flags,
                      _ptr(counts), _stream(dev))
    if rc != _lib.CE_OK:
        raise CEError(rc, "ce_count")
    return counts


class CrossEntropyFunction(torch.autograd.Function):
    """Autograd wrapper: forward stores the gradient in the logits buffer;
    backward scales it by grad_output (ce_bwd) and returns that buffer."""

    @staticmethod
    def forward(ctx, logits, target, weight, ignore_index, lse_square_scale, label_smoothing,
                reduction, softcap, return_z_loss, return_acc, return_pred, batch_counts=None):
        want_grad = logits.requires_grad
        loss, z_loss, acc, pred = _forward(logits, target, weight, ignore_index,
                                           lse_square_scale, label_smoothing, reduction,
                                           softcap, want_grad, return_z_loss, return_acc,
                                           return_pred, batch_counts)
        ctx.reduction = reduction
        if want_grad:
            ctx.save_for_backward(logits.detach())  # now holds dlogits
        extras = [t for t in (z_loss, acc, pred) if t is not None]
        if extras:
            ctx.mark_non_differentiable(*extras)
        return loss, z_loss, acc, pred

    @staticmethod
    def backward(ctx, grad_loss, *unused):
        (dlogits,) = ctx.saved_tensors
        g = grad_loss.to(torch.float32).contiguous()
        per_row = 1 if ctx.reduction == "none" else 0
        with torch.cuda.device(dlogits.device):
            if dlogits.dim() > 2:
                N, C = dlogits.shape[0], dlogits.shape[1]
                rc, where = ce_bwd_nd(_ptr(g), per_row, _ptr(dlogits), _DTYPES[dlogits.dtype], N,
                                      C, math.prod(dlogits.shape[2:]),
                                      _stream(dlogits.device)), "ce_bwd_nd"
            else:
                rows, V = dlogits.shape
                rc, where = ce_bwd(_ptr(g), per_row, _ptr(dlogits), _DTYPES[dlogits.dtype], rows,
                                   V, _stream(dlogits.device)), "ce_bwd"
        if rc != _lib.CE_OK:
            raise CEError(rc, where)
        return dlogits, None, None, None, None, None, None, None, None, None, None, None


def cross_entropy(logits, target, weight=None, ignore_index=-100, lse_square_scale=0.0,
                  label_smoothing=0.0, reduction="mean", softcap=None, return_z_loss=False,
                  return_token_accuracy=False, return_predicted_tokens=False,
                  batch_counts=None):
    """Fused softmax cross-entropy. Returns the loss tensor, or a
    CrossEntropyOutput(loss, z_loss, token_accuracy, predicted_tokens) when
    any return_* flag is set (unrequested fields are None).

    batch_counts: for one shard of a row-sharded batch, the float64 CUDA
    tensor (D, counted rows) of the whole batch (the sum over shards of
    shard_counts, e.g. after an all-reduce). The "mean" loss is then this
    shard's share of the batch mean (the shards' values add up to it) and
    the gradient is that of the batch mean; accuracy likewise."""
    _check_inputs(logits, target, weight)
    if batch_counts is not None:
        if (not isinstance(batch_counts, torch.Tensor) or batch_counts.dtype != torch.float64
                or batch_counts.numel() != 2 or batch_counts.device != logits.device):
            raise ValueError("batch_counts must be a float64 tensor of 2 on the logits' device")
        batch_counts = batch_counts.contiguous()
    if reduction not in _REDUCTIONS:
        raise ValueError(f"reduction must be one of {sorted(_REDUCTIONS)}")
    if not 0.0 <= label_smoothing <= 1.0:
        raise ValueError("label_smoothing must lie in [0, 1]")
    if softcap is not None and not softcap > 0:
        raise ValueError("softcap must be positive or None")
    if not logits.is_contiguous():
        logits = logits.contiguous()
    target = target.contiguous()
    loss, z_loss, acc, pred = CrossEntropyFunction.apply(
        logits, target, weight, ignore_index, lse_square_scale, label_smoothing, reduction,
        softcap, return_z_loss, return_token_accuracy, return_predicted_tokens, batch_counts)
    if return_z_loss or return_token_accuracy or return_predicted_tokens:
        return CrossEntropyOutput(loss, z_loss, acc, pred)
    return loss


class CrossEntropyLoss(torch.nn.Module):
    """Module form of cross_entropy with the profile's constructor
    parameters (§Module Parameters)."""

    def __init__(self, weight=None, ignore_index=-100, lse_square_scale=0.0,
                 label_smoothing=0.0, reduction="mean", softcap=None, return_z_loss=False,
                 return_token_accuracy=False, return_predicted_tokens=False):
        super().__init__()
        self.weight = weight
        self.ignore_index = ignore_index
        self.lse_square_scale = lse_square_scale
        self.label_smoothing = label_smoothing
        self.reduction = reduction
        self.softcap = softcap
        self.return_z_loss = return_z_loss
        self.return_token_accuracy = return_token_accuracy
        self.return_predicted_tokens = return_predicted_tokens

    def forward(self, logits, target):
        return cross_entropy(logits, target, self.weight, self.ignore_index,
                             self.lse_square_scale, self.label_smoothing, self.reduction,
                             self.softcap, self.return_z_loss, self.return_token_accuracy,
                             self.return_predicted_tokens)


def device_status(device=None) -> int:
    """Synchronizes the current stream of `device` and returns (and clears)
    the library's device-side error status for it (CE_OK when clean)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else \
        torch.device(device)
    with torch.cuda.device(dev):
        return ce_device_status(_stream(dev))
