"""The unfused (aten-shaped) form of softmax cross-entropy on libgbce.so.

A decomposed F.cross_entropy graph runs four ops (tt-mlir pull request
#9324, the table of decomposed aten ops; the #9339 description):

    y = log_softmax(x)                                   _log_softmax
    loss, total_weight = nll_loss_forward(y, target)     nll_loss_forward
    dy = nll_loss_backward(g, target, C, total_weight)   nll_loss_backward
    dx = log_softmax_backward_data(dy, y)                _log_softmax_backward_data

Each function below is one C-ABI call (argument marshalling only; the
arithmetic runs in the library's kernels). `LogSoftmax` and `NLLLoss` are
the matching autograd functions and `cross_entropy_unfused` chains them, as
the fallback for graphs that were not fused. Tensors are 2-D (rows, C) CUDA
tensors in float32, bfloat16 or float16; targets int32 or int64.
"""
from __future__ import annotations

import torch

from . import _lib
from ._lib import CEError

_DTYPES = {torch.float32: _lib.CE_F32, torch.bfloat16: _lib.CE_BF16,
           torch.float16: _lib.CE_F16}
_REDUCTIONS = {"none": _lib.CE_RED_NONE, "sum": _lib.CE_RED_SUM, "mean": _lib.CE_RED_MEAN}


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(dev):
    return torch.cuda.current_stream(dev).cuda_stream


def _check_2d(t, name):
    if not isinstance(t, torch.Tensor) or t.dim() != 2 or not t.is_cuda:
        raise ValueError(f"{name} must be a 2-D (rows, C) CUDA tensor")
    if t.dtype not in _DTYPES:
        raise TypeError(f"{name} dtype {t.dtype} is not supported")
    return t.contiguous()


def _target(target, rows, dev):
    if target.dim() != 1 or target.shape[0] != rows or target.device != dev:
        raise ValueError("target must be 1-D with one label per row, on the same device")
    if target.dtype not in (torch.int32, torch.int64):
        raise TypeError("target must be int32 or int64")
    flags = _lib.CE_FLAG_TARGET_I64 if target.dtype == torch.int64 else 0
    return target.contiguous(), flags


def _weight(weight, C, dev):
    if weight is None:
        return None
    if weight.dim() != 1 or weight.shape[0] != C:
        raise ValueError("weight must have shape (C,)")
    return weight.to(device=dev, dtype=torch.float32).contiguous()


def log_softmax(x, out=None):
    """_log_softmax over the last dimension (out may be x itself)."""
    x = _check_2d(x, "x")
    rows, C = x.shape
    out = torch.empty_like(x) if out is None else out
    with torch.cuda.device(x.device):
        rc = _lib.ce_log_softmax(_ptr(x), _ptr(out), _DTYPES[x.dtype], rows, C, _stream(x.device))
    if rc != _lib.CE_OK:
        raise CEError(rc, "ce_log_softmax")
    return out


def nll_loss_forward(logp, target, weight=None, reduction="mean", ignore_index=-100):
    """nll_loss_forward: (output, total_weight), both float32 (output has one
    value per row for "none")."""
    logp = _check_2d(logp, "logp")
    rows, C = logp.shape
    target, flags = _target(target, rows, logp.device)
    w = _weight(weight, C, logp.device)
    f32 = dict(dtype=torch.float32, device=logp.device)
    out = torch.empty((rows,) if reduction == "none" else (), **f32)
    tw = torch.empty((), **f32)
    with torch.cuda.device(logp.device):
        rc = _lib.ce_nll_loss_fwd(_ptr(logp), _DTYPES[logp.dtype], rows, C, _ptr(target), _ptr(w),
                                  int(ignore_index), _REDUCTIONS[reduction], flags, _ptr(out),
                                  _ptr(tw), _stream(logp.device))
    if rc != _lib.CE_OK:
        raise CEError(rc, "ce_nll_loss_fwd")
    return out, tw


def nll_loss_backward(grad_output, target, C, dtype, weight=None, reduction="mean",
                      ignore_index=-100, total_weight=None):
    """nll_loss_backward: the (rows, C) gradient in `dtype`."""
    dev = target.device
    rows = target.shape[0]
    target, flags = _target(target, rows, dev)
    w = _weight(weight, C, dev)
    g = grad_output.to(device=dev, dtype=torch.float32).contiguous()
    tw = None if total_weight is None else total_weight.to(dtype=torch.float32).contiguous()
    grad = torch.empty((rows, C), dtype=dtype, device=dev)
    with torch.cuda.device(dev):
        rc = _lib.ce_nll_loss_bwd(_ptr(g), _ptr(tw), _ptr(grad), _DTYPES[dtype], rows, C,
                                  _ptr(target), _ptr(w), int(ignore_index),
                                  _REDUCTIONS[reduction], flags, _stream(dev))
    if rc != _lib.CE_OK:
        raise CEError(rc, "ce_nll_loss_bwd")
    return grad


def log_softmax_backward_data(grad_output, output, grad_input=None):
    """_log_softmax_backward_data: grad_output - exp(output) * rowsum(grad_output)."""
    dy = _check_2d(grad_output, "grad_output")
    y = _check_2d(output, "output")
    if dy.shape != y.shape or dy.dtype != y.dtype:
        raise ValueError("grad_output and output must have the same shape and dtype")
    rows, C = y.shape
    dx = torch.empty_like(dy) if grad_input is None else grad_input
    with torch.cuda.device(y.device):
        rc = _lib.ce_log_softmax_bwd(_ptr(dy), _ptr(y), _ptr(dx), _DTYPES[y.dtype], rows, C,
                                     _stream(y.device))
    if rc != _lib.CE_OK:
        raise CEError(rc, "ce_log_softmax_bwd")
    return dx


class LogSoftmax(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x):
        y = log_softmax(x)
        ctx.save_for_backward(y)
        return y

    @staticmethod
    def backward(ctx, dy):
        (y,) = ctx.saved_tensors
        return log_softmax_backward_data(dy.to(y.dtype), y)


class NLLLoss(torch.autograd.Function):
    @staticmethod
    def forward(ctx, logp, target, weight, reduction, ignore_index):
        out, tw = nll_loss_forward(logp, target, weight, reduction, ignore_index)
        ctx.save_for_backward(target, tw)
        ctx.weight, ctx.reduction, ctx.ignore_index = weight, reduction, ignore_index
        ctx.shape, ctx.dtype = logp.shape, logp.dtype
        return out

    @staticmethod
    def backward(ctx, g):
        target, tw = ctx.saved_tensors
        grad = nll_loss_backward(g, target, ctx.shape[1], ctx.dtype, ctx.weight, ctx.reduction,
                                 ctx.ignore_index, tw)
        return grad, None, None, None, None


def cross_entropy_unfused(logits, target, weight=None, ignore_index=-100, reduction="mean"):
    """F.cross_entropy as the decomposed graph computes it: _log_softmax,
    then nll_loss (no label smoothing, z-loss or softcap in this form)."""
    if reduction not in _REDUCTIONS:
        raise ValueError(f"reduction must be one of {sorted(_REDUCTIONS)}")
    return NLLLoss.apply(LogSoftmax.apply(logits), target, weight, reduction, ignore_index)
