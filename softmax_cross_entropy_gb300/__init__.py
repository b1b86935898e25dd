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
import os
from collections import namedtuple

import torch

from . import _lib
from ._lib import (CEError, ce_bwd, ce_bwd_nd, ce_count, ce_device_status, ce_flce,
                   ce_flce_workspace_bytes, ce_fwd, ce_fwd_nd, ce_fwd_shard, ce_last_error,
                   ce_scale_round, ce_status_string)

__all__ = ["cross_entropy", "CrossEntropyLoss", "CrossEntropyFunction", "CrossEntropyOutput",
           "CEError", "device_status", "shard_counts", "ce_fwd", "ce_fwd_shard", "ce_count",
           "ce_bwd", "ce_fwd_nd", "ce_bwd_nd", "ce_flce", "ce_flce_workspace_bytes",
           "ce_scale_round", "ce_device_status", "ce_status_string", "ce_last_error",
           "fused_linear_cross_entropy", "FusedLinearCrossEntropyFunction"]

CrossEntropyOutput = namedtuple("CrossEntropyOutput",
                                ["loss", "z_loss", "token_accuracy", "predicted_tokens"])

_REDUCTIONS = {"none": _lib.CE_RED_NONE, "sum": _lib.CE_RED_SUM, "mean": _lib.CE_RED_MEAN}
_DTYPES = {torch.float32: _lib.CE_F32, torch.bfloat16: _lib.CE_BF16,
           torch.float16: _lib.CE_F16}


# NVTX ranges around the library's calls (forward, backward) for profiler
# timelines, when GBCE_NVTX=1 at import; otherwise the ranges cost nothing.
_NVTX = os.environ.get("GBCE_NVTX", "") not in ("", "0")


class _Range:
    __slots__ = ("name",)

    def __init__(self, name):
        self.name = name

    def __enter__(self):
        if _NVTX:
            torch.cuda.nvtx.range_push(self.name)

    def __exit__(self, *exc):
        if _NVTX:
            torch.cuda.nvtx.range_pop()
        return False


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
        with _Range("gbce.cross_entropy.forward"):
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
        with torch.cuda.device(dlogits.device), _Range("gbce.cross_entropy.backward"):
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


def _flce_call(hidden, lm_weight, target, bias, weight, ignore_index, lse_square_scale,
               label_smoothing, reduction, softcap, want_z, want_acc, want_pred, want_grad,
               chunk_rows):
    """Runs ce_flce; returns (loss, z_loss, acc, pred, grad_hidden, grad_weight (fp32),
    grad_bias (fp32)), the gradients None unless want_grad."""
    dev = hidden.device
    dt = _DTYPES[hidden.dtype]
    rows, H = hidden.shape
    V = lm_weight.shape[0]
    red = _REDUCTIONS[reduction]
    out_shape = (rows,) if red == _lib.CE_RED_NONE else ()
    f32 = dict(dtype=torch.float32, device=dev)
    loss = torch.empty(out_shape, **f32)
    z_loss = torch.empty(out_shape, **f32) if want_z else None
    acc = torch.empty(out_shape, **f32) if want_acc else None
    pred = torch.empty((rows,), dtype=torch.int64, device=dev) if want_pred else None
    gh = torch.empty_like(hidden) if want_grad else None
    gw = torch.empty((V, H), **f32) if want_grad else None
    gb = torch.empty((V,), **f32) if (want_grad and bias is not None) else None
    nbytes = ce_flce_workspace_bytes(dt, rows, V, int(chunk_rows))
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)  # 256-byte aligned by the allocator
    flags = ((_lib.CE_FLAG_GRAD if want_grad else 0) | (_lib.CE_FLAG_Z_LOSS if want_z else 0) |
             (_lib.CE_FLAG_ACC if want_acc else 0) | (_lib.CE_FLAG_PRED if want_pred else 0) |
             (_lib.CE_FLAG_TARGET_I64 if target.dtype == torch.int64 else 0))
    b = None if bias is None else bias.to(torch.float32).contiguous()
    w = None if weight is None else weight.to(torch.float32).contiguous()
    with torch.cuda.device(dev):
        rc = ce_flce(_ptr(hidden), _ptr(lm_weight), _ptr(b), dt, rows, H, V, _ptr(target),
                     _ptr(w), int(ignore_index), float(label_smoothing), float(lse_square_scale),
                     float(softcap) if softcap is not None else 0.0, red, flags, _ptr(loss),
                     _ptr(z_loss), _ptr(acc), _ptr(pred), _ptr(gh), _ptr(gw), _ptr(gb),
                     int(chunk_rows), _ptr(ws), nbytes, _stream(dev))
    if rc != _lib.CE_OK:
        raise CEError(rc, "ce_flce")
    return loss, z_loss, acc, pred, gh, gw, gb


class FusedLinearCrossEntropyFunction(torch.autograd.Function):
    """Autograd wrapper of ce_flce: the forward computes the gradients of the
    reduced loss along with it (one chunk of logits at a time); backward
    scales them by the scalar grad_output in the library's kernels."""

    @staticmethod
    def forward(ctx, hidden, lm_weight, target, bias, weight, ignore_index, lse_square_scale,
                label_smoothing, reduction, softcap, return_z_loss, return_acc, return_pred,
                chunk_rows):
        want_grad = hidden.requires_grad or lm_weight.requires_grad or (
            bias is not None and bias.requires_grad)
        if want_grad and reduction == "none":
            raise ValueError("fused_linear_cross_entropy differentiates a scalar loss: use "
                             "reduction 'mean' or 'sum' (or no gradient)")
        with _Range("gbce.fused_linear_cross_entropy.forward"):
            loss, z_loss, acc, pred, gh, gw, gb = _flce_call(
                hidden, lm_weight, target, bias, weight, ignore_index, lse_square_scale,
                label_smoothing, reduction, softcap, return_z_loss, return_acc, return_pred,
                want_grad, chunk_rows)
        ctx.w_dtype = lm_weight.dtype
        ctx.has_bias = bias is not None
        if want_grad:
            ctx.save_for_backward(gh, gw, gb if gb is not None else torch.empty(0))
        extras = [t for t in (z_loss, acc, pred) if t is not None]
        if extras:
            ctx.mark_non_differentiable(*extras)
        return loss, z_loss, acc, pred

    @staticmethod
    def backward(ctx, grad_loss, *unused):
        gh, gw, gb = ctx.saved_tensors
        g = grad_loss.to(torch.float32).reshape(1).contiguous()
        dev = gh.device
        with torch.cuda.device(dev), _Range("gbce.fused_linear_cross_entropy.backward"):
            st = _stream(dev)
            rows, H = gh.shape
            rc = ce_bwd(_ptr(g), 0, _ptr(gh), _DTYPES[gh.dtype], rows, H, st)
            if rc != _lib.CE_OK:
                raise CEError(rc, "ce_bwd")
            gw_out = torch.empty(gw.shape, dtype=ctx.w_dtype, device=dev)
            rc = ce_scale_round(_ptr(gw), _ptr(g), _ptr(gw_out), _DTYPES[ctx.w_dtype],
                                gw.numel(), st)
            if rc != _lib.CE_OK:
                raise CEError(rc, "ce_scale_round")
            gb_out = None
            if ctx.has_bias:
                rc = ce_bwd(_ptr(g), 0, _ptr(gb), _lib.CE_F32, 1, gb.numel(), st)
                if rc != _lib.CE_OK:
                    raise CEError(rc, "ce_bwd")
                gb_out = gb
        return (gh, gw_out, None, gb_out, None, None, None, None, None, None, None, None, None,
                None)


def fused_linear_cross_entropy(hidden, lm_weight, target, bias=None, weight=None,
                               ignore_index=-100, lse_square_scale=0.0, label_smoothing=0.0,
                               reduction="mean", softcap=None, return_z_loss=False,
                               return_token_accuracy=False, return_predicted_tokens=False,
                               chunk_rows=0):
    """Cross-entropy of the logits hidden @ lm_weight^T + bias (the profile's
    closest_existing_kernel, fused_linear_cross_entropy) without forming all
    logits: ce_flce, one chunk of rows at a time. hidden [rows, H] and
    lm_weight [V, H] in float32, bfloat16 or float16; bias [V] or None;
    the other arguments as for cross_entropy. Returns the loss, or a
    CrossEntropyOutput when a return_* flag is set."""
    if not (isinstance(hidden, torch.Tensor) and isinstance(lm_weight, torch.Tensor)):
        raise TypeError("hidden and lm_weight must be tensors")
    if hidden.dim() != 2 or lm_weight.dim() != 2 or hidden.shape[1] != lm_weight.shape[1]:
        raise ValueError("hidden must be [rows, H] and lm_weight [V, H]")
    if not hidden.is_cuda or lm_weight.device != hidden.device:
        raise ValueError("hidden and lm_weight must be on one CUDA device")
    if hidden.dtype not in _DTYPES or lm_weight.dtype != hidden.dtype:
        raise TypeError("hidden and lm_weight must share one of float32, bfloat16, float16")
    if target.dim() != 1 or target.shape[0] != hidden.shape[0]:
        raise ValueError("target must be 1-D with one label per row of hidden")
    if target.dtype not in (torch.int32, torch.int64) or target.device != hidden.device:
        raise TypeError("target must be an int32 or int64 tensor on the hidden's device")
    if reduction not in _REDUCTIONS:
        raise ValueError(f"reduction must be one of {sorted(_REDUCTIONS)}")
    if not 0.0 <= label_smoothing <= 1.0:
        raise ValueError("label_smoothing must lie in [0, 1]")
    if softcap is not None and not softcap > 0:
        raise ValueError("softcap must be positive or None")
    hidden = hidden.contiguous()
    lm_weight = lm_weight.contiguous()
    target = target.contiguous()
    loss, z_loss, acc, pred = FusedLinearCrossEntropyFunction.apply(
        hidden, lm_weight, target, bias, weight, ignore_index, lse_square_scale,
        label_smoothing, reduction, softcap, return_z_loss, return_token_accuracy,
        return_predicted_tokens, chunk_rows)
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
