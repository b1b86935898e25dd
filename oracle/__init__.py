"""CPU float64 oracle for fused softmax cross-entropy.

TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import this package. The CUDA library never
links or calls it, and this package imports nothing from the CUDA library:
the two share no code. The arithmetic lives in ``ce_oracle.c`` (plain C,
double precision, single-threaded); this module compiles it with gcc and
marshals numpy arrays in and out.

Logit storage: ``"f64"``, ``"f32"``, or ``"bf16"`` / ``"f16"`` given as the
raw uint16 bit patterns (the oracle decodes them exactly).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "ce_oracle.c"), os.path.join(_HERE, "aten_oracle.c")]
_LIB_PATH = os.path.join(_HERE, "libceoracle.so")

_DTYPES = {"f64": 0, "f32": 1, "bf16": 2, "f16": 3}
_NP_STORAGE = {"f64": np.float64, "f32": np.float32, "bf16": np.uint16, "f16": np.uint16}
REDUCTIONS = {"none": 0, "sum": 1, "mean": 2}

_lock = threading.Lock()
_lib = None


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compiles ce_oracle.c and aten_oracle.c into a shared object next to
    them (no fast-math: IEEE double semantics are part of the oracle's
    definition)."""
    if force or not os.path.exists(_LIB_PATH) or any(
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(src) for src in _SRCS):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off",
             "-shared", "-fPIC", *_SRCS, "-o", tmp, "-lm"],
            check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i64 = ctypes.c_int64
            d = ctypes.c_double
            lib.orc_ce_forward.argtypes = [P, ctypes.c_int, i64, i64, P, P, i64, d, d, d,
                                           ctypes.c_int, P, P, P, P, P]
            lib.orc_ce_forward.restype = ctypes.c_int
            lib.orc_ce_rows.argtypes = [P, ctypes.c_int, i64, i64, P, P, i64, d, d, d,
                                        ctypes.c_int, P, i64, P, P, P, P, P, P, P]
            lib.orc_ce_rows.restype = ctypes.c_int
            lib.orc_ce_backward.argtypes = [P, i64, i64, P, ctypes.c_int]
            lib.orc_ce_backward.restype = None
            lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.orc_bf16_to_double.restype = d
            lib.orc_f16_to_double.argtypes = [ctypes.c_uint16]
            lib.orc_f16_to_double.restype = d
            lib.orc_decode.argtypes = [P, ctypes.c_int, i64, P]
            lib.orc_decode.restype = None
            ci = ctypes.c_int
            lib.ao_log_softmax.argtypes = [P, i64, i64, P]
            lib.ao_nll_forward.argtypes = [P, P, P, i64, i64, i64, ci, P, P]
            lib.ao_nll_backward.argtypes = [P, P, P, i64, i64, i64, ci, d, P]
            lib.ao_log_softmax_backward.argtypes = [P, P, i64, i64, P]
            for f in (lib.ao_log_softmax, lib.ao_nll_forward, lib.ao_nll_backward,
                      lib.ao_log_softmax_backward):
                f.restype = ci
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _prep(x, dtype, target, weight):
    if dtype not in _DTYPES:
        raise ValueError(f"unknown logit storage {dtype!r}")
    x = np.ascontiguousarray(x, dtype=_NP_STORAGE[dtype])
    if x.ndim != 2:
        raise ValueError("logits must be 2-D (rows, V)")
    target = np.ascontiguousarray(target, dtype=np.int64).reshape(-1)
    if target.shape[0] != x.shape[0]:
        raise ValueError("target must have one entry per row")
    if weight is not None:
        weight = np.ascontiguousarray(weight, dtype=np.float64).reshape(-1)
        if weight.shape[0] != x.shape[1]:
            raise ValueError("weight must have V entries")
    return x, target, weight


def _check(rc):
    if rc == 1:
        raise OracleError("invalid argument")
    if rc == 2:
        raise OracleError("target out of range")
    if rc != 0:
        raise OracleError(f"oracle error {rc}")


def forward(x, target, *, dtype="f64", weight=None, ignore_index=-100,
            label_smoothing=0.0, lse_square_scale=0.0, softcap=None,
            reduction="mean", want_grad=True):
    """Whole-batch forward. Returns a dict with ``loss``, ``z_loss``, ``acc``
    (scalars, or [rows] arrays for reduction "none"), ``pred`` [rows] int64
    and ``grad`` [rows, V] float64 (the gradient of the reduced loss with
    respect to the logits) or None."""
    lib = _load()
    x, target, weight = _prep(x, dtype, target, weight)
    rows, V = x.shape
    red = REDUCTIONS[reduction]
    n_out = rows if red == 0 else 1
    loss = np.zeros(n_out, np.float64)
    zl = np.zeros(n_out, np.float64)
    acc = np.zeros(n_out, np.float64)
    pred = np.zeros(rows, np.int64)
    grad = np.empty((rows, V), np.float64) if want_grad else None
    rc = lib.orc_ce_forward(_ptr(x), _DTYPES[dtype], rows, V, _ptr(target), _ptr(weight),
                            int(ignore_index), float(label_smoothing),
                            float(lse_square_scale),
                            float(softcap) if softcap is not None else 0.0, red,
                            _ptr(loss), _ptr(zl), _ptr(acc), _ptr(pred), _ptr(grad))
    _check(rc)
    if red != 0:
        loss, zl, acc = loss[0], zl[0], acc[0]
    return {"loss": loss, "z_loss": zl, "acc": acc, "pred": pred, "grad": grad}


def forward_nd(x, target, *, dtype="f64", **opts):
    """Forward for N-D logits with the class dimension at axis 1, (N, C, d1,
    ..., dk), and targets (N, d1, ..., dk): the cross-entropy of every
    position's C logits, reduced over all positions. By definition this is
    the 2-D computation on the logits with the class axis moved last and
    the positions flattened into rows; the per-position outputs and the
    gradient are reshaped back. Same keyword options as forward()."""
    x = np.asarray(x)
    if x.ndim < 2:
        raise OracleError("N-D logits need at least (N, C)")
    C = x.shape[1]
    rows2d = np.ascontiguousarray(np.moveaxis(x, 1, -1)).reshape(-1, C)
    t = np.asarray(target).reshape(-1)
    r = forward(rows2d, t, dtype=dtype, **opts)
    pos_shape = (x.shape[0],) + x.shape[2:]
    out = dict(r)
    if opts.get("reduction", "mean") == "none":
        for k in ("loss", "z_loss", "acc"):
            out[k] = r[k].reshape(pos_shape)
    out["pred"] = r["pred"].reshape(pos_shape)
    if r["grad"] is not None:
        out["grad"] = np.moveaxis(r["grad"].reshape(pos_shape + (C,)), -1, 1)
    return out


def rows(x, target, row_idx, *, dtype="f64", weight=None, ignore_index=-100,
         label_smoothing=0.0, lse_square_scale=0.0, softcap=None,
         reduction="mean", want_grad=True):
    """Selected rows of a batch: per-row (unreduced) loss, z-loss, pred,
    0/1 correctness and the reduction-scaled gradient rows, plus the batch
    denominators ``D`` and ``n_valid``."""
    lib = _load()
    x, target, weight = _prep(x, dtype, target, weight)
    nrows, V = x.shape
    idx = np.ascontiguousarray(row_idx, dtype=np.int64).reshape(-1)
    k = idx.shape[0]
    loss = np.zeros(k, np.float64)
    zl = np.zeros(k, np.float64)
    pred = np.zeros(k, np.int64)
    corr = np.zeros(k, np.float64)
    grad = np.empty((k, V), np.float64) if want_grad else None
    D = ctypes.c_double(0.0)
    nv = ctypes.c_int64(0)
    rc = lib.orc_ce_rows(_ptr(x), _DTYPES[dtype], nrows, V, _ptr(target), _ptr(weight),
                         int(ignore_index), float(label_smoothing),
                         float(lse_square_scale),
                         float(softcap) if softcap is not None else 0.0,
                         REDUCTIONS[reduction], _ptr(idx), k, _ptr(loss), _ptr(zl),
                         _ptr(pred), _ptr(corr), _ptr(grad), ctypes.byref(D),
                         ctypes.byref(nv))
    _check(rc)
    return {"loss": loss, "z_loss": zl, "pred": pred, "correct": corr, "grad": grad,
            "D": D.value, "n_valid": nv.value}


def backward(grad, grad_output):
    """Scales a stored gradient in place by grad_output: a scalar, or one
    value per row."""
    lib = _load()
    grad = np.ascontiguousarray(grad, dtype=np.float64)
    go = np.ascontiguousarray(np.atleast_1d(grad_output), dtype=np.float64)
    per_row = 1 if go.shape[0] == grad.shape[0] and go.shape[0] != 1 else 0
    lib.orc_ce_backward(_ptr(grad), grad.shape[0], grad.shape[1], _ptr(go), per_row)
    return grad


def decode(x, dtype):
    """The stored values of an array (``"f64"``, ``"f32"``, or bf16 / fp16 bit
    patterns) as float64, exactly."""
    if dtype not in _DTYPES:
        raise ValueError(f"unknown storage {dtype!r}")
    x = np.ascontiguousarray(x, dtype=_NP_STORAGE[dtype])
    out = np.empty(x.shape, np.float64)
    _load().orc_decode(_ptr(x), _DTYPES[dtype], x.size, _ptr(out))
    return out


def linear(hidden, lm_weight, *, dtype="f64", bias=None):
    """The logits of the fused linear cross-entropy: hidden [rows, H] @
    lm_weight[V, H]^T (+ bias [V]), in float64 from the exactly decoded
    stored values."""
    h = decode(hidden, dtype)
    w = decode(lm_weight, dtype)
    if h.ndim != 2 or w.ndim != 2 or h.shape[1] != w.shape[1]:
        raise OracleError("hidden [rows, H] and lm_weight [V, H] expected")
    logits = h @ w.T
    if bias is not None:
        b = np.ascontiguousarray(bias, dtype=np.float64).reshape(-1)
        if b.shape[0] != w.shape[0]:
            raise OracleError("bias must have V entries")
        logits = logits + b[None, :]
    return logits


def flce_forward(hidden, lm_weight, target, *, dtype="f64", bias=None, weight=None,
                 ignore_index=-100, label_smoothing=0.0, lse_square_scale=0.0, softcap=None,
                 reduction="mean", want_grad=True):
    """Fused linear cross-entropy ("Kernel Profile: CrossEntropy",
    closest_existing_kernel: fused_linear_cross_entropy, the cross-entropy
    kernel with the linear layer fused in): the cross-entropy of the logits
    hidden @ lm_weight^T (+ bias), by definition. hidden [rows, H] and
    lm_weight [V, H] in storage ``dtype`` (decoded exactly), bias [V] float
    or None; ``weight`` is the class weight of the cross-entropy. The logits
    are formed in float64 and handed to forward(); with want_grad the chain
    rule gives grad_hidden = G @ lm_weight, grad_weight = G^T @ hidden and
    grad_bias = the column sums of G, G the gradient forward() returns
    (that of the reduced loss; for "none", of the sum of the row losses)."""
    h = decode(hidden, dtype)
    w = decode(lm_weight, dtype)
    logits = linear(hidden, lm_weight, dtype=dtype, bias=bias)
    r = forward(logits, target, dtype="f64", weight=weight, ignore_index=ignore_index,
                label_smoothing=label_smoothing, lse_square_scale=lse_square_scale,
                softcap=softcap, reduction=reduction, want_grad=want_grad)
    out = dict(r)
    out["logits"] = logits
    if want_grad:
        g = r["grad"]
        out["grad_hidden"] = g @ w
        out["grad_weight"] = g.T @ h
        out["grad_bias"] = g.sum(axis=0)
    return out


def bf16_to_double(bits: int) -> float:
    return _load().orc_bf16_to_double(int(bits) & 0xFFFF)


def f16_to_double(bits: int) -> float:
    return _load().orc_f16_to_double(int(bits) & 0xFFFF)


# ---------------------------------------------------------------- unfused (aten) ops

def _f64_2d(a):
    a = np.ascontiguousarray(a, dtype=np.float64)
    if a.ndim != 2:
        raise ValueError("expected a 2-D (rows, C) array")
    return a


def _check_ao(rc, what):
    if rc == 1:
        raise OracleError(f"{what}: invalid arguments")
    if rc == 2:
        raise OracleError(f"{what}: target index out of range")


def log_softmax(x):
    """_log_softmax over the last dimension, float64."""
    x = _f64_2d(x)
    out = np.empty_like(x)
    _check_ao(_load().ao_log_softmax(_ptr(x), x.shape[0], x.shape[1], _ptr(out)), "log_softmax")
    return out


def nll_forward(logp, target, weight=None, ignore_index=-100, reduction="mean"):
    """nll_loss_forward: returns (output, total_weight); output has one value
    per row for "none", else one."""
    logp = _f64_2d(logp)
    rows, C = logp.shape
    target = np.ascontiguousarray(target, dtype=np.int64).reshape(-1)
    w = None if weight is None else np.ascontiguousarray(weight, dtype=np.float64)
    out = np.empty(max(rows, 1) if reduction == "none" else 1)
    tw = np.zeros(1)
    _check_ao(_load().ao_nll_forward(_ptr(logp), _ptr(target), _ptr(w), rows, C,
                                     int(ignore_index), REDUCTIONS[reduction], _ptr(out),
                                     _ptr(tw)), "nll_forward")
    return (out[:rows] if reduction == "none" else float(out[0])), float(tw[0])


def nll_backward(grad_output, target, C, weight=None, ignore_index=-100, reduction="mean",
                 total_weight=1.0):
    """nll_loss_backward: the (rows, C) gradient of the nll loss."""
    target = np.ascontiguousarray(target, dtype=np.int64).reshape(-1)
    rows = target.shape[0]
    go = np.ascontiguousarray(np.atleast_1d(grad_output), dtype=np.float64)
    w = None if weight is None else np.ascontiguousarray(weight, dtype=np.float64)
    grad = np.empty((rows, C))
    _check_ao(_load().ao_nll_backward(_ptr(go), _ptr(target), _ptr(w), rows, C,
                                      int(ignore_index), REDUCTIONS[reduction],
                                      float(total_weight), _ptr(grad)), "nll_backward")
    return grad


def log_softmax_backward(dy, y):
    """_log_softmax_backward_data: dy - exp(y) * rowsum(dy)."""
    dy, y = _f64_2d(dy), _f64_2d(y)
    dx = np.empty_like(dy)
    _check_ao(_load().ao_log_softmax_backward(_ptr(dy), _ptr(y), dy.shape[0], dy.shape[1],
                                              _ptr(dx)), "log_softmax_backward")
    return dx
