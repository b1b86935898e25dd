"""ctypes binding of libgbce.so: the C ABI declared in include/gbce.h, under
the same names, taking integers for device pointers and streams. Argument
marshalling only; every step of the computation runs in the library's CUDA
kernels. There is no fallback: loading fails loudly if the library has not
been built (``python -m softmax_cross_entropy_gb300.build``)."""
from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgbce.so")

CE_OK, CE_ERR_INVALID_ARG, CE_ERR_UNSUPPORTED, CE_ERR_CUDA, CE_ERR_TARGET_RANGE, \
    CE_ERR_TIMEOUT = range(6)
CE_F32, CE_BF16, CE_F16 = 0, 1, 2
CE_RED_NONE, CE_RED_SUM, CE_RED_MEAN = 0, 1, 2
CE_FLAG_GRAD, CE_FLAG_Z_LOSS, CE_FLAG_ACC, CE_FLAG_PRED, CE_FLAG_TARGET_I64 = 1, 2, 4, 8, 16

# (name, restype, argtypes) for every symbol include/gbce.h declares
_P, _I, _I64, _U32, _F = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint32,
                          ctypes.c_float)
SIGNATURES = {
    "ce_fwd": (_I, [_P, _I, _I64, _I64, _P, _P, _I64, _F, _F, _F, _I, _U32, _P, _P, _P, _P, _P]),
    "ce_fwd_noalloc": (_I, [_P, _I, _I64, _I64, _P, _P, _I64, _F, _F, _F, _I, _U32, _P, _P, _P, _P,
                            _P]),
    "ce_fwd_shard": (_I, [_P, _I, _I64, _I64, _P, _P, _I64, _F, _F, _F, _I, _U32, _P, _P, _P, _P,
                          _P, _P]),
    "ce_count": (_I, [_P, _P, _I64, _I64, _I64, _U32, _P, _P]),
    "ce_fwd_nd": (_I, [_P, _I, _I64, _I64, _I64, _P, _P, _I64, _F, _F, _F, _I, _U32, _P, _P, _P,
                       _P, _P]),
    "ce_bwd_nd": (_I, [_P, _I, _P, _I, _I64, _I64, _I64, _P]),
    "ce_flce_workspace_bytes": (ctypes.c_size_t, [_I, _I64, _I64, _I64]),
    "ce_scale_round": (_I, [_P, _P, _P, _I, _I64, _P]),
    "ce_gemm_abt": (_I, [_P, _P, _I, _I64, _I64, _I64, _P, _P, _P]),
    "ce_gemm": (_I, [_P, _I, _P, _I, _I, _I64, _I64, _I64, _P, _I, _P, _P]),
    "ce_flce": (_I, [_P, _P, _P, _I, _I64, _I64, _I64, _P, _P, _I64, _F, _F, _F, _I, _U32, _P, _P,
                     _P, _P, _P, _P, _P, _I64, _P, ctypes.c_size_t, _P]),
    "ce_bwd": (_I, [_P, _I, _P, _I, _I64, _I64, _P]),
    "ce_log_softmax": (_I, [_P, _P, _I, _I64, _I64, _P]),
    "ce_nll_loss_fwd": (_I, [_P, _I, _I64, _I64, _P, _P, _I64, _I, _U32, _P, _P, _P]),
    "ce_nll_loss_bwd": (_I, [_P, _P, _P, _I, _I64, _I64, _P, _P, _I64, _I, _U32, _P]),
    "ce_log_softmax_bwd": (_I, [_P, _P, _P, _I, _I64, _I64, _P]),
    "ce_device_status": (_I, [_P]),
    "ce_noalloc_status": (_I, [_P]),
    "ce_scratch_areas": (_I64, []),
    "ce_status_string": (ctypes.c_char_p, [_I]),
    "ce_last_error": (ctypes.c_char_p, []),
}

_lock = threading.Lock()
_lib = None


class CEError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = load()
        msg = lib.ce_status_string(status).decode()
        detail = lib.ce_last_error().decode()
        super().__init__(f"{where}: {msg}" + (f" ({detail})" if detail else ""))
        self.status = status


def load():
    """Loads libgbce.so once and declares its signatures."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(
                    f"{LIB_PATH} is missing: build the CUDA library first with "
                    "`python -m softmax_cross_entropy_gb300.build`")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def ce_fwd(logits, dtype, rows, V, target, weight, ignore_index, label_smoothing,
           lse_square_scale, softcap, reduction, flags, loss, z_loss, acc, pred, stream):
    return load().ce_fwd(logits, dtype, rows, V, target, weight, ignore_index,
                         label_smoothing, lse_square_scale, softcap, reduction, flags,
                         loss, z_loss, acc, pred, stream)


def ce_fwd_noalloc(logits, dtype, rows, V, target, weight, ignore_index, label_smoothing,
                   lse_square_scale, softcap, reduction, flags, loss, z_loss, acc, pred, stream):
    return load().ce_fwd_noalloc(logits, dtype, rows, V, target, weight, ignore_index,
                                 label_smoothing, lse_square_scale, softcap, reduction, flags,
                                 loss, z_loss, acc, pred, stream)


def ce_fwd_shard(logits, dtype, rows, V, target, weight, ignore_index, label_smoothing,
                 lse_square_scale, softcap, reduction, flags, loss, z_loss, acc, pred,
                 batch_counts, stream):
    return load().ce_fwd_shard(logits, dtype, rows, V, target, weight, ignore_index,
                               label_smoothing, lse_square_scale, softcap, reduction, flags,
                               loss, z_loss, acc, pred, batch_counts, stream)


def ce_count(target, weight, rows, V, ignore_index, flags, counts, stream):
    return load().ce_count(target, weight, rows, V, ignore_index, flags, counts, stream)


def ce_fwd_nd(logits, dtype, N, C, inner, target, weight, ignore_index, label_smoothing,
              lse_square_scale, softcap, reduction, flags, loss, z_loss, acc, pred, stream):
    return load().ce_fwd_nd(logits, dtype, N, C, inner, target, weight, ignore_index,
                            label_smoothing, lse_square_scale, softcap, reduction, flags,
                            loss, z_loss, acc, pred, stream)


def ce_bwd_nd(grad_output, grad_per_position, dlogits, dtype, N, C, inner, stream):
    return load().ce_bwd_nd(grad_output, grad_per_position, dlogits, dtype, N, C, inner, stream)


def ce_flce_workspace_bytes(dtype, rows, V, chunk_rows):
    return load().ce_flce_workspace_bytes(dtype, rows, V, chunk_rows)


def ce_flce(hidden, lm_weight, bias, dtype, rows, H, V, target, class_weight, ignore_index,
            label_smoothing, lse_square_scale, softcap, reduction, flags, loss, z_loss, acc,
            pred, grad_hidden, grad_weight, grad_bias, chunk_rows, workspace, workspace_bytes,
            stream):
    return load().ce_flce(hidden, lm_weight, bias, dtype, rows, H, V, target, class_weight,
                          ignore_index, label_smoothing, lse_square_scale, softcap, reduction,
                          flags, loss, z_loss, acc, pred, grad_hidden, grad_weight, grad_bias,
                          chunk_rows, workspace, workspace_bytes, stream)


def ce_gemm_abt(A, B, dtype, M, N, K, C, bias, stream):
    return load().ce_gemm_abt(A, B, dtype, M, N, K, C, bias, stream)


CE_GEMM_F32, CE_GEMM_F32_ADD, CE_GEMM_16BIT = 0, 1, 2


def ce_gemm(A, a_mn, B, b_mn, dtype, M, N, K, C, c_mode, bias, stream):
    return load().ce_gemm(A, a_mn, B, b_mn, dtype, M, N, K, C, c_mode, bias, stream)


def ce_scale_round(inp, grad_output, out, dtype, n, stream):
    return load().ce_scale_round(inp, grad_output, out, dtype, n, stream)


def ce_bwd(grad_output, grad_per_row, dlogits, dtype, rows, V, stream):
    return load().ce_bwd(grad_output, grad_per_row, dlogits, dtype, rows, V, stream)


def ce_log_softmax(x, out, dtype, rows, C, stream):
    return load().ce_log_softmax(x, out, dtype, rows, C, stream)


def ce_nll_loss_fwd(logp, dtype, rows, C, target, weight, ignore_index, reduction, flags, out,
                    total_weight, stream):
    return load().ce_nll_loss_fwd(logp, dtype, rows, C, target, weight, ignore_index,
                                  reduction, flags, out, total_weight, stream)


def ce_nll_loss_bwd(grad_output, total_weight, grad_input, dtype, rows, C, target, weight,
                    ignore_index, reduction, flags, stream):
    return load().ce_nll_loss_bwd(grad_output, total_weight, grad_input, dtype, rows, C, target,
                                  weight, ignore_index, reduction, flags, stream)


def ce_log_softmax_bwd(grad_output, output, grad_input, dtype, rows, C, stream):
    return load().ce_log_softmax_bwd(grad_output, output, grad_input, dtype, rows, C, stream)


def ce_device_status(stream):
    return load().ce_device_status(stream)


def ce_noalloc_status(stream):
    return load().ce_noalloc_status(stream)


def ce_scratch_areas():
    return load().ce_scratch_areas()


def ce_status_string(status):
    return load().ce_status_string(status).decode()


def ce_last_error():
    return load().ce_last_error().decode()
