"""Helpers for the GPU parity tests: move a workload case to the device, run
the CUDA path through the C ABI, run the oracle on the same bits, and the
tolerances the comparisons use."""
from __future__ import annotations

import math

import numpy as np

import workloads

# Tolerances. The headline bounds: fp32 loss rel 1e-5 and dlogits abs 1e-6;
# bf16 dlogits abs 4e-3 with the loss (fp32-accumulated) rel 1e-4;
# predicted tokens and accuracy exact. Because mean-scaled gradients are
# small, the gradient checks add a relative bound as well: a bf16 gradient
# must be within one bf16 unit in the last place of the oracle value (the
# kernel computes in fp32 and rounds once), an fp32 gradient within 1e-5
# relative plus 1e-6 of the largest gradient magnitude of the batch.
# The bf16 absolute bound applies wherever |gradient| < 2: there the nearest
# bf16 value lies within half a unit in the last place, at most 2^-8 =
# 3.9e-3 from the exact value (plus fp32 noise of order 1e-6), so 4e-3 is
# attainable. From magnitude 2 up, half a unit is 2^-7 > 4e-3 and the
# one-ulp bound governs.
# fp16 logits (no bound stated for them): the same fp32 arithmetic, so the
# bf16 loss bound; gradients rounded once to fp16, so within one fp16 unit
# in the last place (2^-10 relative) plus the smallest subnormal step 2^-24,
# and, by the same argument as for bf16, 5e-4 absolute wherever |gradient|
# < 2 (half a unit below 2 is at most 2^-11 = 4.9e-4).
LOSS_RTOL = {"f32": 1e-5, "bf16": 1e-4, "f16": 1e-4}
GRAD_ATOL = {"f32": 1e-6, "bf16": 4e-3, "f16": 5e-4}
CE_DTYPE = {"f32": 0, "bf16": 1, "f16": 2}  # ce_dtype of each storage
ATOL_BELOW = 2.0  # 16-bit storage: the absolute bound holds below this magnitude


def to_device(case, device="cuda"):
    import torch
    if case.dtype in ("bf16", "f16"):
        x = torch.from_numpy(np.ascontiguousarray(case.x).view(np.int16)).view(
            torch.bfloat16 if case.dtype == "bf16" else torch.float16)
    else:
        x = torch.from_numpy(np.ascontiguousarray(case.x))
    x = x.to(device)
    t = torch.from_numpy(np.ascontiguousarray(case.target)).to(device)
    w = None if case.weight is None else torch.from_numpy(case.weight).to(device)
    return x, t, w


def run_cuda(case, *, grad=True, want_z=False, want_acc=False, want_pred=False, x=None,
             target=None, reduction=None, stream=None):
    """Calls ce_fwd through the C ABI. Returns a dict of numpy outputs plus
    the device logits buffer (holding dlogits when grad)."""
    import torch
    from softmax_cross_entropy_gb300 import _lib
    dev_x, dev_t, dev_w = to_device(case)
    if x is not None:
        dev_x = x
    if target is not None:
        dev_t = target
    red = reduction or case.reduction
    rows, V = case.rows, case.V
    n = rows if red == "none" else 1
    f32 = dict(dtype=torch.float32, device=dev_x.device)
    loss = torch.full((n,), float("nan"), **f32)
    zl = torch.full((n,), float("nan"), **f32) if want_z else None
    acc = torch.full((n,), float("nan"), **f32) if want_acc else None
    pred = torch.full((rows,), -7, dtype=torch.int64, device=dev_x.device) if want_pred else None
    flags = ((_lib.CE_FLAG_GRAD if grad else 0) | (_lib.CE_FLAG_Z_LOSS if want_z else 0) |
             (_lib.CE_FLAG_ACC if want_acc else 0) | (_lib.CE_FLAG_PRED if want_pred else 0) |
             (_lib.CE_FLAG_TARGET_I64 if dev_t.dtype == torch.int64 else 0))
    st = stream if stream is not None else torch.cuda.current_stream().cuda_stream
    rc = _lib.ce_fwd(dev_x.data_ptr(), CE_DTYPE[case.dtype],
                     rows, V, dev_t.data_ptr(), None if dev_w is None else dev_w.data_ptr(),
                     case.ignore_index, case.label_smoothing, case.lse_square_scale,
                     case.softcap or 0.0, {"none": 0, "sum": 1, "mean": 2}[red], flags,
                     loss.data_ptr(), None if zl is None else zl.data_ptr(),
                     None if acc is None else acc.data_ptr(),
                     None if pred is None else pred.data_ptr(), st)
    assert rc == _lib.CE_OK, (_lib.ce_status_string(rc), _lib.ce_last_error())
    status = _lib.ce_device_status(st)
    out = {"status": status, "x": dev_x,
           "loss": loss.cpu().numpy().astype(np.float64),
           "z_loss": None if zl is None else zl.cpu().numpy().astype(np.float64),
           "acc": None if acc is None else acc.cpu().numpy().astype(np.float64),
           "pred": None if pred is None else pred.cpu().numpy()}
    if red != "none":
        for k in ("loss", "z_loss", "acc"):
            if out[k] is not None:
                out[k] = out[k][0]
    return out


def grad_rows_f64(dev_x, rows_idx=None):
    import torch
    g = dev_x if rows_idx is None else dev_x[torch.as_tensor(rows_idx, device=dev_x.device)]
    return g.float().cpu().numpy().astype(np.float64)


def oracle_full(case, reduction=None, want_grad=True):
    import oracle
    opts = case.options()
    if reduction:
        opts["reduction"] = reduction
    return oracle.forward(case.x, case.target, dtype=case.dtype, weight=case.weight,
                          want_grad=want_grad, **opts)


def oracle_rows(case, idx, reduction=None, want_grad=True):
    import oracle
    opts = case.options()
    if reduction:
        opts["reduction"] = reduction
    return oracle.rows(case.x, case.target, idx, dtype=case.dtype, weight=case.weight,
                       want_grad=want_grad, **opts)


def assert_loss_close(got, want, dtype, what="loss"):
    if isinstance(want, float) and math.isnan(want):
        assert math.isnan(got), f"{what}: expected NaN, got {got}"
        return
    np.testing.assert_allclose(got, want, rtol=LOSS_RTOL[dtype], atol=1e-30, err_msg=what)


def assert_rowloss_close(got, want, dtype, what="row loss"):
    # per-row values: relative bound plus a small absolute floor for rows
    # whose loss is near zero
    np.testing.assert_allclose(got, want, rtol=LOSS_RTOL[dtype], atol=LOSS_RTOL[dtype] * 1e-2,
                               err_msg=what)


def grad_violations(got, want, dtype, gmax=None):
    """Checks gradient values against the bounds above. Returns None when
    every element is within them, else a message naming the first
    offender. ``gmax`` is the largest oracle gradient magnitude of the whole
    batch (taken from ``want`` when None)."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    if got.shape != want.shape:
        return f"shape {got.shape} != {want.shape}"
    aw = np.abs(want)
    err = np.abs(got - want)
    if gmax is None:
        gmax = aw.max(initial=0.0)
    small = aw < ATOL_BELOW if dtype in ("bf16", "f16") else np.ones(want.shape, bool)
    emax = err[small].max(initial=0.0)
    if not emax <= GRAD_ATOL[dtype]:
        return f"max abs err {emax} above {GRAD_ATOL[dtype]}"
    if dtype == "bf16":
        # one bf16 ulp of the oracle value (2^-7 relative covers the binade
        # edge), plus the fp32 compute noise near zero
        bound = aw * 2.0 ** -7 + 1e-6 * gmax + 1e-30
    elif dtype == "f16":
        bound = aw * 2.0 ** -10 + 1e-6 * gmax + 2.0 ** -24
    else:
        bound = 1e-5 * aw + 1e-6 * gmax + 1e-30
    bad = ~(err <= bound)  # NaN counts as out of bound
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        return (f"{int(bad.sum())} elements out of bound; first at {i}: "
                f"got {got[i]!r} want {want[i]!r}")
    return None


def assert_grad_close(got, want, dtype, what="dlogits", gmax=None):
    msg = grad_violations(got, want, dtype, gmax)
    assert msg is None, f"{what}: {msg}"


def host_values(dev_x):
    """The device logits/gradient buffer as a host numpy array of its
    storage (float32, or the raw uint16 bits of bf16 / fp16)."""
    import torch
    if dev_x.dtype == torch.float32:
        return dev_x.cpu().numpy()
    return dev_x.view(torch.int16).cpu().numpy().view(np.uint16)


def storage_to_f64(a, dtype):
    """Exact widening of stored values to float64."""
    if dtype == "f32":
        return a.astype(np.float64)
    if dtype == "bf16":
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.view(np.float16).astype(np.float64)


def assert_grad_whole(case, dev_x, reduction=None, chunk_rows=None, workers=None):
    """Compares every gradient row of the batch with the oracle. The rows go
    to the oracle in contiguous chunks, in a pool of threads (the oracle's C
    code runs without the interpreter lock); each chunk is held to the bounds
    above with its own largest oracle magnitude as ``gmax``, which is never
    larger than the batch's (so this is at least as strict as one
    whole-batch comparison)."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    red = reduction or case.reduction
    host = host_values(dev_x)
    rows, V = case.rows, case.V
    assert host.shape == (rows, V)
    if chunk_rows is None:
        chunk_rows = max(1, min(256, (1 << 22) // max(V, 1)))

    def one(r0):
        idx = np.arange(r0, min(rows, r0 + chunk_rows), dtype=np.int64)
        want = oracle_rows(case, idx, reduction=red)["grad"]
        got = storage_to_f64(host[r0:r0 + idx.size], case.dtype)
        return r0, grad_violations(got, want, case.dtype)

    nw = workers or max(1, min(16, os.cpu_count() or 1))
    with ThreadPoolExecutor(max_workers=nw) as pool:
        for r0, msg in pool.map(one, range(0, rows, chunk_rows)):
            if msg is not None:
                raise AssertionError(f"dlogits, chunk of rows from {r0}: {msg}")


def sample_rows(case, n=24, seed=0):
    """A fixed sample of row indices: some valid, some ignored, first and
    last rows."""
    rng = np.random.default_rng(seed)
    rows = case.rows
    idx = set(rng.choice(rows, size=min(n, rows), replace=False).tolist())
    idx.update({0, rows - 1})
    ign = np.nonzero(case.target == case.ignore_index)[0]
    if ign.size:
        idx.add(int(ign[0]))
    return np.array(sorted(idx), np.int64)




__all__ = ["to_device", "run_cuda", "grad_rows_f64", "oracle_full", "oracle_rows",
           "assert_loss_close", "assert_rowloss_close", "assert_grad_close", "grad_violations",
           "assert_grad_whole", "host_values", "storage_to_f64", "sample_rows", "workloads"]
