"""ce_fwd_noalloc: the forward call for callers that cannot allocate device
memory (an allocator's own callbacks, a memory-capped sandbox, a framework
that forbids allocations after start-up). It must give what ce_fwd gives,
call after call, although its scratch is one fixed device array that every
call reuses. This file is collected last on purpose: if it fails, a run that
stops at the first failure has already run every other test."""

import numpy as np
import pytest

import workloads
from ce_gpu import (assert_grad_close, assert_loss_close, assert_rowloss_close, grad_rows_f64,
                    to_device)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from softmax_cross_entropy_gb300 import build, _lib
    build.build()
    _lib.load()


def _call(entry, case, reduction):
    """Runs one forward entry point through the C ABI on fresh device copies
    of the case's inputs; returns numpy outputs and the gradient buffer."""
    from softmax_cross_entropy_gb300 import _lib
    x, t, w = to_device(case)
    rows, V = case.rows, case.V
    n = rows if reduction == "none" else 1
    f32 = dict(dtype=torch.float32, device=x.device)
    loss = torch.full((n,), float("nan"), **f32)
    zl = torch.full((n,), float("nan"), **f32)
    acc = torch.full((n,), float("nan"), **f32)
    pred = torch.full((rows,), -7, dtype=torch.int64, device=x.device)
    flags = (_lib.CE_FLAG_GRAD | _lib.CE_FLAG_Z_LOSS | _lib.CE_FLAG_ACC | _lib.CE_FLAG_PRED)
    st = torch.cuda.current_stream().cuda_stream
    rc = entry(x.data_ptr(), _lib.CE_BF16 if case.dtype == "bf16" else _lib.CE_F32, rows, V,
               t.data_ptr(), None if w is None else w.data_ptr(), case.ignore_index,
               case.label_smoothing, case.lse_square_scale, case.softcap or 0.0,
               {"none": 0, "sum": 1, "mean": 2}[reduction], flags, loss.data_ptr(),
               zl.data_ptr(), acc.data_ptr(), pred.data_ptr(), st)
    assert rc == _lib.CE_OK, (_lib.ce_status_string(rc), _lib.ce_last_error())
    torch.cuda.synchronize()
    return {"loss": loss.cpu().numpy().astype(np.float64),
            "z_loss": zl.cpu().numpy().astype(np.float64),
            "acc": acc.cpu().numpy(), "pred": pred.cpu().numpy(), "grad": grad_rows_f64(x)}


CASES = [
    ("bf16 V=32768, mean", lambda: workloads.vsweep(V=32768, rows=300), "mean"),
    ("fp32 V=4096 with ignored rows, sum",
     lambda: workloads.tt_fp32(rows=96, V=4096, reduction="sum"), "sum"),
    ("bf16 weighted smoothing, none", lambda: workloads.weighted(rows=70, V=32000, reduction="none"),
     "none"),
    ("odd V (general kernel), mean",
     lambda: workloads.random_case(5, 40, 1001, dtype="f32", label_smoothing=0.1,
                                   lse_square_scale=1e-3), "mean"),
]


@pytest.mark.parametrize("name,make,reduction", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_ce_fwd_on_two_calls_in_a_row(name, make, reduction):
    from softmax_cross_entropy_gb300 import _lib
    case = make()
    ref = _call(_lib.ce_fwd, case, reduction)
    for _ in range(2):  # the second call reuses the array the first one left behind
        got = _call(_lib.ce_fwd_noalloc, case, reduction)
        if reduction == "none":
            assert_rowloss_close(got["loss"], ref["loss"], case.dtype)
            assert_rowloss_close(got["z_loss"], ref["z_loss"], case.dtype, "z_loss")
        else:
            assert_loss_close(float(got["loss"][0]), float(ref["loss"][0]), case.dtype)
            assert_loss_close(float(got["z_loss"][0]), float(ref["z_loss"][0]), case.dtype,
                              "z_loss")
        assert np.array_equal(got["pred"], ref["pred"])
        a, b = got["acc"], ref["acc"]
        assert np.array_equal(a, b) or (np.isnan(a).all() and np.isnan(b).all())
        assert_grad_close(got["grad"], ref["grad"], case.dtype)
