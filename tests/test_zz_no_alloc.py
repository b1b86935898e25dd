"""ce_fwd_noalloc: the forward call for callers that cannot allocate device
memory (an allocator's own callbacks, a memory-capped sandbox, a framework
that forbids allocations after start-up). Its scratch is one fixed device
array that every call reuses, so it must give what the oracle gives, and
what ce_fwd gives, call after call, including right after a call that left
the array dirty (a bounded wait that ran out), and it must never make a
library scratch area. Its errors are read with ce_noalloc_status.

This file is collected last on purpose: if it fails, a run that stops at
the first failure has already run every other test."""

import numpy as np
import pytest

import workloads
from ce_gpu import (assert_grad_close, assert_loss_close, assert_rowloss_close, grad_rows_f64,
                    oracle_full, to_device)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from softmax_cross_entropy_gb300 import build, _lib
    build.build()
    _lib.load()


_DT = {"f32": 0, "bf16": 1, "f16": 2}


def _call(entry, case, reduction, stream):
    """Runs one forward entry point through the C ABI on fresh device copies
    of the case's inputs, on `stream`; returns numpy outputs and the
    gradient."""
    from softmax_cross_entropy_gb300 import _lib
    with torch.cuda.stream(stream):
        x, t, w = to_device(case)
        rows, V = case.rows, case.V
        n = rows if reduction == "none" else 1
        f32 = dict(dtype=torch.float32, device=x.device)
        loss = torch.full((n,), float("nan"), **f32)
        zl = torch.full((n,), float("nan"), **f32)
        acc = torch.full((n,), float("nan"), **f32)
        pred = torch.full((rows,), -7, dtype=torch.int64, device=x.device)
    flags = (_lib.CE_FLAG_GRAD | _lib.CE_FLAG_Z_LOSS | _lib.CE_FLAG_ACC | _lib.CE_FLAG_PRED)
    rc = entry(x.data_ptr(), _DT[case.dtype], rows, V,
               t.data_ptr(), None if w is None else w.data_ptr(), case.ignore_index,
               case.label_smoothing, case.lse_square_scale, case.softcap or 0.0,
               {"none": 0, "sum": 1, "mean": 2}[reduction], flags, loss.data_ptr(),
               zl.data_ptr(), acc.data_ptr(), pred.data_ptr(), stream.cuda_stream)
    assert rc == _lib.CE_OK, (_lib.ce_status_string(rc), _lib.ce_last_error())
    stream.synchronize()
    return {"loss": loss.cpu().numpy().astype(np.float64),
            "z_loss": zl.cpu().numpy().astype(np.float64),
            "acc": acc.cpu().numpy().astype(np.float64), "pred": pred.cpu().numpy(),
            "grad": grad_rows_f64(x)}


def _agree(got, ref, case, reduction):
    """got against ref (the oracle's outputs, or ce_fwd's), with the
    tolerances of the parity tests."""
    if reduction == "none":
        assert_rowloss_close(got["loss"], np.asarray(ref["loss"]), case.dtype)
        assert_rowloss_close(got["z_loss"], np.asarray(ref["z_loss"]), case.dtype, "z_loss")
        assert np.array_equal(np.float32(got["acc"]), np.float32(ref["acc"]))
    else:
        assert_loss_close(float(got["loss"][0]), float(np.ravel(ref["loss"])[0]), case.dtype)
        assert_loss_close(float(got["z_loss"][0]), float(np.ravel(ref["z_loss"])[0]),
                          case.dtype, "z_loss")
        a, b = np.float32(got["acc"][0]), np.float32(np.ravel(ref["acc"])[0])
        assert a == b or (np.isnan(a) and np.isnan(b))
    assert np.array_equal(got["pred"], ref["pred"])
    assert_grad_close(got["grad"], ref["grad"], case.dtype)


CASES = [
    ("bf16 V=32768, mean", lambda: workloads.vsweep(V=32768, rows=300), "mean"),
    ("bf16 V=131072 softcap smoothing z-loss, mean",
     lambda: workloads.softcap_z(rows=40), "mean"),
    ("fp32 V=4096 with ignored rows, sum",
     lambda: workloads.tt_fp32(rows=96, V=4096, reduction="sum"), "sum"),
    ("bf16 weighted smoothing, none", lambda: workloads.weighted(rows=70, V=32000, reduction="none"),
     "none"),
    ("odd V (general kernel), mean",
     lambda: workloads.random_case(5, 40, 1001, dtype="f32", label_smoothing=0.1,
                                   lse_square_scale=1e-3), "mean"),
]


@pytest.mark.parametrize("name,make,reduction", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_oracle_and_ce_fwd_on_two_calls_in_a_row(name, make, reduction):
    from softmax_cross_entropy_gb300 import _lib
    case = make()
    want = oracle_full(case, reduction=reduction)
    ref = _call(_lib.ce_fwd, case, reduction, torch.cuda.current_stream())
    # a stream ce_fwd has never seen: the noalloc calls must not make a
    # library scratch area for it
    fresh = torch.cuda.Stream()
    areas = _lib.ce_scratch_areas()
    for _ in range(2):  # the second call reuses the array the first one left behind
        got = _call(_lib.ce_fwd_noalloc, case, reduction, fresh)
        assert _lib.ce_noalloc_status(fresh.cuda_stream) == _lib.CE_OK
        _agree(got, want, case, reduction)
        _agree(got, ref, case, reduction)
    assert _lib.ce_scratch_areas() == areas


@pytest.mark.parametrize("kernel,V", [("4", 4096), ("2", 65536)])
def test_noalloc_after_a_wait_ran_out(monkeypatch, kernel, V):
    """A call whose bounded wait runs out (test hook: CTA 0 leaves its first
    copy out) leaves the array dirty; ce_noalloc_status reports it, and the
    next call, without the hook, matches the oracle."""
    from softmax_cross_entropy_gb300 import _lib
    monkeypatch.setenv("GBCE_KERNEL", kernel)
    monkeypatch.setenv("GBCE_WAIT_TIMEOUT_MS", "20")
    # no ignored rows: CTA 0 owns row 0, and an ignored row would leave it
    # no copy to leave out
    case = workloads.random_case(17, 48, V, dtype="bf16", ignore_frac=0.0, reduction="mean")
    st = torch.cuda.Stream()
    monkeypatch.setenv("GBCE_TEST_STALL_COPY", "1")
    _call(_lib.ce_fwd_noalloc, case, "mean", st)
    assert _lib.ce_noalloc_status(st.cuda_stream) == _lib.CE_ERR_TIMEOUT
    assert _lib.ce_noalloc_status(st.cuda_stream) == _lib.CE_OK  # read clears it
    monkeypatch.delenv("GBCE_TEST_STALL_COPY")
    want = oracle_full(case)
    for _ in range(2):
        got = _call(_lib.ce_fwd_noalloc, case, "mean", st)
        assert _lib.ce_noalloc_status(st.cuda_stream) == _lib.CE_OK
        _agree(got, want, case, "mean")


def test_noalloc_reports_an_out_of_range_target():
    from softmax_cross_entropy_gb300 import _lib
    case = workloads.vsweep(V=4096, rows=64)
    case.target[5] = case.V + 3  # neither ignore_index nor in [0, V)
    st = torch.cuda.Stream()
    got = _call(_lib.ce_fwd_noalloc, case, "sum", st)
    assert _lib.ce_noalloc_status(st.cuda_stream) == _lib.CE_ERR_TARGET_RANGE
    assert np.all(got["grad"][5] == 0.0)  # the row is treated as ignored
    assert got["pred"][5] == -1


def test_noalloc_refuses_a_launch_beyond_its_slots(monkeypatch):
    """With the usable slots lowered to 4 (test hook), a launch over many
    rows needs more and is refused on the host with nothing enqueued."""
    from softmax_cross_entropy_gb300 import _lib
    monkeypatch.setenv("GBCE_TEST_NOALLOC_SLOTS", "4")
    case = workloads.vsweep(V=4096, rows=2048)
    x, t, _ = to_device(case)
    before = x.clone()
    loss = torch.full((1,), float("nan"), dtype=torch.float32, device=x.device)
    st = torch.cuda.current_stream()
    rc = _lib.ce_fwd_noalloc(x.data_ptr(), _DT[case.dtype], case.rows, case.V, t.data_ptr(),
                             None, case.ignore_index, 0.0, 0.0, 0.0, 2, _lib.CE_FLAG_GRAD,
                             loss.data_ptr(), None, None, None, st.cuda_stream)
    assert rc == _lib.CE_ERR_UNSUPPORTED
    assert "partial-sum slots" in _lib.ce_last_error()
    st.synchronize()
    assert torch.equal(x, before) and torch.isnan(loss).all()
