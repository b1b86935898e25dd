"""Row-sharded batch on one GPU: the shards' counts (ce_count) are added as
an all-reduce would add them, each shard runs ce_fwd_shard with the batch
totals, and the shards' outputs must give the oracle's whole-batch mean
loss, z-loss, accuracy and gradient."""
import math

import numpy as np
import pytest

import workloads
from ce_gpu import CE_DTYPE, assert_grad_close, assert_loss_close, grad_rows_f64, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from softmax_cross_entropy_gb300 import build, _lib
    build.build()
    _lib.load()


def _counts(lib, t, w, V, ignore_index, st):
    c = torch.full((2,), float("nan"), dtype=torch.float64, device="cuda")
    flags = lib.CE_FLAG_TARGET_I64 if t.dtype == torch.int64 else 0
    rc = lib.ce_count(t.data_ptr() if t.numel() else None, None if w is None else w.data_ptr(),
                      t.numel(), V, ignore_index, flags, c.data_ptr(), st)
    assert rc == 0, lib.ce_last_error()
    return c


@pytest.mark.parametrize("dtype,rows,V,cuts,opts", [
    ("bf16", 300, 8192, (0, 97, 200, 300), dict()),
    ("f32", 77, 4096, (0, 40, 77), dict(weight=True, label_smoothing=0.1, lse_square_scale=1e-3)),
    ("bf16", 64, 32000, (0, 0, 30, 64), dict(weight=True, softcap=20.0)),  # an empty shard
    ("f16", 90, 16384, (0, 45, 90), dict(label_smoothing=0.05)),
    ("bf16", 40, 4096, (0, 20, 40), dict(ignore_frac=1.0)),  # every row ignored
])
def test_sharded_mean_matches_whole_batch(dtype, rows, V, cuts, opts):
    import oracle
    from softmax_cross_entropy_gb300 import _lib
    case = workloads.random_case(31 + rows, rows, V, dtype=dtype, **opts)
    x, t, w = to_device(case)
    st = torch.cuda.current_stream().cuda_stream
    shards = list(zip(cuts[:-1], cuts[1:]))
    total = torch.zeros(2, dtype=torch.float64, device="cuda")
    for lo, hi in shards:  # the all-reduce
        total += _counts(_lib, t[lo:hi], w, V, case.ignore_index, st)
    ref = oracle.forward(case.x, case.target, dtype=dtype, weight=case.weight, **case.options())
    ref_acc = oracle.forward(case.x, case.target, dtype=dtype, weight=case.weight,
                             want_grad=False, **{**case.options(), "reduction": "sum"})["acc"]
    n_valid = int(np.sum(case.target != case.ignore_index))
    assert total[1].item() == n_valid
    loss = zl = acc = 0.0
    flags = (_lib.CE_FLAG_GRAD | _lib.CE_FLAG_Z_LOSS | _lib.CE_FLAG_ACC |
             (_lib.CE_FLAG_TARGET_I64 if t.dtype == torch.int64 else 0))
    for lo, hi in shards:
        out = torch.full((3,), float("nan"), device="cuda")
        rc = _lib.ce_fwd_shard(x[lo:hi].data_ptr() if hi > lo else None, CE_DTYPE[dtype], hi - lo,
                               V, t[lo:hi].data_ptr() if hi > lo else None,
                               None if w is None else w.data_ptr(), case.ignore_index,
                               case.label_smoothing, case.lse_square_scale, case.softcap or 0.0,
                               _lib.CE_RED_MEAN, flags, out[0:].data_ptr(), out[1:].data_ptr(),
                               out[2:].data_ptr(), None, total.data_ptr(), st)
        assert rc == 0, _lib.ce_last_error()
        assert _lib.ce_device_status(st) == 0
        o = out.cpu().numpy().astype(np.float64)
        loss, zl, acc = loss + o[0], zl + o[1], acc + o[2]
    if n_valid == 0:
        assert math.isnan(loss) and math.isnan(zl) and math.isnan(acc)
    else:
        assert_loss_close(loss, ref["loss"], dtype)
        assert_loss_close(zl, ref["z_loss"], dtype, "z_loss")
        assert acc == pytest.approx(ref_acc, rel=1e-6)
    # every shard's gradient is already that of the batch mean
    assert_grad_close(grad_rows_f64(x), ref["grad"], dtype)


def test_count_matches_host_count():
    from softmax_cross_entropy_gb300 import _lib
    from softmax_cross_entropy_gb300.distributed import local_denominator
    st = torch.cuda.current_stream().cuda_stream
    for rows, V, weight, i64 in ((0, 10, False, False), (1, 5, True, False), (5000, 300, True, True),
                                 (100000, 50, False, True)):
        case = workloads.random_case(5 + rows, rows, V, dtype="f32",
                                     **(dict(weight=True) if weight else {}))
        t = torch.from_numpy(case.target.astype(np.int64 if i64 else np.int32)).cuda()
        t[:3] = V + 2 if rows >= 3 else t[:3]  # out-of-range targets are not counted
        w = None if case.weight is None else torch.from_numpy(case.weight).cuda()
        got = _counts(_lib, t, w, V, case.ignore_index, st).cpu().numpy()
        D, n = local_denominator(t.cpu().numpy(), case.ignore_index, case.weight, V)
        assert got[1] == n
        assert got[0] == pytest.approx(D, rel=1e-12)
        again = _counts(_lib, t, w, V, case.ignore_index, st).cpu().numpy()
        assert np.array_equal(got, again)  # deterministic
