"""GPU parity: the CUDA path, called through the C ABI, against the CPU
float64 oracle on the same seeded inputs.

Every comparison covers the whole batch, element by element. At the full
workload sizes (the launch configuration the benchmark times) the scalar and
per-row outputs come from the oracle's whole-batch forward and the gradient
from the oracle in chunks of rows (tests/ce_gpu.py, assert_grad_whole);
ignored rows are also checked to be exact +0 bit patterns."""
import math
import os

import numpy as np
import pytest

import workloads
from ce_gpu import (CE_DTYPE, assert_grad_close, assert_grad_whole, assert_loss_close,
                    assert_rowloss_close, grad_rows_f64, oracle_full, oracle_rows, run_cuda,
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


def check_full(case, *, want_z=False, want_acc=False, want_pred=False, reduction=None):
    red = reduction or case.reduction
    out = run_cuda(case, want_z=want_z, want_acc=want_acc, want_pred=want_pred, reduction=red)
    ref = oracle_full(case, reduction=red)
    assert out["status"] == 0
    if red == "none":
        assert_rowloss_close(out["loss"], ref["loss"], case.dtype)
        if want_z:
            assert_rowloss_close(out["z_loss"], ref["z_loss"], case.dtype, "z_loss")
        if want_acc:
            assert np.array_equal(out["acc"], ref["acc"])
    else:
        assert_loss_close(out["loss"], ref["loss"], case.dtype)
        if want_z:
            assert_loss_close(out["z_loss"], ref["z_loss"], case.dtype, "z_loss")
        if want_acc:
            assert out["acc"] == np.float32(ref["acc"]) or (
                math.isnan(out["acc"]) and math.isnan(ref["acc"]))
    if want_pred:
        assert np.array_equal(out["pred"], ref["pred"])
    assert_grad_close(grad_rows_f64(out["x"]), ref["grad"], case.dtype)
    return out, ref


def check_whole(case, *, want_z=False, want_acc=False, want_pred=True, reduction=None):
    """Full-size check: scalars, per-row outputs and predictions from the
    oracle's whole-batch forward, every gradient row from the oracle in
    chunks, and ignored rows as exact +0."""
    red = reduction or case.reduction
    out = run_cuda(case, want_z=want_z, want_acc=want_acc, want_pred=want_pred, reduction=red)
    assert out["status"] == 0
    ref = oracle_full(case, reduction=red, want_grad=False)
    if red == "none":
        assert_rowloss_close(out["loss"], ref["loss"], case.dtype)
    else:
        assert_loss_close(out["loss"], ref["loss"], case.dtype)
    if want_z:
        f = assert_rowloss_close if red == "none" else assert_loss_close
        f(out["z_loss"], ref["z_loss"], case.dtype, "z_loss")
    if want_acc:
        assert np.array_equal(np.float32(out["acc"]), np.float32(ref["acc"]))
    if want_pred:
        assert np.array_equal(out["pred"], ref["pred"])
    assert_grad_whole(case, out["x"], reduction=red)
    ign = np.nonzero(case.target == case.ignore_index)[0]
    if ign.size:
        g = out["x"][torch.as_tensor(ign, device=out["x"].device)]
        assert bool((g.view(torch.int32 if case.dtype == "f32" else torch.int16) == 0).all())
    return out, ref


# ------------------------------------------------------------------ workloads

def test_small_config():
    check_full(workloads.small(), want_acc=True, want_pred=True)


@pytest.mark.parametrize("V", workloads.VSWEEP)
def test_vsweep_reduced_rows(V):
    check_full(workloads.vsweep(V=V, rows=96), want_acc=True, want_pred=True)


@pytest.mark.parametrize("V", workloads.VSWEEP)
def test_vsweep_full_size(V):
    check_whole(workloads.vsweep(V=V), want_acc=True)


@pytest.mark.parametrize("V", [32768, 131072])
def test_f16_full_size(V):
    # fp16 logits at the bench shape (4096 rows), whole batch against the oracle
    case = workloads.random_case(21, 4096, V, dtype="f16", std=3.0, ignore_frac=0.05)
    check_whole(case, want_acc=True)


@pytest.mark.parametrize("reduction", ["mean", "sum"])
def test_tt_fp32_full_size(reduction):
    check_whole(workloads.tt_fp32(reduction=reduction), want_acc=True)


@pytest.mark.parametrize("reduction", ["mean", "sum"])
def test_tt_fp32_reduced_rows(reduction):
    check_full(workloads.tt_fp32(rows=40, reduction=reduction), want_acc=True, want_pred=True)


def test_tt_fp32_all_ignored():
    case = workloads.tt_fp32(variant="all_ignored")
    m = run_cuda(case, want_acc=True, want_pred=True)
    assert math.isnan(m["loss"]) and math.isnan(m["acc"])
    assert bool((m["x"].view(torch.int32) == 0).all())  # every gradient is +0
    assert (m["pred"] == -1).all()
    s = run_cuda(case.with_(reduction="sum"))
    assert s["loss"] == 0.0


def test_tt_fp32_nonfinite_in_ignored_rows():
    plain = workloads.tt_fp32(rows=300)
    bad = workloads.tt_fp32(rows=300, variant="nonfinite_ignored")
    assert np.array_equal(plain.target, bad.target)
    assert not np.isfinite(bad.x).all()
    for red in ("mean", "sum"):
        a = run_cuda(plain.with_(reduction=red), want_pred=True)
        b = run_cuda(bad.with_(reduction=red), want_pred=True)
        assert a["loss"] == b["loss"]
        assert np.array_equal(a["pred"], b["pred"])
        assert torch.equal(a["x"], b["x"])  # valid rows identical, ignored rows +0
    ref = oracle_full(bad)
    assert_loss_close(run_cuda(bad)["loss"], ref["loss"], "f32")


def test_softcap_zloss_reduced_rows():
    check_full(workloads.softcap_z(rows=64), want_z=True, want_acc=True, want_pred=True)


def test_softcap_zloss_full_size():
    check_whole(workloads.softcap_z(), want_z=True, want_acc=True)


@pytest.mark.parametrize("reduction", ["none", "mean"])
def test_weighted_reduced_rows(reduction):
    check_full(workloads.weighted(rows=257, reduction=reduction), want_acc=True,
               want_pred=True)


@pytest.mark.parametrize("reduction", ["none", "mean"])
def test_weighted_full_size(reduction):
    check_whole(workloads.weighted(reduction=reduction), want_acc=True)


# ------------------------------------------------------------------ shapes and options

EDGE_SHAPES = [(1, 1), (3, 2), (5, 3), (63, 127), (4, 4097), (2, 8191), (17, 8), (9, 16),
               (33, 64), (7, 1000), (65, 4096), (3, 262144)]
OPTION_SETS = [
    dict(),
    dict(label_smoothing=0.2, lse_square_scale=1e-3),
    dict(softcap=5.0, label_smoothing=0.1),
    dict(weight=True, label_smoothing=0.3, reduction="sum"),
    dict(weight=True, reduction="none", lse_square_scale=1e-2),
]


@pytest.mark.parametrize("rows,V", EDGE_SHAPES)
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("opt", range(len(OPTION_SETS)))
def test_edge_shapes(rows, V, dtype, opt):
    if rows * V > 2_000_000 and opt > 1:
        pytest.skip("large shape covered by the first option sets")
    case = workloads.random_case(1000 + rows * 7 + V, rows, V, dtype=dtype,
                                 **dict(OPTION_SETS[opt]))
    check_full(case, want_z=True, want_acc=True, want_pred=True)


@pytest.mark.parametrize("cluster", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("dtype,V,rows", [("bf16", 16384, 203), ("f32", 8192, 77),
                                          ("bf16", 32000, 50), ("bf16", 131072, 37)])
def test_forced_cluster_sizes(monkeypatch, cluster, dtype, V, rows):
    monkeypatch.setenv("GBCE_CLUSTER", str(cluster))
    for opts in (dict(), dict(weight=True, label_smoothing=0.1, softcap=20.0,
                               lse_square_scale=1e-3)):
        case = workloads.random_case(7 + cluster, rows, V, dtype=dtype, **opts)
        check_full(case, want_z=True, want_acc=True, want_pred=True)


@pytest.mark.parametrize("cfg", range(6))
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_forced_cta_shapes(monkeypatch, cfg, dtype):
    # every CTA shape of the staged kernel, with the smallest cluster it fits
    monkeypatch.setenv("GBCE_CFG", str(cfg))
    case = workloads.random_case(40 + cfg, 150, 8192, dtype=dtype, label_smoothing=0.05,
                                 lse_square_scale=1e-4)
    check_full(case, want_z=True, want_acc=True, want_pred=True)


def test_general_path_forced(monkeypatch):
    monkeypatch.setenv("GBCE_CLUSTER", "-1")  # skip the staged kernel
    case = workloads.random_case(11, 70, 8192, dtype="bf16", weight=True, label_smoothing=0.1,
                                 softcap=20.0, lse_square_scale=1e-3)
    check_full(case, want_z=True, want_acc=True, want_pred=True)


def test_unaligned_base_pointer():
    case = workloads.random_case(12, 31, 1024, dtype="bf16", label_smoothing=0.1)
    x, _, _ = to_device(case)
    buf = torch.empty(x.numel() + 1, dtype=x.dtype, device=x.device)
    view = buf[1:].view(case.rows, case.V)
    view.copy_(x)
    assert view.data_ptr() % 16 != 0
    out = run_cuda(case, x=view, want_pred=True)
    ref = oracle_full(case)
    assert_loss_close(out["loss"], ref["loss"], "bf16")
    assert np.array_equal(out["pred"], ref["pred"])
    assert_grad_close(grad_rows_f64(view), ref["grad"], "bf16")


def test_argmax_ties_across_cta_slices():
    rows, V = 48, 131072
    case = workloads.vsweep(V=V, rows=rows)
    x = workloads.bf16_bits_to_f32(case.x).copy()
    top = np.float32(64.0)
    cols = [(32767, 32768), (40000, 100000), (131071, 5), (65536, 65535), (98304, 98303)]
    for r in range(rows):
        a, b = cols[r % len(cols)]
        x[r, a] = top
        x[r, b] = top
    case = case.with_(x=workloads.f32_to_bf16_bits(x))
    out = run_cuda(case, want_pred=True, want_acc=True)
    ref = oracle_full(case, want_grad=False)
    valid = case.target != case.ignore_index
    assert np.array_equal(out["pred"], ref["pred"])
    expect = np.array([min(cols[r % len(cols)]) for r in range(rows)])
    assert np.array_equal(out["pred"][valid], expect[valid])


def test_int64_targets():
    case = workloads.random_case(13, 50, 4096, dtype="bf16", label_smoothing=0.1)
    x, t, _ = to_device(case)
    out = run_cuda(case, target=t.to(torch.int64), want_pred=True)
    ref = oracle_full(case)
    assert_loss_close(out["loss"], ref["loss"], "bf16")
    assert np.array_equal(out["pred"], ref["pred"])
    assert_grad_close(grad_rows_f64(out["x"]), ref["grad"], "bf16")


def test_custom_ignore_index():
    case = workloads.random_case(14, 64, 512, dtype="f32", ignore_frac=0.0)
    case.target[::3] = 7
    case = case.with_(ignore_index=7)
    check_full(case, want_acc=True, want_pred=True)


def test_out_of_range_target_is_reported_and_ignored():
    from softmax_cross_entropy_gb300 import _lib
    case = workloads.random_case(15, 20, 256, dtype="f32", ignore_frac=0.0)
    bad = case.target.copy()
    bad[4] = 256
    bad[9] = -3
    out = run_cuda(case.with_(target=bad), want_pred=True)
    assert out["status"] == _lib.CE_ERR_TARGET_RANGE
    as_ignored = bad.copy()
    as_ignored[[4, 9]] = case.ignore_index
    ref = oracle_full(case.with_(target=as_ignored))
    assert_loss_close(out["loss"], ref["loss"], "f32")
    assert_grad_close(grad_rows_f64(out["x"]), ref["grad"], "f32")
    assert out["pred"][4] == -1 and out["pred"][9] == -1
    # the status word is cleared by the read
    assert run_cuda(case)["status"] == 0


def test_empty_batch():
    case = workloads.random_case(16, 0, 64, dtype="f32")
    m = run_cuda(case, want_acc=True, want_z=True)
    assert math.isnan(m["loss"]) and math.isnan(m["z_loss"]) and math.isnan(m["acc"])
    s = run_cuda(case.with_(reduction="sum"))
    assert s["loss"] == 0.0


def test_forward_only_leaves_logits_untouched():
    case = workloads.vsweep(V=65536, rows=64)
    x, _, _ = to_device(case)
    before = x.clone()
    out = run_cuda(case, x=x, grad=False, want_pred=True)
    assert torch.equal(x, before)
    ref = oracle_full(case, want_grad=False)
    assert_loss_close(out["loss"], ref["loss"], "bf16")
    assert np.array_equal(out["pred"], ref["pred"])


@pytest.mark.parametrize("make", [
    lambda: workloads.vsweep(V=131072, rows=300),
    lambda: workloads.softcap_z(rows=200),
    lambda: workloads.tt_fp32(rows=200, reduction="sum"),
    lambda: workloads.weighted(rows=300, reduction="none"),
], ids=["bf16-131072", "softcap-131072", "fp32-128256-sum", "weighted-32000-none"])
def test_forward_only_streams_once_and_matches(make):
    # without CE_FLAG_GRAD the long-row kernel reads each row once; loss,
    # z-loss, accuracy and predictions must still be the oracle's and the
    # logits must be left as they were
    case = make()
    x, _, _ = to_device(case)
    before = x.clone()
    red = case.reduction
    out = run_cuda(case, x=x, grad=False, want_z=True, want_acc=True, want_pred=True)
    assert out["status"] == 0
    assert torch.equal(x, before)
    ref = oracle_full(case, want_grad=False)
    if red == "none":
        assert_rowloss_close(out["loss"], ref["loss"], case.dtype)
        assert_rowloss_close(out["z_loss"], ref["z_loss"], case.dtype, "z_loss")
        assert np.array_equal(out["acc"], ref["acc"])
    else:
        assert_loss_close(out["loss"], ref["loss"], case.dtype)
        assert_loss_close(out["z_loss"], ref["z_loss"], case.dtype, "z_loss")
        assert np.float32(out["acc"]) == np.float32(ref["acc"])
    assert np.array_equal(out["pred"], ref["pred"])


def test_deterministic():
    case = workloads.softcap_z(rows=300)
    a = run_cuda(case, want_z=True)
    b = run_cuda(case, want_z=True)
    assert a["loss"] == b["loss"] and a["z_loss"] == b["z_loss"]
    assert torch.equal(a["x"], b["x"])


# ------------------------------------------------------------------ backward

@pytest.mark.parametrize("dtype,V", [("bf16", 4096), ("f32", 1000), ("bf16", 131072),
                                     ("f16", 4096)])
def test_backward_scales_stored_gradient(dtype, V):
    import oracle
    from softmax_cross_entropy_gb300 import _lib
    rows = 24
    case = workloads.random_case(17, rows, V, dtype=dtype, reduction="none")
    out = run_cuda(case)
    g = out["x"]
    stored = grad_rows_f64(g)
    dt = CE_DTYPE[dtype]
    st = torch.cuda.current_stream().cuda_stream
    one = torch.ones(1, device="cuda")
    assert _lib.ce_bwd(one.data_ptr(), 0, g.data_ptr(), dt, rows, V, st) == 0
    np.testing.assert_array_equal(grad_rows_f64(g), stored)  # factor 1: untouched
    go = torch.from_numpy(np.random.default_rng(0).uniform(-2, 2, rows).astype(np.float32))
    go[3] = 1.0
    assert _lib.ce_bwd(go.cuda().data_ptr(), 1, g.data_ptr(), dt, rows, V, st) == 0
    torch.cuda.synchronize()
    want = oracle.backward(oracle_full(case)["grad"], go.numpy().astype(np.float64))
    assert_grad_close(grad_rows_f64(g), want, dtype)
    half = torch.full((1,), 0.5, device="cuda")
    before = grad_rows_f64(g)
    assert _lib.ce_bwd(half.data_ptr(), 0, g.data_ptr(), dt, rows, V, st) == 0
    if dtype == "f16":
        # halving an fp16 subnormal rounds: numpy's fp16 product rounds the
        # same way (exact product, one rounding to nearest even)
        want_half = (before.astype(np.float16) * np.float16(0.5)).astype(np.float64)
    else:
        want_half = before * 0.5
    np.testing.assert_array_equal(grad_rows_f64(g), want_half)


def test_autograd_api_matches_c_abi():
    import softmax_cross_entropy_gb300 as ce
    case = workloads.weighted(rows=129, V=32000)
    x, t, w = to_device(case)
    x.requires_grad_(True)
    out = ce.cross_entropy(x, t, weight=w, label_smoothing=case.label_smoothing,
                           return_token_accuracy=True, return_predicted_tokens=True)
    (out.loss * 3.0).backward()
    ref = oracle_full(case)
    assert_loss_close(float(out.loss), ref["loss"], "bf16")
    assert np.array_equal(out.predicted_tokens.cpu().numpy(), ref["pred"])
    assert_grad_close(grad_rows_f64(x.grad), 3.0 * ref["grad"], "bf16")
    assert ce.device_status() == 0


def test_module_reduction_none_backward():
    import softmax_cross_entropy_gb300 as ce
    case = workloads.random_case(18, 40, 2048, dtype="f32", reduction="none",
                                 lse_square_scale=1e-3)
    x, t, _ = to_device(case)
    x.requires_grad_(True)
    loss = ce.CrossEntropyLoss(reduction="none", lse_square_scale=1e-3)(x, t)
    go = torch.linspace(-1, 1, 40, device="cuda")
    loss.backward(go)
    import oracle
    ref = oracle_full(case)
    assert_rowloss_close(loss.detach().cpu().numpy(), ref["loss"], "f32")
    want = oracle.backward(ref["grad"], go.cpu().numpy().astype(np.float64))
    assert_grad_close(grad_rows_f64(x.grad), want, "f32")


# ------------------------------------------------------------------ kernel variants

KINDS = {"staged": "1", "stream": "2", "general": "3", "reg": "4"}


@pytest.mark.parametrize("kind", sorted(KINDS) + ["stream8", "stream16"])
@pytest.mark.parametrize("dtype,V,rows", [("bf16", 4096, 300), ("bf16", 32768, 90),
                                          ("f32", 8192, 77), ("bf16", 131072, 20),
                                          ("f32", 24, 33), ("f16", 8192, 50),
                                          ("f16", 131072, 9)])
def test_kernel_kinds(monkeypatch, kind, dtype, V, rows):
    if dtype == "f16" and kind == "staged":
        pytest.skip("the staged kernel has no fp16 variant")
    if kind == "reg" and V * (4 if dtype == "f32" else 2) > 32768:
        pytest.skip("the register-resident kernel takes rows of at most 32 KB")
    if kind in ("stream8", "stream16"):
        monkeypatch.setenv("GBCE_STREAM_WARPS", kind[6:])
        kind = "stream"
    monkeypatch.setenv("GBCE_KERNEL", KINDS[kind])
    for opts in (dict(), dict(label_smoothing=0.1, softcap=20.0, lse_square_scale=1e-3),
                 dict(weight=True, reduction="none")):
        case = workloads.random_case(60 + rows, rows, V, dtype=dtype, **opts)
        check_full(case, want_z=True, want_acc=True, want_pred=True)


@pytest.mark.parametrize("warps", [8, 16])
@pytest.mark.parametrize("groups", [1, 2, 4, 8])
def test_stream_groups(monkeypatch, groups, warps):
    monkeypatch.setenv("GBCE_KERNEL", "2")
    monkeypatch.setenv("GBCE_STREAM_GROUPS", str(groups))
    monkeypatch.setenv("GBCE_STREAM_WARPS", str(warps))
    case = workloads.random_case(70 + groups, 203, 2048, dtype="bf16", label_smoothing=0.1,
                                 lse_square_scale=1e-4)
    check_full(case, want_z=True, want_acc=True, want_pred=True)


@pytest.mark.parametrize("warps", [8, 16])
@pytest.mark.parametrize("dtype,V", [("bf16", 32768), ("f32", 20000), ("bf16", 8200),
                                     ("f16", 16384)])
def test_stream_twice_from_l2(monkeypatch, dtype, V, warps):
    # rows streamed through the ring twice (the large-vocabulary mode), at
    # sizes the oracle checks whole
    monkeypatch.setenv("GBCE_KERNEL", "2")
    monkeypatch.setenv("GBCE_STREAM_TWICE", "1")
    monkeypatch.setenv("GBCE_STREAM_WARPS", str(warps))
    for opts in (dict(), dict(label_smoothing=0.2, softcap=10.0)):
        case = workloads.random_case(80, 61, V, dtype=dtype, **opts)
        check_full(case, want_z=True, want_acc=True, want_pred=True)


@pytest.mark.parametrize("dtype,V,rows,twice", [
    ("bf16", 4096, 150, 0),    # rows resident in the ring
    ("bf16", 32000, 70, 0),    # the weights leave room for three 32 KB slots
    ("bf16", 32000, 70, 1),
    ("f32", 8192, 40, 0),
    ("f32", 20000, 33, 1),
    ("bf16", 49152, 13, 0),    # 192 KB of weights: smaller slots
    ("f32", 24, 33, 0),
    ("f16", 32000, 40, 0),
])
def test_stream_weighted_smoothing(monkeypatch, dtype, V, rows, twice):
    # class weights with label smoothing in the streaming kernel, the weights
    # held in shared memory
    monkeypatch.setenv("GBCE_KERNEL", "2")
    if twice:
        monkeypatch.setenv("GBCE_STREAM_TWICE", "1")
    for opts in (dict(weight=True, label_smoothing=0.05),
                 dict(weight=True, label_smoothing=0.1, softcap=15.0, lse_square_scale=1e-3,
                      reduction="none"),
                 dict(weight=True, label_smoothing=1.0, reduction="sum", ignore_frac=0.3)):
        case = workloads.random_case(90 + rows, rows, V, dtype=dtype, **opts)
        check_full(case, want_z=True, want_acc=True, want_pred=True)


@pytest.mark.parametrize("dtype,V,rows", [
    ("bf16", 1024, 150),    # one warp a row
    ("bf16", 4096, 300),    # the bench sweep's shortest row: 4 warps
    ("bf16", 5000, 97),     # ragged: the last warp's vectors partly past the row
    ("bf16", 16000, 40),    # 8 warps of 8 vectors, the last vectors ragged
    ("bf16", 16384, 33),    # 8 warps of 8 vectors exactly
    ("bf16", 32000, 20),    # 16 vectors a thread only (8 warps)
    ("f32", 8192, 70),
    ("f32", 6000, 21),
    ("f32", 12, 33),        # three vectors: most threads hold nothing
    ("f16", 8192, 50),
])
@pytest.mark.parametrize("nvl", ["8", "16"])
def test_register_kernel(monkeypatch, dtype, V, rows, nvl):
    # the register-resident kernel forced, 8 or 16 vectors a thread, every
    # option set, whole-batch comparison
    if nvl == "8" and V * (4 if dtype == "f32" else 2) > 32768:
        pytest.skip("8 vectors a thread hold rows of at most 32 KB")
    monkeypatch.setenv("GBCE_KERNEL", "4")
    monkeypatch.setenv("GBCE_REG_NVL", nvl)
    for opts in (dict(),
                 dict(label_smoothing=0.1, softcap=20.0, lse_square_scale=1e-3),
                 dict(weight=True, reduction="none"),
                 dict(weight=True, label_smoothing=0.05, reduction="sum"),
                 dict(weight=True, label_smoothing=0.2, softcap=8.0, ignore_frac=0.3)):
        case = workloads.random_case(110 + rows, rows, V, dtype=dtype, **opts)
        check_full(case, want_z=True, want_acc=True, want_pred=True)


@pytest.mark.parametrize("dtype,V,rows", [
    ("bf16", 24576, 41),    # one CTA a row, two slots
    ("bf16", 40000, 37),    # one CTA a row, the last slot ragged
    ("bf16", 65536, 21),    # one CTA a row, every TMEM column
    ("bf16", 65544, 19),    # two CTAs, the second holds one vector
    ("bf16", 131072, 23),   # the softcap bench shape: two CTAs of 64K elements
    ("f32", 128256, 11),    # two CTAs of 16384 vectors, the second ragged
    ("f16", 100000, 13),
    ("bf16", 200000, 5),    # four CTAs (clusters up to eight)
])
def test_tensor_memory_kernel(monkeypatch, dtype, V, rows):
    # the softcap kernel that keeps tanh's intermediate in TMEM, forced,
    # whole-batch comparison for every option it takes (softcap <= 40, no
    # class-weighted smoothing)
    monkeypatch.setenv("GBCE_KERNEL", "6")
    for opts in (dict(softcap=30.0, std=8.0),
                 dict(softcap=30.0, std=8.0, label_smoothing=0.1, lse_square_scale=1e-4),
                 dict(softcap=5.0, std=20.0, label_smoothing=0.05, reduction="none"),
                 dict(softcap=40.0, std=3.0, weight=True, lse_square_scale=1e-3, reduction="sum",
                      ignore_frac=0.3),
                 dict(softcap=1.0, std=3.0, ignore_frac=1.0)):
        case = workloads.random_case(170 + rows, rows, V, dtype=dtype, **opts)
        check_full(case, want_z=True, want_acc=True, want_pred=True)


def test_tensor_memory_kernel_ties_and_forward_only(monkeypatch):
    monkeypatch.setenv("GBCE_KERNEL", "6")
    case = workloads.random_case(191, 9, 131072, dtype="bf16", std=2.0, softcap=20.0,
                                 label_smoothing=0.1, ignore_frac=0.0)
    # the row maximum twice, once in each CTA's slice, and twice in one vector
    case.x[0, 70000] = case.x[0, 5] = workloads.f32_to_bf16_bits(np.array([40.0], np.float32))[0]
    case.x[1, 9] = case.x[1, 10] = workloads.f32_to_bf16_bits(np.array([40.0], np.float32))[0]
    check_full(case, want_z=True, want_acc=True, want_pred=True)
    x, _, _ = to_device(case)
    before = x.clone()
    out = run_cuda(case, x=x, grad=False, want_pred=True)
    assert torch.equal(x, before)
    assert out["pred"][0] == 5 and out["pred"][1] == 9


def test_tensor_memory_kernel_refuses_large_softcaps(monkeypatch):
    from softmax_cross_entropy_gb300 import _lib
    monkeypatch.setenv("GBCE_KERNEL", "6")
    case = workloads.random_case(192, 4, 131072, dtype="bf16", softcap=50.0)
    x, t, _ = to_device(case)
    loss = torch.empty(1, dtype=torch.float32, device="cuda")
    rc = _lib.ce_fwd(x.data_ptr(), 1, case.rows, case.V, t.data_ptr(), None, -100, 0.0, 0.0,
                     50.0, 2, _lib.CE_FLAG_GRAD, loss.data_ptr(), None, None, None,
                     torch.cuda.current_stream().cuda_stream)
    assert rc == _lib.CE_ERR_UNSUPPORTED


@pytest.mark.parametrize("sw,nbuf", [("0", "1"), ("1", "2"), ("0", "2")])
@pytest.mark.parametrize("dtype,V,rows", [("bf16", 32000, 37), ("bf16", 4096, 301),
                                          ("f32", 5000, 45), ("f16", 16384, 29)])
def test_register_kernel_weight_and_buffer_options(monkeypatch, sw, nbuf, dtype, V, rows):
    # class weights from L1/L2 (GBCE_REG_SW=0) or shared memory (the
    # default), one or two row buffers a team (GBCE_REG_NBUF), whole batch
    monkeypatch.setenv("GBCE_KERNEL", "4")
    monkeypatch.setenv("GBCE_REG_SW", sw)
    monkeypatch.setenv("GBCE_REG_NBUF", nbuf)
    for opts in (dict(weight=True, label_smoothing=0.05, reduction="mean", ignore_frac=0.2),
                 dict(weight=True, label_smoothing=0.1, softcap=12.0, lse_square_scale=1e-3,
                      reduction="none"),
                 dict(label_smoothing=0.1, reduction="sum")):
        case = workloads.random_case(150 + rows, rows, V, dtype=dtype, **opts)
        check_full(case, want_z=True, want_acc=True, want_pred=True)


@pytest.mark.parametrize("dtype,V,rows", [
    ("bf16", 65536, 24),    # 2 CTAs of 64 KB
    ("bf16", 131072, 20),   # 4 CTAs
    ("bf16", 98312, 17),    # 4 CTAs, the last holds one vector
    ("bf16", 40000, 30),    # 2 CTAs, the second ragged
    ("f32", 128256, 9),     # 8 CTAs of 16 vectors a thread
    ("f16", 50264, 19),
])
def test_register_cluster_kernel(monkeypatch, dtype, V, rows):
    # a cluster of CTAs a row (row maximum and sums merged through
    # distributed shared memory), every option set, whole-batch comparison
    monkeypatch.setenv("GBCE_KERNEL", "5")
    for opts in (dict(),
                 dict(label_smoothing=0.1, softcap=20.0, lse_square_scale=1e-3),
                 dict(weight=True, reduction="none"),
                 dict(weight=True, label_smoothing=0.05, reduction="sum"),
                 dict(weight=True, label_smoothing=0.2, softcap=8.0, ignore_frac=0.3)):
        case = workloads.random_case(130 + rows, rows, V, dtype=dtype, **opts)
        check_full(case, want_z=True, want_acc=True, want_pred=True)


def test_register_cluster_ties_across_ctas(monkeypatch):
    # the row maximum repeated in several CTAs' slices: the lowest index wins
    monkeypatch.setenv("GBCE_KERNEL", "5")
    V = 131072
    case = workloads.random_case(6, 40, V, dtype="bf16")
    x = case.x.copy()
    top = workloads.f32_to_bf16_bits(np.array([60.0], np.float32))[0]
    firsts = []
    for r in range(case.rows):
        cols = sorted({(r * 7919) % V, (r * 7919 + 40000) % V, (r * 7919 + 90001) % V})
        x[r, cols] = top
        firsts.append(cols[0])
    case = case.with_(x=x)
    out, ref = check_full(case, want_acc=True, want_pred=True)
    valid = case.target != case.ignore_index
    assert np.array_equal(out["pred"][valid], np.array(firsts)[valid])


def test_register_kernel_counts_back_to_back(monkeypatch):
    # Launches of the register kernel (and its count kernel) queued back to
    # back on one stream, with a different D each (weights, ignore
    # fractions, a batch with every row ignored, a single row), each against
    # the oracle.
    from softmax_cross_entropy_gb300 import _lib
    monkeypatch.setenv("GBCE_KERNEL", "4")
    cases = [workloads.random_case(61, 300, 4096, dtype="bf16", weight=True, ignore_frac=0.2),
             workloads.random_case(62, 300, 4096, dtype="bf16", ignore_frac=1.0),
             workloads.random_case(63, 1, 4096, dtype="bf16", weight=True),
             workloads.random_case(64, 977, 2048, dtype="f32", ignore_frac=0.5),
             workloads.random_case(65, 300, 4096, dtype="bf16", weight=True, ignore_frac=0.05)]
    st = torch.cuda.current_stream().cuda_stream
    runs = []
    for case in cases:
        x, t, w = to_device(case)
        loss = torch.full((1,), float("nan"), device="cuda")
        acc = torch.full((1,), float("nan"), device="cuda")
        rc = _lib.ce_fwd(x.data_ptr(), CE_DTYPE[case.dtype], case.rows, case.V, t.data_ptr(),
                         None if w is None else w.data_ptr(), case.ignore_index, 0.0, 0.0, 0.0,
                         2, _lib.CE_FLAG_GRAD | _lib.CE_FLAG_ACC, loss.data_ptr(), None,
                         acc.data_ptr(), None, st)
        assert rc == 0
        runs.append((case, x, t, w, loss, acc))
    assert _lib.ce_device_status(st) == 0
    for case, x, t, w, loss, acc in runs:
        ref = oracle_full(case.with_(label_smoothing=0.0), reduction="mean")
        if math.isnan(ref["loss"]):
            assert math.isnan(float(loss.item())) and math.isnan(float(acc.item()))
        else:
            assert_loss_close(float(loss.item()), ref["loss"], case.dtype)
            assert np.float32(acc.item()) == np.float32(ref["acc"])
        assert_grad_close(grad_rows_f64(x), ref["grad"], case.dtype)


def test_register_kernel_counts_many_rows(monkeypatch):
    # many rows and a short row: many count-kernel CTAs
    monkeypatch.setenv("GBCE_KERNEL", "4")
    case = workloads.random_case(66, 40000, 256, dtype="bf16", weight=True, ignore_frac=0.3)
    check_full(case, want_acc=True)


def test_register_kernel_ties_across_warps(monkeypatch):
    # the row maximum repeated in several warps' vectors: the lowest index
    # wins
    monkeypatch.setenv("GBCE_KERNEL", "4")
    case = workloads.random_case(5, 64, 16384, dtype="bf16")
    x = case.x.copy()
    top = workloads.f32_to_bf16_bits(np.array([60.0], np.float32))[0]
    for r in range(case.rows):
        cols = sorted({(r * 977) % 16384, (r * 977 + 4100) % 16384, (r * 977 + 9000) % 16384})
        x[r, cols] = top
    case = case.with_(x=x)
    out, ref = check_full(case, want_acc=True, want_pred=True)
    valid = case.target != case.ignore_index
    firsts = np.array([min((r * 977) % 16384, (r * 977 + 4100) % 16384,
                           (r * 977 + 9000) % 16384) for r in range(case.rows)])
    assert np.array_equal(out["pred"][valid], firsts[valid])


def test_register_kernel_unaligned_weights_fall_back(monkeypatch):
    # class weights that do not start on a 16-byte boundary: the register
    # kernel's vector weight loads are not used, the result is the same
    case = workloads.random_case(7, 50, 4096, dtype="bf16", weight=True, label_smoothing=0.1)
    import torch as _t
    from softmax_cross_entropy_gb300 import _lib
    x, t, w = to_device(case)
    wbuf = _t.empty(case.V + 1, dtype=_t.float32, device="cuda")
    wbuf[1:] = w
    w_off = wbuf[1:]
    loss = _t.empty(1, device="cuda")
    rc = _lib.ce_fwd(x.data_ptr(), 1, case.rows, case.V, t.data_ptr(), w_off.data_ptr(), -100,
                     0.1, 0.0, 0.0, 2, _lib.CE_FLAG_GRAD, loss.data_ptr(), None, None, None,
                     _t.cuda.current_stream().cuda_stream)
    assert rc == 0
    ref = oracle_full(case)
    assert_loss_close(float(loss.item()), ref["loss"], "bf16")
    assert_grad_close(grad_rows_f64(x), ref["grad"], "bf16")
