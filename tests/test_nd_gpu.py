"""GPU parity of the N-D form (logits (N, C, d1, ..., dk), class dimension 1;
F.cross_entropy's N-D form, tt-mlir pull request #9324 review comments: the
reductions run over every non-class dimension). The CUDA path is called
through the C ABI (ce_fwd_nd, ce_bwd_nd) and through the autograd API, and
compared element by element with the oracle's N-D form on the same seeded
inputs, in every tile layout of the kernel: 16-byte vectors of positions or
single positions, the tile staged in shared memory or read again from
global memory."""
import math
import os

import numpy as np
import pytest

import workloads
from ce_gpu import (CE_DTYPE, assert_grad_close, assert_loss_close, assert_rowloss_close)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

RED = {"none": 0, "sum": 1, "mean": 2}
# GBCE_ND_MODE: 1 vector staged, 2 vector from global, 3 scalar staged,
# 4 scalar from global, 0 automatic
MODES = (0, 1, 2, 3, 4)


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from softmax_cross_entropy_gb300 import build, _lib
    build.build()
    _lib.load()


@pytest.fixture
def nd_mode(monkeypatch):
    def set_mode(m):
        monkeypatch.setenv("GBCE_ND_MODE", str(m))
    yield set_mode


def _dev_logits(case):
    if case.dtype in ("bf16", "f16"):
        x = torch.from_numpy(np.ascontiguousarray(case.x).view(np.int16)).view(
            torch.bfloat16 if case.dtype == "bf16" else torch.float16)
    else:
        x = torch.from_numpy(np.ascontiguousarray(case.x))
    return x.cuda()


def run_nd(case, *, grad=True, want_z=False, want_acc=False, want_pred=False, x=None,
           target=None):
    """ce_fwd_nd through the C ABI; numpy outputs plus the device buffer."""
    from softmax_cross_entropy_gb300 import _lib
    dx = _dev_logits(case) if x is None else x
    dt = torch.from_numpy(np.ascontiguousarray(case.target)).cuda() if target is None else target
    dw = None if case.weight is None else torch.from_numpy(case.weight).cuda()
    shape = case.x.shape
    N, C = shape[0], shape[1]
    inner = math.prod(shape[2:])
    pos = (N,) + tuple(shape[2:])
    n = pos if case.reduction == "none" else (1,)
    f32 = dict(dtype=torch.float32, device="cuda")
    loss = torch.full(n, float("nan"), **f32)
    zl = torch.full(n, float("nan"), **f32) if want_z else None
    acc = torch.full(n, float("nan"), **f32) if want_acc else None
    pred = torch.full(pos, -7, dtype=torch.int64, device="cuda") if want_pred else None
    flags = ((_lib.CE_FLAG_GRAD if grad else 0) | (_lib.CE_FLAG_Z_LOSS if want_z else 0) |
             (_lib.CE_FLAG_ACC if want_acc else 0) | (_lib.CE_FLAG_PRED if want_pred else 0) |
             (_lib.CE_FLAG_TARGET_I64 if dt.dtype == torch.int64 else 0))
    st = torch.cuda.current_stream().cuda_stream
    rc = _lib.ce_fwd_nd(dx.data_ptr(), CE_DTYPE[case.dtype], N, C, inner, dt.data_ptr(),
                        None if dw is None else dw.data_ptr(), case.ignore_index,
                        case.label_smoothing, case.lse_square_scale, case.softcap or 0.0,
                        RED[case.reduction], flags, loss.data_ptr(),
                        None if zl is None else zl.data_ptr(),
                        None if acc is None else acc.data_ptr(),
                        None if pred is None else pred.data_ptr(), st)
    assert rc == _lib.CE_OK, (_lib.ce_status_string(rc), _lib.ce_last_error())
    status = _lib.ce_device_status(st)
    out = {"status": status, "x": dx,
           "loss": loss.cpu().numpy().astype(np.float64),
           "z_loss": None if zl is None else zl.cpu().numpy().astype(np.float64),
           "acc": None if acc is None else acc.cpu().numpy().astype(np.float64),
           "pred": None if pred is None else pred.cpu().numpy()}
    if case.reduction != "none":
        for k in ("loss", "z_loss", "acc"):
            if out[k] is not None:
                out[k] = out[k][0]
    return out


def oracle_nd(case, want_grad=True):
    import oracle
    return oracle.forward_nd(case.x, case.target, dtype=case.dtype, weight=case.weight,
                             want_grad=want_grad, **case.options())


def check(case, *, want_z=False, want_acc=False, want_pred=False):
    out = run_nd(case, want_z=want_z, want_acc=want_acc, want_pred=want_pred)
    ref = oracle_nd(case)
    assert out["status"] == 0
    if case.reduction == "none":
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
    got = out["x"].float().cpu().numpy().astype(np.float64)
    assert_grad_close(got, ref["grad"], case.dtype)
    ign = case.target == case.ignore_index
    assert np.all(np.moveaxis(got, 1, -1)[ign] == 0.0)
    return out, ref


OPTION_SETS = {
    "plain": dict(),
    "wsmooth": dict(weight=True, label_smoothing=0.1),
    "softcap_z": dict(softcap=20.0, lse_square_scale=1e-3, label_smoothing=0.05),
    "weight": dict(weight=True),
}


# tiles of several CTAs with ragged tails: inner a multiple of the vector
# width (8 for 2-byte types, 4 for fp32) and not; one and several N
@pytest.mark.parametrize("shape", [(2, 5, 3), (3, 19, 8, 16), (2, 37, 40, 24), (1, 7, 1, 1, 6),
                                   (5, 3, 100)])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("reduction", ["mean", "none", "sum"])
def test_nd_parity_auto(shape, dtype, reduction):
    case = workloads.nd_case(sum(shape), shape, dtype, std=3.0, reduction=reduction,
                             **OPTION_SETS["plain"])
    check(case, want_acc=True, want_pred=True)


@pytest.mark.parametrize("opts", sorted(OPTION_SETS))
@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_nd_parity_every_layout(nd_mode, opts, mode, dtype):
    nd_mode(mode)
    shape = (3, 21, 16, 24)  # inner 384: vectors fit either dtype
    case = workloads.nd_case(11, shape, dtype, std=4.0, reduction="mean",
                             **dict(OPTION_SETS[opts]))
    check(case, want_z=case.lse_square_scale > 0, want_acc=True, want_pred=True)


@pytest.mark.parametrize("mode", [0, 3, 4])
def test_nd_unaligned_inner_scalar_layouts(nd_mode, mode):
    nd_mode(mode)
    case = workloads.nd_case(5, (4, 13, 7, 9), "bf16", reduction="none", weight=True,
                             label_smoothing=0.2)
    check(case, want_acc=True, want_pred=True)


def test_nd_vector_layout_refused_for_unaligned_inner(nd_mode):
    from softmax_cross_entropy_gb300 import _lib
    nd_mode(1)
    case = workloads.nd_case(5, (2, 13, 7), "bf16")
    x = _dev_logits(case)
    t = torch.from_numpy(case.target).cuda()
    loss = torch.empty(1, device="cuda")
    rc = _lib.ce_fwd_nd(x.data_ptr(), 1, 2, 13, 7, t.data_ptr(), None, -100, 0.0, 0.0, 0.0, 2,
                        _lib.CE_FLAG_GRAD, loss.data_ptr(), None, None, None,
                        torch.cuda.current_stream().cuda_stream)
    assert rc == _lib.CE_ERR_UNSUPPORTED


@pytest.mark.parametrize("shape,dtype", [((2, 1000, 64), "bf16"), ((2, 1500, 33), "f32"),
                                         ((1, 3000, 40), "f32")])
def test_nd_many_classes(shape, dtype):
    # beyond the vector tile (scalar staged) and beyond any staged tile
    # (scalar from global memory)
    case = workloads.nd_case(3, shape, dtype, std=3.0, reduction="mean", label_smoothing=0.1)
    check(case, want_pred=True)


# The split form (GBCE_ND_SPLIT=1): the classes of a tile in chunks of at
# least 64 that separate CTAs take, merged per position. Shapes with several
# chunks, ragged last chunks and ragged tiles, vector and single positions.
@pytest.mark.parametrize("opts", sorted(OPTION_SETS))
@pytest.mark.parametrize("shape,dtype", [((2, 300, 40), "bf16"), ((3, 1000, 24), "f32"),
                                         ((2, 517, 7, 3), "bf16"), ((1, 2049, 16), "f16")])
@pytest.mark.parametrize("reduction", ["mean", "none"])
def test_nd_split_every_option(monkeypatch, opts, shape, dtype, reduction):
    monkeypatch.setenv("GBCE_ND_SPLIT", "1")
    case = workloads.nd_case(13 + sum(shape), shape, dtype, std=3.0, reduction=reduction,
                             **dict(OPTION_SETS[opts]))
    check(case, want_z=case.lse_square_scale > 0, want_acc=True, want_pred=True)


def test_nd_split_ties_across_chunks(monkeypatch):
    # the top logit of every position tied at classes in different chunks:
    # the prediction is the first of them
    monkeypatch.setenv("GBCE_ND_SPLIT", "1")
    case = workloads.nd_case(17, (2, 1000, 64), "bf16", reduction="mean")
    x = case.x.copy()
    top = workloads.f32_to_bf16_bits(np.array([60.0], np.float32))[0]
    for c in (130, 640, 999):
        x[:, c, :] = top
    case = case.with_(x=x)
    out, _ = check(case, want_pred=True, want_acc=True)
    valid = case.target != case.ignore_index
    assert np.all(out["pred"][valid] == 130)


def test_nd_split_matches_single_kernel_layouts(monkeypatch):
    # both forms on the same staged-size input, each against the oracle
    case = workloads.nd_case(19, (4, 40, 96), "bf16", reduction="sum", label_smoothing=0.1)
    for split in ("0", "1"):
        monkeypatch.setenv("GBCE_ND_SPLIT", split)
        check(case, want_acc=True, want_pred=True)


def test_nd_split_large(monkeypatch):
    # the N-D profile's class count at 2 x 32000 x 128 bf16 (8.2M logits),
    # the whole gradient against the oracle
    monkeypatch.delenv("GBCE_ND_SPLIT", raising=False)
    case = workloads.nd_case(23, (2, 32000, 128), "bf16", std=3.0, reduction="mean")
    check(case, want_acc=True, want_pred=True)


# A warp a tile (few classes, vector positions): forced with GBCE_ND_WARP=2
# on small shapes (ragged last tile, several tiles a warp), and taken by
# default on one with enough tiles.
@pytest.mark.parametrize("opts", sorted(OPTION_SETS))
@pytest.mark.parametrize("shape,dtype", [((3, 19, 8, 16), "bf16"), ((2, 48, 40, 24), "f32"),
                                         ((4, 7, 1000), "f16"), ((1, 1, 64), "bf16"),
                                         ((2, 21, 64), "bf16")])
@pytest.mark.parametrize("reduction", ["mean", "none", "sum"])
def test_nd_warp_per_tile(monkeypatch, opts, shape, dtype, reduction):
    monkeypatch.setenv("GBCE_ND_WARP", "2")
    case = workloads.nd_case(29 + sum(shape), shape, dtype, std=3.0, reduction=reduction,
                             **dict(OPTION_SETS[opts]))
    check(case, want_z=case.lse_square_scale > 0, want_acc=True, want_pred=True)


def test_nd_warp_per_tile_default_and_ties():
    # 8 x 19 x 128 x 128 bf16: 512 tiles, the warp form by default; the top
    # logit tied at classes 2, 9 and 18 of every position
    case = workloads.nd_case(31, (8, 19, 128, 128), "bf16", std=3.0, reduction="mean",
                             label_smoothing=0.1)
    x = case.x.copy()
    top = workloads.f32_to_bf16_bits(np.array([40.0], np.float32))[0]
    for c in (2, 9, 18):
        x[:, c] = top
    case = case.with_(x=x)
    out, _ = check(case, want_acc=True, want_pred=True)
    valid = case.target != case.ignore_index
    assert np.all(out["pred"][valid] == 2)


# The single-read tile kernel (more than 48 classes, no softcap, no
# class-weighted smoothing; GBCE_ND_TILE=2 forces it for any class count): a
# cluster holds a tile's classes in shared memory. Shapes with one CTA, a few
# and more than eight a tile (128- and 64-byte class rows), ragged class
# slices, tiles past the end of `inner`, several N.
TILE_OPTS = {"plain": dict(), "weight": dict(weight=True),
             "smooth_z": dict(label_smoothing=0.1, lse_square_scale=1e-3)}


@pytest.mark.parametrize("opts", sorted(TILE_OPTS))
@pytest.mark.parametrize("shape,dtype", [((2, 300, 40), "bf16"), ((3, 1000, 24), "f32"),
                                         ((1, 2049, 16), "f16"), ((2, 4096, 256), "bf16"),
                                         ((4, 100, 8), "bf16"), ((2, 5, 3, 8), "f32"),
                                         ((1, 7000, 72), "f32")])
@pytest.mark.parametrize("reduction", ["mean", "none", "sum"])
def test_nd_tile(monkeypatch, opts, shape, dtype, reduction):
    monkeypatch.setenv("GBCE_ND_TILE", "2")
    case = workloads.nd_case(37 + sum(shape), shape, dtype, std=3.0, reduction=reduction,
                             **dict(TILE_OPTS[opts]))
    check(case, want_z=case.lse_square_scale > 0, want_acc=True, want_pred=True)


@pytest.mark.parametrize("shape,dtype", [((64, 200, 512), "bf16"), ((32, 2000, 256), "bf16"),
                                         ((4, 32000, 128), "bf16"), ((48, 300, 256), "f32")])
@pytest.mark.parametrize("reduction", ["mean", "none"])
def test_nd_tile_several_tiles_a_cluster(monkeypatch, shape, dtype, reduction):
    # more tiles than resident clusters: each cluster's producer reloads its
    # blocks for the next tile as the consumers release them, and the
    # cluster exchanges reuse their buffers by tile parity
    monkeypatch.setenv("GBCE_ND_TILE", "2")
    case = workloads.nd_case(47 + sum(shape), shape, dtype, std=3.0, reduction=reduction,
                             label_smoothing=0.05)
    check(case, want_acc=True, want_pred=True)


def test_nd_tile_large_cluster_and_ties():
    # 2 x 32000 x 128 bf16: more than eight CTAs a tile (64-byte class rows);
    # the top logit tied at classes in different CTAs' slices
    case = workloads.nd_case(41, (2, 32000, 128), "bf16", std=3.0, reduction="mean")
    x = case.x.copy()
    top = workloads.f32_to_bf16_bits(np.array([50.0], np.float32))[0]
    for c in (7001, 15000, 31999):
        x[:, c, :] = top
    case = case.with_(x=x)
    out, _ = check(case, want_acc=True, want_pred=True)
    valid = case.target != case.ignore_index
    assert np.all(out["pred"][valid] == 7001)


def test_nd_tile_forward_only_and_all_ignored():
    case = workloads.nd_case(43, (2, 700, 64), "bf16", std=3.0, reduction="mean")
    x = _dev_logits(case)
    before = x.clone()
    out = run_nd(case, grad=False, want_pred=True, x=x)
    assert torch.equal(x, before)
    assert np.array_equal(out["pred"], oracle_nd(case, want_grad=False)["pred"])
    none = case.with_(target=np.full_like(case.target, case.ignore_index))
    m = run_nd(none, want_acc=True)
    assert math.isnan(m["loss"]) and math.isnan(m["acc"])
    assert bool((m["x"] == 0).all())


def test_nd_inner_one_is_2d():
    case = workloads.nd_case(2, (33, 4096, 1), "bf16", reduction="sum")
    check(case, want_pred=True)


@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
def test_nd_all_ignored(reduction):
    case = workloads.nd_case(4, (2, 11, 8, 8), "f32", reduction=reduction)
    case.target[...] = -100
    out, ref = check(case, want_acc=True, want_pred=True)
    if reduction == "mean":
        assert math.isnan(out["loss"]) and math.isnan(out["acc"])
    assert np.all(out["x"].cpu().numpy() == 0.0)


@pytest.mark.parametrize("mode", [0, 2, 4])
def test_nd_nonfinite_logits_at_ignored_positions(nd_mode, mode):
    nd_mode(mode)
    case = workloads.nd_case(6, (2, 9, 16, 8), "f32", reduction="mean", ignore_frac=0.2)
    rng = np.random.default_rng(0)
    ign = np.argwhere(case.target == case.ignore_index)
    specials = np.array([np.inf, -np.inf, np.nan], np.float32)
    for n, *sp in ign:
        c = rng.integers(0, case.x.shape[1])
        case.x[(n, c) + tuple(sp)] = specials[rng.integers(0, 3)]
    check(case, want_acc=True, want_pred=True)


def test_nd_argmax_ties_first_class():
    case = workloads.nd_case(7, (2, 24, 64), "bf16", reduction="none")
    x = case.x.copy()
    top = workloads.f32_to_bf16_bits(np.array([50.0], np.float32))[0]
    x[:, 3, :] = top   # every position: classes 3, 11 and 20 tie at the top
    x[:, 11, :] = top
    x[:, 20, :] = top
    case = case.with_(x=x)
    out, _ = check(case, want_pred=True, want_acc=True)
    valid = case.target != case.ignore_index
    assert np.all(out["pred"][valid] == 3)


def test_nd_out_of_range_target_reported():
    from softmax_cross_entropy_gb300 import _lib
    case = workloads.nd_case(8, (2, 6, 40), "f32", reduction="sum")
    case.target[1, 5] = 6
    out = run_nd(case)
    assert out["status"] == _lib.CE_ERR_TARGET_RANGE
    case.target[1, 5] = -100
    ref = oracle_nd(case)
    assert_loss_close(out["loss"], ref["loss"], "f32")


def test_nd_int64_targets_and_custom_ignore_index():
    case = workloads.nd_case(9, (3, 10, 5, 8), "bf16", reduction="mean")
    t = case.target.astype(np.int64)
    t[t == -100] = 7
    case = case.with_(target=t, ignore_index=7)
    out = run_nd(case, target=torch.from_numpy(t).cuda(), want_pred=True)
    ref = oracle_nd(case)
    assert_loss_close(out["loss"], ref["loss"], "bf16")
    assert np.array_equal(out["pred"], ref["pred"])


def test_nd_forward_only_leaves_logits():
    case = workloads.nd_case(10, (2, 12, 32), "bf16", reduction="mean")
    x = _dev_logits(case)
    before = x.clone()
    out = run_nd(case, grad=False, x=x, want_pred=True)
    ref = oracle_nd(case, want_grad=False)
    assert torch.equal(x, before)
    assert_loss_close(out["loss"], ref["loss"], "bf16")


@pytest.mark.parametrize("shape,dtype", [((3, 7, 16), "bf16"), ((2, 5, 3, 3), "f32"),
                                         ((2, 4, 40), "f16")])
def test_nd_backward_scales(shape, dtype):
    from softmax_cross_entropy_gb300 import _lib
    case = workloads.nd_case(12, shape, dtype, reduction="none")
    out = run_nd(case)
    x = out["x"]
    N, C = shape[0], shape[1]
    inner = math.prod(shape[2:])
    g_pos = torch.from_numpy(np.random.default_rng(1).uniform(-2, 2, (N,) + shape[2:])
                             .astype(np.float32)).cuda()
    before = x.float().cpu().numpy().astype(np.float64)
    st = torch.cuda.current_stream().cuda_stream
    rc = _lib.ce_bwd_nd(g_pos.data_ptr(), 1, x.data_ptr(), CE_DTYPE[dtype], N, C, inner, st)
    assert rc == _lib.CE_OK
    want = before * np.expand_dims(g_pos.cpu().numpy().astype(np.float64), 1)
    assert_grad_close(x.float().cpu().numpy().astype(np.float64), want, dtype, "per-position")
    g1 = torch.tensor([0.5], device="cuda")
    before = x.float().cpu().numpy().astype(np.float64)
    rc = _lib.ce_bwd_nd(g1.data_ptr(), 0, x.data_ptr(), CE_DTYPE[dtype], N, C, inner, st)
    assert rc == _lib.CE_OK
    torch.cuda.synchronize()
    # halving is exact except for fp16 subnormals, which round once into the dtype
    want = torch.from_numpy(before * 0.5).to(x.dtype).double().numpy()
    np.testing.assert_array_equal(x.double().cpu().numpy(), want)


@pytest.mark.parametrize("reduction", ["mean", "none"])
def test_nd_autograd_api(reduction):
    import softmax_cross_entropy_gb300 as ce
    case = workloads.nd_case(13, (2, 19, 12, 10), "bf16", reduction=reduction, weight=True,
                             label_smoothing=0.1)
    x = _dev_logits(case).requires_grad_()
    t = torch.from_numpy(case.target).cuda()
    w = torch.from_numpy(case.weight).cuda()
    out = ce.cross_entropy(x, t, weight=w, label_smoothing=0.1, reduction=reduction,
                           return_predicted_tokens=True)
    ref = oracle_nd(case)
    g_out = torch.ones_like(out.loss) if reduction == "mean" else \
        torch.linspace(0.5, 1.5, out.loss.numel(), device="cuda").reshape(out.loss.shape)
    out.loss.backward(g_out)
    assert out.loss.shape == (() if reduction == "mean" else t.shape)
    assert out.predicted_tokens.shape == t.shape
    assert np.array_equal(out.predicted_tokens.cpu().numpy(), ref["pred"])
    want = ref["grad"]
    got = x.grad.float().cpu().numpy().astype(np.float64)
    if reduction == "none":
        want = want * np.expand_dims(g_out.cpu().numpy().astype(np.float64), 1)
        assert_rowloss_close(out.loss.detach().cpu().numpy().astype(np.float64), ref["loss"],
                             "bf16")
        # two roundings to bf16: the forward stores the unscaled gradient,
        # the backward rounds its product with grad_output again, so each
        # element is within half a bf16 ulp of each rounding (2^-8 relative,
        # scaled by grad_output <= 1.5 for the first) of the exact value
        err = np.abs(got - want)
        assert np.all(err <= 2.0 ** -7 * 1.5 * np.abs(want) + 1e-6 * np.abs(want).max())
    else:
        assert_loss_close(float(out.loss.detach()), ref["loss"], "bf16")
        assert_grad_close(got, want, "bf16")


def test_nd_rank_one_logits_rejected():
    import softmax_cross_entropy_gb300 as ce
    with pytest.raises(ValueError):
        ce.cross_entropy(torch.zeros(8, device="cuda"), torch.zeros((), dtype=torch.int64,
                                                                    device="cuda"))
