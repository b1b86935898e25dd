"""GPU parity of the fused linear cross-entropy (ce_flce: the cross-entropy of
hidden @ lm_weight^T + bias, one chunk of rows of logits at a time) against
the oracle's flce_forward on the same seeded inputs, element by element.

Tolerances come from the arithmetic. The logits are fp32 sums of exact
products of the stored inputs (bf16 and fp16 products are exact in fp32;
fp32 products round once), so a logit is off by at most
delta_i = H * 2^-23 * max_v sum_k |h_ik w_vk|; a row's loss moves by at most
about twice its largest delta, and the gradient G by a relative 3 delta.
G is rounded once into the storage type before the two gradient GEMMs
(fp32 accumulation over V or over rows), so
  |grad_hidden error| <= (u + 3 delta + V 2^-23) (|G| |W|) + (fp16: 2^-24 |W| row sums)
  |grad_weight error| <= (u + 3 delta + rows 2^-23) (|G|^T |H|) (+ the same subnormal term)
with u = 2^-8 (bf16), 2^-11 (fp16), 1e-5 (fp32, the forward kernel's own
relative error), plus the forward kernel's absolute floor 1e-6 max|G| times
the same row sums, grad_hidden also rounded once to the storage type. The argmax is over fp32 logits: a predicted token
must hold a logit within 2 delta of the oracle's largest, and equal the
oracle's where the top two differ by more."""
import math

import numpy as np
import pytest

import workloads

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

RED = {"none": 0, "sum": 1, "mean": 2}
CE_DT = {"f32": 0, "bf16": 1, "f16": 2}
# relative error of G before the GEMMs: its rounding into the storage type,
# or for fp32 the forward kernel's own fp32 error (1e-5 relative, as its
# parity tests allow)
U = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11, "f32": 1e-5}


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from softmax_cross_entropy_gb300 import build, _lib
    build.build()
    _lib.load()


def make_case(seed, rows, H, V, dtype, ignore_frac=0.1, with_bias=False, class_weight=False):
    """hidden ~ N(0, 1), lm_weight ~ N(0, (3 / sqrt(H))^2) (logits ~ N(0, 3^2)),
    from the seeded generators of workloads."""
    hb = workloads.random_case(seed, rows, H, dtype=dtype, std=1.0, ignore_frac=0.0)
    wb = workloads.random_case(seed + 1, V, H, dtype=dtype, std=3.0 / math.sqrt(H),
                               ignore_frac=0.0)
    tc = workloads.random_case(seed + 2, rows, V, dtype="f32", std=1.0, ignore_frac=ignore_frac,
                               weight=class_weight)
    rng = np.random.default_rng(seed)
    bias = rng.normal(0, 1, V).astype(np.float32) if with_bias else None
    return hb.x, wb.x, tc.target, bias, tc.weight


def dev_tensor(a, dtype):
    if dtype in ("bf16", "f16"):
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(
            torch.bfloat16 if dtype == "bf16" else torch.float16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a))
    return t.cuda()


def run_flce(h, w, t, bias, cw, dtype, reduction, chunk_rows, opts, grad=True):
    from softmax_cross_entropy_gb300 import _lib
    rows, H = h.shape
    V = w.shape[0]
    dh, dw = dev_tensor(h, dtype), dev_tensor(w, dtype)
    dt = torch.from_numpy(t).cuda()
    db = None if bias is None else torch.from_numpy(bias).cuda()
    dcw = None if cw is None else torch.from_numpy(cw).cuda()
    n = rows if reduction == "none" else 1
    f32 = dict(dtype=torch.float32, device="cuda")
    loss = torch.full((n,), float("nan"), **f32)
    zl = torch.full((n,), float("nan"), **f32)
    acc = torch.full((n,), float("nan"), **f32)
    pred = torch.full((rows,), -7, dtype=torch.int64, device="cuda")
    gh = torch.full_like(dh, float("nan")) if grad else None
    gw = torch.full((V, H), float("nan"), **f32) if grad else None
    gb = torch.full((V,), float("nan"), **f32) if (grad and bias is not None) else None
    nbytes = _lib.ce_flce_workspace_bytes(CE_DT[dtype], rows, V, chunk_rows)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    flags = (_lib.CE_FLAG_Z_LOSS | _lib.CE_FLAG_ACC | _lib.CE_FLAG_PRED |
             (_lib.CE_FLAG_GRAD if grad else 0))
    st = torch.cuda.current_stream().cuda_stream
    ptr = lambda x: None if x is None else x.data_ptr()  # noqa: E731
    rc = _lib.ce_flce(dh.data_ptr(), dw.data_ptr(), ptr(db), CE_DT[dtype], rows, H, V,
                      dt.data_ptr(), ptr(dcw), -100, opts.get("label_smoothing", 0.0),
                      opts.get("lse_square_scale", 0.0), opts.get("softcap") or 0.0,
                      RED[reduction], flags, loss.data_ptr(), zl.data_ptr(), acc.data_ptr(),
                      pred.data_ptr(), ptr(gh), ptr(gw), ptr(gb), chunk_rows, ws.data_ptr(),
                      nbytes, st)
    assert rc == _lib.CE_OK, (_lib.ce_status_string(rc), _lib.ce_last_error())
    assert _lib.ce_device_status(st) == 0
    f64 = lambda x: None if x is None else x.double().cpu().numpy()  # noqa: E731
    return {"loss": f64(loss), "z_loss": f64(zl), "acc": f64(acc), "pred": pred.cpu().numpy(),
            "grad_hidden": f64(gh), "grad_weight": f64(gw), "grad_bias": f64(gb)}


def check(h, w, t, bias, cw, dtype, reduction, chunk_rows, opts):
    import oracle
    got = run_flce(h, w, t, bias, cw, dtype, reduction, chunk_rows, opts)
    ref = oracle.flce_forward(h, w, t, dtype=dtype, bias=bias, weight=cw, reduction=reduction,
                              **opts)
    H = h.shape[1]
    hv = np.abs(oracle.decode(h, dtype))
    wv = np.abs(oracle.decode(w, dtype))
    absdot = hv @ wv.T                                   # sum_k |h_ik w_vk|
    delta = H * 2.0 ** -23 * absdot.max(axis=1)          # per row
    counted = t != -100
    # loss
    rel = {"bf16": 1e-4, "f16": 1e-4, "f32": 1e-5}[dtype]
    if reduction == "none":
        bound = 4 * delta + rel * np.abs(ref["loss"]) + 1e-6
        assert np.all(np.abs(got["loss"] - ref["loss"]) <= bound), "row loss"
    else:
        cwt = np.ones(h.shape[0]) if cw is None else np.where(counted, cw[np.clip(t, 0, None)], 0)
        D = cwt[counted].sum() if reduction == "mean" else 1.0
        bound = 4 * (cwt * delta).sum() / max(D, 1e-30) + rel * abs(ref["loss"]) + 1e-6
        assert abs(got["loss"][0] - ref["loss"]) <= bound, (got["loss"][0], ref["loss"])
    # predicted tokens: within 2 delta of the largest logit; exact when the top two differ
    lg = ref["logits"]
    top2 = np.sort(lg, axis=1)[:, -2:] if lg.shape[1] > 1 else np.stack([lg[:, 0] - 1e9, lg[:, 0]], 1)
    gap = top2[:, 1] - top2[:, 0]
    p = got["pred"]
    assert np.all(p[~counted] == -1)
    idx = np.nonzero(counted)[0]
    assert np.all(lg[idx, p[idx]] >= top2[idx, 1] - 2 * delta[idx])
    clear = idx[gap[idx] > 2 * delta[idx]]
    assert np.array_equal(p[clear], ref["pred"][clear])
    # gradients
    G = ref["grad"]
    u = U[dtype]
    sub = 2.0 ** -24 if dtype == "f16" else 0.0
    gfloor = 1e-6 * np.abs(G).max(initial=0.0)
    bh = ((u + 3 * delta.max() + w.shape[0] * 2.0 ** -23) * (np.abs(G) @ wv) +
          (sub + gfloor) * wv.sum(axis=0)[None, :])
    bh += (2.0 ** -8 if dtype == "bf16" else 2.0 ** -11 if dtype == "f16" else 0) * \
        np.abs(ref["grad_hidden"])
    err = np.abs(got["grad_hidden"] - ref["grad_hidden"])
    assert np.all(err <= bh + 1e-30), f"grad_hidden max excess {(err - bh).max()}"
    bw = ((u + 3 * delta.max() + h.shape[0] * 2.0 ** -23) * (np.abs(G).T @ hv) +
          (sub + gfloor) * hv.sum(axis=0)[None, :])
    err = np.abs(got["grad_weight"] - ref["grad_weight"])
    assert np.all(err <= bw + 1e-30), f"grad_weight max excess {(err - bw).max()}"
    if bias is not None:
        bb = ((1e-5 + 3 * delta.max() + h.shape[0] * 2.0 ** -23) * np.abs(G).sum(axis=0) +
              gfloor * h.shape[0] + 1e-12)
        err = np.abs(got["grad_bias"] - ref["grad_bias"])
        assert np.all(err <= bb), f"grad_bias max excess {(err - bb).max()}"
    return got, ref


OPTS = {
    "plain": dict(),
    "smooth_z": dict(label_smoothing=0.1, lse_square_scale=1e-3),
    "softcap": dict(softcap=15.0, label_smoothing=0.05),
}


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("shape,chunk", [((37, 64, 500), 0), ((300, 136, 4096), 64),
                                         ((1, 8, 3), 0), ((70, 256, 20000), 16),
                                         ((129, 96, 1000), 50)])
@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
def test_flce_parity(dtype, shape, chunk, reduction):
    rows, H, V = shape
    h, w, t, _, _ = make_case(rows + H + V, rows, H, V, dtype)
    check(h, w, t, None, None, dtype, reduction, chunk, OPTS["plain"])


@pytest.mark.parametrize("opts", sorted(OPTS))
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_flce_options_bias_class_weights(opts, dtype):
    h, w, t, b, cw = make_case(5, 200, 128, 3000, dtype, with_bias=True, class_weight=True)
    check(h, w, t, b, cw, dtype, "mean", 48, OPTS[opts])


def test_flce_all_ignored():
    h, w, t, b, _ = make_case(9, 40, 32, 100, "bf16", with_bias=True)
    t[:] = -100
    got = run_flce(h, w, t, b, None, "bf16", "mean", 16, {})
    assert math.isnan(got["loss"][0])
    assert np.all(got["grad_hidden"] == 0) and np.all(got["grad_weight"] == 0)
    assert np.all(got["grad_bias"] == 0)


def test_flce_forward_only_matches():
    import oracle
    h, w, t, _, _ = make_case(11, 64, 64, 777, "bf16")
    got = run_flce(h, w, t, None, None, "bf16", "sum", 0, {}, grad=False)
    ref = oracle.flce_forward(h, w, t, dtype="bf16", reduction="sum", want_grad=False)
    assert abs(got["loss"][0] - ref["loss"]) <= 1e-4 * abs(ref["loss"]) + 1e-3


@pytest.mark.parametrize("reduction", ["mean", "sum"])
def test_flce_autograd_api(reduction):
    import oracle
    import softmax_cross_entropy_gb300 as ce
    h, w, t, b, cw = make_case(13, 96, 64, 2000, "bf16", with_bias=True, class_weight=True)
    hh = dev_tensor(h, "bf16").requires_grad_()
    ww = dev_tensor(w, "bf16").requires_grad_()
    bb = torch.from_numpy(b).cuda().requires_grad_()
    out = ce.fused_linear_cross_entropy(hh, ww, torch.from_numpy(t).cuda(), bias=bb,
                                        weight=torch.from_numpy(cw).cuda(),
                                        label_smoothing=0.1, reduction=reduction, chunk_rows=40)
    (out * 0.5).backward()
    ref = oracle.flce_forward(h, w, t, dtype="bf16", bias=b, weight=cw, label_smoothing=0.1,
                              reduction=reduction)
    assert abs(float(out.detach()) - ref["loss"]) <= 1e-3 * abs(ref["loss"])
    assert hh.grad.dtype == torch.bfloat16 and ww.grad.dtype == torch.bfloat16
    G = np.abs(ref["grad"])
    wv = np.abs(oracle.decode(w, "bf16"))
    hv = np.abs(oracle.decode(h, "bf16"))
    gh = hh.grad.double().cpu().numpy()
    assert np.all(np.abs(gh - 0.5 * ref["grad_hidden"]) <=
                  0.5 * 2.0 ** -6 * (G @ wv) + 1e-30)
    gw = ww.grad.double().cpu().numpy()
    assert np.all(np.abs(gw - 0.5 * ref["grad_weight"]) <=
                  0.5 * 2.0 ** -6 * (G.T @ hv) + 2.0 ** -8 * np.abs(0.5 * ref["grad_weight"]))
    gb = bb.grad.double().cpu().numpy()
    assert np.allclose(gb, 0.5 * ref["grad_bias"], rtol=1e-4, atol=1e-7)


def test_flce_rejects_small_workspace():
    from softmax_cross_entropy_gb300 import _lib
    h, w, t, _, _ = make_case(3, 8, 16, 40, "bf16")
    dh, dw = dev_tensor(h, "bf16"), dev_tensor(w, "bf16")
    dt = torch.from_numpy(t).cuda()
    loss = torch.empty(1, device="cuda")
    nbytes = _lib.ce_flce_workspace_bytes(CE_DT["bf16"], 8, 40, 0)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    rc = _lib.ce_flce(dh.data_ptr(), dw.data_ptr(), None, 1, 8, 16, 40, dt.data_ptr(), None,
                      -100, 0.0, 0.0, 0.0, 2, 0, loss.data_ptr(), None, None, None, None, None,
                      None, 0, ws.data_ptr(), nbytes - 256, torch.cuda.current_stream().cuda_stream)
    assert rc == _lib.CE_ERR_INVALID_ARG


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("reduction", ["mean", "none"])
def test_flce_with_cublas_gemms(monkeypatch, dtype, reduction):
    # the three GEMMs on cuBLAS (the path fp32 and unaligned inputs take)
    monkeypatch.setenv("GBCE_FLCE_GEMM", "cublas")
    h, w, t, b, cw = make_case(21, 300, 136, 5000, dtype, with_bias=True, class_weight=True)
    check(h, w, t, b, cw, dtype, reduction, 64, OPTS["smooth_z"])


def test_flce_full_size_sampled_rows(monkeypatch):
    """The bench's fused linear cross-entropy at full size, in its own launch
    configuration (rows 4096, H 4096, V 128256 bf16, the default chunk):
    reduction "none", so a row's loss, predicted token and grad_hidden row
    depend on that row alone and the oracle computes 24 sampled rows one by
    one, within the bounds of check(). grad_weight sums over every row, so
    the oracle cannot sample it: it is compared element by element with the
    same step on cuBLAS's GEMMs (GBCE_FLCE_GEMM=cublas), which consume the
    same rounded gradient G_b; the two differ only in the order of fp32
    accumulation over the 4096 rows, 2 rows 2^-23 (|G_b|^T |H|) an element
    at most, which with random signs is about sqrt(rows) = 64 times |gw|:
    3% relative. The test allows 2^-4 of |gw| plus 2^-2 of the column's
    mean |gw| (a misplaced or transposed tile differs by the entries
    themselves)."""
    import oracle
    rows, H, V = 4096, 4096, 128256
    h, w, t, _, _ = make_case(4096, rows, H, V, "bf16", ignore_frac=0.05)
    got = run_flce(h, w, t, None, None, "bf16", "none", 0, {})
    rng = np.random.default_rng(4096)
    sample = np.sort(rng.choice(rows, 24, replace=False))
    ref = oracle.flce_forward(h[sample], w, t[sample], dtype="bf16", reduction="none",
                              want_grad=False)
    wa = np.abs(oracle.decode(w, "bf16"))
    hv = oracle.decode(h[sample], "bf16")
    delta = H * 2.0 ** -23 * (np.abs(hv) @ wa.T).max(axis=1)
    counted = t[sample] != -100
    bound = 4 * delta + 1e-4 * np.abs(ref["loss"]) + 1e-6
    assert np.all(np.abs(got["loss"][sample] - ref["loss"]) <= bound), "row loss"
    lg = ref["logits"]
    top2 = np.sort(lg, axis=1)[:, -2:]
    p = got["pred"][sample]
    assert np.all(p[~counted] == -1)
    idx = np.nonzero(counted)[0]
    assert np.all(lg[idx, p[idx]] >= top2[idx, 1] - 2 * delta[idx])
    clear = idx[(top2[idx, 1] - top2[idx, 0]) > 2 * delta[idx]]
    assert np.array_equal(p[clear], ref["pred"][clear])
    # grad_hidden rows: G (the oracle's, from these rows' float64 logits) @ W
    G = oracle.forward(lg, t[sample], dtype="f64", reduction="none", want_grad=True)["grad"]
    want = G @ oracle.decode(w, "bf16")
    gbound = (U["bf16"] + 3 * delta[:, None] + V * 2.0 ** -23) * (np.abs(G) @ wa)
    gbound += np.abs(want) * 2.0 ** -8 + 1e-6 * np.abs(G).max() * wa.sum(axis=0)
    assert np.all(np.abs(got["grad_hidden"][sample] - want) <= gbound), "grad_hidden rows"
    # grad_weight against the same step on cuBLAS's GEMMs
    monkeypatch.setenv("GBCE_FLCE_GEMM", "cublas")
    blas = run_flce(h, w, t, None, None, "bf16", "none", 0, {})
    gw, gw_ref = got["grad_weight"], blas["grad_weight"]
    assert np.all(np.isfinite(gw))
    wbound = 2.0 ** -4 * np.abs(gw_ref) + 2.0 ** -2 * np.abs(gw_ref).mean(axis=0)[None, :]
    assert np.all(np.abs(gw - gw_ref) <= wbound), "grad_weight against the cuBLAS GEMMs"
