"""Parity of the unfused (aten-shaped) kernels with the oracle:
ce_log_softmax, ce_nll_loss_fwd, ce_nll_loss_bwd, ce_log_softmax_bwd, and
the chain of all four against the fused oracle.

Tolerances (no bound is stated for these ops; derived from the
arithmetic: fp32 throughout, one rounding into the output dtype):
outputs within one unit in the last place of the dtype of the oracle value
(2^-7 relative for bf16, 2^-10 for fp16, 2^-22 for fp32, which allows a few
fp32 roundings) plus 1e-5 (fp32: 4e-6) absolute for values near zero;
scalar losses relative 1e-5 (sums in double, rounded to fp32 once)."""
import numpy as np
import pytest

import workloads
from ce_gpu import CE_DTYPE, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ULP = {"f32": 2.0 ** -22, "bf16": 2.0 ** -7, "f16": 2.0 ** -10}
ABS = {"f32": 4e-6, "bf16": 1e-5, "f16": 1e-5}
TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from softmax_cross_entropy_gb300 import build, _lib
    build.build()
    _lib.load()


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def _close(got, want, dtype, what, scale=0.0):
    err = np.abs(got - want)
    bound = ULP[dtype] * np.abs(want) + ABS[dtype] + scale
    bad = ~(err <= bound)
    assert not bad.any(), f"{what}: {bad.sum()} out of bound, max err {err.max()}"


def _status():
    from softmax_cross_entropy_gb300 import _lib
    return _lib.ce_device_status(torch.cuda.current_stream().cuda_stream)


def _stored(dtype, a):
    """A float array rounded to the storage dtype, on the device."""
    return torch.from_numpy(np.asarray(a, np.float32)).to(TORCH_DT[dtype]).cuda()


SHAPES = [(1, 1), (3, 7), (5, 8), (17, 1000), (33, 4096), (9, 32000), (4, 131072), (2, 128256)]


@pytest.mark.parametrize("rows,C", SHAPES)
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_log_softmax(rows, C, dtype):
    import oracle
    from softmax_cross_entropy_gb300 import unfused
    case = workloads.random_case(200 + rows + C, rows, C, dtype=dtype, std=4.0)
    x, _, _ = to_device(case)
    y = unfused.log_softmax(x)
    assert _status() == 0
    want = oracle.log_softmax(workloads.logits_f64(case))
    _close(_f64(y), want, dtype, "log_softmax")
    # in place
    unfused.log_softmax(x, out=x)
    _close(_f64(x), want, dtype, "log_softmax in place")


def test_log_softmax_unaligned_and_large_gap():
    import oracle
    from softmax_cross_entropy_gb300 import unfused
    case = workloads.random_case(210, 6, 4096, dtype="bf16")
    x, _, _ = to_device(case)
    buf = torch.empty(x.numel() + 1, dtype=x.dtype, device="cuda")
    view = buf[1:].view(x.shape)  # 2-byte offset: the general kernel
    view.copy_(x)
    _close(_f64(unfused.log_softmax(view)), oracle.log_softmax(workloads.logits_f64(case)),
           "bf16", "unaligned log_softmax")
    g = torch.tensor([[0.0, 1000.0, 0.0, 0.0]], device="cuda")
    out = unfused.log_softmax(g).cpu().numpy()
    assert out[0, 0] == -1000.0 and out[0, 1] == 0.0


@pytest.mark.parametrize("reduction", ["none", "sum", "mean"])
@pytest.mark.parametrize("dtype,rows,C,weight", [("f32", 1023, 1000, False),
                                                 ("bf16", 300, 4096, True),
                                                 ("f16", 77, 333, True), ("f32", 5, 3, False)])
def test_nll_loss_forward(reduction, dtype, rows, C, weight):
    import oracle
    from softmax_cross_entropy_gb300 import unfused
    case = workloads.random_case(220 + rows, rows, C, dtype="f32", weight=weight or None)
    logp_dev = _stored(dtype, oracle.log_softmax(workloads.logits_f64(case)))
    t = torch.from_numpy(case.target).cuda()
    w = None if case.weight is None else torch.from_numpy(case.weight).cuda()
    out, tw = unfused.nll_loss_forward(logp_dev, t, w, reduction)
    assert _status() == 0
    want, want_tw = oracle.nll_forward(_f64(logp_dev), case.target, case.weight,
                                       reduction=reduction)
    np.testing.assert_allclose(out.cpu().numpy().astype(np.float64), want, rtol=1e-5, atol=1e-7)
    assert float(tw) == pytest.approx(want_tw, rel=1e-6)


def test_nll_loss_all_ignored_and_empty():
    from softmax_cross_entropy_gb300 import unfused
    lp = torch.zeros((4, 8), device="cuda")
    t = torch.full((4,), -100, dtype=torch.int64, device="cuda")
    out, tw = unfused.nll_loss_forward(lp, t, reduction="mean")
    assert torch.isnan(out) and float(tw) == 0.0
    g = unfused.nll_loss_backward(torch.ones(()), t, 8, torch.float32, reduction="mean",
                                  total_weight=tw)
    assert bool((g == 0).all())
    out, tw = unfused.nll_loss_forward(torch.zeros((0, 8), device="cuda"),
                                       torch.zeros((0,), dtype=torch.int64, device="cuda"),
                                       reduction="sum")
    assert float(out) == 0.0 and float(tw) == 0.0


@pytest.mark.parametrize("reduction", ["none", "sum", "mean"])
@pytest.mark.parametrize("dtype,rows,C,weight", [("f32", 100, 1000, True),
                                                 ("bf16", 64, 4096, False),
                                                 ("f16", 33, 77, True)])
def test_nll_loss_backward(reduction, dtype, rows, C, weight):
    import oracle
    from softmax_cross_entropy_gb300 import unfused
    case = workloads.random_case(230 + rows, rows, C, dtype="f32", weight=weight or None)
    t = torch.from_numpy(case.target).cuda()
    w = None if case.weight is None else torch.from_numpy(case.weight).cuda()
    rng = np.random.default_rng(0)
    go = rng.uniform(-2, 2, rows if reduction == "none" else 1).astype(np.float32)
    tw = np.float32(37.5)
    got = unfused.nll_loss_backward(torch.from_numpy(go).reshape(-1 if reduction == "none" else ())
                                    .cuda(), t, C, TORCH_DT[dtype], w, reduction,
                                    total_weight=torch.tensor(tw, device="cuda"))
    assert _status() == 0
    want = oracle.nll_backward(go.astype(np.float64), case.target, C, case.weight,
                               reduction=reduction, total_weight=float(tw))
    _close(_f64(got), want, dtype, "nll_loss_backward")


@pytest.mark.parametrize("rows,C", [(3, 7), (33, 4096), (5, 1001), (2, 128256)])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_log_softmax_backward(rows, C, dtype):
    import oracle
    from softmax_cross_entropy_gb300 import unfused
    case = workloads.random_case(240 + C, rows, C, dtype="f32", std=3.0)
    y = _stored(dtype, oracle.log_softmax(workloads.logits_f64(case)))
    dy = _stored(dtype, np.random.default_rng(1).normal(0, 1, (rows, C)))
    dx = unfused.log_softmax_backward_data(dy, y)
    assert _status() == 0
    want = oracle.log_softmax_backward(_f64(dy), _f64(y))
    # the row sum of dy enters every element: allow its fp32 rounding
    scale = 1e-6 * np.abs(_f64(dy)).sum(axis=1, keepdims=True)
    _close(_f64(dx), want, dtype, "log_softmax_backward", scale)
    unfused.log_softmax_backward_data(dy, y, grad_input=dy)  # in place
    _close(_f64(dy), want, dtype, "log_softmax_backward in place", scale)


@pytest.mark.parametrize("reduction", ["none", "sum", "mean"])
@pytest.mark.parametrize("dtype,weight", [("f32", True), ("bf16", False), ("f16", True)])
def test_unfused_chain_matches_fused_oracle(reduction, dtype, weight):
    import oracle
    from softmax_cross_entropy_gb300 import unfused
    case = workloads.random_case(250, 96, 8192, dtype=dtype, weight=weight or None,
                                 reduction=reduction)
    x, t, w = to_device(case)
    x.requires_grad_(True)
    loss = unfused.cross_entropy_unfused(x, t, w, reduction=reduction)
    loss.backward(torch.ones_like(loss))
    assert _status() == 0
    ref = oracle.forward(case.x, case.target, dtype=dtype, weight=case.weight,
                         reduction=reduction)
    # the loss is -logp[t] of log-probs already rounded to the dtype: half
    # a unit in the last place per row (for fp32, the fused bound 1e-5)
    np.testing.assert_allclose(loss.detach().cpu().numpy().astype(np.float64), ref["loss"],
                               rtol=ULP[dtype] if dtype != "f32" else 1e-5, atol=1e-6)
    # dx_j = dy_j - exp(y_j) * S with S the row sum of the nll gradient dy.
    # The chain rounds three times into the dtype (log-probs y, dy, dx); a
    # log-prob rounded by up to ULP * |y| changes exp(y) by that factor, so
    # that term is bounded by ULP * p * |y| * |S| (p, y and S exact here).
    y = oracle.log_softmax(workloads.logits_f64(case))
    _, tw = oracle.nll_forward(y, case.target, case.weight, reduction=reduction)
    go = np.ones(case.rows) if reduction == "none" else np.array([1.0])
    S = oracle.nll_backward(go, case.target, case.V, case.weight, reduction=reduction,
                            total_weight=tw).sum(axis=1, keepdims=True)
    err = np.abs(_f64(x.grad) - ref["grad"])
    bound = (3 * ULP[dtype] * np.abs(ref["grad"]) + 2 * ULP[dtype] * np.exp(y) * (np.abs(y) + 1)
             * np.abs(S) + 1e-6 * np.abs(ref["grad"]).max() + ABS[dtype])
    assert (err <= bound).all(), f"max err {err.max()}"


def test_unfused_chain_tt_fp32_sampled():
    # the decomposed graph's own shape: 1023 x 128256 fp32, mean, sampled rows
    import oracle
    from softmax_cross_entropy_gb300 import unfused
    case = workloads.tt_fp32()
    x, t, _ = to_device(case)
    x.requires_grad_(True)
    loss = unfused.cross_entropy_unfused(x, t, reduction="mean")
    loss.backward()
    assert _status() == 0
    ref = oracle.forward(case.x, case.target, dtype="f32", want_grad=False, **case.options())
    np.testing.assert_allclose(float(loss.detach()), ref["loss"], rtol=1e-5)
    idx = np.array([0, 1, 511, 1022])
    rr = oracle.rows(case.x, case.target, idx, dtype="f32", **case.options())
    got = _f64(x.grad[torch.as_tensor(idx, device="cuda")])
    err = np.abs(got - rr["grad"])
    assert (err <= 3 * ULP["f32"] * np.abs(rr["grad"]) + 1e-6 * np.abs(rr["grad"]).max()
            + 1e-9).all(), err.max()
