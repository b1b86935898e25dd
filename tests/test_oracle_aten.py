"""Pins for the oracle's unfused ops (_log_softmax, nll_loss_forward,
nll_loss_backward, _log_softmax_backward_data): torch CPU float64 (a
library special case), closed forms and invariants, and the chain against
the fused oracle (the decomposition must give the fused loss and
gradient)."""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def orc():
    import oracle
    oracle.build()
    return oracle


def _case(seed, rows, C, ignore_frac=0.2, weight=False):
    rng = np.random.default_rng(seed)
    x = rng.normal(0, 4, (rows, C))
    t = rng.integers(0, C, rows)
    t[rng.random(rows) < ignore_frac] = -100
    w = rng.uniform(0.5, 2.0, C) if weight else None
    return x, t, w


def test_log_softmax_matches_torch(orc):
    x, _, _ = _case(1, 9, 37)
    want = torch.log_softmax(torch.from_numpy(x), dim=-1).numpy()
    np.testing.assert_allclose(orc.log_softmax(x), want, rtol=1e-13, atol=1e-13)


def test_log_softmax_large_gap_and_invariants(orc):
    # a plain log(softmax) gives -inf for the smaller logit past a gap of ~87
    out = orc.log_softmax(np.array([[0.0, 1000.0]]))
    assert out[0, 0] == -1000.0 and out[0, 1] == 0.0
    x, _, _ = _case(2, 6, 50)
    y = orc.log_softmax(x)
    # every row is a log-distribution; a shift of a row leaves it unchanged
    np.testing.assert_allclose(np.log(np.exp(y).sum(axis=1)), 0.0, atol=1e-14)
    np.testing.assert_allclose(orc.log_softmax(x + 123.25), y, atol=1e-12)
    # constant logits: -log C
    np.testing.assert_allclose(orc.log_softmax(np.full((2, 8), 3.0)), -math.log(8), rtol=1e-15)


@pytest.mark.parametrize("reduction", ["none", "sum", "mean"])
@pytest.mark.parametrize("weight", [False, True])
def test_nll_forward_matches_torch(orc, reduction, weight):
    x, t, w = _case(3, 11, 23, weight=weight)
    lp = orc.log_softmax(x)
    got, tw = orc.nll_forward(lp, t, w, reduction=reduction)
    want = torch.nn.functional.nll_loss(
        torch.from_numpy(lp), torch.from_numpy(t), None if w is None else torch.from_numpy(w),
        ignore_index=-100, reduction=reduction).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-13)
    valid = t != -100
    want_tw = 0.0 if reduction == "none" else (w[t[valid]].sum() if weight else valid.sum())
    assert tw == pytest.approx(want_tw, rel=1e-14)


def test_nll_all_ignored(orc):
    lp = orc.log_softmax(np.zeros((3, 4)))
    t = np.full(3, -100)
    loss, tw = orc.nll_forward(lp, t, reduction="mean")
    assert math.isnan(loss) and tw == 0.0
    assert orc.nll_forward(lp, t, reduction="sum")[0] == 0.0
    g = orc.nll_backward(1.0, t, 4, reduction="mean", total_weight=tw)
    assert np.array_equal(g, np.zeros((3, 4)))


def test_nll_target_out_of_range_is_an_error(orc):
    with pytest.raises(orc.OracleError):
        orc.nll_forward(np.zeros((2, 3)), np.array([0, 3]))


@pytest.mark.parametrize("reduction", ["none", "sum", "mean"])
@pytest.mark.parametrize("weight", [False, True])
def test_nll_backward_matches_torch_autograd(orc, reduction, weight):
    x, t, w = _case(4, 10, 17, weight=weight)
    lp = torch.from_numpy(orc.log_softmax(x)).requires_grad_(True)
    tw_t = None if w is None else torch.from_numpy(w)
    loss = torch.nn.functional.nll_loss(lp, torch.from_numpy(t), tw_t, reduction=reduction)
    go = (np.random.default_rng(5).uniform(-2, 2, 10) if reduction == "none"
          else np.array([1.75]))
    (g_want,) = torch.autograd.grad(loss, lp, torch.from_numpy(go if reduction == "none"
                                                                else go.reshape(())))
    _, tw = orc.nll_forward(lp.detach().numpy(), t, w, reduction=reduction)
    got = orc.nll_backward(go, t, 17, w, reduction=reduction, total_weight=tw)
    np.testing.assert_allclose(got, g_want.numpy(), rtol=1e-13, atol=0)


def test_log_softmax_backward_matches_torch_autograd(orc):
    x, _, _ = _case(6, 7, 29)
    xt = torch.from_numpy(x).requires_grad_(True)
    y = torch.log_softmax(xt, dim=-1)
    dy = np.random.default_rng(7).normal(0, 1, (7, 29))
    (want,) = torch.autograd.grad(y, xt, torch.from_numpy(dy))
    got = orc.log_softmax_backward(dy, y.detach().numpy())
    np.testing.assert_allclose(got, want.numpy(), rtol=1e-12, atol=1e-15)
    # each row of the result sums to zero (the softmax Jacobian's rows do)
    np.testing.assert_allclose(got.sum(axis=1), 0.0, atol=1e-12)


@pytest.mark.parametrize("reduction", ["none", "sum", "mean"])
@pytest.mark.parametrize("weight", [False, True])
def test_unfused_chain_equals_fused_oracle(orc, reduction, weight):
    # _log_softmax -> nll_loss_forward, and nll_loss_backward ->
    # _log_softmax_backward_data, against the fused oracle with no
    # smoothing, z-loss or softcap
    x, t, w = _case(8, 13, 41, weight=weight)
    y = orc.log_softmax(x)
    loss, tw = orc.nll_forward(y, t, w, reduction=reduction)
    go = np.ones(13) if reduction == "none" else np.array([1.0])
    dy = orc.nll_backward(go, t, 41, w, reduction=reduction, total_weight=tw)
    dx = orc.log_softmax_backward(dy, y)
    fused = orc.forward(x, t, dtype="f64", weight=w, reduction=reduction)
    np.testing.assert_allclose(loss, fused["loss"], rtol=1e-12)
    np.testing.assert_allclose(dx, fused["grad"], rtol=1e-11, atol=1e-15)
