"""Pins for the oracle's N-D form (class dimension 1): torch CPU float64
F.cross_entropy on N-D inputs (a library special case that reduces over
every non-class dimension) and the reduction to the 2-D form."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def orc():
    import oracle
    oracle.build()
    return oracle


@pytest.mark.parametrize("shape", [(2, 5, 3), (3, 4, 2, 5), (1, 7, 1, 1, 6)])
@pytest.mark.parametrize("reduction", ["none", "sum", "mean"])
@pytest.mark.parametrize("opts", [dict(), dict(weight=True, label_smoothing=0.1),
                                  dict(label_smoothing=0.3)])
def test_nd_matches_torch(orc, shape, reduction, opts):
    rng = np.random.default_rng(sum(shape))
    x = rng.normal(0, 3, shape)
    C = shape[1]
    t = rng.integers(0, C, (shape[0],) + shape[2:])
    t[rng.random(t.shape) < 0.2] = -100
    w = rng.uniform(0.5, 2.0, C) if opts.get("weight") else None
    eps = opts.get("label_smoothing", 0.0)
    r = orc.forward_nd(x, t, weight=w, label_smoothing=eps, reduction=reduction)
    xt = torch.from_numpy(x).requires_grad_(True)
    loss = torch.nn.functional.cross_entropy(
        xt, torch.from_numpy(t), None if w is None else torch.from_numpy(w),
        ignore_index=-100, reduction=reduction, label_smoothing=eps)
    loss.backward(torch.ones_like(loss))
    np.testing.assert_allclose(r["loss"], loss.detach().numpy(), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(r["grad"], xt.grad.numpy(), rtol=1e-11, atol=1e-15)
    assert r["grad"].shape == x.shape


def test_nd_with_no_spatial_dims_is_the_2d_form(orc):
    rng = np.random.default_rng(3)
    x = rng.normal(0, 3, (9, 11))
    t = rng.integers(0, 11, 9)
    a = orc.forward_nd(x, t, reduction="sum", lse_square_scale=1e-3, softcap=7.0)
    b = orc.forward(x, t, reduction="sum", lse_square_scale=1e-3, softcap=7.0)
    assert a["loss"] == b["loss"] and np.array_equal(a["grad"], b["grad"])


def test_nd_argmax_per_position(orc):
    x = np.zeros((1, 3, 2))
    x[0, 2, 0] = 5.0   # position 0: class 2
    x[0, 1, 1] = 5.0   # position 1: classes 1 and 2 tie at the top
    x[0, 2, 1] = 5.0
    r = orc.forward_nd(x, np.array([[2, 2]]), reduction="none")
    assert r["pred"].tolist() == [[2, 1]]
