"""Pins for the oracle's fused linear cross-entropy (the cross-entropy of
hidden @ lm_weight^T + bias; "Kernel Profile: CrossEntropy",
closest_existing_kernel fused_linear_cross_entropy): torch CPU float64
F.linear + F.cross_entropy with autograd (softcap and z-loss composed from
torch's tanh and logsumexp), the identity-hidden special case against the
plain cross-entropy oracle, central finite differences of the loss in every
input, and the exact decoding of stored bf16 / fp16 values."""
import itertools

import numpy as np
import pytest

torch = pytest.importorskip("torch")
F = torch.nn.functional


def torch_flce(h, w, b, t, cw, eps, lam, softcap, reduction, ignore_index=-100):
    ht = torch.tensor(h, dtype=torch.float64, requires_grad=True)
    wt = torch.tensor(w, dtype=torch.float64, requires_grad=True)
    bt = None if b is None else torch.tensor(b, dtype=torch.float64, requires_grad=True)
    tt = torch.tensor(t, dtype=torch.int64)
    cwt = None if cw is None else torch.tensor(cw, dtype=torch.float64)
    x = F.linear(ht, wt, bt)
    z = softcap * torch.tanh(x / softcap) if softcap else x
    loss = F.cross_entropy(z, tt, weight=cwt, ignore_index=ignore_index, label_smoothing=eps,
                           reduction=reduction)
    valid = tt != ignore_index
    zl_rows = lam * torch.logsumexp(z, dim=1) ** 2 * valid
    if reduction == "none":
        zl = zl_rows
    elif reduction == "sum":
        zl = zl_rows.sum()
    else:
        tc = tt.clamp(min=0)
        D = (cwt[tc] * valid).sum() if cwt is not None else valid.sum()
        zl = zl_rows.sum() / D
    total = loss + zl
    total.sum().backward()
    return (total.detach().numpy(), ht.grad.numpy(), wt.grad.numpy(),
            None if bt is None else bt.grad.numpy())


CASES = list(itertools.product([False, True], [False, True], [0.0, 0.1], [0.0, 1e-3],
                               [None, 5.0], ["none", "sum", "mean"]))


@pytest.mark.parametrize("bias,cw,eps,lam,softcap,reduction", CASES)
def test_flce_matches_torch_f64(oracle_mod, bias, cw, eps, lam, softcap, reduction):
    rng = np.random.default_rng(abs(hash((bias, cw, eps, lam, softcap, reduction))) % 2**32)
    rows, H, V = 13, 9, 21
    h = rng.normal(0, 1, (rows, H))
    w = rng.normal(0, 0.7, (V, H))
    b = rng.normal(0, 0.5, V) if bias else None
    t = rng.integers(0, V, rows)
    t[rng.choice(rows, 3, replace=False)] = -100
    c = rng.uniform(0.5, 2.0, V) if cw else None
    loss, gh, gw, gb = torch_flce(h, w, b, t, c, eps, lam, softcap, reduction)
    r = oracle_mod.flce_forward(h, w, t, dtype="f64", bias=b, weight=c, label_smoothing=eps,
                                lse_square_scale=lam, softcap=softcap, reduction=reduction)
    np.testing.assert_allclose(r["loss"], loss, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(r["grad_hidden"], gh, rtol=1e-10, atol=1e-14)
    np.testing.assert_allclose(r["grad_weight"], gw, rtol=1e-10, atol=1e-14)
    if bias:
        np.testing.assert_allclose(r["grad_bias"], gb, rtol=1e-10, atol=1e-14)


def test_flce_identity_hidden_is_plain_ce(oracle_mod):
    # hidden = I: the logits are lm_weight^T itself, grad_weight = G^T
    rng = np.random.default_rng(4)
    H, V = 11, 17
    w = rng.normal(0, 2, (V, H))
    t = rng.integers(0, V, H)
    t[2] = -100
    r = oracle_mod.flce_forward(np.eye(H), w, t, dtype="f64", label_smoothing=0.2,
                                reduction="sum")
    ce = oracle_mod.forward(np.ascontiguousarray(w.T), t, dtype="f64", label_smoothing=0.2,
                            reduction="sum")
    assert r["loss"] == ce["loss"]
    np.testing.assert_array_equal(r["grad_weight"], ce["grad"].T)
    np.testing.assert_allclose(r["grad_hidden"], ce["grad"] @ w, rtol=1e-14)


@pytest.mark.parametrize("reduction", ["sum", "mean"])
def test_flce_finite_differences(oracle_mod, reduction):
    rng = np.random.default_rng(7)
    rows, H, V = 3, 4, 5
    h = rng.normal(0, 1, (rows, H))
    w = rng.normal(0, 1, (V, H))
    b = rng.normal(0, 1, V)
    t = np.array([1, -100, 4])
    cw = rng.uniform(0.5, 2.0, V)
    opts = dict(dtype="f64", weight=cw, label_smoothing=0.1, lse_square_scale=1e-2,
                softcap=3.0, reduction=reduction)
    r = oracle_mod.flce_forward(h, w, t, bias=b, **opts)

    def loss(hh, ww, bb):
        return oracle_mod.flce_forward(hh, ww, t, bias=bb, want_grad=False, **opts)["loss"]

    step = 1e-6
    for name, arr, grad in (("h", h, r["grad_hidden"]), ("w", w, r["grad_weight"]),
                            ("b", b, r["grad_bias"])):
        for idx in np.ndindex(arr.shape):
            up, dn = arr.copy(), arr.copy()
            up[idx] += step
            dn[idx] -= step
            args_up = {"h": (up, w, b), "w": (h, up, b), "b": (h, w, up)}[name]
            args_dn = {"h": (dn, w, b), "w": (h, dn, b), "b": (h, w, dn)}[name]
            fd = (loss(*args_up) - loss(*args_dn)) / (2 * step)
            assert abs(fd - grad[idx]) <= 1e-7 * max(1.0, abs(grad[idx])), (name, idx)


def test_decode_exact(oracle_mod):
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2**16, 4096, dtype=np.uint16)
    bf = oracle_mod.decode(bits, "bf16")
    want = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    np.testing.assert_array_equal(np.isnan(bf), np.isnan(want))
    ok = ~np.isnan(want)
    np.testing.assert_array_equal(bf[ok], want[ok])
    f16 = oracle_mod.decode(bits, "f16")
    want16 = bits.view(np.float16).astype(np.float64)
    ok = ~np.isnan(want16)
    np.testing.assert_array_equal(f16[ok], want16[ok])
