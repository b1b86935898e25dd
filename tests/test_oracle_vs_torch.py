"""Cross-checks the oracle against PyTorch's CPU float64 library routines in
the cases where they coincide with the method: F.cross_entropy (weights,
ignore_index, label smoothing, reductions) and autograd, plus tanh softcap
and the z-loss composed from torch's tanh and logsumexp."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
F = torch.nn.functional


def torch_reference(x, t, weight, eps, lam, softcap, reduction, ignore_index=-100):
    """loss(x) from torch library pieces, differentiated by autograd."""
    xt = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    tt = torch.tensor(t, dtype=torch.int64)
    wt = None if weight is None else torch.tensor(weight, dtype=torch.float64)
    z = softcap * torch.tanh(xt / softcap) if softcap else xt
    loss = F.cross_entropy(z, tt, weight=wt, ignore_index=ignore_index,
                           label_smoothing=eps, reduction=reduction)
    valid = tt != ignore_index
    zl_rows = lam * torch.logsumexp(z, dim=1) ** 2 * valid
    if reduction == "none":
        zl = zl_rows
    elif reduction == "sum":
        zl = zl_rows.sum()
    else:
        tc = tt.clamp(min=0)
        D = (wt[tc] * valid).sum() if wt is not None else valid.sum()
        zl = zl_rows.sum() / D
    total = loss + zl
    total.sum().backward()
    return total.detach().numpy(), zl.detach().numpy(), xt.grad.numpy()


CASES = list(__import__("itertools").product(
    [False, True], [0.0, 0.15], [0.0, 1e-3], [None, 4.0], ["none", "sum", "mean"]))


@pytest.mark.parametrize("weighted,eps,lam,softcap,reduction", CASES)
def test_oracle_matches_torch_f64(oracle_mod, weighted, eps, lam, softcap, reduction):
    rng = np.random.default_rng(abs(hash((weighted, eps, lam, softcap, reduction))) % 2**32)
    rows, V = 23, 57
    x = rng.normal(0, 3, (rows, V))
    t = rng.integers(0, V, rows)
    t[rng.choice(rows, 4, replace=False)] = -100
    w = rng.uniform(0.5, 2.0, V) if weighted else None
    loss, zl, grad = torch_reference(x, t, w, eps, lam, softcap, reduction)
    r = oracle_mod.forward(x, t, dtype="f64", weight=w, label_smoothing=eps,
                           lse_square_scale=lam, softcap=softcap, reduction=reduction)
    np.testing.assert_allclose(r["loss"], loss, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(r["z_loss"], zl, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(r["grad"], grad, rtol=1e-11, atol=1e-15)


def test_oracle_matches_torch_on_bf16_workload(oracle_mod):
    import workloads
    case = workloads.weighted(rows=64, V=512)
    x = workloads.logits_f64(case)
    loss, _, grad = torch_reference(x, case.target.astype(np.int64),
                                    case.weight.astype(np.float64), case.label_smoothing,
                                    0.0, None, "mean")
    r = oracle_mod.forward(case.x, case.target, dtype="bf16", weight=case.weight,
                           **case.options())
    np.testing.assert_allclose(r["loss"], loss, rtol=1e-12)
    np.testing.assert_allclose(r["grad"], grad, rtol=1e-11, atol=1e-16)


def test_all_ignored_matches_torch(oracle_mod):
    x = np.random.default_rng(0).normal(0, 1, (5, 6))
    t = np.full(5, -100)
    xt = torch.tensor(x, requires_grad=True)
    l = F.cross_entropy(xt, torch.tensor(t), reduction="mean")
    l.backward()
    r = oracle_mod.forward(x, t, dtype="f64", reduction="mean")
    assert np.isnan(r["loss"]) and np.isnan(l.item())
    np.testing.assert_array_equal(r["grad"], xt.grad.numpy())
