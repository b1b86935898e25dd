"""Pins the CPU oracle to facts that do not come from the oracle itself:
closed forms, the numbers the pages print, invariants, brute force and
finite differences. A dropped term, a wrong sign or a wrong index anywhere
in the oracle fails at least one of these."""
import itertools
import json
import math
import os

import numpy as np
import pytest

import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ce_facts.json")


def fwd(oracle_mod, x, t, **kw):
    return oracle_mod.forward(np.asarray(x, np.float64), np.asarray(t, np.int64),
                              dtype="f64", **kw)


def softmax(x):
    # scipy's softmax is an independent library routine for p
    from scipy.special import softmax as sp_softmax
    return sp_softmax(np.asarray(x, np.float64), axis=-1)


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("V", [1, 2, 7, 4096])
@pytest.mark.parametrize("c", [-3.0, 0.0, 5.5])
def test_constant_logits_give_log_V(oracle_mod, V, c):
    rows = 3
    x = np.full((rows, V), c)
    t = np.array([0, V - 1, V // 2])
    r = fwd(oracle_mod, x, t, reduction="none")
    np.testing.assert_allclose(r["loss"], math.log(V), rtol=1e-14, atol=1e-15)
    assert (r["pred"] == 0).all()  # every entry ties: the lowest index wins
    onehot = np.zeros((rows, V))
    onehot[np.arange(rows), t] = 1.0
    np.testing.assert_allclose(r["grad"], 1.0 / V - onehot, rtol=0, atol=1e-15)


@pytest.mark.parametrize("lam", [1e-4, 0.5])
def test_constant_logits_zloss_closed_form(oracle_mod, lam):
    V, c = 10, 1.25
    x = np.full((2, V), c)
    r = fwd(oracle_mod, x, [3, 4], lse_square_scale=lam, reduction="none")
    lse = c + math.log(V)
    np.testing.assert_allclose(r["z_loss"], lam * lse * lse, rtol=1e-14)
    np.testing.assert_allclose(r["loss"], math.log(V) + lam * lse * lse, rtol=1e-14)


def test_golden_closed_forms(oracle_mod):
    doc = json.load(open(GOLDEN))
    for case in doc["closed_forms"]:
        r = fwd(oracle_mod, [case["x"]], [case["target"]], reduction="sum",
                label_smoothing=case["label_smoothing"],
                lse_square_scale=case["lse_square_scale"])
        assert r["loss"] == pytest.approx(case["loss"], rel=1e-14), case["name"]
        np.testing.assert_allclose(r["grad"][0], case["grad"], rtol=1e-13, atol=1e-15,
                                   err_msg=case["name"])


def test_golden_logit_gap_stays_finite(oracle_mod):
    # tt-mlir #9339: plain log(softmax) reaches -inf past a gap of ~87; the
    # max-shifted log-sum-exp must not.
    doc = json.load(open(GOLDEN))["logit_gap"]
    for c in doc["cases"]:
        r = fwd(oracle_mod, [[0.0, c["gap"]]], [0], reduction="sum")
        assert math.isfinite(r["loss"])
        assert r["loss"] == pytest.approx(c["loss"], rel=1e-15)
        # the gradient is p - onehot: (p0 - 1, p1) with p1 = 1 - p0
        np.testing.assert_allclose(r["grad"][0], [-1.0, 1.0], atol=2e-22 + math.exp(-c["gap"]))
        # the other target gives log1p(exp(-gap)), exact up to the rounding
        # of lse (an ulp of the gap)
        r1 = fwd(oracle_mod, [[0.0, c["gap"]]], [1], reduction="sum")
        assert r1["loss"] == pytest.approx(math.log1p(math.exp(-c["gap"])),
                                           abs=2 * math.ulp(c["gap"]))


def test_golden_workload_bytes():
    doc = json.load(open(GOLDEN))["workload_bytes"]
    nbytes = doc["rows"] * doc["V"] * doc["bytes_per_element"]
    assert round(nbytes / 2**20) in (doc["mib"], doc["mib"] + 1)  # 500.5 MiB
    case = workloads.tt_fp32(rows=4, V=doc["V"])  # shape and storage of the recipe
    assert case.V == doc["V"] and case.x.dtype == np.float32


def test_golden_vsweep_matches_workloads():
    doc = json.load(open(GOLDEN))["vsweep"]
    assert list(workloads.VSWEEP) == doc["V"]
    assert doc["B"] * doc["T"] == 4096


def test_label_smoothing_closed_form(oracle_mod):
    # Unweighted, no z-loss, no softcap, sum reduction: the gradient is
    # softmax - (1 - eps) onehot - eps / V.
    rng = np.random.default_rng(1)
    rows, V = 5, 11
    x = rng.normal(0, 3, (rows, V))
    t = rng.integers(0, V, rows)
    for eps in (0.0, 0.1, 0.7, 1.0):
        r = fwd(oracle_mod, x, t, label_smoothing=eps, reduction="sum")
        onehot = np.zeros((rows, V))
        onehot[np.arange(rows), t] = 1.0
        np.testing.assert_allclose(r["grad"], softmax(x) - (1 - eps) * onehot - eps / V,
                                   rtol=1e-12, atol=1e-15)


def test_bf16_decoding_is_exact(oracle_mod):
    pins = {0x3F80: 1.0, 0xC000: -2.0, 0x3FC0: 1.5, 0x4049: 3.140625,
            0x0001: 2.0 ** -133, 0x0080: 2.0 ** -126, 0x7F7F: (2 - 2 ** -7) * 2.0 ** 127,
            0x8000: -0.0, 0x7F80: math.inf, 0xFF80: -math.inf}
    for bits, val in pins.items():
        got = oracle_mod.bf16_to_double(bits)
        assert got == val and math.copysign(1, got) == math.copysign(1, val), hex(bits)
    assert math.isnan(oracle_mod.bf16_to_double(0x7FC0))


def test_bf16_storage_matches_f64_storage(oracle_mod):
    rng = np.random.default_rng(2)
    xf = rng.normal(0, 3, (4, 37)).astype(np.float32)
    bits = workloads.f32_to_bf16_bits(xf)
    t = rng.integers(0, 37, 4)
    a = oracle_mod.forward(bits, t, dtype="bf16", reduction="none")
    b = oracle_mod.forward(workloads.bf16_bits_to_f32(bits).astype(np.float64), t,
                           dtype="f64", reduction="none")
    assert np.array_equal(a["loss"], b["loss"]) and np.array_equal(a["grad"], b["grad"])


def test_f16_decoding_matches_numpy_for_every_bit_pattern(oracle_mod):
    # numpy's float16 -> float64 widening is exact (IEEE binary16): it pins
    # the oracle's own decoder on all 65536 patterns, subnormals, signed
    # zeros, infinities and NaNs included
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    want = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle_mod.f16_to_double(int(b)) for b in bits])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))
    # a few values written out
    pins = {0x3C00: 1.0, 0xC000: -2.0, 0x0001: 2.0 ** -24, 0x0400: 2.0 ** -14,
            0x7BFF: 65504.0, 0x3555: 0.333251953125}
    for b, v in pins.items():
        assert oracle_mod.f16_to_double(b) == v, hex(b)


def test_f16_storage_matches_f64_storage(oracle_mod):
    rng = np.random.default_rng(5)
    xf = rng.normal(0, 3, (4, 41)).astype(np.float32)
    bits = workloads.f32_to_f16_bits(xf)
    t = rng.integers(0, 41, 4)
    opts = dict(reduction="none", label_smoothing=0.1, lse_square_scale=1e-3, softcap=9.0)
    a = oracle_mod.forward(bits, t, dtype="f16", **opts)
    b = oracle_mod.forward(bits.view(np.float16).astype(np.float64), t, dtype="f64", **opts)
    assert np.array_equal(a["loss"], b["loss"]) and np.array_equal(a["grad"], b["grad"])


def test_generator_f16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    vals = np.array([1.0, 1.0 + 2 ** -11, 1.0 + 3 * 2 ** -11, -2.5, 70000.0, 1e-8,
                     3e-5, np.inf, -np.inf], np.float32)
    rng = np.random.default_rng(6)
    vals = np.concatenate([vals, rng.normal(0, 10, 1000).astype(np.float32)])
    ours = workloads.f32_to_f16_bits(vals)
    ref = torch.from_numpy(vals).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_generator_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.4e38, 1e-40,
                     np.inf, -np.inf], np.float32)
    rng = np.random.default_rng(3)
    vals = np.concatenate([vals, rng.normal(0, 10, 1000).astype(np.float32)])
    ours = workloads.f32_to_bf16_bits(vals)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


# ---------------------------------------------------------------- invariants

def test_grad_rows_sum_to_zero_without_zloss_and_softcap(oracle_mod):
    rng = np.random.default_rng(4)
    rows, V = 6, 50
    x = rng.normal(0, 4, (rows, V))
    t = rng.integers(0, V, rows)
    w = rng.uniform(0.5, 2.0, V)
    for weight, eps in itertools.product([None, w], [0.0, 0.3]):
        r = fwd(oracle_mod, x, t, weight=weight, label_smoothing=eps, reduction="sum")
        assert np.abs(r["grad"].sum(axis=1)).max() < 1e-13


def test_grad_row_sum_with_zloss_is_2_lambda_lse(oracle_mod):
    rng = np.random.default_rng(5)
    rows, V, lam = 4, 30, 0.02
    x = rng.normal(0, 2, (rows, V))
    t = rng.integers(0, V, rows)
    r = fwd(oracle_mod, x, t, lse_square_scale=lam, reduction="sum")
    from scipy.special import logsumexp
    lse = logsumexp(x, axis=1)
    np.testing.assert_allclose(r["grad"].sum(axis=1), 2 * lam * lse, rtol=1e-12, atol=1e-14)


def test_reductions_are_consistent(oracle_mod):
    rng = np.random.default_rng(6)
    rows, V = 9, 13
    x = rng.normal(0, 3, (rows, V))
    t = rng.integers(0, V, rows)
    t[[1, 4]] = -100
    w = rng.uniform(0.5, 2.0, V)
    opts = dict(weight=w, label_smoothing=0.1, lse_square_scale=1e-2, softcap=5.0)
    none = fwd(oracle_mod, x, t, reduction="none", **opts)
    s = fwd(oracle_mod, x, t, reduction="sum", **opts)
    m = fwd(oracle_mod, x, t, reduction="mean", **opts)
    valid = t != -100
    D = w[t[valid]].sum()
    assert s["loss"] == pytest.approx(none["loss"].sum(), rel=1e-14)
    assert s["z_loss"] == pytest.approx(none["z_loss"].sum(), rel=1e-14)
    assert m["loss"] == pytest.approx(s["loss"] / D, rel=1e-14)
    assert m["z_loss"] == pytest.approx(s["z_loss"] / D, rel=1e-14)
    np.testing.assert_allclose(m["grad"], s["grad"] / D, rtol=1e-14, atol=1e-300)
    np.testing.assert_array_equal(s["grad"], none["grad"])
    assert none["loss"][~valid].tolist() == [0.0, 0.0]


def test_unit_weights_equal_no_weights_bit_exact(oracle_mod):
    rng = np.random.default_rng(7)
    rows, V = 7, 21
    x = rng.normal(0, 3, (rows, V))
    t = rng.integers(0, V, rows)
    t[2] = -100
    for red in ("none", "sum", "mean"):
        a = fwd(oracle_mod, x, t, reduction=red, label_smoothing=0.2, lse_square_scale=1e-3)
        b = fwd(oracle_mod, x, t, reduction=red, label_smoothing=0.2, lse_square_scale=1e-3,
                weight=np.ones(V))
        for k in ("loss", "z_loss", "acc", "pred", "grad"):
            assert np.array_equal(a[k], b[k]), (red, k)


def test_softcap_converges_to_uncapped(oracle_mod):
    rng = np.random.default_rng(8)
    x = rng.normal(0, 3, (3, 17))
    t = rng.integers(0, 17, 3)
    a = fwd(oracle_mod, x, t, reduction="none", label_smoothing=0.1)
    b = fwd(oracle_mod, x, t, reduction="none", label_smoothing=0.1, softcap=1e7)
    np.testing.assert_allclose(b["loss"], a["loss"], rtol=1e-10)
    np.testing.assert_allclose(b["grad"], a["grad"], rtol=1e-9, atol=1e-14)
    # a small cap really changes the result (the term is live)
    c = fwd(oracle_mod, x, t, reduction="none", label_smoothing=0.1, softcap=2.0)
    assert np.abs(c["loss"] - a["loss"]).max() > 1e-2


def test_softcap_bounds_logits(oracle_mod):
    # With softcap s every z lies in (-s, s), so the loss is at most 2s + ln V.
    x = np.array([[1e4, -1e4, 0.0, 3.0]])
    s = 5.0
    r = fwd(oracle_mod, x, [1], softcap=s, reduction="sum")
    assert 0 < r["loss"] <= 2 * s + math.log(4)
    # logits (s*atanh(a)) reproduce a plain CE over logits (s*a)
    a = np.array([[0.1, -0.5, 0.3, 0.9]])
    r1 = fwd(oracle_mod, s * np.arctanh(a), [2], softcap=s, reduction="sum")
    r2 = fwd(oracle_mod, s * a, [2], reduction="sum")
    assert r1["loss"] == pytest.approx(r2["loss"], rel=1e-12)


# ---------------------------------------------------------------- ignore_index

def test_ignored_rows_are_exact_zero(oracle_mod):
    rng = np.random.default_rng(9)
    x = rng.normal(0, 3, (5, 9))
    t = np.array([1, -100, 3, -100, 0])
    r = fwd(oracle_mod, x, t, reduction="mean", label_smoothing=0.2, lse_square_scale=0.1,
            softcap=4.0)
    g = r["grad"][[1, 3]]
    assert (g == 0).all() and not np.signbit(g).any()
    assert r["pred"][[1, 3]].tolist() == [-1, -1]


def test_custom_ignore_index(oracle_mod):
    rng = np.random.default_rng(10)
    x = rng.normal(0, 3, (4, 6))
    t = np.array([5, 2, 5, 0])
    r = fwd(oracle_mod, x, t, ignore_index=5, reduction="none")
    assert r["loss"][[0, 2]].tolist() == [0.0, 0.0]
    assert (r["grad"][[0, 2]] == 0).all() and r["loss"][1] > 0


def test_nonfinite_logits_in_ignored_rows_do_not_leak(oracle_mod):
    rng = np.random.default_rng(11)
    x = rng.normal(0, 3, (6, 40))
    t = rng.integers(0, 40, 6)
    t[[0, 3]] = -100
    y = x.copy()
    y[0, [1, 5, 7]] = [np.inf, -np.inf, np.nan]
    y[3, :] = np.nan
    for red in ("none", "sum", "mean"):
        a = fwd(oracle_mod, x, t, reduction=red, label_smoothing=0.1)
        b = fwd(oracle_mod, y, t, reduction=red, label_smoothing=0.1)
        for k in ("loss", "z_loss", "acc", "pred", "grad"):
            assert np.array_equal(a[k], b[k]), (red, k)
        assert np.isfinite(b["grad"]).all()


def test_all_ignored_batch(oracle_mod):
    rng = np.random.default_rng(12)
    x = rng.normal(0, 3, (4, 8))
    t = np.full(4, -100)
    m = fwd(oracle_mod, x, t, reduction="mean", label_smoothing=0.1, lse_square_scale=0.1)
    assert math.isnan(m["loss"]) and math.isnan(m["z_loss"]) and math.isnan(m["acc"])
    assert (m["grad"] == 0).all() and not np.signbit(m["grad"]).any()
    s = fwd(oracle_mod, x, t, reduction="sum")
    assert s["loss"] == 0.0 and math.isnan(s["acc"]) and (s["grad"] == 0).all()


def test_target_out_of_range_raises(oracle_mod):
    x = np.zeros((2, 4))
    for bad in (4, -1, 99):
        with pytest.raises(oracle_mod.OracleError):
            fwd(oracle_mod, x, [0, bad])


def test_empty_batch(oracle_mod):
    x = np.zeros((0, 5))
    m = fwd(oracle_mod, x, np.zeros(0, np.int64), reduction="mean")
    assert math.isnan(m["loss"])
    s = fwd(oracle_mod, x, np.zeros(0, np.int64), reduction="sum")
    assert s["loss"] == 0.0


# ---------------------------------------------------------------- argmax, accuracy

def test_argmax_lowest_index_on_ties_and_accuracy(oracle_mod):
    rng = np.random.default_rng(13)
    rows, V = 64, 33
    x = np.round(rng.normal(0, 1, (rows, V)))  # integers: many ties
    for r in range(0, rows, 4):                 # forced ties at known columns
        x[r, :] = 0
        x[r, [5, 9, 30]] = 7
    t = rng.integers(0, V, rows)
    t[::4] = 5
    t[1::8] = -100
    out = fwd(oracle_mod, x, t, reduction="mean")
    brute = np.argmax(x, axis=1)  # numpy returns the first occurrence
    valid = t != -100
    assert np.array_equal(out["pred"][valid], brute[valid])
    assert (out["pred"][~valid] == -1).all()
    assert (out["pred"][::4] == 5).all()
    assert out["acc"] == (brute[valid] == t[valid]).sum() / valid.sum()
    none = fwd(oracle_mod, x, t, reduction="none")
    assert np.array_equal(none["acc"], np.where(valid, (brute == t), 0).astype(float))


def test_argmax_uses_raw_logits_under_softcap(oracle_mod):
    # tanh saturates: 100 and 101 map to the same z in double for s=1, but
    # the raw argmax still separates them.
    x = np.array([[100.0, 101.0, -3.0]])
    r = fwd(oracle_mod, x, [0], softcap=1.0, reduction="sum")
    assert r["pred"][0] == 1


# ---------------------------------------------------------------- finite differences

def _fd_grad(oracle_mod, x, t, h=1e-5, **kw):
    g = np.empty_like(x)
    for idx in np.ndindex(*x.shape):
        xp = x.copy()
        xm = x.copy()
        xp[idx] += h
        xm[idx] -= h
        lp = fwd(oracle_mod, xp, t, want_grad=False, **kw)["loss"]
        lm = fwd(oracle_mod, xm, t, want_grad=False, **kw)["loss"]
        g[idx] = (lp - lm) / (2 * h)
    return g


@pytest.mark.parametrize("weighted", [False, True])
@pytest.mark.parametrize("eps", [0.0, 0.25])
@pytest.mark.parametrize("lam", [0.0, 0.05])
@pytest.mark.parametrize("softcap", [None, 3.0])
@pytest.mark.parametrize("reduction", ["sum", "mean"])
def test_gradient_matches_central_differences(oracle_mod, weighted, eps, lam, softcap, reduction):
    rng = np.random.default_rng(hash((weighted, eps, lam, softcap, reduction)) % 2**32)
    rows, V = 4, 7
    x = rng.normal(0, 2, (rows, V))
    t = rng.integers(0, V, rows)
    t[2] = -100
    w = rng.uniform(0.5, 2.0, V) if weighted else None
    kw = dict(weight=w, label_smoothing=eps, lse_square_scale=lam, softcap=softcap,
              reduction=reduction)
    g = fwd(oracle_mod, x, t, **kw)["grad"]
    fd = _fd_grad(oracle_mod, x, t, **kw)
    np.testing.assert_allclose(g, fd, rtol=1e-7, atol=1e-9)


def test_backward_scales_stored_gradient(oracle_mod):
    rng = np.random.default_rng(14)
    x = rng.normal(0, 2, (3, 5))
    t = rng.integers(0, 5, 3)
    g = fwd(oracle_mod, x, t, reduction="none")["grad"]
    go = np.array([0.5, -2.0, 3.0])
    np.testing.assert_array_equal(oracle_mod.backward(g.copy(), go), g * go[:, None])
    np.testing.assert_array_equal(oracle_mod.backward(g.copy(), 0.25), g * 0.25)


def test_rows_entry_matches_whole_batch(oracle_mod):
    case = workloads.random_case(15, rows=12, V=40, dtype="bf16", weight=True,
                                 label_smoothing=0.1, lse_square_scale=1e-3, softcap=6.0)
    whole = oracle_mod.forward(case.x, case.target, dtype="bf16", weight=case.weight,
                               **case.options())
    idx = np.array([11, 0, 5])
    part = oracle_mod.rows(case.x, case.target, idx, dtype="bf16", weight=case.weight,
                           **case.options())
    np.testing.assert_array_equal(part["grad"], whole["grad"][idx])
    np.testing.assert_array_equal(part["pred"], whole["pred"][idx])
    valid = case.target != -100
    assert part["n_valid"] == valid.sum()
    assert part["D"] == pytest.approx(case.weight[case.target[valid]].astype(np.float64).sum(),
                                      rel=1e-15)
