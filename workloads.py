"""Seeded synthetic inputs for fused softmax cross-entropy.

This module only draws inputs: logits, targets and class weights with the
shapes, distributions and ignore fractions of the workloads the pages
describe. It holds no cross-entropy arithmetic, so both the CUDA path's
tests and the CPU oracle can take their inputs from here.

The workloads (all logits row-major (rows, V), class dimension last):

  small       rows=64, V=4096, fp32 N(0, 2^2); 10% of targets ignored;
              mean; also argmax and accuracy.
  vsweep      rows=4096 (B=8, T=512), V in {4096 ... 131072}, bf16
              N(0, 3^2); 5% ignored; mean; fused fwd+bwd in place. This is
              the sweep of the Liger cross-entropy profile (§Benchmarking).
  tt_fp32     rows=1023, V=128256, fp32 N(0, 4^2) with about 1% of entries +30;
              15% ignored; mean and sum. Variants: every row ignored, and
              ignored rows holding +-inf/NaN in 1% of their entries. This is
              the workload of tt-mlir pull request #9324 (problem table).
  softcap_z   rows=4096, V=131072, bf16 N(0, 8^2); softcap 30, label
              smoothing 0.1, lse_square_scale 1e-4 with z_loss; 5% ignored;
              mean.
  weighted    rows=16384, V=32000, bf16 N(0, 3^2); class weights fp32
              U[0.5, 2.0]; label smoothing 0.05; none and mean; 2% ignored.

bf16 logits are produced as float32 draws rounded to nearest-even bf16 and
are returned as their raw uint16 bit patterns.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np

IGNORE_INDEX = -100
VSWEEP = (4096, 8192, 16384, 32768, 65536, 131072)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Rounds float32 values to bf16 (round to nearest, ties to even) and
    returns the uint16 bit patterns. NaN stays a quiet NaN."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    out = ((u + (((u >> 16) & 1) + 0x7FFF)) >> 16).astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        out[nan] = ((u[nan] >> 16) | 0x0040).astype(np.uint16)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass
class Case:
    name: str
    x: np.ndarray             # float32 (rows, V), or uint16 bf16 / fp16 bits (rows, V)
    dtype: str                # "f32" | "bf16" | "f16"
    target: np.ndarray        # int32 (rows,)
    weight: np.ndarray | None = None   # float32 (V,)
    ignore_index: int = IGNORE_INDEX
    label_smoothing: float = 0.0
    lse_square_scale: float = 0.0
    softcap: float | None = None
    reduction: str = "mean"
    return_z_loss: bool = False
    return_acc: bool = False
    return_pred: bool = False
    notes: dict = field(default_factory=dict)

    @property
    def rows(self) -> int:
        return self.x.shape[0]

    @property
    def V(self) -> int:
        return self.x.shape[1]

    def options(self) -> dict:
        return dict(ignore_index=self.ignore_index, label_smoothing=self.label_smoothing,
                    lse_square_scale=self.lse_square_scale, softcap=self.softcap,
                    reduction=self.reduction)

    def with_(self, **kw) -> "Case":
        return replace(self, **kw)


_BLOCK_ELEMS = 1 << 22  # elements per independently seeded block


def f32_to_f16_bits(a: np.ndarray) -> np.ndarray:
    """Rounds float32 values to IEEE binary16 (numpy's conversion: nearest,
    ties to even; overflow to infinity) and returns the uint16 bit patterns."""
    return np.ascontiguousarray(a, dtype=np.float32).astype(np.float16).view(np.uint16)


def _blocked_normal(seed, rows, V, std, storage):
    """N(0, std^2) logits drawn in fixed row blocks, block b from child b of
    SeedSequence([seed, 0]); blocks run on a thread pool (numpy's generators
    and ufuncs release the GIL), so the values do not depend on the number
    of threads."""
    from concurrent.futures import ThreadPoolExecutor
    import os
    out = np.empty((rows, V), np.float32 if storage == "f32" else np.uint16)
    if out.size == 0:
        return out
    brows = max(1, _BLOCK_ELEMS // max(V, 1))
    starts = list(range(0, rows, brows))
    seeds = np.random.SeedSequence([seed, 0]).spawn(len(starts))

    def fill(i):
        r0 = starts[i]
        r1 = min(rows, r0 + brows)
        blk = np.random.default_rng(seeds[i]).standard_normal((r1 - r0, V), dtype=np.float32)
        blk *= np.float32(std)
        if storage == "bf16":
            out[r0:r1] = f32_to_bf16_bits(blk)
        elif storage == "f16":
            out[r0:r1] = f32_to_f16_bits(blk)
        else:
            out[r0:r1] = blk

    if len(starts) == 1:
        fill(0)
    else:
        with ThreadPoolExecutor(max_workers=min(len(starts), os.cpu_count() or 4)) as ex:
            list(ex.map(fill, range(len(starts))))
    return out


def _normal(seed, rows, V, std):
    return _blocked_normal(seed, rows, V, std, "f32")


def _bf16_normal(seed, rows, V, std):
    return _blocked_normal(seed, rows, V, std, "bf16")


def _f16_normal(seed, rows, V, std):
    return _blocked_normal(seed, rows, V, std, "f16")


def _aux_rng(seed):
    """Generator for everything but the logits (targets, weights, outliers)."""
    return np.random.default_rng(np.random.SeedSequence([seed, 1]))


def targets(rng, rows, V, ignore_frac, ignore_index=IGNORE_INDEX):
    """Uniform targets in [0, V) with exactly round(ignore_frac * rows)
    rows set to ignore_index."""
    t = rng.integers(0, V, size=rows, dtype=np.int64).astype(np.int32)
    n_ign = int(round(ignore_frac * rows))
    if n_ign:
        t[rng.choice(rows, size=n_ign, replace=False)] = ignore_index
    return t


def small(seed=0, rows=64, V=4096) -> Case:
    rng = _aux_rng(seed)
    x = _normal(seed, rows, V, 2.0)
    return Case("small", x, "f32", targets(rng, rows, V, 0.10),
                return_acc=True, return_pred=True)


def vsweep(V=131072, seed=0, rows=4096) -> Case:
    rng = _aux_rng(seed)
    x = _bf16_normal(seed, rows, V, 3.0)
    return Case(f"vsweep_V{V}", x, "bf16", targets(rng, rows, V, 0.05))


def tt_fp32(seed=0, rows=1023, V=128256, reduction="mean", variant="plain") -> Case:
    """variant: "plain", "all_ignored" or "nonfinite_ignored"."""
    rng = _aux_rng(seed)
    x = _normal(seed, rows, V, 4.0)
    # about 1% of the entries get +30 (positions drawn with replacement)
    n_out = int(round(0.01 * x.size))
    flat = x.reshape(-1)
    flat[np.unique(rng.integers(0, x.size, size=n_out))] += np.float32(30.0)
    t = targets(rng, rows, V, 0.15)
    if variant == "all_ignored":
        t[:] = IGNORE_INDEX
    elif variant == "nonfinite_ignored":
        ign = np.nonzero(t == IGNORE_INDEX)[0]
        specials = np.array([np.inf, -np.inf, np.nan], np.float32)
        for r in ign:
            cols = rng.choice(V, size=max(1, V // 100), replace=False)
            x[r, cols] = specials[rng.integers(0, 3, size=cols.size)]
    elif variant != "plain":
        raise ValueError(variant)
    return Case(f"tt_fp32_{variant}_{reduction}", x, "f32", t, reduction=reduction)


def softcap_z(seed=0, rows=4096, V=131072) -> Case:
    rng = _aux_rng(seed)
    x = _bf16_normal(seed, rows, V, 8.0)
    return Case("softcap_z", x, "bf16", targets(rng, rows, V, 0.05), softcap=30.0,
                label_smoothing=0.1, lse_square_scale=1e-4, return_z_loss=True)


def weighted(seed=0, rows=16384, V=32000, reduction="mean") -> Case:
    rng = _aux_rng(seed)
    x = _bf16_normal(seed, rows, V, 3.0)
    w = rng.uniform(0.5, 2.0, size=V).astype(np.float32)
    return Case(f"weighted_{reduction}", x, "bf16", targets(rng, rows, V, 0.02),
                weight=w, label_smoothing=0.05, reduction=reduction)


def random_case(seed, rows, V, dtype="f32", std=3.0, ignore_frac=0.1, **opts) -> Case:
    """Generic seeded case for parity sweeps over shapes and options."""
    rng = _aux_rng(seed)
    gen = {"f32": _normal, "bf16": _bf16_normal, "f16": _f16_normal}[dtype]
    x = gen(seed, rows, V, std)
    t = targets(rng, rows, V, ignore_frac)
    w = opts.pop("weight", None)
    if w is True:
        w = rng.uniform(0.5, 2.0, size=V).astype(np.float32)
    return Case(f"random_{rows}x{V}_{dtype}", x, dtype, t, weight=w, **opts)


def nd_case(seed, shape, dtype="f32", std=3.0, ignore_frac=0.1, **opts) -> Case:
    """Seeded case with N-D logits (N, C, d1, ..., dk), the class dimension at
    axis 1, and targets (N, d1, ..., dk). The logits are the blocked normal
    draws of an (N * C, d1 * ... * dk) matrix reshaped; the targets are
    uniform in [0, C) with round(ignore_frac * positions) ignored."""
    shape = tuple(int(d) for d in shape)
    N, C = shape[0], shape[1]
    inner = int(np.prod(shape[2:], dtype=np.int64))
    rng = _aux_rng(seed)
    gen = {"f32": _normal, "bf16": _bf16_normal, "f16": _f16_normal}[dtype]
    x = gen(seed, N * C, inner, std).reshape(shape)
    t = targets(rng, N * inner, C, ignore_frac).reshape((N,) + shape[2:])
    w = opts.pop("weight", None)
    if w is True:
        w = rng.uniform(0.5, 2.0, size=C).astype(np.float32)
    return Case(f"nd_{'x'.join(map(str, shape))}_{dtype}", x, dtype, t, weight=w, **opts)


def logits_f64(case: Case) -> np.ndarray:
    """The logits as float64 values (exact for every storage)."""
    if case.dtype == "bf16":
        return bf16_bits_to_f32(case.x).astype(np.float64)
    if case.dtype == "f16":
        return np.ascontiguousarray(case.x, dtype=np.uint16).view(np.float16).astype(np.float64)
    return case.x.astype(np.float64)
