"""Writes ce_facts.json: hand-derived closed forms and the few numbers the
pages print. It calls only Python's math module (neither the oracle nor the
CUDA library), so every stored value is fixed by mathematics or by a page.

    python tests/golden/make_ce_facts.py
"""
import json
import math
import os

ln = math.log


def closed_forms():
    cases = [
        dict(name="uniform_V4", x=[0.7, 0.7, 0.7, 0.7], target=2,
             label_smoothing=0.0, lse_square_scale=0.0,
             derivation="all logits equal: p_j = 1/4, lse = 0.7 + ln 4, "
                        "loss = lse - z_t = ln 4; gradient p - onehot",
             loss=ln(4), grad=[0.25, 0.25, -0.75, 0.25]),
        dict(name="two_class_ln3", x=[0.0, ln(3)], target=0,
             label_smoothing=0.0, lse_square_scale=0.0,
             derivation="exp(z) = (1, 3): p = (1/4, 3/4), lse = ln 4, loss = ln 4 - 0",
             loss=ln(4), grad=[-0.75, 0.75]),
        dict(name="two_class_ln3_smooth_half", x=[0.0, ln(3)], target=0,
             label_smoothing=0.5, lse_square_scale=0.0,
             derivation="(1-eps)(lse - z_0) + (eps/2)[(lse - z_0) + (lse - z_1)] "
                        "= 0.5 ln4 + 0.25 (2 ln4 - ln3) = ln4 - ln3/4; gradient "
                        "p - (1-eps) onehot - eps/V = (1/4 - 1/2 - 1/4, 3/4 - 1/4)",
             loss=ln(4) - ln(3) / 4, grad=[-0.5, 0.5]),
    ]
    lse, lam = ln(8), 0.01
    cases.append(dict(
        name="zloss_V3", x=[0.0, ln(2), ln(5)], target=2, label_smoothing=0.0,
        lse_square_scale=lam,
        derivation="exp(z) = (1, 2, 5): lse = ln 8, nll = ln 8 - ln 5, z-loss = "
                   "lam (ln 8)^2; gradient p (1 + 2 lam ln 8) - onehot with "
                   "p = (1/8, 2/8, 5/8)",
        loss=(ln(8) - ln(5)) + lam * lse * lse,
        grad=[(1 / 8) * (1 + 2 * lam * lse), (2 / 8) * (1 + 2 * lam * lse),
              (5 / 8) * (1 + 2 * lam * lse) - 1.0]))
    return cases


def main():
    doc = {
        "source": "hand-derived closed forms (mathematics) and the numbers the pages print",
        "closed_forms": closed_forms(),
        "logit_gap": {
            "citation": "tt-mlir pull request #9339 description (quoted in #9324): "
                        "_log_softmax is lowered as a max-shifted log-sum-exp because "
                        "plain log(softmax) reaches -inf past a logit gap of about 87",
            "setup": "two classes, logits (0, gap), target 0; loss = gap + "
                     "log1p(exp(-gap)) stays finite at every gap",
            "cases": [dict(gap=g, loss=g + math.log1p(math.exp(-g)))
                      for g in (50.0, 87.0, 88.0, 104.0, 1000.0)],
        },
        "workload_bytes": {
            "citation": "tt-mlir pull request #9324, problem description table: "
                        "rows=1023, C=128256, f32 log-probabilities of 500 MiB",
            "rows": 1023, "V": 128256, "bytes_per_element": 4, "mib": 500,
        },
        "vsweep": {
            "citation": "Liger-Kernel cross-entropy kernel profile, section "
                        "Benchmarking: V in 4096..131072 at B=8, T=512, bf16",
            "V": [4096, 8192, 16384, 32768, 65536, 131072], "B": 8, "T": 512,
        },
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "ce_facts.json")
    with open(path, "w") as f:
        f.write(json.dumps(doc, indent=1) + "\n")


if __name__ == "__main__":
    main()
