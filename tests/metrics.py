"""Parity graders: the tolerances of the adapted layer's acceptance criteria.

* fp32 contexts: max_i |g_i - r_i| / max(|r_i|, 1e-2 rms(r)) <= 1e-4.  The
  floor makes the relative error defined near zero crossings.  On the tiny
  fp32 workload a strictly sequential float32 sum of xW scores 1.25-1.5e-4
  under a 1e-3 rms(r) floor and NumPy's blocked sgemm 4.7e-5; the GPU's
  split-precision tf32 GEMM (three products) scores 2.2e-4 there and 5.6e-5
  under the 1e-2 floor used here (test_tiny_fp32 prints both).
* bf16 outputs: max |g - r| <= 3e-2, except where half a bf16 spacing of r
  exceeds 1.5e-2 (|r| >= 4): there the output is graded as
  |g - RN_bf16(r)| <= 1 bf16 spacing (rounding alone would break 3e-2).
* adapter effect: Delta = y - xW; per adapter a,
  sum |Dg - Dr| / sum |Dr| over its rows and all columns <= 1%, graded on fp32
  outputs (a bf16 output's own rounding is ~0.9% of a rank-16 LoRA effect).
"""
import numpy as np

from workloads import bf16_bits, bf16_values

FP32_REL_TOL = 1e-4
BF16_ABS_TOL = 3e-2
EFFECT_TOL = 0.01


FP32_FLOOR = 1e-2


def fp32_rel_err(g, r, floor_frac=FP32_FLOOR):
    g = np.asarray(g, np.float64)
    r = np.asarray(r, np.float64)
    floor = floor_frac * np.sqrt(np.mean(r * r))
    return float(np.max(np.abs(g - r) / np.maximum(np.abs(r), floor)))


def round_bf16(r):
    """The float64 values rounded to bf16 (round-to-nearest-even through
    float32), as float64."""
    r = np.asarray(r, np.float64)
    return bf16_values(bf16_bits(r.astype(np.float32))).astype(np.float64).reshape(r.shape)


def normwise_err(g, r):
    g = np.asarray(g, np.float64)
    r = np.asarray(r, np.float64)
    return float(np.max(np.abs(g - r)) / np.max(np.abs(r)))


def bf16_spacing(v):
    """Distance between consecutive bf16 values around |v| (8 significant bits)."""
    a = np.maximum(np.abs(np.asarray(v, np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def grade_bf16_out(g, r):
    """Returns (max abs error where the 3e-2 bound applies, max error in bf16
    spacings where it does not, count of the latter)."""
    g = np.asarray(g, np.float64)
    r = np.asarray(r, np.float64)
    big = 0.5 * bf16_spacing(r) > 1.5e-2
    small_err = float(np.max(np.abs(g - r)[~big])) if np.any(~big) else 0.0
    if np.any(big):
        rn = bf16_values(bf16_bits(r[big].astype(np.float32))).astype(np.float64)
        big_err = float(np.max(np.abs(g[big] - rn) / bf16_spacing(rn)))
    else:
        big_err = 0.0
    return small_err, big_err, int(np.sum(big))


def assert_bf16_out(g, r, what=""):
    small, big, nbig = grade_bf16_out(g, r)
    assert small <= BF16_ABS_TOL, f"{what}: max abs error {small:.4g} > {BF16_ABS_TOL}"
    assert big <= 1.0 + 1e-9, f"{what}: {big:.3g} bf16 spacings from RN(r) on {nbig} large elements"


def effect_errors(g, r, base, ids):
    """Per adapter id: sum |Dg - Dr| / sum |Dr| (ids with no effect skipped)."""
    g = np.asarray(g, np.float64)
    r = np.asarray(r, np.float64)
    base = np.asarray(base, np.float64)
    out = {}
    for a in np.unique(ids):
        if a < 0:
            continue
        rows = ids == a
        dr = r[rows] - base[rows]
        den = np.sum(np.abs(dr))
        if den <= 1e-12 * max(1.0, np.sum(np.abs(r[rows]))):
            continue
        out[int(a)] = float(np.sum(np.abs((g[rows] - base[rows]) - dr)) / den)
    return out
