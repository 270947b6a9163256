"""Scale-aware parity bars for the bf16 path (test infrastructure; uses the oracle only).

The absolute bar for bf16 inputs is max |o - o_ref| <= 2e-2.  At the pages' workloads |o| is
itself about that size (RMS-normed values averaged over tens of thousands of keys), so that
bar alone would pass an all-zero output.  Next to it, every full-size comparison here also
asks the kernel's error to look like the error bf16 P must cause, following "Kernel
reference: ring_attention_const_max_fwd", section "Adapting this kernel" (Validation: run
exact attention on the CPU in fp32 and in bf16, compare both error distributions with the
kernel's):

  relative   max err <= 1e-2 * max |o_ref|
  element    err_id <= 1.5 * 2^-8 * sum_j p_ij |v_jd| / sum_j p_ij  (+ 1e-6 max |o_ref|):
             rounding a weight to bf16 moves it by at most 2^-8 of itself, so this bounds
             what the P rounding can do to each element; the 1.5 leaves room for the fp32
             sums (the row sum and the PV accumulation), which are far smaller
  quantiles  the median and the 99th percentile of |err| at most 4x those of the oracle's
             bf16-P reference (oracle.attention_bf16p at the oracle's own fixed-m shift),
             plus the same tiny floor.  Quantiles, not the maximum: on a row that one key
             dominates, the rounding of that one weight is a single draw, different in the
             kernel and in the reference.

All three are computed from oracle outputs; nothing here comes from the CUDA path except
the array being judged.
"""
from __future__ import annotations

import numpy as np

import oracle

TOL_BF16 = 2e-2      # absolute bar, bf16 inputs with fp32 accumulation
REL_BAR = 1e-2       # max error over max |o_ref|
ELEMENT_SLACK = 1.5  # on the rigorous 2^-8 bound of the P rounding
QUANTILE_FACTOR = 4.0
FLOOR_REL = 1e-6


TOL_F32 = 1e-5  # absolute bar, fp32 inputs


def f32_bar(q, k, scale=None):
    """The 1e-5 bar for fp32 inputs, widened in proportion to the logits' bound U
    above 8.  fp32 rounds a dot product q.k to within about 2^-24 sqrt(D) sum_d |q_d k_d|,
    and sum_d |q_d k_d| <= |q| |k|, so a base-2 logit carries an error proportional to
    U = alpha * max|q| * max|k| (the method's own Cauchy-Schwarz bound), which every weight
    inherits.  At the fp32 workload's inputs U is below 8 and the bar is 1e-5; keys a hundred
    times louder than the rest widen it accordingly."""
    q, k = _np(q), _np(k)
    D = q.shape[-1]
    alpha = (1.0 / np.sqrt(D) if scale is None else scale) * np.log2(np.e)
    qn = np.sqrt((q ** 2).sum(-1)).max() if q.size else 0.0
    kn = np.sqrt((k ** 2).sum(-1)).max() if k.size else 0.0
    return TOL_F32 * max(1.0, alpha * qn * kn / 8.0)


class Reference:
    """Oracle outputs for the rows under test: exact o, the bf16-P reference at the oracle's
    fixed-m shift, and sum_j p |v| / sum_j p (the weighted mean of |v|)."""

    def __init__(self, q, k, v, shift):
        self.o = oracle.attention(q, k, v)
        self.model = oracle.attention_bf16p(q, k, v, shift=shift)
        self.abs_v = oracle.attention(q, k, np.abs(_np(v)))

    def check(self, got, what=""):
        return assert_bf16_parity(got, self.o, self.model, self.abs_v, what)


def _np(x):
    if hasattr(x, "detach"):
        return x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def bf16_parity_report(got, ref, model, abs_v):
    got, ref, model, abs_v = _np(got), _np(ref), _np(model), _np(abs_v)
    assert got.shape == ref.shape == model.shape == abs_v.shape, (got.shape, ref.shape, model.shape, abs_v.shape)
    err = np.abs(got - ref)
    merr = np.abs(model - ref)
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    floor = FLOOR_REL * max(scale, 1e-30)
    bound = ELEMENT_SLACK * 2.0 ** -8 * abs_v + floor
    with np.errstate(invalid="ignore"):
        over = np.where(np.isfinite(err), err / bound, np.inf)
    return {
        "max_err": float(err.max()) if err.size else 0.0,
        "rms_err": float(np.sqrt(np.mean(err ** 2))) if err.size else 0.0,
        "max_ref": scale,
        "floor": floor,
        "p50": float(np.quantile(err, 0.5)) if err.size else 0.0,
        "p99": float(np.quantile(err, 0.99)) if err.size else 0.0,
        "model_p50": float(np.quantile(merr, 0.5)) if merr.size else 0.0,
        "model_p99": float(np.quantile(merr, 0.99)) if merr.size else 0.0,
        "model_max": float(merr.max()) if merr.size else 0.0,
        "worst_over_element_bound": float(over.max()) if over.size else 0.0,
        "finite": bool(np.all(np.isfinite(got))),
    }


def assert_bf16_parity(got, ref, model, abs_v, what=""):
    """Every bar of this module; returns the figures."""
    r = bf16_parity_report(got, ref, model, abs_v)
    tag = f"{what}: {r}"
    assert r["finite"], tag
    assert r["max_err"] <= TOL_BF16, tag
    assert r["max_err"] <= REL_BAR * r["max_ref"], tag
    assert r["worst_over_element_bound"] <= 1.0, tag
    assert r["p50"] <= QUANTILE_FACTOR * r["model_p50"] + r["floor"], tag
    assert r["p99"] <= QUANTILE_FACTOR * r["model_p99"] + r["floor"], tag
    return r
