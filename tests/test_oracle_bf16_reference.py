"""Pins of the oracle's bf16 reference (``oracle.attention_bf16p``) to things other than itself.

The pages' validation advice ("Kernel reference: ring_attention_const_max_fwd", section
"Adapting this kernel", Validation) is to run exact attention on the CPU in fp32 and in bf16
and to compare both error distributions with the kernel's.  The bf16 reference here rounds
each numerator weight p_ij = 2^(z_ij - b_i) to bf16's 8-bit significand (round to nearest,
ties to even) and keeps the denominator exact.  These tests fix it by hand-rounded closed
forms, an exact special case, an invariance, a rigorous error bound and an independent
bit-level rounding, so that a slip (rounding the denominator too, 7 bits instead of 8, the
shift's sign, truncation instead of rounding) fails one of them.
"""
import math

import numpy as np
import pytest

import oracle

LOG2E = math.log2(math.e)
UNIT_ALPHA_SCALE = 1.0 / LOG2E  # softmax scale that makes alpha = scale*log2(e) = 1


def bits_round_sig8(x):
    """fp64 values rounded to 8 significant bits by integer arithmetic on their bit patterns
    (add half an ulp of the kept part, plus one if the kept part is odd, then clear the 45
    dropped bits): an implementation that shares nothing with the oracle's."""
    b = np.asarray(x, dtype=np.float64).copy().view(np.uint64)
    lsb = (b >> np.uint64(45)) & np.uint64(1)
    b = (b + np.uint64((1 << 44) - 1) + lsb) & ~np.uint64((1 << 45) - 1)
    return b.view(np.float64)


def test_bit_rounding_helper_itself():
    # hand-rounded values: spacing 2^-7 in [1, 2), 2^-6 in [2, 4)
    x = np.array([1 + 1 / 512, 1 + 3 / 512, 1 + 5 / 512, 1 + 7 / 512, 3 + 5 / 256, 0.3, 1 + 2 / 512, 1 + 6 / 512])
    want = np.array([1.0, 1 + 4 / 512, 1 + 4 / 512, 1 + 8 / 512, 3 + 4 / 256, 154 / 512, 1.0, 1 + 8 / 512])
    assert np.array_equal(bits_round_sig8(x), want)


def test_power_of_two_weights_are_exact():
    """Integer base-2 logits and an integer shift: every weight is a power of two, which bf16
    holds exactly, so the bf16 reference equals plain attention."""
    r = np.random.default_rng(0)
    keys = np.zeros((40, 3))
    keys[:, 0] = r.integers(-20, 21, size=40)
    v = r.normal(size=(40, 3))
    q = np.zeros((4, 3))
    q[:, 0] = [1.0, 2.0, -1.0, 0.0]
    exact = oracle.attention(q[None], keys[None], v[None], scale=UNIT_ALPHA_SCALE)
    for shift in (None, np.array([[0.0, 3.0, -5.0, 11.0]])):
        got = oracle.attention_bf16p(q[None], keys[None], v[None], shift=shift, scale=UNIT_ALPHA_SCALE)
        assert np.max(np.abs(got - exact)) < 1e-13


@pytest.mark.parametrize("p2,r2", [(1 + 1 / 512, 1.0), (1 + 3 / 512, 1 + 4 / 512), (1 + 5 / 512, 1 + 4 / 512),
                                   (1 + 7 / 512, 1 + 8 / 512), (1.75 + 1 / 1024, 1.75), (3 + 5 / 256, 3 + 4 / 256),
                                   (0.3, 154 / 512)])
def test_two_key_closed_forms(p2, r2):
    """Two keys with weights 1 and p2 at shift 0 (alpha = 1): o = (v1 + bf16(p2) v2) / (1 + p2),
    the rounded weight in the numerator only.  bf16(p2) is rounded by hand."""
    q = np.array([[[1.0, 0.0]]])
    k = np.array([[[0.0, 0.0], [math.log2(p2), 0.0]]])
    v = np.array([[[0.25, -1.0], [1.0, 2.0]]])
    got = oracle.attention_bf16p(q, k, v, shift=np.zeros((1, 1)), scale=UNIT_ALPHA_SCALE)[0, 0]
    want = (np.array([0.25, -1.0]) + r2 * np.array([1.0, 2.0])) / (1.0 + p2)
    assert np.max(np.abs(got - want)) < 1e-14, (got, want)
    # the exact attention differs from it by the rounding of the one weight
    exact = oracle.attention(q, k, v, scale=UNIT_ALPHA_SCALE)[0, 0]
    assert np.max(np.abs((got - exact) - (r2 - p2) * np.array([1.0, 2.0]) / (1.0 + p2))) < 1e-14


def test_integer_shift_changes_nothing_and_a_fractional_one_moves_within_the_bound():
    r = np.random.default_rng(3)
    q, k, v = r.normal(size=(2, 30, 16)), r.normal(size=(2, 400, 16)), r.normal(size=(2, 400, 16))
    b = r.normal(size=(2, 30)) * 5.0
    a = oracle.attention_bf16p(q, k, v, shift=b)
    assert np.max(np.abs(a - oracle.attention_bf16p(q, k, v, shift=b + 7.0))) < 1e-12
    assert np.max(np.abs(a - oracle.attention_bf16p(q, k, v, shift=b - 3.0))) < 1e-12
    c = oracle.attention_bf16p(q, k, v, shift=b + 0.5)
    assert np.max(np.abs(a - c)) > 1e-6  # other significands, other roundings


def test_error_within_the_rigorous_bound_and_not_zero():
    """Round to nearest moves each weight by at most 2^-8 of itself, so element by element
    |o_bf16 - o| <= 2^-8 * sum_j p_j |v_jd| / sum_j p_j; and the rounding is really there."""
    r = np.random.default_rng(4)
    q, k, v = r.normal(size=(3, 25, 16)), r.normal(size=(3, 600, 16)), r.normal(size=(3, 600, 16))
    scale = 0.7
    shift = r.normal(size=(3, 25))
    got = oracle.attention_bf16p(q, k, v, shift=shift, scale=scale)
    exact = oracle.attention(q, k, v, scale=scale)
    s = scale * np.einsum("grd,gnd->grn", q, k)
    p = np.exp(s - s.max(axis=-1, keepdims=True))
    bound = 2.0 ** -8 * np.einsum("grn,gnd->grd", p, np.abs(v)) / p.sum(-1)[..., None]
    err = np.abs(got - exact)
    assert np.all(err <= bound * (1 + 1e-9) + 1e-15)
    assert err.max() > 1e-5
    # typical rounding errors are a fraction of the worst case, not all of it
    assert np.sqrt(np.mean(err ** 2)) < 0.2 * np.sqrt(np.mean(bound ** 2))


def test_single_key_rows_match_bit_level_rounding():
    """With one key per row, o = bf16(p)/p * v for p = 2^(z - b): the ratio must equal the
    bit-level rounding of p (cases within 1e-9 of a rounding tie are skipped)."""
    r = np.random.default_rng(5)
    G, D = 400, 8
    q, k, v = r.normal(size=(G, 1, D)), r.normal(size=(G, 1, D)), r.normal(size=(G, 1, D)) + 3.0
    scale = 0.45
    b = r.normal(size=(G, 1)) * 3.0
    got = oracle.attention_bf16p(q, k, v, shift=b, scale=scale)
    z = scale * LOG2E * np.einsum("gid,gid->gi", q, k)
    p = np.exp2(z - b)
    frac = np.frexp(p)[0] * 256.0
    away = np.abs(frac - np.floor(frac) - 0.5) > 1e-9
    assert away.sum() > 350
    ratio = bits_round_sig8(p) / p
    want = ratio[..., None] * v
    assert np.max(np.abs(got - want)[away]) < 1e-12
    assert np.any(ratio != 1.0)
