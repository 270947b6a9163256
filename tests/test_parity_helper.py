"""The scale-aware parity bars (tests/parity.py) can fail: CPU checks with oracle outputs only.

At the pages' workloads |o| is about as large as the absolute 2e-2 bar, so that bar alone
passes an all-zero output.  These tests show that the added bars reject the outputs a broken
kernel would produce -- zero, scaled by 0.9, ten times noisier than bf16 P, a row from the
wrong query, a chunk of keys left out -- and accept the oracle's own bf16-P reference and
another legitimate bf16 rounding (the reference at each row's max instead of the fixed-m
shift).  No kernel is broken to show this.
"""
import numpy as np
import pytest

import oracle
import workloads
from tests import parity


@pytest.fixture(scope="module")
def case():
    # the H40 S4096 workload's recipe and key count, 256 query rows of two heads
    q, k, v = workloads.make_inputs("h40_s4096", device="cpu", heads=[0, 1], Sq=256)
    ob = oracle.bounds(q, k, v, centering=False)
    ref = parity.Reference(q[0], k[0], v[0], ob["shift"][0])
    # the premise: |o| is of the order of the absolute bar
    assert np.abs(ref.o).max() < 2 * parity.TOL_BF16
    return q, k, v, ref


def test_accepts_bf16_references(case):
    q, k, v, ref = case
    parity.assert_bf16_parity(ref.model, ref.o, ref.model, ref.abs_v, "bf16-P at the fixed-m shift")
    other = oracle.attention_bf16p(q[0], k[0], v[0])  # rounded at each row's max instead
    parity.assert_bf16_parity(other, ref.o, ref.model, ref.abs_v, "bf16-P at the row max")


def test_zero_output_passes_the_absolute_bar_but_not_these(case):
    _, _, _, ref = case
    zero = np.zeros_like(ref.o)
    assert np.abs(zero - ref.o).max() <= parity.TOL_BF16  # what the absolute bar alone lets through
    with pytest.raises(AssertionError):
        parity.assert_bf16_parity(zero, ref.o, ref.model, ref.abs_v)


@pytest.mark.parametrize("factor", [0.9, 0.99, 1.01])
def test_scaled_output_fails(case, factor):
    _, _, _, ref = case
    with pytest.raises(AssertionError):
        parity.assert_bf16_parity(factor * ref.o, ref.o, ref.model, ref.abs_v)


def test_ten_times_the_bf16_error_fails(case):
    _, _, _, ref = case
    noisy = ref.o + 10.0 * (ref.model - ref.o)
    with pytest.raises(AssertionError):
        parity.assert_bf16_parity(noisy, ref.o, ref.model, ref.abs_v)


def test_a_row_from_the_wrong_query_fails(case):
    _, _, _, ref = case
    bad = ref.model.copy()
    bad[1, 77] = ref.model[1, 78]  # one row of 512 taken from its neighbour
    with pytest.raises(AssertionError):
        parity.assert_bf16_parity(bad, ref.o, ref.model, ref.abs_v)


def test_a_dropped_chunk_fails(case):
    q, k, v, ref = case
    partial = oracle.attention(q[0], k[0, :, :3000], v[0, :, :3000])  # the last 1096 keys lost
    with pytest.raises(AssertionError):
        parity.assert_bf16_parity(partial, ref.o, ref.model, ref.abs_v)


def test_a_non_finite_element_fails(case):
    _, _, _, ref = case
    bad = ref.model.copy()
    bad[0, 3, 5] = np.nan
    with pytest.raises(AssertionError):
        parity.assert_bf16_parity(bad, ref.o, ref.model, ref.abs_v)


def test_f32_bar_is_the_plain_1e5_at_the_fp32_workload():
    q, k, _ = workloads.make_inputs("tiny")
    assert parity.f32_bar(q[0], k[0]) == parity.TOL_F32
    # a key a hundred times louder widens it in proportion to the bound U
    k2 = k.clone()
    k2[0, 0, 3] *= 100.0
    assert parity.f32_bar(q[0, :1], k2[0, :1]) > 5 * parity.TOL_F32
