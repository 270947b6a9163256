"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test checks the oracle against what the pages print or what mathematics fixes:
closed forms, invariants, brute force on tiny inputs, a library routine, and the
constants and adversarial verdicts printed on the PR #477 page.  They are chosen so
that a plausible slip in the oracle (a dropped term, a wrong sign or index, a
transposed operand, a missing max subtraction or normalisation) fails one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.conftest import golden

LOG2E = math.log2(math.e)


def rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- attention (T1, T2)

def brute_force_attention(q, k, v, scale):
    """Independent naive triple loop with math.exp and no max subtraction (tiny, tame inputs)."""
    R, D = q.shape
    N = k.shape[0]
    out = np.zeros((R, D))
    for i in range(R):
        w = [math.exp(scale * sum(q[i, d] * k[j, d] for d in range(D))) for j in range(N)]
        tot = sum(w)
        for d in range(D):
            out[i, d] = sum(w[j] * v[j, d] for j in range(N)) / tot
    return out


def test_attention_matches_brute_force_loop():
    r = rng(0)
    q, k, v = r.normal(size=(5, 6)), r.normal(size=(7, 6)), r.normal(size=(7, 6))
    got = oracle.attention(q[None], k[None], v[None], scale=0.37)[0]
    want = brute_force_attention(q, k, v, 0.37)
    assert np.max(np.abs(got - want)) < 1e-13


def test_attention_matches_torch_softmax_fp64():
    r = rng(1)
    B, H, S, N, D = 1, 3, 33, 41, 16
    q, k, v = r.normal(size=(B, H, S, D)), r.normal(size=(B, H, N, D)), r.normal(size=(B, H, N, D))
    got = oracle.attention(q, k, v)
    t = torch.softmax(torch.from_numpy(q) @ torch.from_numpy(k).transpose(-1, -2) / math.sqrt(D), dim=-1)
    want = (t @ torch.from_numpy(v)).numpy()
    assert got.shape == (B, H, S, D)
    assert np.max(np.abs(got - want)) < 1e-13


def test_attention_lse_matches_logsumexp():
    r = rng(2)
    q, k, v = r.normal(size=(1, 9, 8)), r.normal(size=(1, 13, 8)), r.normal(size=(1, 13, 8))
    _, lse = oracle.attention(q, k, v, scale=0.5, return_lse=True)
    s = 0.5 * np.einsum("grd,gnd->grn", q, k)
    want = torch.logsumexp(torch.from_numpy(s), dim=-1).numpy()
    assert np.max(np.abs(lse - want)) < 1e-12


def test_shift_invariance_key_offset():
    """Adding one vector c to every key shifts each row's scores by q_i.c: output unchanged.

    Large c makes raw exp overflow, so this also pins the max subtraction (T1)."""
    r = rng(3)
    q, k, v = r.normal(size=(1, 20, 16)), r.normal(size=(1, 30, 16)), r.normal(size=(1, 30, 16))
    c = 40.0 * r.normal(size=(16,))
    a = oracle.attention(q, k, v)
    b = oracle.attention(q, k + c, v)
    assert np.all(np.isfinite(b))
    assert np.max(np.abs(a - b)) < 1e-12


def test_value_affine_and_key_permutation():
    r = rng(4)
    q, k, v = r.normal(size=(1, 11, 8)), r.normal(size=(1, 17, 8)), r.normal(size=(1, 17, 8))
    o = oracle.attention(q, k, v)
    # weights sum to one: an affine map of V passes through
    o2 = oracle.attention(q, k, 3.0 * v - 2.0)
    assert np.max(np.abs(o2 - (3.0 * o - 2.0))) < 1e-12
    # keys and values are paired: permuting them together changes nothing
    p = r.permutation(17)
    o3 = oracle.attention(q, k[:, p], v[:, p])
    assert np.max(np.abs(o3 - o)) < 1e-13
    # but permuting only the values does (catches a k_j / v_j pairing slip)
    o4 = oracle.attention(q, k, v[:, p])
    assert np.max(np.abs(o4 - o)) > 1e-3


def test_closed_forms():
    r = rng(5)
    D = 8
    v = r.normal(size=(1, 12, D))
    k = r.normal(size=(1, 12, D))
    # Q = 0: uniform weights -> mean of V
    o = oracle.attention(np.zeros((1, 3, D)), k, v)
    assert np.max(np.abs(o - v.mean(axis=1, keepdims=True))) < 1e-14
    # all keys identical: uniform weights again
    o = oracle.attention(r.normal(size=(1, 3, D)), np.repeat(k[:, :1], 12, axis=1), v)
    assert np.max(np.abs(o - v.mean(axis=1, keepdims=True))) < 1e-14
    # one key: output is that value
    o = oracle.attention(r.normal(size=(1, 3, D)), k[:, :1], v[:, :1])
    assert np.max(np.abs(o - v[:, :1])) < 1e-15
    # one overwhelmingly aligned key: output is its value
    kk = r.normal(size=(1, 12, D)) * 0.01
    kk[0, 5] = 50.0 * np.ones(D)
    o = oracle.attention(np.ones((1, 2, D)), kk, v, scale=1.0)
    assert np.max(np.abs(o - v[:, 5:6])) < 1e-12
    # empty key set: zeros
    o = oracle.attention(np.ones((1, 2, D)), np.zeros((1, 0, D)), np.zeros((1, 0, D)))
    assert np.all(o == 0.0)


def test_closed_form_qk_zero_v_one():
    rows = dict((r[0], r[1:]) for r in golden("closed_forms.txt"))
    expected = float(rows["qk_zero_v_one"][0])
    o = oracle.attention(np.zeros((1, 4, 16)), np.zeros((1, 9, 16)), np.ones((1, 9, 16)))
    assert np.all(o == expected)


def test_sum_clamp_matches_85_nats():
    rows = dict((r[0], r[1:]) for r in golden("closed_forms.txt"))
    clamp, nats = float(rows["sum_clamp"][0]), float(rows["sum_clamp"][1])
    # a row whose terms are all e^-x reaches the clamp at x = -ln(clamp)
    assert abs(-math.log(clamp) - nats) < 1.0


# ---------------------------------------------------------------- constants (T6)

def test_constants_printed_values():
    for row in golden("constants.txt"):
        n, vmax = int(row[0]), int(row[1])
        C, W, gate = oracle.constants(n, vmax)
        for want, got in zip(row[2:5], (C, W, gate)):
            if want != "-":
                assert int(want) == got, (row, (C, W, gate))


def test_legacy_window_triples():
    # W = C + 125 and gate = floor(W/2) reproduce the legacy (88, 213, 106) and new triple
    for c, w, g in golden("legacy_window.txt"):
        c, w, g = int(c), int(w), int(g)
        # find an N with this C (at Vmax = 256) when one exists, else check W/gate arithmetic
        n = 2 ** (127 - 8 - c)
        C, W, gate = oracle.constants(n, 256)
        assert (C, W, gate) == (c, w, g)


def test_ceil_log2_brute_force():
    for n in list(range(1, 300)) + [4095, 4096, 4097, 37800, 75600, 2 ** 40, 2 ** 40 + 1]:
        want = 0
        while (1 << want) < n:
            want += 1
        assert oracle.ceil_log2(n) == want, n


# ---------------------------------------------------------------- bounds (closed forms)

def test_bounds_closed_form_norms_and_mean():
    """Planted norms and an exactly known key mean.  U is in base-2 logit units: it bounds
    alpha*q.k with alpha = scale*log2(e), the exponent the kernels feed to exp2."""
    D, Sq, N = 16, 300, 64
    r = rng(6)
    c = r.normal(size=(D,))
    u = r.normal(size=(N // 2, D))
    u /= np.linalg.norm(u, axis=1, keepdims=True)
    k = np.concatenate([u, -u]) + c  # mean exactly c, centered norms exactly 1
    k[[3, 40]] = k[[40, 3]]
    q = r.normal(size=(Sq, D))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    planted = {5: 3.0, 130: 7.5, 299: 2.25}  # row -> norm, one per Q-block
    for i, nrm in planted.items():
        q[i] *= nrm
    v = r.normal(size=(N, D))
    b = oracle.bounds(q[None], k[None], v[None], scale=0.25, centering=True)
    assert np.max(np.abs(b["kbar"][0] - c)) < 1e-14
    assert abs(b["kmax_sq"][0] - 1.0) < 1e-12
    qmax = b["qmax_sq"][0]
    assert qmax.shape == (3,)
    assert np.allclose(qmax, [9.0, 56.25, 5.0625], rtol=1e-13)
    alpha = 0.25 * LOG2E
    assert np.allclose(b["U"][0], alpha * np.array([3.0, 7.5, 2.25]), rtol=1e-13)
    assert np.allclose(b["qkbar"][0], alpha * (q @ c), rtol=1e-12, atol=1e-12)
    assert b["vmax_sq"] == pytest.approx(np.max(v * v), rel=0, abs=0)
    # raw keys: the norm is that of k itself, and the mean is not used
    b2 = oracle.bounds(q[None], k[None], v[None], scale=0.25, centering=False)
    assert np.all(b2["kbar"] == 0.0)
    assert b2["kmax_sq"][0] == pytest.approx(np.max(np.sum(k * k, axis=1)), rel=1e-14)


def test_bounds_v_check_boundary():
    """|V| <= 256 passes, anything above fails every tile; an unsafe dtype fails too."""
    D = 8
    q = np.zeros((1, 10, D))
    k = np.zeros((1, 10, D))
    v = np.zeros((1, 10, D))
    v[0, 3, 2] = -256.0
    assert oracle.bounds(q, k, v)["flag"].all()
    v[0, 3, 2] = 256.5
    assert not oracle.bounds(q, k, v)["flag"].any()
    v[0, 3, 2] = 1.0
    assert not oracle.bounds(q, k, v, dtype_safe=False)["flag"].any()


def _aligned_case(U_target, N=4096, D=8, scale=None):
    """Row 0 parallel to the longest key, row 1 anti-parallel: attains z = +U and -U."""
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    alpha = scale * LOG2E
    e = np.zeros(D)
    e[0] = 1.0
    k = np.zeros((N, D))
    k[: N // 2] = e
    k[N // 2:] = -e  # exactly centered
    qn = U_target / alpha  # |k| = 1
    q = np.zeros((2, D))
    q[0] = qn * e
    q[1] = -qn * e
    return q, k, scale, alpha


def brute_exponents(q, k, kbar, alpha, m):
    z = alpha * (q @ (k - kbar).T)
    return z.min() - m, z.max() - m


@pytest.mark.parametrize("N", [256, 4096, 16384, 75600])
def test_gate_is_the_edge_of_the_stated_invariant(N):
    """For the worst case (a row attaining +U and -U), the flag is set exactly when
    every shifted exponent z - m stays in [-125, C]; checked by brute force over U
    around the gate.  A wrong sign in m, a dropped C or a wrong gate fails here."""
    C, W, gate = oracle.constants(N)
    for U_target in np.arange(gate - 2.0, gate + 2.0, 0.125):
        q, k, scale, alpha = _aligned_case(U_target, N=N)
        v = np.ones((N, 8))
        b = oracle.bounds(q[None], k[None], v[None], scale=scale, centering=True, bq=128)
        lo, hi = brute_exponents(q, k, b["kbar"][0], alpha, b["m"][0, 0])
        ok = (lo >= -125) and (hi <= C)
        assert bool(b["flag"][0, 0]) == ok, (N, U_target, lo, hi, b["m"][0, 0])
        # the upper end is nearly attained: m is not larger than it needs to be
        assert C - 1 < hi <= C


def test_invariant_on_generated_eligible_tiles():
    """T3 on a small draw of each bf16 workload recipe: eligible tiles keep z - m in [-125, C]."""
    import workloads
    for name, Sq, N, cen in [("h40_s4096", 256, 512, False), ("mix", 256, 512, False),
                             ("mix", 256, 512, True), ("adversarial", 256, 512, True),
                             ("wan", 256, 512, True)]:
        q, k, v = workloads.make_inputs(name, heads=[0, 1, 25], Sq=Sq, N=N)
        b = oracle.bounds(q, k, v, centering=cen)
        qa, ka = q.double().numpy(), k.double().numpy()
        for h in range(q.shape[1]):
            z = b["alpha"] * qa[0, h] @ (ka[0, h] - b["kbar"][0, h]).T
            for qb in range(b["m"].shape[2]):
                if not b["flag"][0, h, qb]:
                    continue
                zz = z[qb * 128:(qb + 1) * 128] - b["m"][0, h, qb]
                assert zz.min() >= -125 and zz.max() <= b["C"], (name, h, qb)


def test_per_row_shift_keeps_every_row_in_the_window():
    """Per-row bounds (the page's recommended granularity): each row's own shift keeps all
    its exponents in [-125, C] (brute force), is never above its block's, and for the row
    that attains its bound the top exponent sits in (C-1, C]."""
    import workloads
    for name, cen in (("mix", False), ("mix", True), ("wan", True), ("adversarial", True)):
        q, k, v = workloads.make_inputs(name, heads=[0, 3, 30], Sq=300, N=700)
        b = oracle.bounds(q, k, v, centering=cen, per_row=True)
        blk = oracle.bounds(q, k, v, centering=cen, per_row=False)
        qa, ka = q.double().numpy(), k.double().numpy()
        for h in range(3):
            z = b["alpha"] * qa[0, h] @ (ka[0, h] - b["kbar"][0, h]).T
            e = z - b["shift"][0, h][:, None] + b["qkbar"][0, h][:, None]  # z - m_i (centering term apart)
            zc = b["alpha"] * qa[0, h] @ ka[0, h].T - b["shift"][0, h][:, None]  # the kernels' exponent
            assert np.allclose(e, zc, atol=1e-9)
            for qb in range(b["flag"].shape[2]):
                if not b["flag"][0, h, qb]:
                    continue
                ee = e[qb * 128:(qb + 1) * 128]
                assert ee.min() >= -125 and ee.max() <= b["C"], (name, h, qb)
            assert np.all(b["m_row"][0, h] <= np.repeat(blk["m"][0, h], 128)[:300])
            assert np.all(b["shift"][0, h] <= blk["shift"][0, h] + 1e-12)
    # a row parallel to the longest key attains its own bound: top exponent in (C-1, C]
    q, k, scale, alpha = _aligned_case(40.5, N=4096)
    b = oracle.bounds(q[None], k[None], np.ones((1, 4096, 8)), scale=scale, centering=True, per_row=True)
    top = (alpha * q[0] @ k.T).max() - b["shift"][0, 0]
    assert b["C"] - 1 < top <= b["C"]


# ---------------------------------------------------------------- adversarial verdicts (T4, T5, T7)

def test_adversarial_gate_rejects_231():
    """T4: N=4096, exactly centered keys, a query whose bound is 231.01: the full window
    W=232 would admit it; the shipped gate 116 does not.  Under W's shift a quieter row in
    the same block loses the mass of its negative logits (flushed to zero)."""
    (n, U, W, gate, by_w, by_gate), = golden("adversarial_gate.txt")
    n, U, W, gate = int(n), float(U), int(W), int(gate)
    C, W_o, gate_o = oracle.constants(n)
    assert (W_o, gate_o) == (W, gate)
    q, k, scale, alpha = _aligned_case(U, N=n)
    D = q.shape[1]
    # a quiet second row whose logits spread over a few units either side of zero
    r = rng(7)
    k = k.copy()
    k[: n // 2, 1:] = 0.3 * r.normal(size=(n // 2, D - 1))
    k[n // 2:] = -k[: n // 2]
    kn = np.linalg.norm(k, axis=1).max()
    q = np.zeros((2, D))
    q[0, 0] = U / (alpha * kn)
    q[0] *= 1.0  # row 0 bound: alpha*|q0|*max|k| = U
    q[1, 1:] = 3.0 / alpha * np.ones(D - 1) / math.sqrt(D - 1)
    v = r.normal(size=(n, D))
    b = oracle.bounds(q[None], k[None], v[None], scale=scale, centering=True)
    assert abs(b["U"][0, 0] - U) < 1e-9
    assert bool(b["flag"][0, 0]) == bool(int(by_gate))      # rejected by floor(W/2)
    assert (b["U"][0, 0] <= W) == bool(int(by_w))           # W would have admitted it
    # the shift W would have allowed, applied to the quiet row: terms flush, mass is lost
    m_w = math.ceil(b["U"][0, 0]) - C
    em = oracle.fixed_m_emulate_f32(q[1:2], k, v, np.array([m_w]), scale=scale, kbar=b["kbar"][0])
    exact = oracle.attention(q[None, 1:2], k[None], v[None], scale=scale)[0]
    assert em["n_flushed"][0] > 0
    assert np.max(np.abs(em["o"] - exact)) > 1e-3
    # the same row under its own admissible shift (U <= gate) keeps every term
    qq = q[1:2]
    b1 = oracle.bounds(qq[None], k[None], v[None], scale=scale, centering=True)
    assert b1["flag"][0, 0]
    em1 = oracle.fixed_m_emulate_f32(qq, k, v, np.array([b1["m"][0, 0] + b1["qkbar"][0, 0]]),
                                     scale=scale, kbar=None)
    assert em1["n_flushed"][0] == 0 and em1["n_overflow"][0] == 0
    assert np.max(np.abs(em1["o"] - exact)) < 1e-5


def test_matched_pair_raw_bound_with_centered_logits_overflows():
    """T5: 4095 keys equal to a (|a| = 100), one key -a, q a unit vector in z units along -a.
    The raw bound (100) passes gate 116; centered logits reach about +200, and the shift
    built from the raw bound puts the exponent past 128: fp32 overflow.  Centered bounds
    (the matched pair) reject the tile instead."""
    (n, knorm, raw_bound, gate, cen_logit, ovf), = golden("matched_pair.txt")
    n, knorm, gate, ovf = int(n), float(knorm), int(gate), float(ovf)
    D = 8
    scale = 1.0 / math.sqrt(D)
    alpha = scale * LOG2E
    a = np.zeros(D)
    a[0] = knorm
    k = np.tile(a, (n, 1))
    k[-1] = -a
    q = np.zeros((1, D))
    q[0, 0] = -1.0 / alpha  # alpha*|q| = 1
    v = np.ones((n, D))
    raw = oracle.bounds(q[None], k[None], v[None], scale=scale, centering=False)
    assert raw["gate"] == gate
    assert abs(raw["U"][0, 0] - float(raw_bound)) < 1e-9
    assert raw["flag"][0, 0] == 1
    cen = oracle.bounds(q[None], k[None], v[None], scale=scale, centering=True)
    z_cen_max = (alpha * q @ (k - cen["kbar"][0]).T).max()
    assert abs(z_cen_max - float(cen_logit)) < 1.0
    assert z_cen_max - raw["m"][0, 0] > ovf
    em = oracle.fixed_m_emulate_f32(q, k, v, np.array([raw["m"][0, 0]]), scale=scale, kbar=cen["kbar"][0])
    assert em["n_overflow"][0] > 0 and not np.all(np.isfinite(em["o"]))
    assert cen["flag"][0, 0] == 0  # centered bound ~200 > 116


def test_sink_head_falls_back_everywhere():
    """T7: one head with a huge key; every tile of that head is ineligible, others are not."""
    r = rng(8)
    q, k, v = r.normal(size=(1, 2, 512, 16)), r.normal(size=(1, 2, 512, 16)), r.normal(size=(1, 2, 512, 16))
    k[0, 1, 77] *= 400.0
    b = oracle.bounds(q, k, v, centering=False)
    assert b["flag"][0, 0].all()
    assert not b["flag"][0, 1].any()


# ---------------------------------------------------------------- emulator pins

def test_emulator_closed_forms():
    r = rng(9)
    N, D = 64, 8
    k, v = r.normal(size=(N, D)), r.normal(size=(N, D))
    q = np.zeros((3, D))
    em = oracle.fixed_m_emulate_f32(q, k, v, np.array([0.0, -200.0, 200.0]))
    assert em["acc_sum"][0] == N and np.max(np.abs(em["o"][0] - v.mean(0))) < 1e-6
    assert em["n_overflow"][1] == N and em["n_flushed"][1] == 0
    assert em["n_flushed"][2] == N and em["acc_sum"][2] == 0.0
    # an admissible exact shift reproduces plain attention to fp32 accuracy
    qq = r.normal(size=(4, D))
    alpha = LOG2E / math.sqrt(D)
    mrow = (alpha * qq @ k.T).max(axis=1)
    em = oracle.fixed_m_emulate_f32(qq, k, v, mrow)
    exact = oracle.attention(qq[None], k[None], v[None])[0]
    assert np.max(np.abs(em["o"] - exact)) < 1e-5


# ---------------------------------------------------------------- key sinks

INT32_MAX = 2**31 - 1


def _planted_keys(norms, D=4):
    """Key j = norms[j] * (+/-) e_(j mod D): exactly the given norms, mean of small norm."""
    k = np.zeros((len(norms), D))
    for j, n in enumerate(norms):
        k[j, j % D] = n if (j // D) % 2 == 0 else -n
    return k


def test_sinks_closed_form_selection():
    """Planted norms: the n loudest keys are the sinks, the key max is the next norm down."""
    norms = [1.0, 2.0, 300.0, 3.0, 100.0, 4.0, 200.0, 5.0]
    k = _planted_keys(norms)[None]
    q = np.ones((1, 3, 4))
    v = np.zeros((1, 8, 4))
    for n, sinks, kmax in [(1, [2], 200.0), (2, [2, 6], 100.0), (3, [2, 4, 6], 5.0),
                           (5, [2, 4, 6, 7, 5], 3.0)]:
        b = oracle.bounds(q, k, v, sink_keys=n)
        assert list(b["sink_idx"][0]) == sorted(sinks), (n, b["sink_idx"])
        assert b["kmax_sq"][0] == pytest.approx(kmax ** 2, rel=1e-12)
        assert b["U"][0, 0] == pytest.approx(b["alpha"] * 2.0 * kmax, rel=1e-12)  # |q| = 2
    b0 = oracle.bounds(q, k, v)
    assert b0["kmax_sq"][0] == pytest.approx(300.0 ** 2, rel=1e-12) and b0["sink_idx"].shape == (1, 0)


def test_sinks_ties_and_short_sequences():
    """Keys tied with the first kept one are not sinks (the set is the keys strictly above
    it); with fewer keys than sinks + 1 every nonzero key is a sink and the bound is 0."""
    k = _planted_keys([7.0, 1.0, 7.0, 2.0])[None]
    q, v = np.ones((1, 2, 4)), np.zeros((1, 4, 4))
    b = oracle.bounds(q, k, v, sink_keys=1)
    assert list(b["sink_idx"][0]) == [INT32_MAX]
    assert b["kmax_sq"][0] == pytest.approx(49.0) and b["sink_gap"][0] == pytest.approx(0.0, abs=1e-12)
    b = oracle.bounds(q, k, v, sink_keys=2)
    assert list(b["sink_idx"][0]) == [0, 2] and b["kmax_sq"][0] == pytest.approx(4.0)
    k2 = _planted_keys([3.0, 0.0])[None]
    b = oracle.bounds(q, k2, np.zeros((1, 2, 4)), sink_keys=4)
    assert list(b["sink_idx"][0]) == [0, INT32_MAX, INT32_MAX, INT32_MAX]
    assert b["kmax_sq"][0] == 0.0 and b["U"][0, 0] == 0.0 and b["m"][0, 0] == -b["C"]
    assert b["sink_gap"][0] == math.inf


def test_sinks_use_the_centered_norms():
    """With centering the loudness of a key is measured as |k - kbar|: keys along the mean
    are quiet once it is removed."""
    D, N = 4, 20
    base = np.array([10.0, 0.0, 0.0, 0.0])
    k = np.tile(base, (N, 1))
    k[1] = np.array([11.0, 0.0, 0.0, 0.0])   # loudest raw (121), along the mean: quiet centered
    k[4] = np.array([10.0, 3.0, 0.0, 0.0])   # 109 raw, loudest once the mean is removed
    q, v = np.ones((1, 2, D)), np.zeros((1, N, D))
    raw = oracle.bounds(q, k[None], v, sink_keys=1)
    cen = oracle.bounds(q, k[None], v, sink_keys=1, centering=True)
    assert list(raw["sink_idx"][0]) == [1]
    assert list(cen["sink_idx"][0]) == [4]
    d = k - k.mean(0)
    assert cen["kmax_sq"][0] == pytest.approx(np.sort((d * d).sum(1))[-2], rel=1e-12)


def test_sink_workload_needs_the_sinks_folded_exactly():
    """The sinks workload: with its 4 planted sinks left out of the key max every tile is
    eligible and every kept key stays in [-125, C] (T3), while a sink through the same shift
    leaves the window and overflows fp32.  Folding the sinks back exactly (an online merge
    of the kept keys' fixed-m sums with the sink terms) gives plain attention."""
    import workloads
    q, k, v = workloads.make_inputs("sinks", heads=[0], Sq=256, N=600)
    b0 = oracle.bounds(q, k, v)
    b = oracle.bounds(q, k, v, sink_keys=4)
    assert not b0["flag"].any() and b["flag"].all()
    sinks = list(b["sink_idx"][0, 0])
    assert sinks == workloads.sink_positions(600)
    qa, ka, va = q[0, 0].double().numpy(), k[0, 0].double().numpy(), v[0, 0].double().numpy()
    keep = np.setdiff1d(np.arange(600), sinks)
    z = b["alpha"] * qa @ ka.T
    shift = b["shift"][0, 0][:, None]
    e = z - shift
    assert e[:, keep].min() >= -125 and e[:, keep].max() <= b["C"]
    assert e[:, sinks].max() > 128  # 2^e is not an fp32 number
    em_all = oracle.fixed_m_emulate_f32(qa, ka, va, b["shift"][0, 0])
    assert em_all["n_overflow"].sum() > 0
    em = oracle.fixed_m_emulate_f32(qa, ka[keep], va[keep], b["shift"][0, 0])
    assert em["n_overflow"].sum() == 0
    # online merge of the kept keys' (o, sum) at shift b_i with the sink terms
    zs = z[:, sinks]
    new = np.maximum(b["shift"][0, 0], zs.max(1))
    sc = np.exp2(b["shift"][0, 0] - new)
    ps = np.exp2(zs - new[:, None])
    num = em["acc_o"].astype(np.float64) * sc[:, None] + ps @ va[sinks]
    den = em["acc_sum"].astype(np.float64) * sc + ps.sum(1)
    exact = oracle.attention(qa[None], ka[None], va[None])[0]
    assert np.max(np.abs(num / den[:, None] - exact)) < 1e-5
