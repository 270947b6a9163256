"""GPU parity of the CUDA path (through the C ABI) against the fp64 CPU oracle.

Bars: m and flag bit-exact outside the tie band (|U - nearest integer| or |U - gate|
below 1e-4*max(1,U), where fp32 device sums may legitimately round the other way);
outputs within max-abs 1e-5 for fp32 inputs and 2e-2 for bf16 inputs; the fixed-m and
the online-fallback path within the same tolerance of each other.  Because |o| is about
2e-2 itself at the pages' sizes, bf16 outputs also meet the scale-aware bars of
tests/parity.py (max error within 1e-2 of max |o|, every element within the bound bf16 P
can cause, and an error distribution like the oracle's bf16-P reference).  Small cases are
compared element by element; the full-size workloads on sampled (head, row) sets that
include every ragged tail.
"""
import math

import numpy as np
import pytest
import torch

import fixed_max_softmax_gb300 as fm
import oracle
import workloads
from tests.parity import Reference

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2
TOL_F32 = 1e-5


@pytest.fixture(scope="session")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fixed_max_softmax_gb300 import build as fmbuild

    fmbuild.build()
    fm.load()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def run(q, k, v, chunks=None, centering=False, force_online=False, out_dtype=torch.float32, with_lse=False,
        per_row=False, sink_keys=0):
    B, H, Sq, D = q.shape
    fa = fm.FixedMAttention(B, H, Sq, k.shape[2], D, q.device, centering=centering, force_online=force_online,
                            out_dtype=out_dtype, per_row=per_row, sink_keys=sink_keys)
    o = fa.forward(q, k, v, chunks, with_lse=with_lse)
    fm.fm_sync_status()
    return fa, o


def maxerr(a, b):
    a = a.detach().cpu().double().numpy() if hasattr(a, "detach") else np.asarray(a)
    b = b.detach().cpu().double().numpy() if hasattr(b, "detach") else np.asarray(b)
    assert a.shape == b.shape, (a.shape, b.shape)
    return float(np.max(np.abs(a - b))) if a.size else 0.0


def reference(q, k, v, heads=None, rows=None, centering=False, per_row=False, sink_keys=0):
    """Oracle reference for the rows under test, of every batch entry and the given heads:
    exact o, the bf16-P reference at the oracle's own row shift, and the weighted |v|.  The
    shifts come from bounds over every row and key of those heads."""
    q, k, v = q.cpu(), k.cpu(), v.cpu()
    if heads is not None:
        q, k, v = q[:, heads], k[:, heads], v[:, heads]
    ob = oracle.bounds(q, k, v, centering=centering, per_row=per_row, sink_keys=sink_keys)
    shift = ob["shift"]
    if rows is not None:
        q, shift = q[:, :, rows], shift[:, :, rows]
    return Reference(q, k, v, shift)


def pick(o, heads=None, rows=None):
    """The [B, heads, rows, D] part of a device output, matching reference()'s selection."""
    if heads is not None:
        o = o[:, heads]
    if rows is not None:
        o = o[:, :, rows]
    return o


def check_bounds(fa, ob, heads=None, check_vmax=True):
    """GPU bounds vs oracle bounds (optionally for a subset of heads of batch 0)."""
    sel = (lambda x: x) if heads is None else (lambda x: x[:, heads])
    m_g = sel(fa.bounds.m.cpu().numpy())
    f_g = sel(fa.bounds.flag.cpu().numpy())
    U = ob["U"]
    safe = ob["margin"] > 1e-4 * np.maximum(1.0, U)
    assert np.array_equal(m_g[safe], ob["m"][safe]), "m differs outside the tie band"
    assert np.array_equal(f_g[safe], ob["flag"][safe]), "flag differs outside the tie band"
    assert np.all(np.abs(m_g.astype(np.int64) - ob["m"]) <= 1)
    np.testing.assert_allclose(sel(fa.bounds.qmax_sq.cpu().numpy()), ob["qmax_sq"], rtol=2e-5, atol=1e-30)
    np.testing.assert_allclose(sel(fa.bounds.kmax_sq.cpu().numpy()), ob["kmax_sq"], rtol=2e-5, atol=1e-12)
    np.testing.assert_allclose(sel(fa.bounds.kbar.cpu().numpy()), ob["kbar"], rtol=1e-5, atol=2e-6)
    qk = sel(fa.bounds.qkbar.cpu().numpy())[..., : ob["qkbar"].shape[-1]]
    np.testing.assert_allclose(qk, ob["qkbar"], rtol=1e-4, atol=1e-4)
    if check_vmax:
        # v^2 of a bf16 value is exact in fp32; of an fp32 value it takes one rounding
        g = float(fa.bounds.vmax_sq.item())
        assert abs(g - ob["vmax_sq"]) <= 2.0 ** -23 * ob["vmax_sq"], (g, ob["vmax_sq"])
    # the row shift b_i = m_i + qkbar_i: exact integer part outside the tie band, plus qkbar
    sh = sel(fa.bounds.shift.cpu().numpy())[..., : ob["shift"].shape[-1]].astype(np.float64)
    if fa.bounds.out.per_row:
        safe_rows = ob["margin_row"] > 1e-4 * np.maximum(1.0, ob["U_row"])
    else:
        Sq = ob["shift"].shape[-1]
        safe_rows = np.repeat(safe, 128, axis=-1)[..., :Sq]
    d = np.abs(sh - ob["shift"])
    assert np.all(d[safe_rows] <= 1e-4 * np.maximum(1.0, np.abs(ob["shift"][safe_rows]))), float(d[safe_rows].max())
    assert np.all(d <= 1.0 + 1e-4 * np.maximum(1.0, np.abs(ob["shift"])))
    b = fa.bounds.out
    assert (b.C, b.W, b.gate) == (ob["C"], ob["W"], ob["gate"])
    assert b.magic == fm.FM_BOUNDS_MAGIC
    return int((~safe).sum())


# ------------------------------------------------------------------ small, element by element

def test_tiny_fp32_element_by_element(dev):
    w = workloads.WORKLOADS["tiny"]
    q, k, v = workloads.make_inputs("tiny", device=dev)
    fa, o = run(q, k, v, workloads.chunk_bounds(w), centering=False)
    ref = oracle.attention(q.cpu(), k.cpu(), v.cpu())
    assert maxerr(o, ref) <= TOL_F32
    check_bounds(fa, oracle.bounds(q.cpu(), k.cpu(), v.cpu(), centering=False))
    _, o2 = run(q, k, v, workloads.chunk_bounds(w), force_online=True)
    assert maxerr(o2, ref) <= TOL_F32


@pytest.mark.parametrize("centering", [False, True])
@pytest.mark.parametrize("force_online", [False, True])
@pytest.mark.parametrize("shape", [(1, 3, 300, 333, [(0, 128), (128, 100), (228, 105)]),
                                   (2, 2, 128, 128, [(0, 128)]),
                                   (1, 2, 77, 1000, [(0, 999), (999, 1)]),
                                   (1, 1, 513, 257, [(0, 129), (129, 128)])])
def test_bf16_ragged_chunks_element_by_element(dev, shape, centering, force_online):
    B, H, Sq, N, chunks = shape
    q, k, v = workloads.make_inputs("wan", device="cpu", heads=range(H), Sq=Sq, N=N)
    if B > 1:
        q2, k2, v2 = workloads.make_inputs("h40_s4096", device="cpu", heads=range(H), Sq=Sq, N=N)
        q, k, v = torch.cat([q, q2]), torch.cat([k, k2]), torch.cat([v, v2])
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    fa, o = run(qd, kd, vd, chunks, centering=centering, force_online=force_online)
    reference(q, k, v, centering=centering).check(o, f"{shape} centering={centering} online={force_online}")
    check_bounds(fa, oracle.bounds(q, k, v, centering=centering))


def test_fp32_d128_and_bf16_d64_use_the_cuda_core_path(dev):
    for name, D in (("tiny", 64), ("h40_s4096", 128)):
        q, k, v = workloads.make_inputs(name, device="cpu", heads=[0, 1], Sq=200, N=300)
        for dt, tol in ((torch.float32, TOL_F32), (torch.bfloat16, TOL_BF16)):
            qq, kk, vv = q.to(dt), k.to(dt), v.to(dt)
            _, o = run(qq.to(dev), kk.to(dev), vv.to(dev), [(0, 150), (150, 150)], centering=True)
            assert maxerr(o, oracle.attention(qq, kk, vv)) <= tol, (name, dt)


def test_token_major_layout_and_bf16_output(dev):
    """Inputs laid out [B, S, H, D] (the pages' token-major layout) seen through strides."""
    q, k, v = workloads.make_inputs("wan", device="cpu", heads=range(4), Sq=260, N=390)
    tq = q.permute(0, 2, 1, 3).contiguous().to(dev).permute(0, 2, 1, 3)
    tk = k.permute(0, 2, 1, 3).contiguous().to(dev).permute(0, 2, 1, 3)
    tv = v.permute(0, 2, 1, 3).contiguous().to(dev).permute(0, 2, 1, 3)
    assert not tq.is_contiguous()
    ref = oracle.attention(q, k, v)
    _, o = run(tq, tk, tv, [(0, 200), (200, 190)], centering=True, out_dtype=torch.bfloat16)
    assert o.dtype == torch.bfloat16
    assert maxerr(o, ref) <= TOL_BF16


def test_strided_head_dim_layout(dev):
    """D not contiguous ([B, H, D, S] storage seen as [B, H, S, D]): the bounds pass takes its
    scalar-load path and the chunks the CUDA-core kernel; results still match the oracle."""
    q, k, v = workloads.make_inputs("mix", device="cpu", heads=range(2), Sq=300, N=260)
    tq = q.transpose(2, 3).contiguous().to(dev).transpose(2, 3)
    tk = k.transpose(2, 3).contiguous().to(dev).transpose(2, 3)
    tv = v.transpose(2, 3).contiguous().to(dev).transpose(2, 3)
    assert tq.stride(3) != 1
    for cen in (False, True):
        fa, o = run(tq, tk, tv, [(0, 130), (130, 130)], centering=cen)
        check_bounds(fa, oracle.bounds(q, k, v, centering=cen))
        assert maxerr(o, oracle.attention(q, k, v)) <= TOL_BF16


def test_empty_and_degenerate_inputs(dev):
    # a single key: output equals its value (up to bf16 P rounding, exact here: p=1 scale)
    q, k, v = workloads.make_inputs("wan", device="cpu", heads=[0], Sq=5, N=1)
    _, o = run(q.to(dev), k.to(dev), v.to(dev))
    assert maxerr(o, v.expand(1, 1, 5, 128).float()) <= TOL_BF16
    # an empty first chunk initialises; the next one accumulates
    q, k, v = workloads.make_inputs("wan", device="cpu", heads=[0, 1], Sq=140, N=200)
    _, o = run(q.to(dev), k.to(dev), v.to(dev), [(0, 0), (0, 200)], centering=True)
    assert maxerr(o, oracle.attention(q, k, v)) <= TOL_BF16
    # Sq = 0 and H = 0 are no-ops
    z = torch.empty(1, 2, 0, 128, dtype=torch.bfloat16, device=dev)
    kk = torch.randn(1, 2, 10, 128, device=dev).bfloat16()
    run(z, kk, kk)
    # Q = K = 0, V = 1 gives exactly 1 (the case fp16 fixed-m gets wrong)
    zq = torch.zeros(1, 1, 130, 128, dtype=torch.bfloat16, device=dev)
    ones = torch.ones(1, 1, 300, 128, dtype=torch.bfloat16, device=dev)
    _, o = run(zq, torch.zeros_like(ones), ones, [(0, 150), (150, 150)])
    assert torch.all(torch.isfinite(o)) and maxerr(o, torch.ones_like(o)) <= TOL_BF16


def test_schedule_invariance_bitwise(dev):
    """Repeated runs are bit-identical (deterministic reductions, fixed tile order)."""
    q, k, v = workloads.make_inputs("mix", device=dev, heads=range(6), Sq=700, N=900)
    outs = []
    for _ in range(2):
        fa, o = run(q, k, v, [(0, 450), (450, 450)], centering=True)
        outs.append((o.clone(), fa.bounds.m.clone(), fa.bounds.kbar.clone(), fa.acc_sum.clone()))
    for a, b in zip(*outs):
        assert torch.equal(a, b)


@pytest.mark.parametrize("name,centering", [("wan", True), ("mix", False), ("adversarial", True)])
def test_per_row_shift_parity(dev, name, centering):
    """Per-row bounds: shifts match the oracle's per-row m_i + qkbar_i, outputs match the
    oracle, and per-row and per-block runs agree within the tolerance."""
    q, k, v = workloads.make_inputs(name, device="cpu", heads=[0, 5, 33], Sq=390, N=700)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    fa, o = run(qd, kd, vd, [(0, 350), (350, 350)], centering=centering, per_row=True)
    check_bounds(fa, oracle.bounds(q, k, v, centering=centering, per_row=True))
    ref = oracle.attention(q, k, v)
    assert maxerr(o, ref) <= TOL_BF16
    _, o_blk = run(qd, kd, vd, [(0, 350), (350, 350)], centering=centering, per_row=False)
    assert maxerr(o, o_blk) <= TOL_BF16


TOL_LSE = 1e-4  # fp32 S and sums, ex2.approx: about 1e-5 absolute on |lse| < 100


@pytest.mark.parametrize("force_online", [False, True])
def test_lse_matches_oracle(dev, force_online):
    """LSE (natural log of the scaled scores' exp-sum) from acc_max and acc_sum, both paths."""
    for name, centering, dt in (("wan", True, torch.bfloat16), ("mix", False, torch.bfloat16),
                                ("tiny", False, torch.float32)):
        q, k, v = workloads.make_inputs(name, device="cpu", heads=range(3), Sq=300, N=333)
        q, k, v = q.to(dt), k.to(dt), v.to(dt)
        fa, o = run(q.to(dev), k.to(dev), v.to(dev), [(0, 200), (200, 133)], centering=centering,
                    force_online=force_online, with_lse=True)
        ref, ref_lse = oracle.attention(q, k, v, return_lse=True)
        assert maxerr(fa.lse, ref_lse) <= TOL_LSE * max(1.0, float(np.max(np.abs(ref_lse)))), name
        assert maxerr(o, ref) <= (TOL_F32 if dt == torch.float32 else TOL_BF16)
    # an empty key set gives -inf
    z = torch.zeros(1, 1, 5, 128, dtype=torch.bfloat16, device=dev)
    fa, _ = run(z, z[:, :, :0], z[:, :, :0], [(0, 0)], with_lse=True)
    assert torch.all(torch.isneginf(fa.lse))


@pytest.mark.parametrize("force_online", [False, True])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_fused_final_chunk_equals_chunk_plus_finalize(dev, force_online, out_dtype):
    """fm_attn_chunk_final (fold + normalise in one pass) gives the same bits as
    fm_attn_chunk followed by fm_finalize_lse, and matches the oracle."""
    q, k, v = workloads.make_inputs("mix", device="cpu", heads=range(3), Sq=333, N=600)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    chunks = [(0, 256), (256, 344)]
    outs = []
    for fused in (True, False):
        fa = fm.FixedMAttention(1, 3, 333, 600, 128, dev, centering=False, force_online=force_online,
                                out_dtype=out_dtype)
        o = fa.forward(qd, kd, vd, chunks, with_lse=True, fused_final=fused).clone()
        fm.fm_sync_status()
        outs.append((o, fa.lse.clone(), fa.acc_sum.clone(), fa.acc_max.clone()))
    for a, b in zip(*outs):
        assert torch.equal(a, b)
    ref, ref_lse = oracle.attention(q, k, v, return_lse=True)
    assert maxerr(outs[0][0], ref) <= TOL_BF16
    assert maxerr(outs[0][1], ref_lse) <= TOL_LSE * max(1.0, float(np.max(np.abs(ref_lse))))
    # an output layout the kernel cannot store to directly (D not contiguous) takes the
    # chunk + finalize route inside the same call
    fa = fm.FixedMAttention(1, 3, 333, 600, 128, dev, centering=False, force_online=force_online)
    o_t = torch.empty(1, 3, 128, 333, dtype=out_dtype, device=dev).transpose(2, 3)
    fm.fm_bounds(qd, kd, vd, fa.opt, fa.bounds, fa.workspace)
    fm.fm_attn_chunk(qd, kd[:, :, :256], vd[:, :, :256], fa.bounds, fa.opt, fa.acc_o, fa.acc_sum, fa.acc_max, False)
    fm.fm_attn_chunk_final(qd, kd[:, :, 256:], vd[:, :, 256:], fa.bounds, fa.opt, fa.acc_o, fa.acc_sum, fa.acc_max,
                           True, o_t)
    fm.fm_sync_status()
    assert torch.equal(o_t, outs[0][0])


def test_long_key_sequence_and_batches(dev):
    """2^20 keys (C(N) = 99, gate = 112) folded in 3 uneven chunks, and B = 2."""
    N = 1 << 20
    q, k, v = workloads.make_inputs("wan", device=dev, heads=[0], Sq=200, N=N)
    chunks = [(0, 300001), (300001, 500000), (800001, N - 800001)]
    fa, o = run(q, k, v, chunks, centering=True)
    assert (fa.bounds.out.C, fa.bounds.out.gate) == oracle.constants(N)[0:3:2]
    reference(q, k, v, centering=True).check(o, "2^20 keys")
    # two batches with different recipes
    q1, k1, v1 = workloads.make_inputs("mix", device="cpu", heads=range(3), Sq=1000, N=1500)
    q2, k2, v2 = workloads.make_inputs("wan", device="cpu", heads=range(3), Sq=1000, N=1500)
    q, k, v = torch.cat([q1, q2]), torch.cat([k1, k2]), torch.cat([v1, v2])
    fa, o = run(q.to(dev), k.to(dev), v.to(dev), [(0, 700), (700, 800)], centering=True)
    check_bounds(fa, oracle.bounds(q, k, v, centering=True))
    reference(q, k, v, centering=True).check(o, "B = 2")


def test_device_flags_follow_the_gate_edge(dev):
    """Queries whose bound sits just under / over the gate: the device flags match the
    oracle's decision exactly (both values are far from the tie band)."""
    N, D = 4096, 128
    C, W, gate = oracle.constants(N)
    g = torch.Generator().manual_seed(11)
    k = torch.randn(1, 1, N, D, generator=g)
    v = torch.randn(1, 1, N, D, generator=g)
    q = torch.randn(1, 1, 4 * 128, D, generator=g)
    kb = k.bfloat16().double()
    kmax = (kb - kb.mean(dim=2, keepdim=True)).norm(dim=-1).max().item()
    alpha = math.log2(math.e) / math.sqrt(D)
    # one loud row per Q-block, its bound set to gate - 1.5, gate - 0.5, gate + 0.5, gate + 1.5
    # (bf16 rounding of the query moves U by about 0.2)
    for blk, u in enumerate((gate - 1.5, gate - 0.5, gate + 0.5, gate + 1.5)):
        qr = q[0, 0, blk * 128]
        q[0, 0, blk * 128] = qr / qr.norm() * (u / (alpha * kmax))
    qb, kbf, vb = q.bfloat16(), k.bfloat16(), v.bfloat16()
    fa, o = run(qb.to(dev), kbf.to(dev), vb.to(dev), [(0, 2000), (2000, 2096)], centering=True)
    ob = oracle.bounds(qb, kbf, vb, centering=True)
    check_bounds(fa, ob)
    # the oracle's verdict on the rounded values rules, outside the tie band
    safe = ob["margin"][0, 0] > 1e-4 * np.maximum(1.0, ob["U"][0, 0])
    assert np.array_equal(fa.bounds.flag.cpu().numpy()[0, 0][safe], ob["flag"][0, 0][safe])
    assert list(ob["flag"][0, 0]) == [1, 1, 0, 0], ob["U"][0, 0]
    assert maxerr(o, oracle.attention(qb, kbf, vb)) <= TOL_BF16


@pytest.mark.parametrize("force_online", [False, True])
def test_chunks_in_one_launch(dev, force_online):
    """fm_attn_chunks folds several ragged chunks in one launch (O and sums on chip across
    them): matches the oracle and the one-call-per-chunk path (different fp32 summation
    order, so within the tolerance, not bitwise); 11 chunks take two launches."""
    q, k, v = workloads.make_inputs("mix", device="cpu", heads=range(3), Sq=300, N=1500)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    ref, ref_lse = oracle.attention(q, k, v, return_lse=True)
    for chunks in ([(0, 200), (200, 1), (201, 0), (201, 1299)],
                   [(i * 136, 136 if i < 10 else 140) for i in range(11)]):
        assert sum(n for _, n in chunks) == 1500
        fa = fm.FixedMAttention(1, 3, 300, 1500, 128, dev, centering=False, force_online=force_online)
        o1 = fa.forward(qd, kd, vd, chunks, with_lse=True, one_launch=True).clone()
        lse1 = fa.lse.clone()
        fm.fm_sync_status()
        fb = fm.FixedMAttention(1, 3, 300, 1500, 128, dev, centering=False, force_online=force_online)
        o2 = fb.forward(qd, kd, vd, chunks).clone()
        fm.fm_sync_status()
        assert maxerr(o1, ref) <= TOL_BF16
        assert maxerr(o1, o2) <= TOL_BF16
        assert maxerr(lse1, ref_lse) <= TOL_LSE * max(1.0, float(np.max(np.abs(ref_lse))))
        assert fa.bounds.out.kv_seen == 1500


@pytest.mark.parametrize("one_launch", [False, True])
def test_cuda_graph_capture_and_replay(dev, one_launch):
    """The whole path (bounds, chunks, fused normalise) captured once in a CUDA graph and
    replayed on new data in the same buffers gives the eager result bit for bit."""
    Sq, N = 700, 900
    chunks = [(0, 450), (450, 450)]
    q, k, v = workloads.make_inputs("mix", device=dev, heads=range(3), Sq=Sq, N=N)
    q2, k2, v2 = workloads.make_inputs("wan", device=dev, heads=range(3), Sq=Sq, N=N)
    fa = fm.FixedMAttention(1, 3, Sq, N, 128, dev, centering=True)
    fa.forward(q, k, v, chunks, one_launch=one_launch)  # first calls on the device happen before capture
    fm.fm_sync_status()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fa.forward(q, k, v, chunks, one_launch=one_launch)
    q.copy_(q2)
    k.copy_(k2)
    v.copy_(v2)
    g.replay()
    torch.cuda.synchronize()
    fm.fm_sync_status()
    fb = fm.FixedMAttention(1, 3, Sq, N, 128, dev, centering=True)
    ref = fb.forward(q2, k2, v2, chunks, one_launch=one_launch)
    fm.fm_sync_status()
    assert torch.equal(fa.out, ref)
    assert maxerr(fa.out, oracle.attention(q2.cpu(), k2.cpu(), v2.cpu())) <= TOL_BF16


def test_bounded_wait_reports_timeout_and_context_survives(dev):
    """Failure detection without a fault: a wait on a barrier nothing completes gives up
    after 50 ms, fm_sync_status reports FM_ERR_TIMEOUT once, and work continues."""
    fm.fm_probe_wait_timeout(50)
    with pytest.raises(fm.FMError) as e:
        fm.fm_sync_status()
    assert e.value.code == fm.FM_ERR_TIMEOUT and "role 5" in str(e.value)
    fm.fm_sync_status()  # cleared
    q, k, v = workloads.make_inputs("wan", device="cpu", heads=[0], Sq=130, N=140)
    _, o = run(q.to(dev), k.to(dev), v.to(dev), centering=True)
    assert maxerr(o, oracle.attention(q, k, v)) <= TOL_BF16


def test_host_pipeline_matches_device_path(dev):
    """HostPipeline (overlapped upload / compute / read-back) gives the device path's bits."""
    Sq, N = 700, 900
    batches, refs = [], []
    for i in range(3):
        q, k, v = workloads.make_inputs("mix", device="cpu", heads=range(2 + i % 2, 4 + i % 2), Sq=Sq, N=N)
        _, o = run(q.to(dev), k.to(dev), v.to(dev), [(0, 450), (450, 450)], centering=True)
        refs.append(o.cpu())
        batches.append((q.pin_memory(), k.pin_memory(), v.pin_memory(), torch.empty(o.shape).pin_memory()))
    fa = fm.FixedMAttention(1, 2, Sq, N, 128, dev, centering=True)
    fm.HostPipeline(fa, torch.bfloat16, dev).run(batches, [(0, 450), (450, 450)])
    fm.fm_sync_status()
    for (_, _, _, oh), ref in zip(batches, refs):
        assert torch.equal(oh, ref)


# ------------------------------------------------------------------ full-size workloads (sampled rows)

def test_h40_s4096_full(dev):
    w = workloads.WORKLOADS["h40_s4096"]
    q, k, v = workloads.make_inputs("h40_s4096", device=dev)
    fa, o = run(q, k, v, workloads.chunk_bounds(w), centering=False)
    check_bounds(fa, oracle.bounds(q.cpu(), k.cpu(), v.cpu(), centering=False))
    assert bool(fa.bounds.flag.all())
    heads = [0, 13, 26, 39]
    rows = list(range(0, 128)) + list(range(1000, 1050)) + list(range(2000, 2100)) + list(range(3968, 4096))
    ref = reference(q, k, v, heads, rows)
    ref.check(pick(o, heads, rows), "h40_s4096 fixed-m")
    _, o2 = run(q, k, v, workloads.chunk_bounds(w), force_online=True)
    ref.check(pick(o2, heads, rows), "h40_s4096 online")
    assert maxerr(pick(o2, heads, rows), pick(o, heads, rows)) <= TOL_BF16


def test_wan_full_size(dev):
    w = workloads.WORKLOADS["wan"]
    q, k, v = workloads.make_inputs("wan", device=dev)
    fa, o = run(q, k, v, workloads.chunk_bounds(w), centering=True)
    heads = [0, 17, 39]
    ob = oracle.bounds(q[:, heads].cpu(), k[:, heads].cpu(), v[:, heads].cpu(), centering=True)
    check_bounds(fa, ob, heads=heads, check_vmax=False)
    # the V maximum spans every head: the oracle's, over groups of heads (keys stand in
    # for nothing here, they only give the call the shape it wants)
    vmax = max(oracle.bounds(q[:, h0:h0 + 4, :1].cpu(), v[:, h0:h0 + 4].cpu(), v[:, h0:h0 + 4].cpu())["vmax_sq"]
               for h0 in range(0, 40, 4))
    assert float(fa.bounds.vmax_sq.item()) == vmax
    nqb = fa.bounds.out.n_qblocks
    assert nqb == 591
    # rows: the first Q-block pair, the Q-blocks around row 37,800 (where the key chunks
    # meet), the last full block and the ragged 80-row tail; eight heads across the range
    rows = (list(range(0, 256)) + list(range(37632, 37888)) + list(range(75392, 75520))
            + list(range(75520, 75600)))
    heads = [0, 5, 11, 17, 22, 28, 33, 39]
    ref = reference(q, k, v, heads, rows, centering=True)
    r = ref.check(pick(o, heads, rows), "wan fixed-m")
    assert r["max_ref"] > 5 * r["max_err"] and r["max_ref"] > 1e-2  # |o| is far above the error
    # the LSE of two heads' rows, from the accumulators of this call: acc_sum and acc_max are
    # current after the fused final chunk (acc_o is not, so the o this writes is thrown away)
    lse = torch.empty_like(fa.acc_sum)
    fm.fm_finalize_lse(fa.acc_o, fa.acc_sum, fa.acc_max, torch.empty_like(fa.out), lse)
    _, ref_lse = oracle.attention(q[0, [0, 17]][:, rows].cpu(), k[0, [0, 17]].cpu(), v[0, [0, 17]].cpu(),
                                  return_lse=True)
    assert maxerr(lse[0, [0, 17]][:, rows], ref_lse) <= TOL_LSE * max(1.0, float(np.max(np.abs(ref_lse))))
    _, o2 = run(q, k, v, workloads.chunk_bounds(w), centering=True, force_online=True)
    ref.check(pick(o2, heads, rows), "wan online")
    assert maxerr(pick(o2, heads, rows), pick(o, heads, rows)) <= TOL_BF16


@pytest.mark.parametrize("centering", [False, True])
def test_mix_fallback_full(dev, centering):
    q, k, v = workloads.make_inputs("mix", device=dev)
    fa, o = run(q, k, v, None, centering=centering)
    ob = oracle.bounds(q.cpu(), k.cpu(), v.cpu(), centering=centering)
    check_bounds(fa, ob)
    flags = fa.bounds.flag.cpu().numpy()[0]
    heads_on = [h for h in range(40) if flags[h].all()]
    heads_off = [h for h in range(40) if not flags[h].any()]
    if not centering:
        assert heads_off, "without centering some heads must fall back"
    rows = list(range(0, 128)) + list(range(8192, 8320)) + list(range(16256, 16384))
    for hs in (heads_on[:2], heads_off[:2]):
        if hs:
            reference(q, k, v, hs, rows, centering=centering).check(pick(o, hs, rows), f"mix heads {hs}")


def test_adversarial_full(dev):
    w = workloads.WORKLOADS["adversarial"]
    q, k, v = workloads.make_inputs("adversarial", device=dev)
    fa, o = run(q, k, v, None, centering=True)
    ob = oracle.bounds(q.cpu(), k.cpu(), v.cpu(), centering=True)
    check_bounds(fa, ob)
    flags = fa.bounds.flag.cpu().numpy()[0]
    adv = w.extra["adv_heads"]
    assert not flags[:adv, 0].any(), "the query with bound 231.01 must be rejected"
    assert flags[:adv, 1:].all() and flags[adv:].all()
    rows = list(range(0, 256)) + list(range(3968, 4096))
    heads = [0, 7, 19, 25]
    ref = reference(q, k, v, heads, rows, centering=True)
    ref.check(pick(o, heads, rows), "adversarial auto")
    _, o2 = run(q, k, v, None, centering=True, force_online=True)
    ref.check(pick(o2, heads, rows), "adversarial online")
    assert maxerr(pick(o2, heads, rows), pick(o, heads, rows)) <= TOL_BF16


# ------------------------------------------------------------------ key sinks

def check_sinks(fa, ob, heads=None):
    """Device sink lists equal the oracle's wherever the n-th and (n+1)-th loudest keys are
    apart by more than fp32 norms can blur (elsewhere the two sets may differ in near-ties,
    which changes no output: every key is still counted once).  Returns the heads compared."""
    n = ob["sink_idx"].shape[-1]
    got = fa.bounds.sink_idx.cpu().numpy()
    if heads is not None:
        got = got[:, heads]
    got = got.reshape(-1, fm.FM_MAX_SINKS)
    ref = ob["sink_idx"].reshape(-1, n)
    gap = ob["sink_gap"].reshape(-1)
    tau = ob["kmax_sq"].reshape(-1)
    compared = 0
    for g in range(ref.shape[0]):
        assert np.all(got[g, n:] == 2**31 - 1)
        if gap[g] > 1e-4 * max(1.0, tau[g]):
            assert np.array_equal(got[g, :n], ref[g]), (g, got[g], ref[g])
            compared += 1
    return compared


@pytest.mark.parametrize("centering", [False, True])
@pytest.mark.parametrize("force_online", [False, True])
@pytest.mark.parametrize("chunks", [[(0, 300), (300, 400)], [(0, 353), (353, 347)], [(0, 700)]])
def test_key_sinks_element_by_element(dev, chunks, force_online, centering):
    """The sinks workload (4 loud keys at 0, 1, N/2+3, N-1 in heads 0-19): with the 4 sinks
    left out of the key max every tile is eligible, the chunks skip the sinks (two in one tile,
    one at a chunk start or mid-chunk, one in a ragged tail) and the fold merges them back:
    the output is plain attention over every key."""
    q, k, v = workloads.make_inputs("sinks", device="cpu", heads=[0, 1, 25], Sq=300, N=700)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    fa, o = run(qd, kd, vd, chunks, centering=centering, force_online=force_online, sink_keys=4, with_lse=True)
    ob = oracle.bounds(q, k, v, centering=centering, sink_keys=4)
    check_bounds(fa, ob)
    assert check_sinks(fa, ob) >= 2  # the two sink heads at least
    assert list(fa.bounds.sink_idx[0, 0, :4].cpu().numpy()) == workloads.sink_positions(700)
    if not force_online:
        assert bool(fa.bounds.flag.all())
    ref, ref_lse = oracle.attention(q, k, v, return_lse=True)
    reference(q, k, v, centering=centering, sink_keys=4).check(o, f"sinks {chunks}")
    assert maxerr(fa.lse, ref_lse) <= TOL_LSE * max(1.0, float(np.max(np.abs(ref_lse))))
    # without sinks the sink heads fall back to online softmax everywhere; same output
    fb, o_plain = run(qd, kd, vd, chunks, centering=centering, force_online=force_online)
    if not centering and not force_online:
        assert not fb.bounds.flag[0, :2].any()
    assert maxerr(o, o_plain) <= TOL_BF16


@pytest.mark.parametrize("sink_keys", [1, 2, 8])
def test_key_sink_counts_and_paths(dev, sink_keys):
    """Fewer sinks than loud keys (the rest stay in, their heads still fall back), more sinks
    than loud keys (ordinary keys become sinks too), on the fused-final, separate-finalize
    (explicit fm_fold_sinks) and one-launch paths, which agree bit for bit where they share
    the arithmetic."""
    q, k, v = workloads.make_inputs("sinks", device="cpu", heads=[0, 30], Sq=260, N=900)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    chunks = [(0, 450), (450, 450)]
    ref = oracle.attention(q, k, v)
    ob = oracle.bounds(q, k, v, sink_keys=sink_keys)
    outs = {}
    for mode in ("fused", "separate", "one_launch"):
        fa = fm.FixedMAttention(1, 2, 260, 900, 128, dev, sink_keys=sink_keys)
        o = fa.forward(qd, kd, vd, chunks, fused_final=mode == "fused", one_launch=mode == "one_launch").clone()
        fm.fm_sync_status()
        check_bounds(fa, ob)
        check_sinks(fa, ob)
        assert np.array_equal(fa.bounds.flag.cpu().numpy(), ob["flag"])
        assert maxerr(o, ref) <= TOL_BF16, mode
        assert fa.bounds.out.sinks_folded == 1
        outs[mode] = o
    assert torch.equal(outs["fused"], outs["separate"])
    assert maxerr(outs["one_launch"], outs["fused"]) <= TOL_BF16


def test_key_sinks_cuda_core_path_and_edges(dev):
    """fp32 inputs (CUDA-core kernel, exact fp32) with sinks; a key set made only of sinks
    (every key left out of the chunks, the fold alone gives the output); no chunk may follow
    the fold."""
    q, k, v = workloads.make_inputs("sinks", device="cpu", heads=[0, 1], Sq=200, N=300)
    q32, k32, v32 = q.float(), k.float(), v.float()
    fa, o = run(q32.to(dev), k32.to(dev), v32.to(dev), [(0, 150), (150, 150)], sink_keys=4)
    ob = oracle.bounds(q32, k32, v32, sink_keys=4)
    check_bounds(fa, ob)
    check_sinks(fa, ob)
    assert maxerr(o, oracle.attention(q32, k32, v32)) <= TOL_F32
    # three keys, four sinks: all three are sinks, tau = 0, m = -C
    qs, ks, vs = q[:, :, :130], k[:, :, 5:8], v[:, :, 5:8]
    fa, o = run(qs.to(dev), ks.to(dev), vs.to(dev), [(0, 2), (2, 1)], sink_keys=4)
    assert list(fa.bounds.sink_idx[0, 0].cpu().numpy()[:3]) == [0, 1, 2]
    assert float(fa.bounds.kmax_sq.max().item()) == 0.0
    assert maxerr(o, oracle.attention(qs, ks, vs)) <= TOL_BF16
    with pytest.raises(fm.FMError) as e:
        fm.fm_attn_chunk(qs.to(dev), ks.to(dev), vs.to(dev), fa.bounds, fa.opt, fa.acc_o, fa.acc_sum, fa.acc_max, True)
    assert e.value.code == fm.FM_ERR_BOUNDS_MISMATCH
    # D = 64 (fp32, CUDA-core kernel) with per-row shifts and sinks
    qt, kt, vt = workloads.make_inputs("tiny", device="cpu")
    kt[0, 0, [3, 200]] *= 30.0
    fa, o = run(qt.to(dev), kt.to(dev), vt.to(dev), [(0, 100), (100, 156)], per_row=True, sink_keys=2)
    check_bounds(fa, oracle.bounds(qt, kt, vt, per_row=True, sink_keys=2))
    assert list(fa.bounds.sink_idx[0, 0, :2].cpu().numpy()) == [3, 200]
    assert maxerr(o, oracle.attention(qt, kt, vt)) <= TOL_F32
    # no keys at all: no sinks, an empty key set gives 0
    z = torch.zeros(1, 1, 130, 128, dtype=torch.bfloat16, device=dev)
    fa, o = run(z, z[:, :, :0], z[:, :, :0], [(0, 0)], sink_keys=3)
    assert torch.all(fa.bounds.sink_idx == 2**31 - 1) and torch.all(o == 0)


def test_sinks_full(dev):
    """The sinks workload at full size (H=40, S=16384, 4 chunks of 4096): 4 sinks make every
    tile eligible; sampled rows match the oracle and the run without sinks."""
    w = workloads.WORKLOADS["sinks"]
    q, k, v = workloads.make_inputs("sinks", device=dev)
    fa, o = run(q, k, v, workloads.chunk_bounds(w), sink_keys=4)
    ob = oracle.bounds(q.cpu(), k.cpu(), v.cpu(), sink_keys=4)
    check_bounds(fa, ob)
    assert check_sinks(fa, ob) >= w.extra["sink_heads"]
    assert bool(fa.bounds.flag.all())
    rows = list(range(0, 128)) + list(range(8190, 8300)) + list(range(16256, 16384))
    heads = [0, 19, 39]
    ref = reference(q, k, v, heads, rows, sink_keys=4)
    ref.check(pick(o, heads, rows), "sinks, 4 sink keys")
    fb, o2 = run(q, k, v, workloads.chunk_bounds(w))
    assert not fb.bounds.flag[0, :w.extra["sink_heads"]].any()
    r = ref.check(pick(o2, heads, rows), "sinks, no sink keys")
    # online rows that continue from the earlier chunks' shift give a later chunk's loud key a
    # weight of up to 2^8 in bf16: about 1.8e-3 of error here, which must not grow
    assert r["max_err"] <= 3e-3, r
    assert maxerr(pick(o2, heads, rows), pick(o, heads, rows)) <= TOL_BF16


def test_key_sinks_with_per_row_centering_and_batches(dev):
    """Key sinks combined with per-row shifts, centering and B = 2 (each batch entry and head
    picks its own sinks); LSE included."""
    q1, k1, v1 = workloads.make_inputs("sinks", device="cpu", heads=[0, 30], Sq=300, N=500)
    q2, k2, v2 = workloads.make_inputs("sinks", device="cpu", heads=[5, 6], Sq=300, N=500)
    q, k, v = torch.cat([q1, q2]), torch.cat([k1, k2]), torch.cat([v1, v2])
    fa, o = run(q.to(dev), k.to(dev), v.to(dev), [(0, 260), (260, 240)], centering=True, per_row=True,
                sink_keys=3, with_lse=True)
    ob = oracle.bounds(q, k, v, centering=True, per_row=True, sink_keys=3)
    check_bounds(fa, ob)
    check_sinks(fa, ob)
    ref, ref_lse = oracle.attention(q, k, v, return_lse=True)
    assert maxerr(o, ref) <= TOL_BF16
    assert maxerr(fa.lse, ref_lse) <= TOL_LSE * max(1.0, float(np.max(np.abs(ref_lse))))


@pytest.mark.parametrize("one_launch", [False, True])
def test_head_and_batch_placement_bitwise(dev, one_launch):
    """Scheduling changes that leave each (batch, head) problem's arithmetic alone give the same
    bits (the bit-invariance pattern of PR444's heads_per_tile): heads in reverse order, and
    the heads laid out as batch entries instead, so that a different CTA of the grid computes
    each problem."""
    q, k, v = workloads.make_inputs("mix", device=dev, heads=range(4), Sq=333, N=700)
    chunks = [(0, 300), (300, 400)]

    def go(qq, kk, vv):
        fa = fm.FixedMAttention(qq.shape[0], qq.shape[1], 333, 700, 128, dev, centering=False)
        o = fa.forward(qq, kk, vv, chunks, with_lse=True, one_launch=one_launch).clone()
        fm.fm_sync_status()
        return o, fa.lse.clone(), fa.bounds.m.clone(), fa.bounds.shift.clone()

    base = go(q, k, v)
    rev = go(q.flip(1).contiguous(), k.flip(1).contiguous(), v.flip(1).contiguous())
    bat = go(q.transpose(0, 1).contiguous(), k.transpose(0, 1).contiguous(), v.transpose(0, 1).contiguous())
    for a, r, bb in zip(base, rev, bat):
        assert torch.equal(a, r.flip(1))
        assert torch.equal(a, bb.transpose(0, 1))


def test_key_sink_positions_and_ties_on_the_device(dev):
    """Sinks at the edges of the bounds pass's 256-key blocks and of the 128-key tiles
    (positions 127, 128, 255, 256, 512 of 513 keys), split across chunks at 256; and a tie:
    two identical loudest keys with sink_keys = 1 give no sink at all (only keys strictly
    louder than the first kept one are sinks), on the device as in the oracle."""
    q, k, v = workloads.make_inputs("h40_s4096", device="cpu", heads=[0, 1], Sq=140, N=513)
    pos = [127, 128, 255, 256, 512]
    k[:, 0, pos] *= 60.0
    k[:, 1, 300] = k[:, 1, 40] * 80.0   # head 1: two identical loud keys
    k[:, 1, 40] = k[:, 1, 300]
    ob = oracle.bounds(q, k, v, sink_keys=5)
    fa, o = run(q.to(dev), k.to(dev), v.to(dev), [(0, 256), (256, 257)], sink_keys=5)
    check_bounds(fa, ob)
    assert list(fa.bounds.sink_idx[0, 0, :5].cpu().numpy()) == pos
    assert maxerr(o, oracle.attention(q, k, v)) <= TOL_BF16
    ob1 = oracle.bounds(q, k, v, sink_keys=1)
    fb, o1 = run(q.to(dev), k.to(dev), v.to(dev), [(0, 513)], sink_keys=1)
    assert list(ob1["sink_idx"][0, 1]) == [2**31 - 1]
    assert int(fb.bounds.sink_idx[0, 1, 0].item()) == 2**31 - 1
    assert float(fb.bounds.kmax_sq[0, 1].item()) == pytest.approx(float(ob1["kmax_sq"][0, 1]), rel=2e-5)
    assert maxerr(o1, oracle.attention(q, k, v)) <= TOL_BF16


@pytest.mark.parametrize("force_online", [False, True])
def test_ring_order_of_chunks(dev, force_online):
    """The ring hands each device the KV chunks in a rotated order.  The fixed-m merge is a pure
    add, and the online one a max-rescaled add, so folding the chunks in any order gives the same
    result up to fp32 summation order (within the bf16 tolerance, and close to each other)."""
    q, k, v = workloads.make_inputs("mix", device="cpu", heads=range(2), Sq=300, N=900)
    qd = q.to(dev)
    parts = [(0, 300), (300, 300), (600, 300)]
    ref = oracle.attention(q, k, v)
    outs = []
    for order in ([0, 1, 2], [1, 2, 0], [2, 0, 1]):
        kk = torch.cat([k[:, :, s:s + n] for s, n in (parts[i] for i in order)], dim=2).to(dev)
        vv = torch.cat([v[:, :, s:s + n] for s, n in (parts[i] for i in order)], dim=2).to(dev)
        _, o = run(qd, kk, vv, parts, force_online=force_online)
        assert maxerr(o, ref) <= TOL_BF16
        outs.append(o.clone())
    assert maxerr(outs[0], outs[1]) <= 1e-3 and maxerr(outs[0], outs[2]) <= 1e-3


def test_cuda_graph_capture_with_key_sinks(dev):
    """The key-sink path (selection in the bounds pass, masked chunks, the fold with the
    normalise) has no host synchronisation either: captured once and replayed on new data it
    gives the eager bits."""
    Sq, N = 400, 900
    chunks = [(0, 450), (450, 450)]
    q, k, v = workloads.make_inputs("sinks", device=dev, heads=[0, 1, 30], Sq=Sq, N=N)
    q2, k2, v2 = workloads.make_inputs("sinks", device=dev, heads=[2, 3, 31], Sq=Sq, N=N)
    fa = fm.FixedMAttention(1, 3, Sq, N, 128, dev, sink_keys=4)
    fa.forward(q, k, v, chunks, with_lse=True)
    fm.fm_sync_status()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fa.forward(q, k, v, chunks, with_lse=True)
    q.copy_(q2)
    k.copy_(k2)
    v.copy_(v2)
    g.replay()
    torch.cuda.synchronize()
    fm.fm_sync_status()
    fb = fm.FixedMAttention(1, 3, Sq, N, 128, dev, sink_keys=4)
    ref = fb.forward(q2, k2, v2, chunks, with_lse=True)
    fm.fm_sync_status()
    assert torch.equal(fa.out, ref) and torch.equal(fa.lse, fb.lse)
    assert torch.equal(fa.bounds.sink_idx, fb.bounds.sink_idx)
    assert maxerr(fa.out, oracle.attention(q2.cpu(), k2.cpu(), v2.cpu())) <= TOL_BF16


def test_randomised_shapes_and_options(dev):
    """Forty seeded random cases against the oracle: batch, heads, query and key lengths
    (ragged everywhere), chunk splits (empty chunks included), dtype and head dimension, and
    every option (centering, per-row shifts, key sinks, forced fallback, LSE, one launch)."""
    rng = np.random.default_rng(1234)
    for case in range(40):
        B = int(rng.integers(1, 3))
        H = int(rng.integers(1, 4))
        Sq = int(rng.integers(1, 400))
        N = int(rng.integers(1, 700))
        D = 128 if rng.random() < 0.8 else 64
        dt = torch.bfloat16 if (D == 128 and rng.random() < 0.8) else torch.float32
        g = torch.Generator().manual_seed(case)
        scale = float(rng.choice([0.3, 1.0, 3.0]))
        q = (torch.randn(B, H, Sq, D, generator=g) * scale).to(dt)
        k = (torch.randn(B, H, N, D, generator=g) + float(rng.normal()) * 2.0).to(dt)
        v = torch.randn(B, H, N, D, generator=g).to(dt)
        n_chunks = int(rng.integers(1, 5))
        cuts = np.sort(rng.integers(0, N + 1, size=n_chunks - 1))
        edges = [0, *cuts.tolist(), N]
        chunks = [(edges[i], edges[i + 1] - edges[i]) for i in range(n_chunks)]
        opts = dict(centering=bool(rng.random() < 0.5), per_row=bool(rng.random() < 0.3),
                    force_online=bool(rng.random() < 0.2), sink_keys=int(rng.choice([0, 0, 1, 3])))
        fa = fm.FixedMAttention(B, H, Sq, N, D, dev, **opts)
        one = bool(rng.random() < 0.3)
        o = fa.forward(q.to(dev), k.to(dev), v.to(dev), chunks, with_lse=True, one_launch=one)
        fm.fm_sync_status()
        ref, ref_lse = oracle.attention(q, k, v, return_lse=True)
        tol = TOL_F32 if dt == torch.float32 else TOL_BF16
        desc = (case, B, H, Sq, N, D, dt, chunks, opts, one)
        assert maxerr(o, ref) <= tol, desc
        if dt == torch.bfloat16:
            reference(q, k, v, centering=opts["centering"], per_row=opts["per_row"],
                      sink_keys=opts["sink_keys"]).check(o, str(desc))
        assert maxerr(fa.lse, ref_lse) <= TOL_LSE * max(1.0, float(np.max(np.abs(ref_lse)))), desc
        ob = oracle.bounds(q, k, v, centering=opts["centering"], per_row=opts["per_row"],
                           sink_keys=opts["sink_keys"])
        check_bounds(fa, ob)


@pytest.mark.parametrize("force_online", [False, True])
@pytest.mark.parametrize("mode", ["chunks", "fused", "one_launch", "sinks"])
def test_persistent_schedule_gives_the_grid_bits(dev, mode, force_online):
    """The persistent schedule (one CTA per SM walking work items) and the grid schedule (one
    CTA per work item) do the same fp32 arithmetic in the same order: identical bits, on more
    work items (20 heads x 8 Q-tile pairs, the last pair half past Sq) than a GB300 has SMs."""
    H, Sq, N = 20, 1900, 1500
    name = "sinks" if mode == "sinks" else "mix"
    q, k, v = workloads.make_inputs(name, device="cpu", heads=range(H), Sq=Sq, N=N)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    chunks = [(0, 700), (700, 1), (701, 799)]
    outs = {}
    for sched in ("grid", "persistent"):
        fa = fm.FixedMAttention(1, H, Sq, N, 128, dev, centering=mode != "sinks", force_online=force_online,
                                sink_keys=4 if mode == "sinks" else 0, schedule=sched)
        o = fa.forward(qd, kd, vd, chunks, with_lse=True, fused_final=mode != "chunks",
                       one_launch=mode == "one_launch").clone()
        fm.fm_sync_status()
        outs[sched] = (o, fa.lse.clone(), fa.acc_sum.clone(), fa.acc_max.clone())
    for a, b in zip(outs["grid"], outs["persistent"]):
        assert torch.equal(a, b)
    heads = [0, 7, 19]
    rows = list(range(0, 128)) + list(range(1792, 1900))
    reference(q, k, v, heads, rows, centering=mode != "sinks", sink_keys=4 if mode == "sinks" else 0).check(
        pick(outs["persistent"][0], heads, rows), f"persistent {mode} online={force_online}")


def test_schedule_option_is_validated(dev):
    q, k, v = workloads.make_inputs("wan", device=dev, heads=[0], Sq=130, N=140)
    fa = fm.FixedMAttention(1, 1, 130, 140, 128, dev, schedule=3)
    fm.fm_bounds(q, k, v, fa.opt, fa.bounds, fa.workspace)
    with pytest.raises(fm.FMError) as e:
        fm.fm_attn_chunk(q, k, v, fa.bounds, fa.opt, fa.acc_o, fa.acc_sum, fa.acc_max, False)
    assert e.value.code == fm.FM_ERR_ARG
