"""The bounds of a ring of ranks, and chunks folded in ring order, on one GPU.

Each "rank" below is simulated in turn in one process: its own query rows, one shard of the keys
and values.  The exchanges a ring makes with collectives (the key sums all-reduced, the
statistics blocks all-gathered) are done here with plain tensor sums and concatenation in rank
order.  No kernel ever waits on another rank's kernel.  The combined bounds must match the
oracle's bounds over every key exactly as fm_bounds' do (m and flag outside the fp32 tie band,
the key sinks, the norms), and folding the shards in ring order -- rank r takes shard r, r-1, ...
with each shard's global key offset -- must give attention over every key.
"""
import types

import numpy as np
import pytest
import torch

import fixed_max_softmax_gb300 as fm
import oracle
import workloads
from tests.test_gpu_parity import check_bounds, check_sinks, reference

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fixed_max_softmax_gb300 import build as fmbuild

    fmbuild.build()
    fm.load()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def ring_bounds(dev, qs, ks, vs, lens, opt):
    """Steps 1-3 of the ring bounds for every simulated rank; returns each rank's Bounds."""
    R = len(lens)
    starts = [sum(lens[:r]) for r in range(R)]
    N = sum(lens)
    B, H, _, D = qs[0].shape
    ws_bytes = max(fm.fm_bounds_workspace_size(B, H, max(n, 1), D) for n in lens)
    ws = torch.empty(ws_bytes // 4 + 4, dtype=torch.float32, device=dev)
    ksum_total = None
    if opt.centering:
        ksum_total = torch.zeros(B, H, D, dtype=torch.float32, device=dev)
        part = torch.empty_like(ksum_total)
        for r in range(R):  # the all-reduce, in rank order
            fm.fm_ring_key_sums(ks[r], part, ws)
            ksum_total += part
    sb = fm.fm_ring_stats_bytes(B, H, D, opt.sink_keys)
    stats = [torch.empty(sb, dtype=torch.uint8, device=dev) for _ in range(R)]
    bounds = [fm.Bounds(B, H, qs[r].shape[2], D, dev) for r in range(R)]
    for r in range(R):
        fm.fm_bounds_local(qs[r], ks[r], vs[r], starts[r], N, ksum_total, opt, bounds[r], stats[r], ws)
        assert bounds[r].out.magic == fm.FM_BOUNDS_LOCAL_MAGIC
    stats_all = torch.cat(stats)  # the all-gather, in rank order
    for r in range(R):
        fm.fm_bounds_combine(stats_all, R, opt, bounds[r])
    fm.fm_sync_status()
    return bounds, starts


@pytest.mark.parametrize("lens", [[500, 400], [350, 300, 250], [500, 0, 400]])
@pytest.mark.parametrize("centering,sink_keys,per_row", [(False, 0, False), (True, 0, False), (False, 4, False),
                                                         (True, 4, True)])
def test_ring_bounds_and_ring_order(dev, lens, centering, sink_keys, per_row):
    R = len(lens)
    N = sum(lens)
    sq = [300, 260, 340][:R]
    name = "sinks" if sink_keys else "mix"
    q_all, k, v = workloads.make_inputs(name, device="cpu", heads=[0, 1, 25], Sq=sum(sq), N=N)
    starts_q = [sum(sq[:r]) for r in range(R)]
    qs = [q_all[:, :, starts_q[r]:starts_q[r] + sq[r]] for r in range(R)]
    starts_k = [sum(lens[:r]) for r in range(R)]
    ks = [k[:, :, starts_k[r]:starts_k[r] + lens[r]].to(dev) for r in range(R)]
    vs = [v[:, :, starts_k[r]:starts_k[r] + lens[r]].to(dev) for r in range(R)]
    opt = fm.opts(centering=centering, per_row=per_row, sink_keys=sink_keys)
    bounds, starts = ring_bounds(dev, [x.to(dev) for x in qs], ks, vs, lens, opt)
    kd, vd = k.to(dev), v.to(dev)
    for r in range(R):
        b = bounds[r]
        assert b.out.magic == fm.FM_BOUNDS_MAGIC and b.out.N_total == N
        ob = oracle.bounds(qs[r], k, v, centering=centering, per_row=per_row, sink_keys=sink_keys)
        check_bounds(types.SimpleNamespace(bounds=b), ob)
        if sink_keys:
            check_sinks(types.SimpleNamespace(bounds=b), ob)
        # the same sinks as the single-GPU bounds pass over every key, in the two heads whose
        # loud keys stand far above the rest (elsewhere near-ties may pick another set, which the
        # oracle check above allows)
        fa = fm.FixedMAttention(1, 3, sq[r], N, 128, dev, centering=centering, per_row=per_row, sink_keys=sink_keys)
        qd = qs[r].to(dev)
        fm.fm_bounds(qd, kd, vd, fa.opt, fa.bounds, fa.workspace)
        fm.fm_sync_status()
        if sink_keys:
            assert torch.equal(fa.bounds.sink_idx[:, :2], b.sink_idx[:, :2])
        assert float(fa.bounds.vmax_sq.item()) == float(b.vmax_sq.item())
        np.testing.assert_allclose(b.kbar.cpu().numpy(), fa.bounds.kbar.cpu().numpy(), rtol=1e-5, atol=1e-6)
        # the ring: rank r folds shard r, r-1, ... at each shard's global key offset
        acc_o, acc_sum, acc_max = fa.acc_o, fa.acc_sum, fa.acc_max
        out = torch.empty(1, 3, sq[r], 128, dtype=torch.float32, device=dev)
        for step in range(R):
            src = (r - step) % R
            b.out.next_key_offset = starts[src]
            if step == R - 1:
                fm.fm_attn_chunk_final(qd, ks[src], vs[src], b, opt, acc_o, acc_sum, acc_max, step > 0, out)
            else:
                fm.fm_attn_chunk(qd, ks[src], vs[src], b, opt, acc_o, acc_sum, acc_max, step > 0)
        fm.fm_sync_status()
        assert b.out.kv_seen == N and b.out.next_key_offset == -1
        reference(qs[r], k, v, centering=centering, per_row=per_row, sink_keys=sink_keys).check(
            out, f"rank {r} of {R}, shards {lens}")


def test_ring_bounds_contracts(dev):
    q, k, v = workloads.make_inputs("wan", device=dev, heads=[0], Sq=130, N=200)
    opt = fm.opts(centering=True)
    b = fm.Bounds(1, 1, 130, 128, dev)
    ws = torch.empty(fm.fm_bounds_workspace_size(1, 1, 200, 128) // 4 + 4, dtype=torch.float32, device=dev)
    stats = torch.empty(fm.fm_ring_stats_bytes(1, 1, 128), dtype=torch.uint8, device=dev)
    # the shard must lie inside the ring's keys; centering needs the ring-wide key sums
    with pytest.raises(fm.FMError) as e:
        fm.fm_bounds_local(q, k, v, 100, 250, None, opt, b, stats, ws)
    assert e.value.code == fm.FM_ERR_ARG
    with pytest.raises(fm.FMError) as e:
        fm.fm_bounds_local(q, k, v, 0, 200, None, opt, b, stats, ws)
    assert e.value.code == fm.FM_ERR_ARG
    # combine only after a local pass, with the same options
    b2 = fm.Bounds(1, 1, 130, 128, dev)
    with pytest.raises(fm.FMError) as e:
        fm.fm_bounds_combine(stats, 1, opt, b2)
    assert e.value.code == fm.FM_ERR_BOUNDS_MISMATCH
    ksum = torch.empty(1, 1, 128, dtype=torch.float32, device=dev)
    fm.fm_ring_key_sums(k, ksum, ws)
    fm.fm_bounds_local(q, k, v, 0, 200, ksum, opt, b, stats, ws)
    with pytest.raises(fm.FMError) as e:
        fm.fm_bounds_combine(stats, 1, fm.opts(centering=False), b)
    assert e.value.code == fm.FM_ERR_BOUNDS_MISMATCH
    # chunks before the combine are refused: the bounds are not complete
    fa = fm.FixedMAttention(1, 1, 130, 200, 128, dev, centering=True)
    with pytest.raises(fm.FMError) as e:
        fm.fm_attn_chunk(q, k, v, b, opt, fa.acc_o, fa.acc_sum, fa.acc_max, False)
    assert e.value.code == fm.FM_ERR_BOUNDS_MISMATCH
    fm.fm_bounds_combine(stats, 1, opt, b)
    # a chunk whose keys would lie past N_total at the given offset is refused
    b.out.next_key_offset = 150
    with pytest.raises(fm.FMError) as e:
        fm.fm_attn_chunk(q, k, v, b, opt, fa.acc_o, fa.acc_sum, fa.acc_max, False)
    assert e.value.code == fm.FM_ERR_BOUNDS_MISMATCH
    fm.fm_sync_status()


@pytest.mark.parametrize("force_online", [False, True])
def test_key_sinks_in_rotated_chunk_order(dev, force_online):
    """Key sinks are found by global key index, so chunks folded in ring order (not key order)
    must skip exactly the keys that the bounds left out: the output is still attention over
    every key."""
    q, k, v = workloads.make_inputs("sinks", device="cpu", heads=[0, 1, 30], Sq=300, N=900)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    for order in ([(300, 300), (0, 300), (600, 300)], [(600, 300), (300, 300), (0, 300)]):
        fa = fm.FixedMAttention(1, 3, 300, 900, 128, dev, sink_keys=4, force_online=force_online)
        o = fa.forward(qd, kd, vd, order, with_lse=True)
        fm.fm_sync_status()
        assert list(fa.bounds.sink_idx[0, 0, :4].cpu().numpy()) == workloads.sink_positions(900)
        reference(q, k, v, sink_keys=4).check(o, f"sinks, chunk order {order}")
        ref_o, ref_lse = oracle.attention(q, k, v, return_lse=True)
        assert np.max(np.abs(fa.lse.cpu().numpy() - ref_lse)) <= 1e-4 * max(1.0, float(np.max(np.abs(ref_lse))))
