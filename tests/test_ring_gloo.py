"""The ring driver (fixed_max_softmax_gb300/ring.py) on CPU gloo ranks, 2 and 3 of them.

What is tested is the host logic: the exchange before the ring (key sums all-reduced, statistics
blocks all-gathered in rank order), the rotation of the K/V shards one hop per step through the
rotating buffers, the global key offset of each step, the accumulate flags, and that the final
step normalises.  The library's kernels need a GPU, so the ranks run the driver with CPU stand-ins
of the calls: exact online-softmax partial folds in fp64, written here for this test only.  If
every shard reaches every rank exactly once, intact and with its own offset, each rank's output
equals the oracle's attention of its query rows over all keys.
"""
import os
import socket
import types

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from fixed_max_softmax_gb300.ring import RingAttention, RingSchedule

B, H, D = 1, 2, 16
SHARDS = {2: [70, 45], 3: [33, 64, 20]}
SQ = [40, 23, 31]


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def full_inputs(world):
    g = torch.Generator().manual_seed(100 + world)
    N = sum(SHARDS[world])
    k = torch.randn(B, H, N, D, generator=g)
    v = torch.randn(B, H, N, D, generator=g)
    qs = [torch.randn(B, H, SQ[r], D, generator=g) for r in range(world)]
    return qs, k, v


def stand_in_ops(log):
    """CPU stand-ins for the library calls the driver makes (fp64 arithmetic, exact folds)."""
    ns = types.SimpleNamespace()

    class Bounds:
        def __init__(self, B_, H_, Sq, D_, device):
            self.out = types.SimpleNamespace(next_key_offset=-1)

    ns.Bounds = Bounds
    ns.opts = lambda scale, centering, force_online, per_row, sink_keys: types.SimpleNamespace(
        centering=centering, sink_keys=sink_keys)
    ns.fm_bounds_workspace_size = lambda B_, H_, N, D_: 64
    ns.fm_ring_stats_bytes = lambda B_, H_, D_, n: 16

    def key_sums(k, ksum, ws):
        ksum.copy_(k.double().sum(2).float())
        log["ksum_local"] = k.double().sum(2)

    def bounds_local(q, k, v, off, N, ksum, opt, b, stats, ws):
        log["local"] = (off, k.shape[2], N, None if ksum is None else ksum.clone())
        words = stats.view(torch.float32)
        words[0], words[1], words[2], words[3] = float(off), float(k.shape[2]), float(N), float(dist.get_rank())

    def combine(stats_all, R, opt, b):
        log["combined"] = stats_all.view(torch.float32).reshape(R, 4).tolist()

    def fold(q, kc, vc, b, opt, acc_o, acc_sum, acc_max, accumulate):
        log.setdefault("calls", []).append((b.out.next_key_offset, kc.shape[2], kc.clone(), bool(accumulate)))
        s = torch.einsum("bhrd,bhnd->bhrn", q.double(), kc.double()) / np.sqrt(D)
        mc = s.amax(-1)
        p = torch.exp(s - mc[..., None])
        oc, lc = torch.einsum("bhrn,bhnd->bhrd", p, vc.double()), p.sum(-1)
        if accumulate:
            m0, o0, l0 = acc_max.double(), acc_o.double(), acc_sum.double()
            m = torch.maximum(m0, mc)
            a0, a1 = torch.exp(m0 - m), torch.exp(mc - m)
            oc, lc, mc = o0 * a0[..., None] + oc * a1[..., None], l0 * a0 + lc * a1, m
        acc_o.copy_(oc)
        acc_sum.copy_(lc)
        acc_max.copy_(mc)
        b.out.next_key_offset = -1

    def fold_final(q, kc, vc, b, opt, acc_o, acc_sum, acc_max, accumulate, out, lse):
        fold(q, kc, vc, b, opt, acc_o, acc_sum, acc_max, accumulate)
        out.copy_(acc_o / acc_sum[..., None])
        log["final"] = True

    ns.fm_ring_key_sums = key_sums
    ns.fm_bounds_local = bounds_local
    ns.fm_bounds_combine = combine
    ns.fm_attn_chunk = fold
    ns.fm_attn_chunk_final = fold_final
    return ns


def _rank(rank, world, port, centering, prefetch, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        qs, k, v = full_inputs(world)
        lens = SHARDS[world]
        s0 = sum(lens[:rank])
        kr, vr = k[:, :, s0:s0 + lens[rank]].clone(), v[:, :, s0:s0 + lens[rank]].clone()
        log = {}
        ra = RingAttention(B, H, SQ[rank], D, lens, "cpu", dtype=torch.float32, centering=centering,
                           prefetch=prefetch, ops=stand_in_ops(log))
        o = ra.forward(qs[rank], kr, vr)
        results[rank] = {
            "o": o.numpy().copy(),
            "calls": [(off, n, c.numpy().copy(), acc) for off, n, c, acc in log["calls"]],
            "local": (log["local"][0], log["local"][1], log["local"][2],
                      None if log["local"][3] is None else log["local"][3].numpy().copy()),
            "combined": log["combined"],
            "final": log.get("final", False),
        }
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,centering,prefetch", [(2, True, 2), (3, True, 2), (3, False, 1)])
def test_ring_delivers_every_shard_in_order_with_its_offset(world, centering, prefetch):
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:  # no fork of this (threaded) process
        results = m.dict()
        mp.start_processes(_rank, args=(world, port, centering, prefetch, results), nprocs=world,
                           start_method="spawn", join=True)
        res = dict(results)
    qs, k, v = full_inputs(world)
    lens = SHARDS[world]
    starts = [sum(lens[:r]) for r in range(world)]
    N = sum(lens)
    for r in range(world):
        got = res[r]
        # the exchange: ring-wide key sums; every rank's block, in rank order, on every rank
        off, n, NN, ksum = got["local"]
        assert (off, n, NN) == (starts[r], lens[r], N)
        if centering:
            np.testing.assert_allclose(ksum, k.double().sum(2).numpy(), rtol=1e-6, atol=1e-5)
        else:
            assert ksum is None
        assert got["combined"] == [[float(starts[i]), float(lens[i]), float(N), float(i)] for i in range(world)]
        # the ring: step s folds the shard of rank (r - s) mod R, at its offset, intact
        assert len(got["calls"]) == world
        for step, (off, n, kc, acc) in enumerate(got["calls"]):
            src = (r - step) % world
            assert (off, n, acc) == (starts[src], lens[src], step > 0)
            assert np.array_equal(kc, k[:, :, starts[src]:starts[src] + lens[src]].numpy())
        assert got["final"]
        # and so each rank's output is attention over every key
        want = oracle.attention(qs[r], k, v)
        assert np.max(np.abs(got["o"] - want)) < 1e-5


def test_schedule_host_logic():
    s = RingSchedule(2, 4, [10, 20, 30, 40])
    assert [s.source(t) for t in range(4)] == [2, 1, 0, 3]
    assert [s.key_offset(t) for t in range(4)] == [30, 10, 0, 60]
    assert [s.length(t) for t in range(4)] == [30, 20, 10, 40]
    assert (s.send_to, s.recv_from, s.N, s.max_len) == (3, 1, 100, 40)
    with pytest.raises(ValueError):
        RingSchedule(0, 2, [1, 2, 3])
