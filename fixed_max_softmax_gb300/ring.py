"""Fixed-m attention over a ring of ranks (torch.distributed; one process per GPU).

Each rank keeps its own query rows and holds one shard of the keys and values.  The shards
rotate one hop per step, so after R steps every rank has folded every shard into its own
unnormalised fp32 accumulators, by plain addition on the fixed-m tiles ("Kernel reference:
ring_attention_const_max_fwd", sections "A static bound makes the ring reduction pure addition"
and "The ring loop").  Before the ring, one exchange makes the bounds ring-wide: the key sums
for the mean (all-reduce, sum) when centering, then every rank's key max, V max and key-sink
candidates (all-gather), which each rank combines into the same bounds ("Global key max";
PR #478 Summary, "Global Virtual K-Centering").

The ring loop: step s folds the shard that started on rank (rank - s) mod R, at its global key
offset.  Its K/V arrive in one of `prefetch + 1` rotating buffers; the transfer for step
s + prefetch (this rank forwards what it held at step s + prefetch - 1 to rank + 1 and receives
from rank - 1) is issued before step s computes, so the hops overlap the attention.  Every
transfer lands in this rank's own memory before a kernel reads it.  Step 0 initialises the
accumulators; the last step folds and normalises in one pass.

All arithmetic runs in the library's kernels (through ``ops``, the package module by default);
this module only orders the calls and moves bytes with torch.distributed.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


class RingSchedule:
    """Which shard each rank folds at each step, and where it comes from (host logic only)."""

    def __init__(self, rank: int, world: int, shard_lens):
        if len(shard_lens) != world:
            raise ValueError("one shard length per rank")
        self.rank, self.world = rank, world
        self.lens = [int(n) for n in shard_lens]
        self.starts = [sum(self.lens[:r]) for r in range(world)]
        self.N = sum(self.lens)
        self.max_len = max(self.lens) if self.lens else 0

    def source(self, step: int) -> int:
        """The rank whose shard this rank folds at `step` (the ring turns one hop per step)."""
        return (self.rank - step) % self.world

    def key_offset(self, step: int) -> int:
        return self.starts[self.source(step)]

    def length(self, step: int) -> int:
        return self.lens[self.source(step)]

    @property
    def send_to(self) -> int:
        return (self.rank + 1) % self.world

    @property
    def recv_from(self) -> int:
        return (self.rank - 1) % self.world


class RingAttention:
    """Buffers and the call sequence of a ring forward on one rank.

    q: [B, H, Sq, D] this rank's queries; k_shard, v_shard: [B, H, shard_lens[rank], D].
    `group` is the process group (None: the default group).  `prefetch` is the number of
    ring steps ahead that a transfer is issued (clamped to [1, R - 1]).
    """

    def __init__(self, B, H, Sq, D, shard_lens, device, dtype=torch.bfloat16, group=None, centering=False,
                 per_row=False, sink_keys=0, softmax_scale=0.0, prefetch=2, out_dtype=torch.float32, ops=None):
        if ops is None:
            import fixed_max_softmax_gb300 as ops
        self.ops = ops
        self.group = group
        rank = dist.get_rank(group)
        world = dist.get_world_size(group)
        self.sched = RingSchedule(rank, world, shard_lens)
        self.prefetch = max(1, min(int(prefetch), world - 1)) if world > 1 else 0
        self.opt = ops.opts(softmax_scale, centering, False, per_row, sink_keys)
        self.centering = centering
        self.B, self.H, self.Sq, self.D = B, H, Sq, D
        self.bounds = ops.Bounds(B, H, Sq, D, device)
        nbytes = ops.fm_bounds_workspace_size(B, H, max(self.sched.max_len, 1), D)
        self.workspace = torch.empty(max(nbytes, 16) // 4 + 4, dtype=torch.float32, device=device)
        self.ksum = torch.zeros(B, H, D, dtype=torch.float32, device=device)
        sb = ops.fm_ring_stats_bytes(B, H, D, sink_keys)
        self.stats = torch.zeros(sb, dtype=torch.uint8, device=device)
        self.stats_all = torch.zeros(world * sb, dtype=torch.uint8, device=device)
        self.acc_o = torch.empty(B, H, Sq, D, dtype=torch.float32, device=device)
        self.acc_sum = torch.empty(B, H, Sq, dtype=torch.float32, device=device)
        self.acc_max = torch.empty(B, H, Sq, dtype=torch.float32, device=device)
        self.out = torch.empty(B, H, Sq, D, dtype=out_dtype, device=device)
        n_buf = self.prefetch + 1
        L = self.sched.max_len
        self.kbuf = [torch.empty(B, H, L, D, dtype=dtype, device=device) for _ in range(n_buf)]
        self.vbuf = [torch.empty(B, H, L, D, dtype=dtype, device=device) for _ in range(n_buf)]
        # gloo runs transfers asynchronously with no order between them: forward a buffer only
        # once it has arrived.  NCCL keeps one communicator's transfers in issue order on its stream.
        self.strict = dist.get_backend(group) != "nccl"

    # ---- the exchange before the ring
    def bounds_ring_wide(self, q, k_shard, v_shard):
        ops, s = self.ops, self.sched
        ksum = None
        if self.centering:
            ops.fm_ring_key_sums(k_shard, self.ksum, self.workspace)
            dist.all_reduce(self.ksum, op=dist.ReduceOp.SUM, group=self.group)
            ksum = self.ksum
        ops.fm_bounds_local(q, k_shard, v_shard, s.starts[s.rank], s.N, ksum, self.opt, self.bounds, self.stats,
                            self.workspace)
        dist.all_gather(list(self.stats_all.chunk(s.world)), self.stats, group=self.group)
        ops.fm_bounds_combine(self.stats_all, s.world, self.opt, self.bounds)

    # ---- the ring loop
    def _issue(self, t, pending):
        """Start the transfer that brings step t's shard into buffer t % (prefetch + 1)."""
        nb = self.prefetch + 1
        src, dst = (t - 1) % nb, t % nb
        if self.strict and (t - 1) in pending:
            for r in pending.pop(t - 1):
                r.wait()
        P2P = dist.P2POp
        ops = [P2P(dist.isend, self.kbuf[src], self.sched.send_to, self.group),
               P2P(dist.isend, self.vbuf[src], self.sched.send_to, self.group),
               P2P(dist.irecv, self.kbuf[dst], self.sched.recv_from, self.group),
               P2P(dist.irecv, self.vbuf[dst], self.sched.recv_from, self.group)]
        pending[t] = dist.batch_isend_irecv(ops)

    def forward(self, q, k_shard, v_shard, lse=None):
        ops, s = self.ops, self.sched
        self.bounds_ring_wide(q, k_shard, v_shard)
        n0 = s.lens[s.rank]
        self.kbuf[0][:, :, :n0].copy_(k_shard)
        self.vbuf[0][:, :, :n0].copy_(v_shard)
        pending = {}
        for t in range(1, self.prefetch + 1):
            if t < s.world:
                self._issue(t, pending)
        nb = self.prefetch + 1
        for step in range(s.world):
            for r in pending.pop(step, []):
                r.wait()
            n = s.length(step)
            kc = self.kbuf[step % nb][:, :, :n]
            vc = self.vbuf[step % nb][:, :, :n]
            self.bounds.out.next_key_offset = s.key_offset(step)
            last = step == s.world - 1
            if last:
                ops.fm_attn_chunk_final(q, kc, vc, self.bounds, self.opt, self.acc_o, self.acc_sum, self.acc_max,
                                        step > 0, self.out, lse)
            else:
                ops.fm_attn_chunk(q, kc, vc, self.bounds, self.opt, self.acc_o, self.acc_sum, self.acc_max, step > 0)
            if step + self.prefetch < s.world:
                self._issue(step + self.prefetch, pending)
        return self.out
