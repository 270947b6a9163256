"""Seeded synthetic workloads for fixed-m attention.

This module only draws random numbers and shapes them into the five workloads; it
holds none of the method's arithmetic (no norms-to-bounds, no constants, no gate).
Both the CUDA path's tests/bench and the CPU oracle take their inputs from here; the
oracle always receives the exact tensors the GPU saw (copied to host), so the device
the generator runs on does not matter for parity.

Each head is drawn from its own generator, seeded with (seed, head), so a subset of
heads can be regenerated alone (the CPU baseline times one head of the large case).

Workloads (the shapes and value recipes of the pages' Wan2.2 DiT attention and of the
pages' adversarial examples; no dataset or trained weights are involved):

  tiny         B=1 H=2  S=256    D=64  fp32  q,k,v = 0.5 N(0,1); 1 chunk; no centering
  h40_s4096    B=1 H=40 S=4096   D=128 bf16  q,k,v = N(0,1) * D^(-1/4); 4 chunks of 1024
  wan          B=1 H=40 S=75600  D=128 bf16  N(0,1) then each (token, head) vector RMS-
                                             normalised to RMS 1 (gain 1); 2 chunks of
                                             37,800; centering on
  mix          B=1 H=40 S=16384  D=128 bf16  k = N(0,1) + a per-head offset (random
                                             direction, norm ~ U[0,60]); every query of a
                                             head has norm s_h ~ U[1,40]; v = N(0,1)
  adversarial  B=1 H=40 S=4096   D=128 bf16  heads 0-19: keys are +/- pairs of unit vectors
                                             (mean exactly zero), query row 0 has the norm
                                             that puts its bound at 231.01, other rows
                                             N(0,1); heads 20-39: N(0,1); centering on
  sinks        B=1 H=40 S=16384  D=128 bf16  q,k,v = N(0,1) * D^(-1/4) as h40_s4096; in heads
                                             0-19 the keys at positions 0, 1, N/2+3 and N-1
                                             are scaled x100 (massive-activation key sinks,
                                             a norm spread in the pages' 100-1000x range);
                                             4 chunks of 4096; centering off
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Sq: int
    N: int
    D: int
    dtype: str  # "f32" | "bf16"
    chunks: tuple
    centering: tuple  # the centering settings this workload is run with
    seed: int
    note: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def flops(self, heads: int | None = None, rows: int | None = None, keys: int | None = None) -> float:
        """4 * H * Sq * Sk * D: the two contractions (QK^T and PV) of attention."""
        h = self.B * self.H if heads is None else heads
        r = self.Sq if rows is None else rows
        n = self.N if keys is None else keys
        return 4.0 * h * r * n * self.D


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 256, 256, 64, "f32", (256,), (False,), 1,
                     "q,k,v = 0.5*N(0,1)"),
    "h40_s4096": Workload("h40_s4096", 1, 40, 4096, 4096, 128, "bf16", (1024,) * 4, (False,), 2,
                          "q,k,v = N(0,1)*D^-1/4"),
    "wan": Workload("wan", 1, 40, 75600, 75600, 128, "bf16", (37800, 37800), (True,), 3,
                    "N(0,1), per-(token,head) RMS-norm to RMS 1"),
    "mix": Workload("mix", 1, 40, 16384, 16384, 128, "bf16", (16384,), (False, True), 4,
                    "k = N(0,1) + per-head offset |o|~U[0,60]; |q| = s_h ~ U[1,40]"),
    "adversarial": Workload("adversarial", 1, 40, 4096, 4096, 128, "bf16", (4096,), (True,), 5,
                            "heads 0-19: +/- unit key pairs, row 0 bound 231.01; heads 20-39 N(0,1)",
                            {"target_bound": 231.01, "adv_heads": 20}),
    "sinks": Workload("sinks", 1, 40, 16384, 16384, 128, "bf16", (4096,) * 4, (False, True), 6,
                      "N(0,1)*D^-1/4; heads 0-19: keys 0, 1, N/2+3, N-1 scaled x100",
                      {"sink_heads": 20, "sink_scale": 100.0}),
}


def sink_positions(N: int) -> list:
    """Key positions the sinks workload plants its loud keys at (distinct, in range)."""
    return sorted({p for p in (0, 1, N // 2 + 3, N - 1) if 0 <= p < N})


def _gen(seed: int, head: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1_000_003 + head)
    return g


def _head(w: Workload, h: int, Sq: int, N: int, device) -> tuple:
    """q [Sq, D], k [N, D], v [N, D] in fp32 for head h of workload w."""
    g = _gen(w.seed, h, device)
    D = w.D

    def randn(*shape):
        return torch.randn(*shape, generator=g, device=device, dtype=torch.float32)

    if w.name == "tiny":
        return 0.5 * randn(Sq, D), 0.5 * randn(N, D), 0.5 * randn(N, D)
    if w.name in ("h40_s4096", "sinks"):
        s = D ** -0.25
        q, k, v = s * randn(Sq, D), s * randn(N, D), s * randn(N, D)
        if w.name == "sinks" and h % w.H < w.extra["sink_heads"]:
            k[sink_positions(N)] *= w.extra["sink_scale"]
        return q, k, v
    if w.name == "wan":
        def rms(x):
            return x * torch.rsqrt(x.pow(2).mean(dim=-1, keepdim=True) + 1e-6)
        return rms(randn(Sq, D)), rms(randn(N, D)), rms(randn(N, D))
    if w.name == "mix":
        u = randn(D)
        u = u / u.norm()
        a = 60.0 * torch.rand((), generator=g, device=device)
        s_h = 1.0 + 39.0 * torch.rand((), generator=g, device=device)
        k = randn(N, D) + a * u
        q = randn(Sq, D)
        q = q / q.norm(dim=-1, keepdim=True) * s_h
        return q, k, randn(N, D)
    if w.name == "adversarial":
        if h < w.extra["adv_heads"]:
            half = N // 2
            u = randn(half, D)
            u = u / u.norm(dim=-1, keepdim=True)
            u = u.to(w.torch_dtype).float()  # round first so that -u is exactly the negation
            k = torch.stack([u, -u], dim=1).reshape(2 * half, D)
            if k.shape[0] < N:  # odd N: one zero key keeps the mean at zero
                k = torch.cat([k, torch.zeros(N - k.shape[0], D, device=device)], 0)
            q = randn(Sq, D)
            # row 0: the norm at which scale*log2(e)*|q|*max|k| reaches the target bound
            kmax = k.norm(dim=-1).max()
            target = w.extra["target_bound"] * math.sqrt(D) / math.log2(math.e) / kmax
            q0 = randn(D)
            q[0] = q0 / q0.norm() * target
            return q, k, randn(N, D)
        return randn(Sq, D), randn(N, D), randn(N, D)
    raise KeyError(w.name)


def make_inputs(name: str, device="cpu", heads=None, Sq: int | None = None, N: int | None = None):
    """q [B, Hs, Sq, D], k, v [B, Hs, N, D] in the workload's dtype on `device`.

    heads: None for all heads, or an iterable of head indices (each head is
    reproducible alone).  Sq / N override the sequence lengths (same recipe),
    for reduced-size cases.
    """
    w = WORKLOADS[name]
    Sq = w.Sq if Sq is None else Sq
    N = w.N if N is None else N
    hs = list(range(w.H)) if heads is None else list(heads)
    dt = w.torch_dtype
    q = torch.empty(w.B, len(hs), Sq, w.D, dtype=dt, device=device)
    k = torch.empty(w.B, len(hs), N, w.D, dtype=dt, device=device)
    v = torch.empty(w.B, len(hs), N, w.D, dtype=dt, device=device)
    for b in range(w.B):
        for i, h in enumerate(hs):
            qh, kh, vh = _head(w, b * w.H + h, Sq, N, device)
            q[b, i].copy_(qh)
            k[b, i].copy_(kh)
            v[b, i].copy_(vh)
    return q, k, v


def chunk_bounds(w: Workload, N: int | None = None) -> list:
    """[(start, length)] of the sequential KV chunks ("ring steps") of a workload."""
    N = w.N if N is None else N
    if N == w.N:
        out, s = [], 0
        for c in w.chunks:
            out.append((s, c))
            s += c
        return out
    n = len(w.chunks)
    base = N // n
    out, s = [], 0
    for i in range(n):
        c = base if i < n - 1 else N - s
        out.append((s, c))
        s += c
    return out
