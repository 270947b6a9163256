"""Out-of-bounds write checks: NaN-patterned guard bands around every buffer a kernel writes.

Each output the library writes -- the accumulators acc_o / acc_sum / acc_max, the output o
(contiguous, and with padded rows whose padding must stay untouched), the LSE and every
bounds array -- is placed inside a larger allocation whose bytes before and after it (and
the row padding of o) hold a fixed NaN bit pattern.  Every path of the library runs on query
lengths that end a Q-block early, exactly, one row late and at the Wan length: the per-chunk
tensor-core kernel (bulk-tensor store and reduce epilogue), the fused final chunk, the
one-launch form, the key-sink fold (fused and separate), the forced online fallback and the
CUDA-core kernel.  After each run the guard bytes must be bit-for-bit what they were, and
the outputs must match the oracle.  A write one row past a ragged tail, or past a head's last
row into the next allocation, changes a guard byte.
"""
import numpy as np
import pytest
import torch

import fixed_max_softmax_gb300 as fm
import oracle
import workloads
from tests.parity import Reference, f32_bar

pytestmark = pytest.mark.gpu

GUARD = 4096  # elements on each side (a multiple of 16 bytes for every element type)
PATTERN = {torch.float32: (torch.int32, 0x7FC0DEAD), torch.bfloat16: (torch.int16, 0x7FC1),
           torch.int32: (torch.int32, 0x5A5A5A5A), torch.uint8: (torch.uint8, 0xA5)}


class Guarded:
    """A tensor of `shape` inside a flat allocation with guard bands on both sides; with
    pad > 0 its last dimension is also padded by `pad` guarded elements per row."""

    def __init__(self, shape, dtype, dev, pad=0):
        self.shape, self.dtype, self.pad = tuple(shape), dtype, pad
        last = shape[-1] + pad
        inner = int(np.prod(shape[:-1], dtype=np.int64)) * last
        self.n_inner = inner
        it, pat = PATTERN[dtype]
        self.flat_bits = torch.full((inner + 2 * GUARD,), pat, dtype=it, device=dev)
        self.flat = self.flat_bits.view(dtype)
        body = self.flat[GUARD:GUARD + inner].view(*shape[:-1], last)
        self.t = body[..., :shape[-1]] if pad else body
        self.pattern = pat

    def intact(self):
        bits = self.flat_bits.cpu().numpy().astype(np.int64) & ((1 << (8 * self.flat_bits.element_size())) - 1)
        pat = self.pattern
        ok = bool(np.all(bits[:GUARD] == pat) and np.all(bits[GUARD + self.n_inner:] == pat))
        if self.pad:
            body = bits[GUARD:GUARD + self.n_inner].reshape(-1, self.shape[-1] + self.pad)
            ok = ok and bool(np.all(body[:, self.shape[-1]:] == pat))
        return ok

    def fully_written(self):
        """No element of the tensor itself still holds the fill pattern."""
        bits = self.flat_bits.cpu().numpy().astype(np.int64) & ((1 << (8 * self.flat_bits.element_size())) - 1)
        body = bits[GUARD:GUARD + self.n_inner].reshape(-1, self.shape[-1] + self.pad)[:, :self.shape[-1]]
        return bool(np.all(body != self.pattern))


def guarded_bounds(B, H, Sq, D, dev):
    """fm.Bounds whose device arrays live inside guard bands; returns (bounds, guards)."""
    nqb = (Sq + fm.FM_BLOCK_Q - 1) // fm.FM_BLOCK_Q
    b = fm.Bounds(B, H, Sq, D, dev)
    specs = {"m": ((B, H, nqb), torch.int32), "flag": ((B, H, nqb), torch.uint8),
             "qmax_sq": ((B, H, nqb), torch.float32), "kmax_sq": ((B, H), torch.float32),
             "kbar": ((B, H, D), torch.float32), "qkbar": ((B, H, Sq), torch.float32),
             "shift": ((B, H, Sq), torch.float32), "vmax_sq": ((1,), torch.float32),
             "sink_idx": ((B, H, fm.FM_MAX_SINKS), torch.int32),
             "sink_k": ((B, H, fm.FM_MAX_SINKS, D), torch.float32),
             "sink_v": ((B, H, fm.FM_MAX_SINKS, D), torch.float32)}
    guards = {}
    for name, (shape, dt) in specs.items():
        g = Guarded(shape, dt, dev)
        guards[name] = g
        setattr(b, name, g.t)
        setattr(b.out, name, g.t.data_ptr())
    return b, guards


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fixed_max_softmax_gb300 import build as fmbuild

    fmbuild.build()
    fm.load()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


N_KEYS = 700
CHUNKS = [(0, 350), (350, 350)]
PATHS = ["chunks", "fused", "fused_bf16_out", "one_launch", "sinks_fused", "sinks_separate", "online",
         "cuda_core"]
_refs = {}


def inputs_and_reference(Sq, dtype):
    """The sinks recipe (head 0 has four loud keys, head 25 none) at Sq query rows; oracle
    output, LSE and, for bf16, the scale-aware reference.  Computed once per (Sq, dtype)."""
    key = (Sq, dtype)
    if key not in _refs:
        q, k, v = workloads.make_inputs("sinks", device="cpu", heads=[0, 25], Sq=Sq, N=N_KEYS)
        q, k, v = q.to(dtype), k.to(dtype), v.to(dtype)
        o, lse = oracle.attention(q, k, v, return_lse=True)
        ref = None
        if dtype == torch.bfloat16:
            ob = oracle.bounds(q, k, v)
            ref = Reference(q, k, v, ob["shift"])
        _refs[key] = (q, k, v, o, lse, ref)
    return _refs[key]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("Sq", [1, 127, 129, 300, 75600])
def test_no_write_outside_any_buffer(dev, Sq, path):
    dtype = torch.float32 if path == "cuda_core" else torch.bfloat16
    q, k, v, o_ref, lse_ref, ref = inputs_and_reference(Sq, dtype)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    B, H, D = 1, 2, 128
    sinks = 2 if path.startswith("sinks") else 0
    opt = fm.opts(centering=path == "online", force_online=path == "online", sink_keys=sinks)
    bounds, guards = guarded_bounds(B, H, Sq, D, dev)
    acc_o = Guarded((B, H, Sq, D), torch.float32, dev)
    acc_sum = Guarded((B, H, Sq), torch.float32, dev)
    acc_max = Guarded((B, H, Sq), torch.float32, dev)
    lse = Guarded((B, H, Sq), torch.float32, dev)
    # o: contiguous fp32 on the separate-finalize paths; elsewhere rows padded by 32 guarded
    # columns (a row stride the fused epilogue can store to), fp32 or bf16
    if path in ("chunks", "sinks_separate"):
        out = Guarded((B, H, Sq, D), torch.float32, dev)
    else:
        out = Guarded((B, H, Sq, D), torch.bfloat16 if path == "fused_bf16_out" else torch.float32, dev, pad=32)
    guards.update(acc_o=acc_o, acc_sum=acc_sum, acc_max=acc_max, lse=lse, o=out)
    nbytes = fm.fm_bounds_workspace_size(B, H, N_KEYS, D)
    ws = Guarded((nbytes // 4 + 4,), torch.float32, dev)
    guards["workspace"] = ws
    fm.fm_bounds(qd, kd, vd, opt, bounds, ws.t)
    kc = [kd[:, :, s:s + n] for s, n in CHUNKS]
    vc = [vd[:, :, s:s + n] for s, n in CHUNKS]
    a = (acc_o.t, acc_sum.t, acc_max.t)
    if path in ("chunks", "sinks_separate", "cuda_core"):
        fm.fm_attn_chunk(qd, kc[0], vc[0], bounds, opt, *a, False)
        if path == "cuda_core":
            fm.fm_attn_chunk_final(qd, kc[1], vc[1], bounds, opt, *a, True, out.t, lse.t)
        else:
            fm.fm_attn_chunk(qd, kc[1], vc[1], bounds, opt, *a, True)
            fm.fm_fold_sinks(qd, bounds, opt, *a)
            fm.fm_finalize_lse(*a, out.t, lse.t)
    elif path == "one_launch":
        fm.fm_attn_chunks(qd, kc, vc, bounds, opt, *a, False, out.t, lse.t)
    else:  # fused final, with or without sinks, fixed-m or forced online
        fm.fm_attn_chunk(qd, kc[0], vc[0], bounds, opt, *a, False)
        fm.fm_attn_chunk_final(qd, kc[1], vc[1], bounds, opt, *a, True, out.t, lse.t)
    fm.fm_sync_status()
    broken = [name for name, g in guards.items() if not g.intact()]
    assert not broken, f"writes outside {broken} (Sq={Sq}, path={path})"
    # every bounds array the pass fills is written in full (each started as the fill pattern),
    # the key mean included: the oracle's with centering, zeros without
    unwritten = [n for n in ("m", "flag", "qmax_sq", "kmax_sq", "kbar", "qkbar", "shift", "vmax_sq")
                 if not guards[n].fully_written()]
    assert not unwritten, f"bounds arrays not fully written: {unwritten} (Sq={Sq}, path={path})"
    ob = oracle.bounds(q, k, v, centering=path == "online")
    np.testing.assert_allclose(bounds.kbar.cpu().numpy(), ob["kbar"], rtol=1e-5, atol=2e-6)
    got = out.t.float().cpu().numpy()
    if dtype == torch.float32:  # 1e-5, widened for the head whose keys are a hundred times louder
        for h in range(H):
            assert np.max(np.abs(got[:, h] - o_ref[:, h])) <= f32_bar(q[:, h], k[:, h]), h
    elif out.dtype == torch.bfloat16:  # o itself rounded to bf16: the absolute and relative bars
        err = np.max(np.abs(got - o_ref))
        assert err <= 2e-2 and err <= 1e-2 * np.max(np.abs(o_ref)), err
    else:
        ref.check(got, f"Sq={Sq} {path}")
    assert np.max(np.abs(lse.t.cpu().numpy() - lse_ref)) <= 1e-4 * max(1.0, float(np.max(np.abs(lse_ref))))
