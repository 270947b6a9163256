"""fixed_max_softmax_gb300 -- fixed-m (const-max) attention forward on GB300.

A thin ctypes binding of ``libfm.so`` (C ABI: ``include/fm.h``).  Every step of the
path -- bounds, chunk folding, finalize -- runs in the library's CUDA kernels; this
module only marshals torch tensors into ``fm_tensor`` descriptors, passes raw
pointers and the current CUDA stream, and turns error codes into exceptions.
PyTorch provides device memory and streams and nothing else.

Functions with the ABI's names (same arguments, torch tensors in place of pointers):
``fm_bounds_workspace_size``, ``fm_bounds``, ``fm_bounds_noalloc``, ``fm_attn_chunk``,
``fm_attn_chunk_final``, ``fm_attn_chunks``, ``fm_fold_sinks``, ``fm_finalize``,
``fm_finalize_lse``, ``fm_sync_status``,
``fm_probe_wait_timeout``,
``fm_last_error``, ``fm_version``.

``FixedMAttention`` owns the buffers of one problem shape and runs the whole path
(bounds, one ``fm_attn_chunk`` per KV chunk, finalize); ``attention()`` is the
one-call form.

There is no CPU path: if the library is not built, ``load()`` raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libfm.so")
DEBUG_LIB_PATH = os.path.join(_HERE, "_build_debug", "libfm.so")  # build(debug=True): kernel index checks

FM_F32, FM_BF16, FM_F16, FM_F8E4M3, FM_F8E5M2 = 0, 1, 2, 3, 4
FM_OK, FM_ERR_ARG, FM_ERR_SHAPE, FM_ERR_DTYPE, FM_ERR_UNSUPPORTED = 0, 1, 2, 3, 4
FM_ERR_BOUNDS_MISMATCH, FM_ERR_CUDA, FM_ERR_TIMEOUT, FM_ERR_INDEX = 5, 6, 7, 8
FM_BOUNDS_MAGIC = 0x314D4246
FM_BOUNDS_LOCAL_MAGIC = 0x314C4246
FM_BLOCK_Q = 128
ERROR_NAMES = {0: "FM_OK", 1: "FM_ERR_ARG", 2: "FM_ERR_SHAPE", 3: "FM_ERR_DTYPE", 4: "FM_ERR_UNSUPPORTED",
               5: "FM_ERR_BOUNDS_MISMATCH", 6: "FM_ERR_CUDA", 7: "FM_ERR_TIMEOUT", 8: "FM_ERR_INDEX"}
ABI_SYMBOLS = ("fm_bounds_workspace_size", "fm_bounds", "fm_attn_chunk", "fm_finalize", "fm_sync_status",
               "fm_last_error", "fm_version", "fm_bounds_noalloc", "fm_finalize_lse", "fm_probe_wait_timeout",
               "fm_attn_chunk_final", "fm_attn_chunks", "fm_fold_sinks", "fm_ring_stats_bytes", "fm_ring_key_sums",
               "fm_bounds_local", "fm_bounds_combine", "fm_attention_host")
FM_MAX_CHUNKS = 8
FM_MAX_SINKS = 8
FM_NOALLOC_SCRATCH_BYTES = 4 << 20


class FMError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERROR_NAMES.get(code, code)}: {msg}")
        self.code = code


class fm_tensor(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("B", ctypes.c_int64), ("H", ctypes.c_int64), ("S", ctypes.c_int64), ("D", ctypes.c_int64),
                ("stride", ctypes.c_int64 * 4)]


class fm_opts(ctypes.Structure):
    _fields_ = [("softmax_scale", ctypes.c_float), ("centering", ctypes.c_int32),
                ("force_online", ctypes.c_int32), ("per_row", ctypes.c_int32), ("sink_keys", ctypes.c_int32),
                ("schedule", ctypes.c_int32)]


class fm_bounds_out(ctypes.Structure):
    _fields_ = [("m", ctypes.c_void_p), ("flag", ctypes.c_void_p), ("qmax_sq", ctypes.c_void_p),
                ("kmax_sq", ctypes.c_void_p), ("kbar", ctypes.c_void_p), ("qkbar", ctypes.c_void_p),
                ("shift", ctypes.c_void_p), ("vmax_sq", ctypes.c_void_p),
                ("sink_idx", ctypes.c_void_p), ("sink_k", ctypes.c_void_p), ("sink_v", ctypes.c_void_p),
                ("B", ctypes.c_int64), ("H", ctypes.c_int64), ("Sq", ctypes.c_int64), ("D", ctypes.c_int64),
                ("n_qblocks", ctypes.c_int64), ("N_total", ctypes.c_int64),
                ("C", ctypes.c_int32), ("W", ctypes.c_int32), ("gate", ctypes.c_int32),
                ("centered", ctypes.c_int32), ("per_row", ctypes.c_int32), ("n_sink", ctypes.c_int32),
                ("alpha", ctypes.c_float), ("dtype", ctypes.c_int32),
                ("kv_seen", ctypes.c_int64), ("next_key_offset", ctypes.c_int64), ("online_lock", ctypes.c_int32),
                ("sinks_folded", ctypes.c_int32),
                ("magic", ctypes.c_uint32)]


class fm_host_buffers(ctypes.Structure):
    _fields_ = [("q", fm_tensor * 2), ("k", fm_tensor * 2), ("v", fm_tensor * 2), ("o", fm_tensor * 2),
                ("acc_o", ctypes.c_void_p), ("acc_sum", ctypes.c_void_p), ("acc_max", ctypes.c_void_p),
                ("bounds", ctypes.POINTER(fm_bounds_out)), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t)]


_lib = None


def load(path: str | None = None):
    """Load libfm.so (build it first with fixed_max_softmax_gb300.build.build())."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise FMError(FM_ERR_CUDA, f"{p} is missing: the CUDA library is not built "
                                   "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(p)
    P, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.fm_bounds_workspace_size.argtypes = [i64, i64, i64, i64, ctypes.POINTER(ctypes.c_size_t)]
    lib.fm_bounds.argtypes = [P, P, P, P, P, P, ctypes.c_size_t, P]
    lib.fm_attn_chunk.argtypes = [P, P, P, P, P, P, P, P, ctypes.c_int, P]
    lib.fm_finalize.argtypes = [P, P, P, P]
    lib.fm_bounds_noalloc.argtypes = [P, P, P, P, P, P]
    lib.fm_finalize_lse.argtypes = [P, P, P, P, P, P]
    lib.fm_probe_wait_timeout.argtypes = [ctypes.c_uint, P]
    lib.fm_attn_chunk_final.argtypes = [P, P, P, P, P, P, P, P, ctypes.c_int, P, P, P]
    lib.fm_attn_chunks.argtypes = [P, P, P, ctypes.c_int, P, P, P, P, P, ctypes.c_int, P, P, P]
    lib.fm_fold_sinks.argtypes = [P, P, P, P, P, P, P]
    lib.fm_ring_stats_bytes.argtypes = [i64, i64, i64, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]
    lib.fm_ring_key_sums.argtypes = [P, P, P, ctypes.c_size_t, P]
    lib.fm_bounds_local.argtypes = [P, P, P, i64, i64, P, P, P, P, P, ctypes.c_size_t, P]
    lib.fm_bounds_combine.argtypes = [P, ctypes.c_int, P, P, P]
    lib.fm_attention_host.argtypes = [P, P, P, P, ctypes.c_int, P, ctypes.c_int, P, P, P]
    lib.fm_sync_status.argtypes = [P]
    lib.fm_last_error.restype = ctypes.c_char_p
    lib.fm_last_error.argtypes = []
    lib.fm_version.argtypes = []
    for name in ("fm_bounds_workspace_size", "fm_bounds", "fm_attn_chunk", "fm_finalize", "fm_sync_status",
                 "fm_version", "fm_bounds_noalloc", "fm_finalize_lse", "fm_probe_wait_timeout",
                 "fm_attn_chunk_final", "fm_attn_chunks", "fm_fold_sinks", "fm_ring_stats_bytes", "fm_ring_key_sums",
                 "fm_bounds_local", "fm_bounds_combine", "fm_attention_host"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


_DTYPES = {torch.float32: FM_F32, torch.bfloat16: FM_BF16, torch.float16: FM_F16}
if hasattr(torch, "float8_e4m3fn"):
    _DTYPES[torch.float8_e4m3fn] = FM_F8E4M3
if hasattr(torch, "float8_e5m2"):
    _DTYPES[torch.float8_e5m2] = FM_F8E5M2


def tensor(t: torch.Tensor) -> fm_tensor:
    """Describe a 4-D [B, H, S, D] torch tensor (any strides) as an fm_tensor."""
    if t.dim() != 4:
        raise FMError(FM_ERR_SHAPE, f"expected a 4-D [B, H, S, D] tensor, got shape {tuple(t.shape)}")
    d = fm_tensor()
    d.ptr = t.data_ptr() or None
    d.dtype = _DTYPES.get(t.dtype, -1)
    d.B, d.H, d.S, d.D = t.shape
    for i, s in enumerate(t.stride()):
        d.stride[i] = s
    return d


FM_SCHEDULE_AUTO, FM_SCHEDULE_GRID, FM_SCHEDULE_PERSISTENT = 0, 1, 2
SCHEDULES = {"auto": FM_SCHEDULE_AUTO, "grid": FM_SCHEDULE_GRID, "persistent": FM_SCHEDULE_PERSISTENT}


def opts(softmax_scale: float = 0.0, centering: bool = False, force_online: bool = False,
         per_row: bool = False, sink_keys: int = 0, schedule="auto") -> fm_opts:
    sched = SCHEDULES[schedule] if isinstance(schedule, str) else int(schedule)
    return fm_opts(float(softmax_scale), int(bool(centering)), int(bool(force_online)), int(bool(per_row)),
                   int(sink_keys), sched)


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(rc: int):
    if rc != FM_OK:
        raise FMError(rc, load().fm_last_error().decode())
    return rc


def fm_version() -> int:
    return load().fm_version()


def fm_last_error() -> str:
    return load().fm_last_error().decode()


def fm_bounds_workspace_size(B: int, H: int, N_total: int, D: int) -> int:
    n = ctypes.c_size_t()
    _check(load().fm_bounds_workspace_size(B, H, N_total, D, ctypes.byref(n)))
    return n.value


class Bounds:
    """Device arrays of one fm_bounds_out (allocated with torch) plus the struct itself."""

    def __init__(self, B: int, H: int, Sq: int, D: int, device):
        nqb = (Sq + FM_BLOCK_Q - 1) // FM_BLOCK_Q
        kw = dict(device=device)
        self.m = torch.zeros(B, H, nqb, dtype=torch.int32, **kw)
        self.flag = torch.zeros(B, H, nqb, dtype=torch.uint8, **kw)
        self.qmax_sq = torch.zeros(B, H, nqb, dtype=torch.float32, **kw)
        self.kmax_sq = torch.zeros(B, H, dtype=torch.float32, **kw)
        self.kbar = torch.zeros(B, H, D, dtype=torch.float32, **kw)
        self.qkbar = torch.zeros(B, H, max(Sq, 1), dtype=torch.float32, **kw)
        self.shift = torch.zeros(B, H, max(Sq, 1), dtype=torch.float32, **kw)
        self.vmax_sq = torch.zeros(1, dtype=torch.float32, **kw)
        self.sink_idx = torch.zeros(B, H, FM_MAX_SINKS, dtype=torch.int32, **kw)
        self.sink_k = torch.zeros(B, H, FM_MAX_SINKS, D, dtype=torch.float32, **kw)
        self.sink_v = torch.zeros(B, H, FM_MAX_SINKS, D, dtype=torch.float32, **kw)
        self.out = fm_bounds_out()
        self.out.m, self.out.flag = self.m.data_ptr(), self.flag.data_ptr()
        self.out.qmax_sq, self.out.kmax_sq = self.qmax_sq.data_ptr(), self.kmax_sq.data_ptr()
        self.out.kbar, self.out.qkbar, self.out.vmax_sq = (self.kbar.data_ptr(), self.qkbar.data_ptr(),
                                                           self.vmax_sq.data_ptr())
        self.out.shift = self.shift.data_ptr()
        self.out.sink_idx, self.out.sink_k, self.out.sink_v = (self.sink_idx.data_ptr(), self.sink_k.data_ptr(),
                                                               self.sink_v.data_ptr())


def fm_bounds(q, k_full, v_full, opt: fm_opts, bounds: Bounds, workspace: torch.Tensor | None, stream=None):
    tq, tk, tv = tensor(q), tensor(k_full), tensor(v_full)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return _check(load().fm_bounds(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv), ctypes.byref(opt),
                                   ctypes.byref(bounds.out), _ptr(workspace), ws_bytes, _stream(stream)))


def fm_bounds_noalloc(q, k_full, v_full, opt: fm_opts, bounds: Bounds, stream=None):
    """fm_bounds without a workspace: the library's static device scratch is used instead
    (for callers that cannot allocate; see include/fm.h)."""
    tq, tk, tv = tensor(q), tensor(k_full), tensor(v_full)
    return _check(load().fm_bounds_noalloc(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv), ctypes.byref(opt),
                                           ctypes.byref(bounds.out), _stream(stream)))


def fm_ring_stats_bytes(B: int, H: int, D: int, sink_keys: int = 0) -> int:
    n = ctypes.c_size_t()
    _check(load().fm_ring_stats_bytes(B, H, D, int(sink_keys), ctypes.byref(n)))
    return n.value


def fm_ring_key_sums(k_shard, ksum, workspace, stream=None):
    """ksum [B, H, D] f32 <- the sums of this rank's keys (step 1 of the ring bounds)."""
    tk = tensor(k_shard)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return _check(load().fm_ring_key_sums(ctypes.byref(tk), _ptr(ksum), _ptr(workspace), ws_bytes, _stream(stream)))


def fm_bounds_local(q, k_shard, v_shard, key_offset: int, N_total: int, ksum_total, opt: fm_opts, bounds: Bounds,
                    stats, workspace, stream=None):
    """This rank's part of the bounds: bounds' query-side arrays and its statistics block (step 2)."""
    tq, tk, tv = tensor(q), tensor(k_shard), tensor(v_shard)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return _check(load().fm_bounds_local(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv), int(key_offset),
                                         int(N_total), _ptr(ksum_total), ctypes.byref(opt), ctypes.byref(bounds.out),
                                         _ptr(stats), _ptr(workspace), ws_bytes, _stream(stream)))


def fm_bounds_combine(stats_all, n_ranks: int, opt: fm_opts, bounds: Bounds, stream=None):
    """Every rank's statistics blocks (rank order) -> the rest of the bounds (step 3)."""
    return _check(load().fm_bounds_combine(_ptr(stats_all), int(n_ranks), ctypes.byref(opt), ctypes.byref(bounds.out),
                                           _stream(stream)))


def fm_attn_chunk(q, k_chunk, v_chunk, bounds: Bounds, opt: fm_opts, acc_o, acc_sum, acc_max,
                  accumulate: bool, stream=None):
    tq, tk, tv = tensor(q), tensor(k_chunk), tensor(v_chunk)
    return _check(load().fm_attn_chunk(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv),
                                       ctypes.byref(bounds.out), ctypes.byref(opt), _ptr(acc_o), _ptr(acc_sum),
                                       _ptr(acc_max), int(bool(accumulate)), _stream(stream)))


def fm_attn_chunk_final(q, k_chunk, v_chunk, bounds: Bounds, opt: fm_opts, acc_o, acc_sum, acc_max,
                        accumulate: bool, o_out, lse=None, stream=None):
    tq, tk, tv, to = tensor(q), tensor(k_chunk), tensor(v_chunk), tensor(o_out)
    return _check(load().fm_attn_chunk_final(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv),
                                             ctypes.byref(bounds.out), ctypes.byref(opt), _ptr(acc_o),
                                             _ptr(acc_sum), _ptr(acc_max), int(bool(accumulate)), ctypes.byref(to),
                                             _ptr(lse), _stream(stream)))


def fm_attn_chunks(q, k_chunks, v_chunks, bounds: Bounds, opt: fm_opts, acc_o, acc_sum, acc_max,
                   accumulate: bool, o_out=None, lse=None, stream=None):
    """Fold a list of consecutive KV chunks in one pass (and normalise into o_out if given)."""
    n = len(k_chunks)
    ks = (fm_tensor * n)(*[tensor(t) for t in k_chunks])
    vs = (fm_tensor * n)(*[tensor(t) for t in v_chunks])
    to = tensor(o_out) if o_out is not None else None
    return _check(load().fm_attn_chunks(ctypes.byref(tensor(q)), ks, vs, n, ctypes.byref(bounds.out),
                                        ctypes.byref(opt), _ptr(acc_o), _ptr(acc_sum), _ptr(acc_max),
                                        int(bool(accumulate)), None if to is None else ctypes.byref(to), _ptr(lse),
                                        _stream(stream)))


def fm_fold_sinks(q, bounds: Bounds, opt: fm_opts, acc_o, acc_sum, acc_max, stream=None):
    """Merge the key sinks set aside by fm_bounds back into the accumulators (after the last
    chunk, before fm_finalize); a no-op without sinks."""
    tq = tensor(q)
    return _check(load().fm_fold_sinks(ctypes.byref(tq), ctypes.byref(bounds.out), ctypes.byref(opt), _ptr(acc_o),
                                       _ptr(acc_sum), _ptr(acc_max), _stream(stream)))


def fm_finalize(acc_o, acc_sum, o_out, stream=None):
    to = tensor(o_out)
    return _check(load().fm_finalize(_ptr(acc_o), _ptr(acc_sum), ctypes.byref(to), _stream(stream)))


def fm_finalize_lse(acc_o, acc_sum, acc_max, o_out, lse, stream=None):
    to = tensor(o_out)
    return _check(load().fm_finalize_lse(_ptr(acc_o), _ptr(acc_sum), _ptr(acc_max), ctypes.byref(to), _ptr(lse),
                                         _stream(stream)))


def fm_sync_status(stream=None):
    return _check(load().fm_sync_status(_stream(stream)))


def fm_probe_wait_timeout(timeout_ms: int, stream=None):
    return _check(load().fm_probe_wait_timeout(int(timeout_ms), _stream(stream)))


class FixedMAttention:
    """Buffers and the call sequence of one fixed-m attention forward of a fixed shape.

    forward(q, k, v, chunks) runs fm_bounds over all of K/V, one fm_attn_chunk per
    (start, length) slice of the key sequence (the ring's steps, sequentially) and writes
    `out` (fp32 or the input dtype): by default the last chunk goes through
    fm_attn_chunk_final (fold and normalise in one pass); fused_final=False uses a separate
    fm_finalize.  one_launch=True folds all chunks with fm_attn_chunks instead (one launch per
    FM_MAX_CHUNKS chunks, accumulators on chip across them).  with_lse=True also fills
    `lse` [B, H, Sq] (natural log).  sink_keys > 0 leaves that many of each head's loudest
    keys out of the key max; they are folded back exactly before the normalise.  schedule:
    "auto", "grid" or "persistent" (fm_opts.schedule; the same bits either way).
    """

    def __init__(self, B, H, Sq, N, D, device="cuda", centering=False, softmax_scale=0.0,
                 force_online=False, out_dtype=torch.float32, per_row=False, sink_keys=0, schedule="auto"):
        self.shape = (B, H, Sq, N, D)
        self.opt = opts(softmax_scale, centering, force_online, per_row, sink_keys, schedule)
        self.bounds = Bounds(B, H, Sq, D, device)
        nbytes = fm_bounds_workspace_size(B, H, N, D)
        self.workspace = torch.empty(max(nbytes, 16) // 4 + 4, dtype=torch.float32, device=device)
        self.acc_o = torch.empty(B, H, Sq, D, dtype=torch.float32, device=device)
        self.acc_sum = torch.empty(B, H, Sq, dtype=torch.float32, device=device)
        self.acc_max = torch.empty(B, H, Sq, dtype=torch.float32, device=device)
        self.out = torch.empty(B, H, Sq, D, dtype=out_dtype, device=device)
        self.lse = None

    def forward(self, q, k, v, chunks=None, stream=None, with_lse=False, fused_final=True, one_launch=False):
        N = k.shape[2]
        chunks = [(0, N)] if chunks is None else chunks
        fm_bounds(q, k, v, self.opt, self.bounds, self.workspace, stream)
        if with_lse and self.lse is None:
            self.lse = torch.empty(self.acc_sum.shape, dtype=torch.float32, device=self.acc_sum.device)
        lse = self.lse if with_lse else None
        if one_launch:  # every chunk (up to FM_MAX_CHUNKS per call) and the normalise in one pass
            for g0 in range(0, len(chunks), FM_MAX_CHUNKS):
                grp = chunks[g0:g0 + FM_MAX_CHUNKS]
                last = g0 + FM_MAX_CHUNKS >= len(chunks)
                if any(grp[i][0] + grp[i][1] != grp[i + 1][0] for i in range(len(grp) - 1)):
                    raise ValueError("one_launch folds consecutive key ranges only")
                self.bounds.out.next_key_offset = grp[0][0]
                fm_attn_chunks(q, [k[:, :, s:s + n] for s, n in grp], [v[:, :, s:s + n] for s, n in grp],
                               self.bounds, self.opt, self.acc_o, self.acc_sum, self.acc_max, g0 > 0,
                               self.out if last else None, lse if last else None, stream)
            return self.out
        for i, (s, n) in enumerate(chunks):
            kc, vc = k[:, :, s:s + n], v[:, :, s:s + n]
            self.bounds.out.next_key_offset = s  # the chunk's global key offset: any order works
            if fused_final and i == len(chunks) - 1:
                fm_attn_chunk_final(q, kc, vc, self.bounds, self.opt, self.acc_o, self.acc_sum, self.acc_max, i > 0,
                                    self.out, lse, stream)
                return self.out
            fm_attn_chunk(q, kc, vc, self.bounds, self.opt, self.acc_o, self.acc_sum, self.acc_max, i > 0, stream)
        fm_fold_sinks(q, self.bounds, self.opt, self.acc_o, self.acc_sum, self.acc_max, stream)
        if with_lse:
            fm_finalize_lse(self.acc_o, self.acc_sum, self.acc_max, self.out, self.lse, stream)
        else:
            fm_finalize(self.acc_o, self.acc_sum, self.out, stream)
        return self.out

    __call__ = forward


def attention(q, k, v, chunks=None, centering=False, softmax_scale=0.0, force_online=False,
              out_dtype=torch.float32, stream=None, per_row=False, sink_keys=0):
    """One-call fixed-m attention forward: returns o [B, H, Sq, D]."""
    B, H, Sq, D = q.shape
    fa = FixedMAttention(B, H, Sq, k.shape[2], D, q.device, centering, softmax_scale, force_online, out_dtype,
                         per_row, sink_keys)
    return fa.forward(q, k, v, chunks, stream).clone()


class HostPipeline:
    """Fixed-m attention over a stream of batches that live in (pinned) host memory, through
    fm_attention_host: batch i+1's inputs are copied to the device on one stream while batch i
    computes on another, and batch i-1's output is read back on a third.  Every batch still makes
    the full host -> device -> host round trip, but the copies hide behind the kernels.  Two
    device copies of the inputs and of the output alternate between batches; the bounds,
    accumulators and workspace of `fa` are reused in order.
    """

    def __init__(self, fa: FixedMAttention, in_dtype, device="cuda"):
        B, H, Sq, N, D = fa.shape
        self.fa = fa
        self.device = torch.device(device)
        self.q = [torch.empty(B, H, Sq, D, dtype=in_dtype, device=device) for _ in range(2)]
        self.k = [torch.empty(B, H, N, D, dtype=in_dtype, device=device) for _ in range(2)]
        self.v = [torch.empty(B, H, N, D, dtype=in_dtype, device=device) for _ in range(2)]
        self.o = [torch.empty_like(fa.out) for _ in range(2)]
        self.streams = [torch.cuda.Stream(device=device) for _ in range(3)]
        self.dev = fm_host_buffers()
        for i in range(2):
            self.dev.q[i], self.dev.k[i], self.dev.v[i], self.dev.o[i] = (tensor(self.q[i]), tensor(self.k[i]),
                                                                          tensor(self.v[i]), tensor(self.o[i]))
        self.dev.acc_o, self.dev.acc_sum, self.dev.acc_max = (fa.acc_o.data_ptr(), fa.acc_sum.data_ptr(),
                                                              fa.acc_max.data_ptr())
        self.dev.bounds = ctypes.pointer(fa.bounds.out)
        self.dev.workspace = fa.workspace.data_ptr()
        self.dev.workspace_bytes = fa.workspace.numel() * fa.workspace.element_size()

    def run(self, batches, chunks=None):
        """batches: a list of (q_host, k_host, v_host, o_host); o_host is filled.  chunks: the
        (start, length) key ranges, consecutive from 0.  Returns when every output is back in
        host memory."""
        batches = list(batches)
        N = self.k[0].shape[2]
        chunks = [(0, N)] if chunks is None else chunks
        if [s for s, _ in chunks] != [sum(n for _, n in chunks[:i]) for i in range(len(chunks))]:
            raise ValueError("chunks must be consecutive key ranges from 0")
        n = len(batches)
        qs = (fm_tensor * max(n, 1))(*[tensor(b[0]) for b in batches])
        ks = (fm_tensor * max(n, 1))(*[tensor(b[1]) for b in batches])
        vs = (fm_tensor * max(n, 1))(*[tensor(b[2]) for b in batches])
        os_ = (fm_tensor * max(n, 1))(*[tensor(b[3]) for b in batches])
        lens = (ctypes.c_int64 * len(chunks))(*[c for _, c in chunks])
        st = (ctypes.c_void_p * 3)(*[s.cuda_stream for s in self.streams])
        return _check(load().fm_attention_host(qs, ks, vs, os_, n, lens, len(chunks), ctypes.byref(self.fa.opt),
                                               ctypes.byref(self.dev), st))
