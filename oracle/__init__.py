"""CPU oracle for fixed-m (const-max) attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import this package.  The product path (``fixed_max_softmax_gb300``) never does: it
shares no code, header, table or constant with this oracle.

The arithmetic lives in ``fm_oracle.c`` (plain fp64 C, OpenMP over rows); this module
only compiles it with gcc on first use, loads it with ctypes and marshals numpy arrays.
Sources and the reading of each step are in the C file's header:

* ``attention``  -- plain softmax attention (the exact result fixed-m reaches, by the
  shift invariance of softmax in "Kernel reference: ring_attention_const_max_fwd",
  section "What you should know before reading").
* ``constants`` / ``bounds`` -- C(N), W, gate, U, m (per Q-block or per row), the row
  shift and the eligibility flag from
  "feat(attention): fixed-m splash attention kernel with dynamic bounds and safety
  fallbacks", Summary ("Dynamic eligibility bounding", "Virtual K-centering"); with
  ``sink_keys``, the loudest keys left out of the key max ("Kernel reference:
  ring_attention_const_max_fwd", section "Adapting this kernel").
* ``attention_bf16p`` -- the same attention with the numerator's weights rounded to bf16
  at a given per-row shift: the bf16 reference that "Kernel reference:
  ring_attention_const_max_fwd", section "Adapting this kernel" (Validation), says to
  compare a kernel's error distribution against.
* ``fixed_m_emulate_f32`` -- fp32 fixed-m sum with an arbitrary shift and
  flush-to-zero, to demonstrate the failure modes the gate exists to prevent.

Nothing here is "parity unpinned" except the 0.882 softmax-mass figure that the
PR #477 page prints without its key set; the gate decision it illustrates is pinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

VMAX_DEFAULT = 256  # the V bound of the PR #477 commit message
BQ_DEFAULT = 128  # rows per Q-block (the granularity of m and of the flag)


def build(force: bool = False) -> str:
    """Compile fm_oracle.c into a shared library with gcc (OpenMP when available)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64 = ctypes.c_int64
        lib.fmo_ceil_log2.restype = ctypes.c_int
        lib.fmo_ceil_log2.argtypes = [i64]
        lib.fmo_constants.restype = None
        lib.fmo_constants.argtypes = [i64, i64, P, P, P]
        lib.fmo_num_threads.restype = ctypes.c_int
        lib.fmo_attention.restype = None
        lib.fmo_attention.argtypes = [P, P, P, i64, i64, i64, i64, ctypes.c_double, P, P, ctypes.c_int]
        lib.fmo_attention_bf16p.restype = None
        lib.fmo_attention_bf16p.argtypes = [P, P, P, i64, i64, i64, i64, ctypes.c_double, P, P, ctypes.c_int]
        lib.fmo_bounds.restype = None
        lib.fmo_bounds.argtypes = [P, P, P, i64, i64, i64, i64, i64, ctypes.c_double, ctypes.c_int,
                                   ctypes.c_int, i64, P, P, P, P, P, P, P, P, P, ctypes.c_int, P, P, P, i64, P, P]
        lib.fmo_fixed_m_emulate_f32.restype = None
        lib.fmo_fixed_m_emulate_f32.argtypes = [P, P, P, i64, i64, i64, ctypes.c_double, P, P, P, P,
                                                P, P]
        _lib = lib
        return lib


def _f64(x) -> np.ndarray:
    """Any array-like (numpy or a CPU torch tensor) -> C-contiguous float64 numpy."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().fmo_num_threads())


def ceil_log2(n: int) -> int:
    return int(_load().fmo_ceil_log2(int(n)))


def constants(n_total: int, vmax: int = VMAX_DEFAULT) -> tuple[int, int, int]:
    """(C, W, gate) for a total KV length n_total and V bound vmax."""
    c, w, g = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _load().fmo_constants(int(n_total), int(vmax), ctypes.byref(c), ctypes.byref(w), ctypes.byref(g))
    return c.value, w.value, g.value


def _as3(x) -> np.ndarray:
    a = _f64(x)
    if a.ndim == 4:
        a = a.reshape(a.shape[0] * a.shape[1], a.shape[2], a.shape[3])
    if a.ndim == 2:
        a = a[None]
    assert a.ndim == 3, a.shape
    return np.ascontiguousarray(a)


def attention(q, k, v, scale: float | None = None, threads: int = 0, return_lse: bool = False):
    """Plain softmax attention in fp64.

    q: [..., R, D] rows to evaluate; k, v: [..., N, D].  Leading dims ([B, H] or [G])
    must match.  Returns o with q's shape (and lse [..., R] if asked).
    """
    qa, ka, va = _as3(q), _as3(k), _as3(v)
    G, R, D = qa.shape
    N = ka.shape[1]
    assert ka.shape == (G, N, D) and va.shape == (G, N, D), (qa.shape, ka.shape, va.shape)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    o = np.zeros((G, R, D), dtype=np.float64)
    lse = np.zeros((G, R), dtype=np.float64) if return_lse else None
    _load().fmo_attention(_ptr(qa), _ptr(ka), _ptr(va), G, R, N, D, float(scale), _ptr(o), _ptr(lse),
                          int(threads))
    shape = tuple(np.shape(q)) if not hasattr(q, "shape") else tuple(q.shape)
    o = o.reshape(shape)
    if return_lse:
        return o, lse.reshape(shape[:-1])
    return o


def attention_bf16p(q, k, v, shift=None, scale: float | None = None, threads: int = 0):
    """Attention with bf16 P: the "bf16 reference" of "Kernel reference:
    ring_attention_const_max_fwd", section "Adapting this kernel" (Validation).

    Each numerator weight p_ij = 2^(z_ij - shift_i) (z = scale*log2(e)*q.k, base-2 units)
    is rounded to bf16's 8-bit significand; the denominator keeps the exact weights; fp64
    otherwise.  shift: [..., R] per-row base-2 shifts (e.g. bounds(...)["shift"] for the rows
    evaluated), or None for each row's max.  q: [..., R, D]; k, v: [..., N, D].
    """
    qa, ka, va = _as3(q), _as3(k), _as3(v)
    G, R, D = qa.shape
    N = ka.shape[1]
    assert ka.shape == (G, N, D) and va.shape == (G, N, D), (qa.shape, ka.shape, va.shape)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    sh = None
    if shift is not None:
        sh = np.ascontiguousarray(_f64(shift).reshape(G, R))
    o = np.zeros((G, R, D), dtype=np.float64)
    _load().fmo_attention_bf16p(_ptr(qa), _ptr(ka), _ptr(va), G, R, N, D, float(scale), _ptr(sh), _ptr(o),
                                int(threads))
    shape = tuple(np.shape(q)) if not hasattr(q, "shape") else tuple(q.shape)
    return o.reshape(shape)


def bounds(q, k, v, scale: float | None = None, centering: bool = False, dtype_safe: bool = True,
           vmax: int = VMAX_DEFAULT, bq: int = BQ_DEFAULT, per_row: bool = False, sink_keys: int = 0) -> dict:
    """Bounds of one fixed-m call in fp64 (norms, kbar, U, m, flag, C, W, gate).

    q: [B, H, Sq, D] (or [G, Sq, D]); k, v: [B, H, N, D] -- N is the TOTAL KV length
    over every chunk of the call.  Arrays come back with leading dims [B, H] when the
    inputs were 4-D.  sink_keys > 0 leaves that many loudest keys per head out of the key
    max ("sink_idx", ascending, padded with 2**31-1; "sink_gap" is the distance of the
    last sink's squared norm to the first kept one).
    """
    q4 = np.shape(q)
    qa, ka, va = _as3(q), _as3(k), _as3(v)
    G, Sq, D = qa.shape
    N = ka.shape[1]
    nqb = (Sq + bq - 1) // bq
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    qmax_sq = np.zeros((G, nqb))
    kbar = np.zeros((G, D))
    kmax_sq = np.zeros((G,))
    vmax_sq = np.zeros((1,))
    U = np.zeros((G, nqb))
    m = np.zeros((G, nqb), dtype=np.int32)
    flag = np.zeros((G, nqb), dtype=np.uint8)
    qkbar = np.zeros((G, Sq))
    U_row = np.zeros((G, Sq))
    m_row = np.zeros((G, Sq), dtype=np.int32)
    shift = np.zeros((G, Sq))
    consts = np.zeros((4,), dtype=np.int32)
    ns = int(sink_keys)
    sink_idx = np.zeros((G, max(ns, 1)), dtype=np.int32)
    sink_gap = np.zeros((G,))
    _load().fmo_bounds(_ptr(qa), _ptr(ka), _ptr(va), G, Sq, N, D, bq, float(scale), int(bool(centering)),
                       int(bool(dtype_safe)), int(vmax), _ptr(qmax_sq), _ptr(kbar), _ptr(kmax_sq),
                       _ptr(vmax_sq), _ptr(U), _ptr(m), _ptr(flag), _ptr(qkbar), _ptr(consts), int(bool(per_row)),
                       _ptr(U_row), _ptr(m_row), _ptr(shift), ns, _ptr(sink_idx), _ptr(sink_gap))
    lead = tuple(q4[:-2]) if len(q4) == 4 else (G,)
    # distance of U to the nearest integer and to the gate: where fp32 device sums can
    # legitimately round across an integer (the tie band of the parity tests)
    margin = np.minimum(np.abs(U - np.round(U)), np.abs(U - consts[2]))
    return {
        "qmax_sq": qmax_sq.reshape(lead + (nqb,)),
        "kbar": kbar.reshape(lead + (D,)),
        "kmax_sq": kmax_sq.reshape(lead),
        "vmax_sq": float(vmax_sq[0]),
        "U": U.reshape(lead + (nqb,)),
        "m": m.reshape(lead + (nqb,)),
        "flag": flag.reshape(lead + (nqb,)),
        "qkbar": qkbar.reshape(lead + (Sq,)),
        "U_row": U_row.reshape(lead + (Sq,)),
        "m_row": m_row.reshape(lead + (Sq,)),
        "shift": shift.reshape(lead + (Sq,)),
        "margin_row": np.minimum(np.abs(U_row - np.round(U_row)), np.abs(U_row - consts[2])).reshape(lead + (Sq,)),
        "margin": margin.reshape(lead + (nqb,)),
        "C": int(consts[0]),
        "W": int(consts[1]),
        "gate": int(consts[2]),
        "v_ok": bool(consts[3]),
        "alpha": float(scale) * float(np.log2(np.e)),
        "N": int(N),
        "sink_idx": sink_idx[:, :ns].reshape(lead + (ns,)),
        "sink_gap": sink_gap.reshape(lead),
    }


def fixed_m_emulate_f32(q, k, v, m_row, scale: float | None = None, kbar=None) -> dict:
    """fp32 fixed-m accumulation of one problem with an arbitrary per-row shift.

    q: [R, D], k, v: [N, D], m_row: [R] (base-2 units).  Returns acc_o, acc_sum
    (float32), the ratio o = acc_o/acc_sum, and per-row counts of flushed
    (subnormal -> 0) and overflowing terms.
    """
    qa = _f64(q).reshape(-1, np.shape(q)[-1])
    ka = _f64(k)
    va = _f64(v)
    R, D = qa.shape
    N = ka.shape[0]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    mr = _f64(m_row).reshape(R)
    kb = None if kbar is None else _f64(kbar).reshape(D)
    acc_o = np.zeros((R, D), dtype=np.float32)
    acc_sum = np.zeros((R,), dtype=np.float32)
    nf = np.zeros((R,), dtype=np.int64)
    nov = np.zeros((R,), dtype=np.int64)
    _load().fmo_fixed_m_emulate_f32(_ptr(qa), _ptr(ka), _ptr(va), R, N, D, float(scale), _ptr(kb), _ptr(mr),
                                    _ptr(acc_o), _ptr(acc_sum), _ptr(nf), _ptr(nov))
    with np.errstate(divide="ignore", invalid="ignore"):
        o = acc_o.astype(np.float64) / acc_sum.astype(np.float64)[:, None]
    return {"acc_o": acc_o, "acc_sum": acc_sum, "o": o, "n_flushed": nf, "n_overflow": nov}
