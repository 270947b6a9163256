"""C-ABI checks that need no GPU: the library loads, exports exactly what include/fm.h
declares, and its host-side validation rejects bad calls with the documented codes
before touching the device (fake device pointers are never dereferenced)."""
import ctypes
import os
import re

import pytest
import torch

import fixed_max_softmax_gb300 as fm
from fixed_max_softmax_gb300 import build as fmbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 0x10000  # an aligned, never-dereferenced "device" address


@pytest.fixture(scope="module")
def lib():
    fmbuild.build()
    return fm.load()


def header_symbols():
    text = open(os.path.join(ROOT, "include", "fm.h")).read()
    return set(re.findall(r"FM_API\s+[\w\s\*]+?\b(fm_\w+)\s*\(", text))


def test_exports_every_declared_symbol(lib):
    declared = header_symbols()
    assert declared == set(fm.ABI_SYMBOLS)
    for name in declared:
        assert hasattr(lib, name), name


def test_exports_nothing_else():
    out = os.popen(f"nm -D --defined-only {fm.LIB_PATH}").read().split("\n")
    names = {ln.split()[-1] for ln in out if ln.strip() and " T " in ln}
    assert names == header_symbols()


def test_struct_layouts_match_header(tmp_path):
    """The ctypes mirrors of fm_tensor, fm_opts, fm_bounds_out and fm_host_buffers have the size
    and field offsets the C compiler gives the header's structs."""
    import subprocess
    structs = {"fm_tensor": fm.fm_tensor, "fm_opts": fm.fm_opts, "fm_bounds_out": fm.fm_bounds_out,
               "fm_host_buffers": fm.fm_host_buffers}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "fm.h"', "int main(void) {"]
    for name, cls in structs.items():
        lines.append(f'  printf("{name} size %zu\\n", sizeof({name}));')
        for f, _ in cls._fields_:
            lines.append(f'  printf("{name} {f} %zu\\n", offsetof({name}, {f}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    seen = 0
    for ln in out:
        if not ln.strip():
            continue
        name, field, val = ln.split()
        cls = structs[name]
        got = ctypes.sizeof(cls) if field == "size" else getattr(cls, field).offset
        assert got == int(val), (name, field, got, val)
        seen += 1
    assert seen == sum(len(c._fields_) + 1 for c in structs.values())


def test_version_and_workspace(lib):
    assert fm.fm_version() >> 16 == 1
    n = fm.fm_bounds_workspace_size(1, 40, 75600, 128)
    assert n > 0 and n % 256 == 0
    assert fm.fm_bounds_workspace_size(0, 0, 0, 128) >= 0


def fake(B, H, S, D, dtype=fm.FM_BF16, strides=None):
    t = fm.fm_tensor()
    t.ptr = FAKE
    t.dtype = dtype
    t.B, t.H, t.S, t.D = B, H, S, D
    st = strides or (H * S * D, S * D, D, 1)
    for i in range(4):
        t.stride[i] = st[i]
    return t


def call_bounds(lib, q, k, v, opt=None, out=None, ws=FAKE, ws_bytes=1 << 30):
    opt = opt or fm.opts()
    if out is None:
        out = fm.fm_bounds_out()
        for f in ("m", "flag", "qmax_sq", "kmax_sq", "kbar", "qkbar", "shift", "vmax_sq"):
            setattr(out, f, FAKE)
    return lib.fm_bounds(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), ctypes.byref(opt), ctypes.byref(out),
                         ws, ws_bytes, None)


def test_bounds_rejects_fp16_and_fp8(lib):
    for dt in (fm.FM_F16, fm.FM_F8E4M3, fm.FM_F8E5M2):
        rc = call_bounds(lib, fake(1, 2, 256, 128, dt), fake(1, 2, 256, 128, dt), fake(1, 2, 256, 128, dt))
        assert rc == fm.FM_ERR_DTYPE
        assert "fp16" in fm.fm_last_error()


def test_bounds_shape_and_support_errors(lib):
    q, k, v = fake(1, 2, 256, 128), fake(1, 2, 300, 128), fake(1, 2, 300, 128)
    assert call_bounds(lib, q, k, fake(1, 2, 299, 128)) == fm.FM_ERR_SHAPE          # k/v lengths
    assert call_bounds(lib, q, fake(2, 2, 300, 128), fake(2, 2, 300, 128)) == fm.FM_ERR_SHAPE  # batch
    assert call_bounds(lib, q, fake(1, 1, 300, 128), fake(1, 1, 300, 128)) == fm.FM_ERR_UNSUPPORTED  # GQA
    assert call_bounds(lib, fake(1, 2, 256, 96), fake(1, 2, 300, 96), fake(1, 2, 300, 96)) == fm.FM_ERR_UNSUPPORTED
    assert call_bounds(lib, q, fake(1, 2, 300, 128, fm.FM_F32), v) == fm.FM_ERR_DTYPE  # mixed types
    assert call_bounds(lib, q, k, v, ws_bytes=16) == fm.FM_ERR_ARG                   # workspace too small
    bad = fm.fm_bounds_out()
    for f in ("flag", "qmax_sq", "kmax_sq", "kbar", "qkbar", "shift", "vmax_sq"):
        setattr(bad, f, FAKE)
    assert call_bounds(lib, q, k, v, out=bad) == fm.FM_ERR_ARG


def good_bounds(B=1, H=2, Sq=256, D=128, N=300, centered=0, alpha=None):
    b = fm.fm_bounds_out()
    for f in ("m", "flag", "qmax_sq", "kmax_sq", "kbar", "qkbar", "shift", "vmax_sq"):
        setattr(b, f, FAKE)
    b.B, b.H, b.Sq, b.D = B, H, Sq, D
    b.n_qblocks = (Sq + 127) // 128
    b.N_total = N
    b.centered = centered
    b.alpha = alpha if alpha is not None else float(ctypes.c_float((1 / D ** 0.5) * 1.4426950408889634).value)
    b.dtype = fm.FM_BF16
    b.kv_seen = 0
    b.online_lock = -1
    b.magic = fm.FM_BOUNDS_MAGIC
    return b


def call_chunk(lib, b, nc=150, opt=None, accumulate=0, Sq=256):
    q, k, v = fake(1, 2, Sq, 128), fake(1, 2, nc, 128), fake(1, 2, nc, 128)
    opt = opt or fm.opts()
    return lib.fm_attn_chunk(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), ctypes.byref(b), ctypes.byref(opt),
                             FAKE, FAKE, FAKE, accumulate, None)


def test_chunk_bounds_mismatch(lib):
    b = good_bounds()
    b.magic = 0
    assert call_chunk(lib, b) == fm.FM_ERR_BOUNDS_MISMATCH
    # legacy / mis-shaped bounds: one Q-block count for another query length
    assert call_chunk(lib, good_bounds(Sq=128)) == fm.FM_ERR_BOUNDS_MISMATCH
    assert call_chunk(lib, good_bounds(H=1)) == fm.FM_ERR_BOUNDS_MISMATCH
    # matched pair: raw-key bounds may not serve centered logits (and vice versa)
    assert call_chunk(lib, good_bounds(centered=0), opt=fm.opts(centering=True)) == fm.FM_ERR_BOUNDS_MISMATCH
    assert "centering" in fm.fm_last_error()
    assert call_chunk(lib, good_bounds(centered=1), opt=fm.opts(centering=False)) == fm.FM_ERR_BOUNDS_MISMATCH
    # another softmax scale than the bounds were built with
    assert call_chunk(lib, good_bounds(), opt=fm.opts(softmax_scale=0.5)) == fm.FM_ERR_BOUNDS_MISMATCH
    # more keys than the bounds cover (C(N) would no longer hold)
    assert call_chunk(lib, good_bounds(N=100), nc=150) == fm.FM_ERR_BOUNDS_MISMATCH
    # accumulate before any init chunk
    assert call_chunk(lib, good_bounds(), accumulate=1) == fm.FM_ERR_BOUNDS_MISMATCH
    # force_online may not change inside one call
    b = good_bounds()
    b.online_lock = 0
    b.kv_seen = 100
    assert call_chunk(lib, b, nc=100, accumulate=1, opt=fm.opts(force_online=True)) == fm.FM_ERR_BOUNDS_MISMATCH


def test_chunk_kv_accounting(lib):
    b = good_bounds(N=300)
    b.online_lock = 0
    b.kv_seen = 200
    assert call_chunk(lib, b, nc=150, accumulate=1) == fm.FM_ERR_BOUNDS_MISMATCH  # 350 > 300
    assert b.kv_seen == 200  # a refused call changes nothing


def test_chunk_flag_values(lib):
    assert call_chunk(lib, good_bounds(), accumulate=2) == fm.FM_ERR_ARG
    o = fm.fm_opts(0.0, 2, 0, 0)
    assert call_chunk(lib, good_bounds(), opt=o) == fm.FM_ERR_ARG
    q, k = fake(1, 2, 256, 128), fake(1, 2, 300, 128)
    assert call_bounds(lib, q, k, k, opt=fm.fm_opts(0.0, 0, 0, 3)) == fm.FM_ERR_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device error path")
def test_valid_call_without_a_gpu_reports_cuda_error(lib):
    rc = call_chunk(lib, good_bounds())
    assert rc == fm.FM_ERR_CUDA


def test_finalize_validation(lib):
    o = fake(1, 2, 256, 128, fm.FM_F16)
    assert lib.fm_finalize(FAKE, FAKE, ctypes.byref(o), None) == fm.FM_ERR_DTYPE
    o = fake(1, 2, 256, 128)
    assert lib.fm_finalize(None, FAKE, ctypes.byref(o), None) == fm.FM_ERR_ARG
    assert lib.fm_finalize(FAKE + 4, FAKE, ctypes.byref(o), None) == fm.FM_ERR_ARG  # acc_o misaligned


def test_product_path_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "fixed_max_softmax_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"\bimport\s+oracle\b|\bfrom\s+oracle\b|fm_oracle|liboracle", text), f


def test_binding_fails_loudly_without_the_library(tmp_path):
    import importlib
    saved = fm._lib
    try:
        fm._lib = None
        with pytest.raises(fm.FMError):
            fm.load(str(tmp_path / "missing.so"))
    finally:
        fm._lib = saved
        importlib.invalidate_caches()


def test_noalloc_refuses_oversized_problems_on_the_host(lib):
    t = fake(1, 200, 75600, 128)
    out = fm.fm_bounds_out()
    rc = lib.fm_bounds_noalloc(ctypes.byref(t), ctypes.byref(t), ctypes.byref(t), ctypes.byref(fm.opts()),
                               ctypes.byref(out), None)
    assert rc == fm.FM_ERR_UNSUPPORTED and "scratch" in fm.fm_last_error()
    # invalid dtype is still reported as such by the shared validation
    t16 = fake(1, 2, 100, 128, fm.FM_F16)
    rc = lib.fm_bounds_noalloc(ctypes.byref(t16), ctypes.byref(t16), ctypes.byref(t16), ctypes.byref(fm.opts()),
                               ctypes.byref(out), None)
    assert rc in (fm.FM_ERR_DTYPE, fm.FM_ERR_CUDA)


def test_key_sink_validation(lib):
    q, k = fake(1, 2, 256, 128), fake(1, 2, 300, 128)
    # sink_keys outside [0, FM_MAX_SINKS]
    assert call_bounds(lib, q, k, k, opt=fm.opts(sink_keys=fm.FM_MAX_SINKS + 1)) == fm.FM_ERR_ARG
    assert call_bounds(lib, q, k, k, opt=fm.opts(sink_keys=-1)) == fm.FM_ERR_ARG
    # sinks asked for without the arrays to hold them
    assert call_bounds(lib, q, k, k, opt=fm.opts(sink_keys=2)) == fm.FM_ERR_ARG
    assert "sink" in fm.fm_last_error()
    # the chunks must skip exactly the keys the bounds left out of the key max
    b = good_bounds()
    assert call_chunk(lib, b, opt=fm.opts(sink_keys=2)) == fm.FM_ERR_BOUNDS_MISMATCH
    b.n_sink = 2
    assert call_chunk(lib, b) == fm.FM_ERR_BOUNDS_MISMATCH
    # nothing may follow the fold of the sinks
    b = good_bounds()
    b.n_sink, b.online_lock, b.kv_seen, b.sinks_folded = 2, 0, 100, 1
    b.sink_idx = b.sink_k = b.sink_v = FAKE
    assert call_chunk(lib, b, nc=100, accumulate=1, opt=fm.opts(sink_keys=2)) == fm.FM_ERR_BOUNDS_MISMATCH
    assert "fold" in fm.fm_last_error()


def test_fold_sinks_validation(lib):
    q = fake(1, 2, 256, 128)

    def fold(b, opt=None):
        return lib.fm_fold_sinks(ctypes.byref(q), ctypes.byref(b), ctypes.byref(opt or fm.opts(sink_keys=2)), FAKE,
                                 FAKE, FAKE, None)
    b = good_bounds()
    b.n_sink = 2
    b.sink_idx = b.sink_k = b.sink_v = FAKE
    assert fold(b) == fm.FM_ERR_BOUNDS_MISMATCH          # no chunk folded yet
    b.online_lock = 0
    assert fold(b, fm.opts(sink_keys=1)) == fm.FM_ERR_BOUNDS_MISMATCH  # other sink count
    b.sinks_folded = 1
    assert fold(b) == fm.FM_ERR_BOUNDS_MISMATCH          # folded twice
    b2 = good_bounds()
    b2.online_lock = 0
    assert lib.fm_fold_sinks(ctypes.byref(q), ctypes.byref(b2), ctypes.byref(fm.opts()), FAKE, FAKE, FAKE,
                             None) == fm.FM_OK           # no sinks: nothing to do, nothing enqueued


def test_plain_c_program_uses_the_abi(lib, tmp_path):
    """The boundary is a C ABI: a C program that includes only include/fm.h links against
    libfm.so and calls it (version, workspace size, a call refused on the host) with no
    Python in between."""
    import subprocess
    src = tmp_path / "use_fm.c"
    src.write_text(r'''
#include <stdio.h>
#include <string.h>
#include "fm.h"
int main(void) {
  size_t ws = 0;
  if (fm_bounds_workspace_size(1, 40, 75600, 128, &ws) != FM_OK || ws == 0) return 1;
  fm_tensor t;
  memset(&t, 0, sizeof t);
  t.ptr = (void *)0x10000;
  t.dtype = FM_F16;
  t.B = 1; t.H = 2; t.S = 64; t.D = 128;
  t.stride[0] = 2 * 64 * 128; t.stride[1] = 64 * 128; t.stride[2] = 128; t.stride[3] = 1;
  fm_opts o;
  memset(&o, 0, sizeof o);
  fm_bounds_out b;
  memset(&b, 0, sizeof b);
  int rc = fm_bounds(&t, &t, &t, &o, &b, NULL, 0, NULL);
  printf("%d %d %zu %s\n", fm_version() >> 16, rc, ws, fm_last_error());
  return rc == FM_ERR_DTYPE ? 0 : 2;
}
''')
    exe = tmp_path / "use_fm"
    libdir = os.path.dirname(fm.LIB_PATH)
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe), "-L", libdir,
                    "-lfm", f"-Wl,-rpath,{libdir}"], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, (r.stdout, r.stderr)
    major, rc, ws, *msg = r.stdout.split()
    assert int(major) == 1 and int(rc) == fm.FM_ERR_DTYPE and int(ws) == fm.fm_bounds_workspace_size(1, 40, 75600, 128)
    assert "fp16" in " ".join(msg)


def test_debug_build_exports_the_same_abi():
    """The debug build (-DFM_DEBUG, the kernels' index checks on) is the same C ABI: the same
    exported symbols and nothing else."""
    from fixed_max_softmax_gb300 import build as fmbuild

    dbg = fmbuild.build(debug=True)
    assert dbg == fm.DEBUG_LIB_PATH and os.path.exists(dbg)
    names = lambda p: {ln.split()[-1] for ln in os.popen(f"nm -D --defined-only {p}").read().split("\n")
                       if ln.strip() and ln.split()[-1].startswith("fm_")}
    assert names(dbg) == names(fm.LIB_PATH) == set(fm.ABI_SYMBOLS)
