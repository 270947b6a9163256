"""fm_bounds_noalloc: the bounds pass for callers that cannot allocate device memory.

Some callers plan all of their device memory before they run (an inference engine that
reserves its arena up front, a plug-in living in another framework's memory pool) or
must keep cudaMalloc's implicit device synchronisation off a latency-critical stream.
For them the library keeps the bounds pass's scratch in a static device array instead
of a caller workspace.  These tests call that entry point through the C ABI and check
that it gives what fm_bounds gives, on two calls in a row (the array keeps the previous
call's contents, which must not matter), and that a problem too large for the array is
refused.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import fixed_max_softmax_gb300 as fm
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fixed_max_softmax_gb300 import build as fmbuild

    fmbuild.build()
    torch.cuda.set_device(0)
    return fm.load()


def bounds_both_ways(lib, q, k, v, centering):
    """Run fm_bounds (torch workspace) and fm_bounds_noalloc (static scratch) via the C ABI."""
    B, H, Sq, D = q.shape
    N = k.shape[2]
    opt = fm.opts(centering=centering)
    tq, tk, tv = fm.tensor(q), fm.tensor(k), fm.tensor(v)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ref = fm.Bounds(B, H, Sq, D, q.device)
    ws_bytes = fm.fm_bounds_workspace_size(B, H, N, D)
    ws = torch.empty(ws_bytes // 4 + 4, dtype=torch.float32, device=q.device)
    rc = lib.fm_bounds(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv), ctypes.byref(opt),
                       ctypes.byref(ref.out), ctypes.c_void_p(ws.data_ptr()), ws.numel() * 4, stream)
    assert rc == fm.FM_OK, fm.fm_last_error()
    got = fm.Bounds(B, H, Sq, D, q.device)
    rc = lib.fm_bounds_noalloc(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv), ctypes.byref(opt),
                               ctypes.byref(got.out), stream)
    assert rc == fm.FM_OK, fm.fm_last_error()
    assert lib.fm_sync_status(stream) == fm.FM_OK, fm.fm_last_error()
    return ref, got


def assert_same(ref, got):
    # integer outputs bit-exact; the reductions are fixed-order, so floats match exactly too
    # (the tolerance the parity tests use for them is kept as the bar)
    assert torch.equal(ref.m, got.m)
    assert torch.equal(ref.flag, got.flag)
    for name in ("qmax_sq", "kmax_sq", "kbar", "qkbar", "shift", "vmax_sq"):
        a, b = getattr(ref, name).cpu().numpy(), getattr(got, name).cpu().numpy()
        np.testing.assert_allclose(b, a, rtol=2e-5, atol=2e-6, err_msg=name)
    for f in ("B", "H", "Sq", "D", "n_qblocks", "N_total", "C", "W", "gate", "centered", "alpha", "magic"):
        assert getattr(ref.out, f) == getattr(got.out, f), f


def test_noalloc_matches_fm_bounds_two_calls_in_a_row(lib):
    dev = torch.device("cuda:0")
    # first call: the mix workload with centering (large key offsets, fallback heads)
    q, k, v = workloads.make_inputs("mix", device=dev, heads=range(8), Sq=1500, N=2200)
    assert_same(*bounds_both_ways(lib, q, k, v, centering=True))
    # second call reuses the scratch left by the first, with another shape and another mode
    q, k, v = workloads.make_inputs("wan", device=dev, heads=range(5), Sq=700, N=3100)
    assert_same(*bounds_both_ways(lib, q, k, v, centering=False))
    # and the bounds it produced drive a full attention call like fm_bounds' would
    q, k, v = workloads.make_inputs("wan", device=dev, heads=range(3), Sq=300, N=333)
    ref, got = bounds_both_ways(lib, q, k, v, centering=True)
    outs = []
    for b in (ref, got):
        fa = fm.FixedMAttention(1, 3, 300, 333, 128, dev, centering=True)
        fa.bounds = b
        fm.fm_attn_chunk(q, k, v, b, fa.opt, fa.acc_o, fa.acc_sum, fa.acc_max, False)
        fm.fm_finalize(fa.acc_o, fa.acc_sum, fa.out)
        fm.fm_sync_status()
        outs.append(fa.out.clone())
    assert torch.equal(outs[0], outs[1])


def test_noalloc_refuses_problems_beyond_its_scratch(lib):
    # 200 heads of 75,600 keys need about 11.3 MB of scratch (about 56 KB per head at
    # D = 128): more than the 4 MiB array.
    need = fm.fm_bounds_workspace_size(1, 200, 75600, 128)
    assert need > fm.FM_NOALLOC_SCRATCH_BYTES, f"{need} bytes fit in the static scratch"
    t = fm.fm_tensor()
    t.ptr = 0x10000
    t.dtype = fm.FM_BF16
    t.B, t.H, t.S, t.D = 1, 200, 75600, 128
    for i, s in enumerate((200 * 75600 * 128, 75600 * 128, 128, 1)):
        t.stride[i] = s
    out = fm.fm_bounds_out()
    opt = fm.opts()
    rc = lib.fm_bounds_noalloc(ctypes.byref(t), ctypes.byref(t), ctypes.byref(t), ctypes.byref(opt),
                               ctypes.byref(out), None)
    assert rc == fm.FM_ERR_UNSUPPORTED
    assert "scratch" in fm.fm_last_error()
    assert out.magic == 0  # nothing was written
