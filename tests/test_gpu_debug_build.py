"""The debug build (nvcc -DFM_DEBUG): the tensor-core chunk kernels check every access of their
epilogues to the accumulators and to o against the buffers' extents; the first failure of a
launch goes to the device error word, the access is skipped, and fm_sync_status reports
FM_ERR_INDEX.  Release builds compile the checks away.

Each library runs in a child process of its own (a process loads one libfm).  On every path that
writes the accumulators or o -- per-chunk adds on both schedules, the fused final chunk in bf16
into padded rows and in fp32, the one-launch form, the separate finalize, forced online tiles --
at ragged sizes, the debug library must report nothing and give the release library's bits.
With FM_DEBUG_SHRINK_ROWS=1 (the accumulators declared one row short) it must report
FM_ERR_INDEX on every path and still give the release bits on every other row; the flagged
accesses are skipped, so nothing touches memory outside the buffers.
"""
import json
import os
import subprocess
import sys

import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

H, SQ, N = 3, 300, 700
CHUNKS = [(0, 300), (300, 1), (301, 399)]
CASES = {  # name: (schedule, out dtype, padded o rows, fused final, one launch, forced online)
    "grid_bf16_padded": ("grid", torch.bfloat16, True, True, False, False),
    "persistent_bf16_padded": ("persistent", torch.bfloat16, True, True, False, False),
    "grid_f32": ("grid", torch.float32, False, True, False, False),
    "one_launch_bf16": ("grid", torch.bfloat16, False, True, True, False),
    "separate_finalize": ("grid", torch.float32, False, False, False, False),
    "online_bf16": ("grid", torch.bfloat16, False, True, False, True),
}


def child(lib, out_path):
    sys.path.insert(0, ROOT)
    import fixed_max_softmax_gb300 as fm
    import workloads

    fm.load(lib)
    dev = torch.device("cuda:0")
    q, k, v = workloads.make_inputs("mix", device="cpu", heads=range(H), Sq=SQ, N=N)
    q, k, v = q.to(dev), k.to(dev), v.to(dev)
    results, status = {}, {}
    for name, (sched, dt, padded, fused, one, online) in CASES.items():
        fa = fm.FixedMAttention(1, H, SQ, N, 128, dev, centering=True, force_online=online, out_dtype=dt,
                                schedule=sched)
        if padded:  # o rows 32 elements apart beyond D, the gap filled with a fixed pattern
            full = torch.full((1, H, SQ, 160), -7.0, dtype=dt, device=dev)
            fa.out = full[..., :128]
        try:
            fa.forward(q, k, v, CHUNKS, with_lse=True, fused_final=fused, one_launch=one)
            fm.fm_sync_status()
            status[name] = "ok"
        except fm.FMError as e:
            status[name] = fm.ERROR_NAMES.get(e.code, str(e.code))
            torch.cuda.synchronize()
        results[name] = {"o": (full if padded else fa.out).float().cpu(), "lse": fa.lse.cpu(),
                         "acc_sum": fa.acc_sum.cpu()}
    torch.save(results, out_path)
    print(json.dumps(status))


def run_child(lib, out_path, extra_env=None):
    env = dict(os.environ)
    env.update(extra_env or {})
    r = subprocess.run([sys.executable, os.path.abspath(__file__), lib, out_path], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    return json.loads(r.stdout.strip().splitlines()[-1]), torch.load(out_path)


@pytest.mark.gpu
def test_debug_build_checks_the_epilogue_accesses(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fixed_max_softmax_gb300 import build as fmbuild

    rel = fmbuild.build()
    dbg = fmbuild.build(debug=True)
    st_rel, rel_out = run_child(rel, str(tmp_path / "rel.pt"))
    st_dbg, dbg_out = run_child(dbg, str(tmp_path / "dbg.pt"))
    assert all(v == "ok" for v in st_rel.values()), st_rel
    assert all(v == "ok" for v in st_dbg.values()), st_dbg
    for name in CASES:
        for key in ("o", "lse", "acc_sum"):
            assert torch.equal(rel_out[name][key].view(-1).view(torch.int32), dbg_out[name][key].view(-1).view(torch.int32)), (name, key)
    st_shr, shr_out = run_child(dbg, str(tmp_path / "shr.pt"), {"FM_DEBUG_SHRINK_ROWS": "1"})
    assert all(v == "FM_ERR_INDEX" for v in st_shr.values()), st_shr
    for name in CASES:
        # every row but the last one of the last head is the release result
        o_r, o_s = rel_out[name]["o"], shr_out[name]["o"]
        assert torch.equal(o_r[:, :H - 1], o_s[:, :H - 1]) and torch.equal(o_r[:, H - 1, :SQ - 1], o_s[:, H - 1, :SQ - 1]), name
        assert torch.equal(rel_out[name]["lse"].view(-1)[:-1], shr_out[name]["lse"].view(-1)[:-1]), name


if __name__ == "__main__":
    child(sys.argv[1], sys.argv[2])
