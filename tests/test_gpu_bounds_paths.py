"""The bounds pass takes one of three norms kernels by the inputs' layout; all give the same bits.

bf16 rows of D = 128 stored back to back within each head go through the norms pass staged by
bulk copies into shared memory; other rows that start on 16-byte boundaries through the
pass with 16-byte register loads; anything else through the element-wise pass.  The staged
and the register-load pass use the same lane layout and order of additions, so for the same
values every output of fm_bounds -- m, flags, norms, the centering terms, the row shifts and
the key sinks -- must be bit-identical between a packed tensor and a row-strided copy of it.
The oracle pins the packed results too (ragged tails, heads of several batches).
"""
import numpy as np
import pytest
import torch

import fixed_max_softmax_gb300 as fm
import oracle
import workloads
from tests.test_gpu_parity import check_bounds, check_sinks

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


def row_strided(x):
    """The same values with a row stride of 2*D (so rows are not back to back)."""
    B, H, S, D = x.shape
    y = torch.zeros(B, H, S, 2 * D, dtype=x.dtype, device=x.device)
    y[..., :D] = x
    return y[..., :D]


def bounds_of(q, k, v, centering, per_row, sink_keys):
    B, H, Sq, D = q.shape
    fa = fm.FixedMAttention(B, H, Sq, k.shape[2], D, q.device, centering=centering, per_row=per_row,
                            sink_keys=sink_keys)
    fm.fm_bounds(q, k, v, fa.opt, fa.bounds, fa.workspace)
    fm.fm_sync_status()
    return fa


FIELDS = ["m", "flag", "qmax_sq", "kmax_sq", "kbar", "qkbar", "shift", "vmax_sq"]


@pytest.mark.parametrize("Sq,N", [(1, 1), (127, 129), (300, 257), (1000, 700), (4096, 4096)])
@pytest.mark.parametrize("centering,per_row,sink_keys", [(False, False, 0), (True, False, 0), (True, True, 4),
                                                         (False, False, 2)])
def test_staged_and_register_norms_give_the_same_bits(dev, Sq, N, centering, per_row, sink_keys):
    name = "sinks" if sink_keys else "mix"
    q, k, v = workloads.make_inputs(name, device="cpu", heads=[0, 1, 25], Sq=Sq, N=N)
    q, k, v = (torch.cat([x, x.flip(2)], 0).to(dev) for x in (q, k, v))  # two batch entries
    a = bounds_of(q, k, v, centering, per_row, sink_keys)
    b = bounds_of(row_strided(q), row_strided(k), row_strided(v), centering, per_row, sink_keys)
    for f in FIELDS:
        x, y = getattr(a.bounds, f), getattr(b.bounds, f)
        assert torch.equal(x.view(torch.uint8) if x.dtype == torch.float32 else x,
                           y.view(torch.uint8) if y.dtype == torch.float32 else y), f
    if sink_keys:
        for f in ["sink_idx", "sink_k", "sink_v"]:
            assert torch.equal(getattr(a.bounds, f), getattr(b.bounds, f)), f
    # and the packed (staged) results against the oracle, batch entry by batch entry
    for bi in range(2):
        ob = oracle.bounds(q[bi:bi + 1].cpu(), k[bi:bi + 1].cpu(), v[bi:bi + 1].cpu(), centering=centering,
                           per_row=per_row, sink_keys=sink_keys)
        one = bounds_of(q[bi:bi + 1], k[bi:bi + 1], v[bi:bi + 1], centering, per_row, sink_keys)
        for f in ["qmax_sq", "kmax_sq", "qkbar", "shift"]:
            assert torch.equal(getattr(one.bounds, f)[0], getattr(a.bounds, f)[bi]), f
        check_bounds(one, ob)
        if sink_keys:
            check_sinks(one, ob)


def test_staged_norms_at_the_wan_size(dev):
    """The staged pass on the full Wan layout (every CTA walks hundreds of blocks), two heads:
    the same bits as the register-load pass on a row-strided copy."""
    q, k, v = workloads.make_inputs("wan", device=dev, heads=[0, 21])
    a = bounds_of(q, k, v, True, False, 0)
    b = bounds_of(row_strided(q), row_strided(k), row_strided(v), True, False, 0)
    for f in FIELDS:
        x, y = getattr(a.bounds, f), getattr(b.bounds, f)
        assert torch.equal(x, y), f
    assert np.all(a.bounds.flag.cpu().numpy() == 1)
