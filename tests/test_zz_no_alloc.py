"""RMSNorm backward without allocation, checked against the regular entry point.

mt_rmsnorm_bwd_noalloc serves callers that cannot allocate device memory
(stream capture, a foreign framework's allocator, allocation-free hot loops):
its scratch is a fixed array inside the library.  Here it is called through
the C ABI twice in a row on different inputs, and each result is compared
with mt_rmsnorm_bwd given a caller-allocated scratch buffer.  This file is
collected last so that a run stopping at the first failure has already run
every other test.
"""
import ctypes as C

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import host_memory_centric_gb300 as mt  # noqa: E402
from host_memory_centric_gb300 import ops  # noqa: E402

_v = C.c_void_p


def _noalloc():
    fn = mt.lib().mt_rmsnorm_bwd_noalloc
    fn.restype = C.c_int32
    fn.argtypes = [_v, _v, _v, _v, _v, C.c_int64, C.c_int32, _v, _v, _v]
    return fn


def _call_noalloc(dy, x, g, r, dres, dx, dg):
    T, H = x.shape
    return _noalloc()(dy.data_ptr(), x.data_ptr(), g.data_ptr(), r.data_ptr(),
                      None if dres is None else dres.data_ptr(), T, H, dx.data_ptr(), dg.data_ptr(),
                      torch.cuda.current_stream().cuda_stream)


def _case(T, H, seed):
    gen = torch.Generator().manual_seed(seed)
    x = torch.randn(T, H, generator=gen).to(torch.bfloat16).cuda()
    g = (1 + 0.1 * torch.randn(H, generator=gen)).to(torch.bfloat16).cuda()
    dy = torch.randn(T, H, generator=gen).to(torch.bfloat16).cuda()
    dres = torch.randn(T, H, generator=gen).to(torch.bfloat16).cuda()
    y = torch.empty_like(x)
    r = torch.empty(T, dtype=torch.float32, device="cuda")
    ops.rmsnorm_fwd(x, g, 1e-6, y, r)
    return dy, x, g, r, dres


def _rel_l2(a, b):
    a, b = a.double().cpu().numpy(), b.double().cpu().numpy()
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


@pytest.mark.parametrize("T,H", [(333, 520), (4096, 2048)])
def test_noalloc_matches_allocating_entry_point_twice(T, H):
    for seed in (1, 2):  # two calls in a row: the shared array keeps the first call's contents
        dy, x, g, r, dres = _case(T, H, seed)
        dx_a, dg_a = torch.empty_like(x), torch.empty(H, dtype=torch.bfloat16, device="cuda")
        scratch = torch.empty(ops.rmsnorm_bwd_scratch_bytes(T, H), dtype=torch.uint8, device="cuda")
        ops.rmsnorm_bwd(dy, x, g, r, dres, dx_a, dg_a, scratch)
        dx_b, dg_b = torch.empty_like(x), torch.empty(H, dtype=torch.bfloat16, device="cuda")
        assert _call_noalloc(dy, x, g, r, dres, dx_b, dg_b) == 0
        torch.cuda.synchronize()
        # the same kernels in the same fixed summation order, only the scratch
        # differs: the results agree bit for bit
        assert torch.equal(dx_b, dx_a) and torch.equal(dg_b, dg_a), (_rel_l2(dx_b, dx_a), _rel_l2(dg_b, dg_a))


def test_noalloc_at_its_limit_and_beyond():
    """At exactly the array's size the call runs and matches the allocating
    entry point; one size past it is refused before anything is launched.
    Both calls get real buffers of the full [T, H] size, so that a broken size
    check shows up as a wrong status or wrong values, never as an access past
    the end of a buffer."""
    T = 9728  # the smallest T that gives the maximum of 304 blocks (32 rows each)
    assert ops.rmsnorm_bwd_scratch_bytes(T, 8192) == 4 * 304 * 8192
    dy, x, g, r, dres = _case(T, 8192, 3)
    dx_a, dg_a = torch.empty_like(x), torch.empty(8192, dtype=torch.bfloat16, device="cuda")
    scratch = torch.empty(ops.rmsnorm_bwd_scratch_bytes(T, 8192), dtype=torch.uint8, device="cuda")
    ops.rmsnorm_bwd(dy, x, g, r, dres, dx_a, dg_a, scratch)
    dx_b, dg_b = torch.empty_like(x), torch.empty(8192, dtype=torch.bfloat16, device="cuda")
    assert _call_noalloc(dy, x, g, r, dres, dx_b, dg_b) == 0
    torch.cuda.synchronize()
    assert torch.equal(dx_b, dx_a) and torch.equal(dg_b, dg_a)
    del dy, x, g, r, dres, dx_a, dg_a, dx_b, dg_b, scratch

    H = 8200  # 304 partial rows of 8200 floats: one column more than the array holds
    assert ops.rmsnorm_bwd_scratch_bytes(T, H) > 4 * 304 * 8192
    dy, x, g, r, dres = _case(T, H, 4)
    dx = torch.full_like(x, 7.0)
    dg = torch.full((H,), 7.0, dtype=torch.bfloat16, device="cuda")
    assert _call_noalloc(dy, x, g, r, dres, dx, dg) == -1  # MT_ERR_ARG
    torch.cuda.synchronize()
    assert bool((dx == 7.0).all()) and bool((dg == 7.0).all())  # nothing was launched
