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


def test_noalloc_rejects_sizes_beyond_its_array():
    T, H = 65536, 12288  # 304 partial rows of 12288 floats > the 304 x 8192 array
    assert ops.rmsnorm_bwd_scratch_bytes(T, H) > 4 * 304 * 8192
    t = torch.empty(8, dtype=torch.bfloat16, device="cuda")
    r = torch.empty(8, dtype=torch.float32, device="cuda")
    st = _noalloc()(t.data_ptr(), t.data_ptr(), t.data_ptr(), r.data_ptr(), None, T, H, t.data_ptr(),
                    t.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == -1  # MT_ERR_ARG, nothing launched
