"""Failure detection, exercised with host-side faults only.

Every host wait of the library has a deadline (timeout_ms) and latches the
model into an error state; every mbarrier wait inside the tensor-core kernels
is bounded and reports through the kernel error word.  Faults are injected on
the host (mt_fault_inject): a stalled Adam worker, a throwing worker, a failed
pinned allocation, and a GEMM whose producer issues nothing so that its
consumers' bounded waits expire.  No test faults, traps or hangs a GPU.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import host_memory_centric_gb300 as mt  # noqa: E402
from host_memory_centric_gb300 import configs, inputs, ops  # noqa: E402


@pytest.fixture(autouse=True)
def _clear_injection():
    for k in (1, 2, 3, 4):
        mt.lib().mt_fault_inject(k, 0)
    yield
    for k in (1, 2, 3, 4):
        mt.lib().mt_fault_inject(k, 0)
    torch.cuda.synchronize()
    ops.kernel_error(clear=True)


def test_pinned_allocation_failure_reports_host_oom():
    assert mt.lib().mt_fault_inject(3, 1) == 0
    with pytest.raises(mt.MtError) as ei:
        mt.Model(configs.get("tiny"))
    assert ei.value.status == -3  # MT_ERR_HOST_OOM
    m = mt.Model(configs.get("tiny"))  # the next allocation succeeds again
    m.close()


def test_stalled_adam_worker_times_out_slab_acquire_and_latches():
    c = configs.get("tiny")
    m = mt.Model(c, n_grad_slabs=1, timeout_ms=300)
    m.set_tokens(inputs.tokens_for(c, 0))
    assert mt.lib().mt_fault_inject(1, 1500) == 0  # every Adam job sleeps 1.5 s first
    with pytest.raises(mt.MtError) as ei:
        m.train_step(0)
    assert ei.value.status == -5  # MT_ERR_TIMEOUT: the one slab never came back in time
    assert "slab" in m.last_error()
    with pytest.raises(mt.MtError) as ei:
        m.sync()
    assert ei.value.status == -2  # latched: every later call is refused
    mt.lib().mt_fault_inject(1, 0)
    m.close()  # shuts down with work in flight


def test_worker_exception_is_reported():
    c = configs.get("tiny")
    m = mt.Model(c, timeout_ms=5000)
    m.set_tokens(inputs.tokens_for(c, 0))
    assert mt.lib().mt_fault_inject(2, 1) == 0
    with pytest.raises(mt.MtError):
        m.train_step(0)
        m.sync()
    assert "injected host worker fault" in m.last_error()
    m.close()


def test_destroy_with_work_in_flight_then_train_again():
    c = configs.get("tiny")
    m = mt.Model(c)
    m.set_tokens(inputs.tokens_for(c, 0))
    m.train_step(0, want_loss=False)
    m.close()  # no sync first
    m2 = mt.Model(c)
    m2.set_tokens(inputs.tokens_for(c, 0))
    loss = m2.train_step(0)
    m2.sync()
    assert np.isfinite(loss)
    m2.close()


def test_gemm_bounded_wait_expires_and_context_survives():
    A = torch.randn(256, 128).to(torch.bfloat16).cuda()
    B = torch.randn(256, 128).to(torch.bfloat16).cuda()
    D = torch.empty(256, 256, dtype=torch.bfloat16, device="cuda")
    ops.kernel_error(clear=True)
    assert mt.lib().mt_fault_inject(4, 1) == 0  # the next GEMM's producer issues no loads
    ops.gemm(A, B, 256, 256, 128, D=D)
    torch.cuda.synchronize()
    assert ops.kernel_error(clear=True) != 0  # its waits ran out and it said so
    ops.gemm(A, B, 256, 256, 128, D=D)  # the context is still usable
    torch.cuda.synchronize()
    assert ops.kernel_error(clear=True) == 0
    ref = A.float() @ B.float().T
    assert torch.allclose(D.float(), ref, rtol=2e-2, atol=2e-1)


def test_bad_arguments_are_rejected_without_latching():
    c = configs.get("tiny")
    m = mt.Model(c)
    with pytest.raises(mt.MtError) as ei:
        m.set_tokens(np.full(m.T, c["vocab"], dtype=np.int32))  # token id out of range
    assert ei.value.status == -1
    m.set_tokens(inputs.tokens_for(c, 0))
    with pytest.raises(mt.MtError) as ei:
        m.train_step(5)  # wrong step index
    assert ei.value.status == -2
    assert np.isfinite(m.train_step(0))
    m.sync()
    m.close()


def test_moe_route_wait_times_out_and_latches():
    """An MoE forward visit waits on the host, bounded, for the router's
    per-expert counts (Route-Ready).  A GEMM made to stall (its bounded waits
    run out after about 2 s, with the context intact) delays that event past
    a 1 s limit: train_step returns MT_ERR_TIMEOUT, the model latches, and a
    fresh model trains normally afterwards."""
    c = configs.get("tiny_moe")
    m = mt.Model(c, timeout_ms=1000)
    # one normal step first: the first launch of a kernel not yet loaded
    # (CUDA's lazy module loading) waits for the device, which would hold the
    # host behind the stalled GEMM before it reaches the bounded wait
    m.set_tokens(inputs.tokens_for(c, 0))
    m.train_step(0)
    m.sync()
    m.set_tokens(inputs.tokens_for(c, 1))
    ops.kernel_error(clear=True)
    assert mt.lib().mt_fault_inject(4, 1) == 0  # layer 1's first GEMM (QKV) issues no loads
    with pytest.raises(mt.MtError) as ei:
        m.train_step(1)
    assert ei.value.status == -5
    assert "routing" in m.last_error()
    with pytest.raises(mt.MtError) as ei:
        m.train_step(1)
    assert ei.value.status == -2  # latched
    m.close()
    torch.cuda.synchronize()
    assert ops.kernel_error(clear=True) != 0
    m2 = mt.Model(c)
    m2.set_tokens(inputs.tokens_for(c, 0))
    assert np.isfinite(m2.train_step(0))
    m2.sync()
    assert ops.kernel_error(clear=True) == 0
    m2.close()


def test_expired_kernel_wait_latches_at_sync():
    """A GEMM made to stall (its bounded waits run out after about 2 s and it
    records a code, the context intact) inside a training step: mt_sync
    reports MT_ERR_TIMEOUT and the model latches; once the code is cleared a
    fresh model trains normally."""
    c = configs.get("tiny")
    m = mt.Model(c)
    m.set_tokens(inputs.tokens_for(c, 0))
    m.train_step(0)  # first step: lazy loading out of the way
    m.sync()
    ops.kernel_error(clear=True)
    m.set_tokens(inputs.tokens_for(c, 1))
    assert mt.lib().mt_fault_inject(4, 1) == 0  # the next GEMM issues no loads
    m.train_step(1, want_loss=False)
    with pytest.raises(mt.MtError) as ei:
        m.sync()
    assert ei.value.status == -5
    assert "bounded wait" in m.last_error()
    with pytest.raises(mt.MtError) as ei:
        m.train_step(2)
    assert ei.value.status == -2  # latched
    m.close()
    torch.cuda.synchronize()
    assert ops.kernel_error(clear=True) != 0
    m2 = mt.Model(c)
    m2.set_tokens(inputs.tokens_for(c, 0))
    assert np.isfinite(m2.train_step(0))
    m2.sync()
    assert ops.kernel_error(clear=True) == 0
    m2.close()


@pytest.mark.parametrize("name,rt", [("tiny", dict(ckpt_interval=2, pin_store=0)), ("tiny_moe", {})])
def test_debug_guards_hold_over_steps(name, rt):
    """With debug_guards every carved device piece and every pinned region has
    a canary after it; training steps leave all of them intact."""
    c = configs.get(name)
    m = mt.Model(c, debug_guards=1, **rt)
    for s in range(2):
        m.set_tokens(inputs.tokens_for(c, s))
        assert np.isfinite(m.train_step(s))
        m.sync()  # checks every guard
    m.close()


@pytest.mark.parametrize("where", ["device", "host"])
def test_debug_guards_catch_an_overwrite(where):
    """A byte written into a guard (test hook, ordinary memory writes) is
    reported by the next mt_sync, which latches the model."""
    import ctypes as C
    c = configs.get("tiny")
    m = mt.Model(c, debug_guards=1)
    m.set_tokens(inputs.tokens_for(c, 0))
    m.train_step(0)
    m.sync()
    n = C.c_int32()
    assert mt.lib().mt_debug_poke_guard(m.h, 1 << 30, C.byref(n)) == -1 and n.value > 10
    which = 5 if where == "device" else n.value - 1
    assert mt.lib().mt_debug_poke_guard(m.h, which, None) == 0
    with pytest.raises(mt.MtError) as ei:
        m.sync()
    assert ei.value.status == -6 and "guard" in m.last_error()
    assert (where == "device") == ("device guard" in m.last_error())
    m.close()
