"""Failure handling on the GPU without a fault: a bounded device wait that
runs out.

With the stall hook on, the softmax warps of every attention kernel first
wait on a barrier that no thread ever arrives at, so their wait runs out
after the (short) limit.  The kernel must then record PKX_ETIMEOUT, raise its
abort flag so the other warps leave their own bounded waits, let the tensor
core and its copies finish, free its tensor memory and return.  The next
call, with the hook off and the default limit, must give the same bits as a
clean call before it (the context stays usable)."""
import math

import pytest
import torch

from paged_kv_extend_gb300 import pkx
from paged_kv_extend_gb300 import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from gpu_cases import DEV, DeviceWorkload


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pkx.load_library()


def _stalled(fn):
    """Run ``fn`` with the stall hook on and a 1 ms wait limit; both are
    reset afterwards whatever happens."""
    pkx.set_wait_limit_ns(1_000_000)
    pkx.set_stall_injection(True)
    try:
        return fn()
    finally:
        pkx.set_stall_injection(False)
        pkx.set_wait_limit_ns(0)


def _check_timeout_then_recovery(call):
    o0, l0, ws0 = call()
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws0) == pkx.PKX_OK
    _, _, ws1 = _stalled(call)
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws1) == pkx.PKX_ETIMEOUT
    o2, l2, ws2 = call()
    torch.cuda.synchronize()
    assert pkx.workspace_status(ws2) == pkx.PKX_OK
    assert torch.equal(o2, o0) and torch.equal(l2, l0)


def test_timeout_extend_unified():
    wl = W.draw(W.small_spec(batch=3, hq=16, hkv=4, prefix=[300, 0, 1000], extend=[77, 5, 260],
                             seed=41))
    dw = DeviceWorkload(wl)
    _check_timeout_then_recovery(dw.unified)


def test_timeout_decode():
    spec = W.WorkloadSpec("dec", batch=5, hq=32, hkv=8, lq=128, lv=128,
                          prefix=[0, 100, 4000, 63, 900], extend=[1] * 5, num_slots=1 << 14,
                          seed=42, decode=True)
    dw = DeviceWorkload(W.draw(spec))
    _check_timeout_then_recovery(dw.decode)


def test_timeout_mla():
    spec = W.small_spec(batch=2, hq=16, hkv=1, lq=576, lv=512, prefix=[200, 40], extend=[70, 9],
                        std=0.5, v_aliases_k=True, sm_scale=1.0 / math.sqrt(192.0), seed=43)
    dw = DeviceWorkload(W.draw(spec))
    _check_timeout_then_recovery(dw.extend)


def test_wait_limit_alone_changes_nothing():
    """A shorter (but ample) limit without the stall hook gives the same bits."""
    wl = W.draw(W.small_spec(batch=2, hq=8, hkv=2, prefix=[50, 700], extend=[30, 90], seed=44))
    dw = DeviceWorkload(wl)
    o0, l0, _ = dw.extend()
    pkx.set_wait_limit_ns(200_000_000)
    try:
        o1, l1, ws1 = dw.extend()
        torch.cuda.synchronize()
    finally:
        pkx.set_wait_limit_ns(0)
    assert pkx.workspace_status(ws1) == pkx.PKX_OK
    assert torch.equal(o1, o0) and torch.equal(l1, l0)
