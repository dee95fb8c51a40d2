"""The 8-bit step kernel's bounded wait, made to run out on purpose, and how that
is reported.

The staged 8-bit step waits for the copies of each group's inputs into shared
memory, at most about a second.  A test hook lowers that limit to zero (give up at
the first poll that finds the copies still in flight) for one call; nothing
faults, traps or hangs: the kernel counts the give-up, lets the copies it issued
land, and stops.  Then:

* the device counter (lema_kernel_wait_timeouts) has grown;
* a direct call: the next lema_adamw_step_q8 returns LEMA_ERR_TIMEOUT and launches
  nothing;
* through the pool: lema_pool_sync returns LEMA_ERR_TIMEOUT once the work is done;
* with the limit back to its default, a fresh run matches the oracle bit for bit.
"""
from __future__ import annotations

import pytest
import torch

from oracle.runner import run_config_q8
from adamw_step_gb300 import lema
from adamw_step_gb300.runner import DeviceGrads, ResidentRunnerQ8, StreamedRunnerQ8
from gpu_common import ensure_library, small_config
from test_gpu_q8 import compare as compare_resident
from test_gpu_stream_q8 import compare as compare_streamed

pytestmark = pytest.mark.gpu
SIZES = [4 * 8192, 3 * 2048, 8192 + 5]      # whole groups, and a ragged end


@pytest.fixture(scope="module", autouse=True)
def lib():
    return ensure_library()


@pytest.fixture
def wait_limit_zero():
    lema.lema_test_kernel_wait_limit(0)
    try:
        yield
    finally:
        lema.lema_test_kernel_wait_limit(-1)


def test_direct_step_gives_up_and_the_next_call_reports_it(wait_limit_zero):
    cfg = small_config(SIZES, K=2, steps=1)
    before = lema.lema_kernel_wait_timeouts()
    r = ResidentRunnerQ8(cfg, DeviceGrads(cfg), fused=True)
    r.step(0)                                   # enqueued normally
    torch.cuda.synchronize()
    lema.lema_test_kernel_wait_limit(-1)
    assert lema.lema_kernel_wait_timeouts() > before
    snap = [{f: x.clone() for f, x in t.items()} for t in r.state.tensors]
    with pytest.raises(lema.LemaError) as e:
        r.adamw(0)
    assert e.value.status == lema.LEMA_ERR_TIMEOUT and "gave up" in e.value.message
    torch.cuda.synchronize()
    for t, s in zip(r.state.tensors, snap):     # nothing was launched
        for f in t:
            assert torch.equal(t[f].view(torch.uint8), s[f].view(torch.uint8)), f
    # reported once: the limit is back to its default and a fresh run is exact
    fresh = ResidentRunnerQ8(cfg, DeviceGrads(cfg), fused=True)
    mark = lema.lema_kernel_wait_timeouts()
    fresh.step(0)
    torch.cuda.synchronize()
    assert lema.lema_kernel_wait_timeouts() == mark
    compare_resident(fresh, run_config_q8(cfg, fused=True), "after the give-up")


def test_pool_step_gives_up_and_sync_reports_it(wait_limit_zero):
    cfg = small_config(SIZES, K=2, steps=1, units=[0, 0, 1])
    before = lema.lema_kernel_wait_timeouts()
    sr = StreamedRunnerQ8(cfg, DeviceGrads(cfg))
    try:
        sr.step(0)
        with pytest.raises(lema.LemaError) as e:
            sr.pool.sync(60_000)
        assert e.value.status == lema.LEMA_ERR_TIMEOUT and "gave up" in e.value.message
        lema.lema_test_kernel_wait_limit(-1)
        assert lema.lema_kernel_wait_timeouts() > before
        sr.pool.sync(60_000)                    # reported once
        # the same pool, fresh states, the default limit: exact
        fresh = StreamedRunnerQ8(cfg, DeviceGrads(cfg))
        fresh.pool.close()
        fresh.pool = sr.pool
        mark = lema.lema_kernel_wait_timeouts()
        fresh.step(0)
        fresh.pool.sync(60_000)
        assert lema.lema_kernel_wait_timeouts() == mark
        compare_streamed(fresh.state, run_config_q8(cfg, fused=True), "pool after the give-up")
        fresh.state.close()
    finally:
        sr.close()
