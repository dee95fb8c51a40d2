"""8-bit states in the streamed residency (pinned host RAM through the slot pool,
lema_stream_layers_q8) on the GPU: every field (codes, block scales, master,
delta, bf16 weight, host accumulator) bit for bit against the oracle's 8-bit form
with the last micro-batch grad folded into the step, and against the resident
8-bit path on the same inputs."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle.runner import run_config_q8
from adamw_step_gb300 import configs, lema
from adamw_step_gb300.runner import DeviceGrads, ResidentRunnerQ8, StreamedRunnerQ8
from adamw_step_gb300.state import HostStateQ8, LayersQ8, Pool, hparams
from gpu_common import ensure_library, small_config

pytestmark = pytest.mark.gpu
SIZES = [1, 7, 8, 9, 0, 255, 256, 257, 511, 1023, 1024, 1025, 8191, 8192, 8193, 16640,
         100_003]
UNITS = [i // 4 for i in range(len(SIZES))]
FIELDS = ("master", "delta", "w", "m_q", "m_scale", "r_q", "r_scale", "acc_q", "acc_scale")


@pytest.fixture(scope="module", autouse=True)
def lib():
    return ensure_library()


def run_streamed(cfg, host_grads=False, n_slots=2, packed=True):
    sr = StreamedRunnerQ8(cfg, DeviceGrads(cfg, pin_host=host_grads), n_slots=n_slots,
                          packed=packed)
    for t in range(cfg.steps):
        sr.step(t)
    sr.pool.sync(600_000)
    torch.cuda.synchronize()
    return sr


def compare(state, ref, label, tensors=None):
    for j in (ref if tensors is None else tensors):
        st = ref[j]
        got = state.numpy_views(j)
        want = {"master": st.master, "delta": st.delta, "w": st.w, "m_q": st.m_q,
                "m_scale": st.m_scale, "r_q": st.r_q, "r_scale": st.r_scale,
                "acc_q": st.acc_q, "acc_scale": st.acc_scale}
        for f in FIELDS:
            same = got[f].view(np.uint8) == want[f].view(np.uint8)
            assert same.all(), \
                f"{label} tensor {j} {f}: first mismatch at byte {np.flatnonzero(~same)[:3]}"


@pytest.mark.parametrize("first_only", [False, True], ids=["every-unit", "first-unit"])
@pytest.mark.parametrize("host_grads", [False, True], ids=["device-grads", "host-grads"])
def test_q8_streamed_sliced_units(host_grads, first_only):
    """Packed 8-bit units split into up to 4 slices of whole chunks (every unit, or
    only each call's first): every field bit for bit against the oracle."""
    cfg = small_config(SIZES, K=3, steps=2, units=UNITS)
    sr = StreamedRunnerQ8(cfg, DeviceGrads(cfg, pin_host=host_grads), n_slots=2, packed=True)
    sr.pool.slices(4, 8192, first_unit_only=first_only)
    try:
        for t in range(cfg.steps):
            sr.step(t)
        sr.pool.sync(600_000)
        compare(sr.state, run_config_q8(cfg, fused=True), "q8 sliced")
    finally:
        sr.close()


@pytest.mark.parametrize("packed", [True, False], ids=["packed", "per-tensor"])
@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_q8_streamed_bit_exact(K, packed):
    cfg = small_config(SIZES, K=K, steps=3, units=UNITS)
    sr = run_streamed(cfg, packed=packed)
    try:
        compare(sr.state, run_config_q8(cfg, fused=True), f"q8 streamed K={K}")
    finally:
        sr.close()


@pytest.mark.parametrize("K", [1, 2, 3])
@pytest.mark.parametrize("host_grads,slices,packed", [(False, 1, True), (True, 1, False),
                                                      (False, 4, True)],
                         ids=["device-grads", "host-grads-per-tensor", "sliced"])
def test_q8_streamed_device_accumulators(K, host_grads, slices, packed):
    """8-bit accumulators (codes and scales) kept in HBM while the other states
    stream: every field bit for bit against the oracle."""
    cfg = small_config(SIZES, K=K, steps=3, units=UNITS)
    sr = StreamedRunnerQ8(cfg, DeviceGrads(cfg, pin_host=host_grads), n_slots=2,
                          packed=packed, acc_on_device=True)
    assert all(t["acc_q"].is_cuda and t["acc_scale"].is_cuda for t in sr.state.tensors)
    sr.pool.slices(slices, 8192)
    try:
        for t in range(cfg.steps):
            sr.step(t)
        sr.pool.sync(600_000)
        compare(sr.state, run_config_q8(cfg, fused=True), f"q8 device acc K={K}")
    finally:
        sr.close()


def test_q8_streamed_mixed_accumulator_residency_rejected():
    """Codes on the device with scales in pinned RAM (one tensor) is a mixed unit:
    rejected before anything is enqueued."""
    cfg = small_config(SIZES, K=2, steps=1, units=UNITS)
    sr = StreamedRunnerQ8(cfg, DeviceGrads(cfg), n_slots=2)
    try:
        j = cfg.unit_tensors(0)[0]
        sr.state.tensors[j]["acc_q"] = torch.zeros_like(sr.state.tensors[j]["acc_q"],
                                                        device="cuda")
        layers = LayersQ8(sr.state, [cfg.unit_tensors(u) for u in range(cfg.n_units)],
                          packed=False)
        arr, keep = layers.build([sr.grads(i, 0, 0) for i in range(len(SIZES))])
        with pytest.raises(lema.LemaError) as e:
            lema.lema_stream_layers_q8(sr.pool.handle, arr, 1, sr.hp, 1)
        assert e.value.status == lema.LEMA_ERR_ARG and "must all be pinned host" in e.value.message
    finally:
        sr.close()


def test_q8_streamed_host_grads_three_slots_matches_resident():
    cfg = small_config(SIZES, K=3, steps=3, units=UNITS)
    sr = run_streamed(cfg, host_grads=True, n_slots=3)
    res = ResidentRunnerQ8(cfg, DeviceGrads(cfg), fused=True)
    for t in range(cfg.steps):
        res.step(t)
    torch.cuda.synchronize()
    try:
        for j in range(len(SIZES)):
            a, b = sr.state.numpy_views(j), res.state.numpy_views(j)
            for f in FIELDS:
                assert np.array_equal(a[f].view(np.uint8), b[f].view(np.uint8)), (j, f)
    finally:
        sr.close()


def test_q8_streamed_268m_full():
    """The 268M-parameter streamed workload (4 units of 4 tensors, K=8) with 8-bit
    states: every element of every tensor against the oracle."""
    from oracle_cache import oracle_states_q8
    cfg = configs.CONFIGS[3]
    sr = run_streamed(cfg)
    try:
        compare(sr.state, oracle_states_q8(cfg, fused=True), "q8 config 3")
    finally:
        sr.close()


def test_q8_streamed_rejects_bad_units():
    cfg = small_config([5000, 3000], K=2, steps=1, units=[0, 0])
    grads = DeviceGrads(cfg)
    st = HostStateQ8([torch.zeros(5000, dtype=torch.bfloat16),
                      torch.zeros(3000, dtype=torch.bfloat16)], units=[[0, 1]])
    hp = hparams(cfg.hyper, 2)
    g = [grads(0, 0, 0), grads(1, 0, 0)]
    small = Pool(2, 4096)                             # the unit needs 5120 + 3072 elements
    arr, keep = LayersQ8(st, [[0, 1]]).build(g)
    with pytest.raises(lema.LemaError) as e:
        lema.lema_stream_layers_q8(small.handle, arr, 1, hp, 1)
    assert e.value.status == lema.LEMA_ERR_ARG and "slot" in e.value.message
    pool = Pool(2, 8192)
    per_tensor = HostStateQ8([torch.zeros(5000, dtype=torch.bfloat16),
                              torch.zeros(3000, dtype=torch.bfloat16)])
    arr, keep = LayersQ8(per_tensor, [[0, 1]], packed=True).build(g)
    with pytest.raises(lema.LemaError) as e:
        lema.lema_stream_layers_q8(pool.handle, arr, 1, hp, 1)
    assert e.value.status == lema.LEMA_ERR_ARG and "packed" in e.value.message
    pageable = [torch.zeros(5000, dtype=torch.bfloat16), torch.zeros(3000, dtype=torch.bfloat16)]
    arr, keep = LayersQ8(st, [[0, 1]]).build(pageable)
    with pytest.raises(lema.LemaError) as e:
        lema.lema_stream_layers_q8(pool.handle, arr, 1, hp, 1)
    assert e.value.status == lema.LEMA_ERR_ARG and "grad" in e.value.message
    for p in (small, pool):
        p.close()
    st.close()
    per_tensor.close()


def test_q8_injected_copy_failure_then_recovery():
    """The 8-bit streamed path reports a copy-enqueue failure made on the host by the
    test hook; the same pool then runs a fresh sequence correctly."""
    cfg = small_config(SIZES, K=2, steps=2, units=UNITS)
    sr = StreamedRunnerQ8(cfg, DeviceGrads(cfg))
    lema.lema_test_fail_copy(5)
    try:
        with pytest.raises(lema.LemaError) as e:
            sr.step(0)
        assert e.value.status == lema.LEMA_ERR_CUDA and "injected" in e.value.message
    finally:
        lema.lema_test_fail_copy(0)
    sr.pool.sync(60_000)
    fresh = StreamedRunnerQ8(cfg, DeviceGrads(cfg))
    fresh.pool.close()
    fresh.pool = sr.pool                      # reuse the pool that saw the failure
    for t in range(cfg.steps):
        fresh.step(t)
    fresh.pool.sync(60_000)
    torch.cuda.synchronize()
    try:
        compare(fresh.state, run_config_q8(cfg, fused=True), "q8 after failure")
    finally:
        fresh.close()
        sr.state.close()
