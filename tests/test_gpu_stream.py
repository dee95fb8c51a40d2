"""Streamed residency (pinned host states through the VRAM slot pool) on the GPU:
same results as the oracle and as the resident path, error handling."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from adamw_step_gb300 import configs, inputs, lema
from adamw_step_gb300.runner import DeviceGrads, ResidentRunner, StreamedRunner
from adamw_step_gb300.state import HostState, Layers, Pool, _State, hparams
from gpu_common import RAGGED, ensure_library, small_config
from oracle_cache import oracle_states
from parity import check_tensor, oracle_dict, state_dict

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    return ensure_library()


def run_streamed(cfg, host_grads=False, n_slots=2, steps=None, packed=True):
    sr = StreamedRunner(cfg, DeviceGrads(cfg, pin_host=host_grads), n_slots=n_slots,
                        packed=packed)
    for t in range(cfg.steps if steps is None else steps):
        sr.step(t)
    sr.pool.sync(600_000)
    return sr


def last_step_acc(cfg, j):
    """After a streamed step the host acc holds the partial sum of micro-steps
    1..K-1 of that step (the last micro-step is added on the device only); with
    K = 1 it is never written and keeps its initial +0."""
    orc = oracle.Oracle()
    gs = inputs.GradSource(cfg)
    acc = np.zeros(cfg.tensors[j].numel, np.float32)
    for k in range(cfg.accum_steps - 1):
        orc.accum(acc, inputs.as_u16(gs(j, cfg.steps - 1, k)))
    return acc


def check_streamed(cfg, sr, ref, tensors=None, label=""):
    bad = 0
    for j in (ref if tensors is None else tensors):
        want = oracle_dict(ref[j])
        want = dict(want, acc=last_step_acc(cfg, j))
        rep = check_tensor(state_dict(sr.state, j), want, f"{label} tensor {j}")
        bad += sum(rep.values())
    return bad


def ragged_units():
    return [i // 3 for i in range(len(RAGGED))]


@pytest.mark.parametrize("packed", [True, False], ids=["packed", "per-tensor"])
@pytest.mark.parametrize("host_grads,n_slots", [(False, 2), (True, 2), (False, 3)])
def test_streamed_small_matches_oracle(host_grads, n_slots, packed):
    cfg = small_config(RAGGED, K=3, steps=3, units=ragged_units())
    sr = run_streamed(cfg, host_grads=host_grads, n_slots=n_slots, packed=packed)
    assert check_streamed(cfg, sr, oracle_states(cfg), label="streamed") == 0
    sr.close()


@pytest.mark.parametrize("first_only", [False, True], ids=["every-unit", "first-unit"])
@pytest.mark.parametrize("host_grads", [False, True], ids=["device-grads", "host-grads"])
def test_streamed_sliced_units_match_oracle(host_grads, first_only):
    """Packed units split into up to 4 slices of whole chunks (slice boundaries
    inside tensors and between them; every unit, or only each call's first): same
    bits as the oracle."""
    cfg = small_config(RAGGED, K=3, steps=3, units=ragged_units())
    sr = StreamedRunner(cfg, DeviceGrads(cfg, pin_host=host_grads), n_slots=2, packed=True)
    sr.pool.slices(4, 8192, first_unit_only=first_only)
    for t in range(cfg.steps):
        sr.step(t)
    sr.pool.sync(600_000)
    assert check_streamed(cfg, sr, oracle_states(cfg), label="sliced") == 0
    sr.close()


@pytest.mark.parametrize("K", [1, 2, 3])
@pytest.mark.parametrize("host_grads,slices,packed", [(False, 1, True), (True, 1, False),
                                                      (False, 4, True), (True, 4, True),
                                                      (False, 2, True)],
                         ids=["device-grads", "host-grads-per-tensor", "sliced",
                              "host-grads-sliced", "first-unit-sliced"])
def test_streamed_device_accumulators_match_oracle(K, host_grads, slices, packed):
    """Accumulators kept in HBM while the optimizer states stream: the same bits as
    the oracle, the device acc holding micro-steps 1..K-1 of the last step (as the
    host acc would)."""
    cfg = small_config(RAGGED, K=K, steps=3, units=ragged_units())
    sr = StreamedRunner(cfg, DeviceGrads(cfg, pin_host=host_grads), n_slots=2, packed=packed,
                        acc_on_device=True)
    assert all(t["acc"].is_cuda for t in sr.state.tensors)
    sr.pool.slices(slices, 8192, first_unit_only=slices == 2)
    try:
        for t in range(cfg.steps):
            sr.step(t)
        sr.pool.sync(600_000)
        assert check_streamed(cfg, sr, oracle_states(cfg), label=f"device acc K={K}") == 0
    finally:
        sr.close()


def test_streamed_device_accumulators_per_unit_and_mixed_unit_rejected():
    """Units may differ (unit 0's accumulators in HBM, the others' in pinned RAM);
    a unit that mixes the two is rejected before anything is enqueued."""
    cfg = small_config(RAGGED, K=3, steps=2, units=ragged_units())
    sr = StreamedRunner(cfg, DeviceGrads(cfg), n_slots=2)
    unit0 = cfg.unit_tensors(0)
    try:
        # a mixed unit: the first tensor's accumulator alone on the device
        host_acc = sr.state.tensors[unit0[0]]["acc"]
        sr.state.tensors[unit0[0]]["acc"] = torch.zeros(host_acc.numel(), device="cuda")
        mixed = Layers(sr.state, [cfg.unit_tensors(u) for u in range(cfg.n_units)], packed=False)
        arr, keep = mixed.build([sr.grads(j, 0, 0) for j in range(len(cfg.tensors))])
        with pytest.raises(lema.LemaError) as e:
            sr.pool.stream_layers(arr, 1, sr.hp, 1)
        assert e.value.status == lema.LEMA_ERR_ARG and "must all be pinned host" in e.value.message
        # the whole of unit 0 on the device, packed like the host block
        P = sum(-(-sr.state.tensors[j]["acc"].numel() // 64) * 64 for j in unit0)
        block = torch.zeros(P, device="cuda")
        o = 0
        for j in unit0:
            n = sr.state.tensors[j]["orig"].numel()
            sr.state.tensors[j]["acc"] = block[o:o + n]
            o += -(-n // 64) * 64
        sr.layers = Layers(sr.state, [cfg.unit_tensors(u) for u in range(cfg.n_units)],
                           packed=False)
        sr._built.clear()
        for t in range(cfg.steps):
            sr.step(t)
        sr.pool.sync(600_000)
        assert check_streamed(cfg, sr, oracle_states(cfg), label="unit 0 on the device") == 0
    finally:
        sr.close()


def test_copies_only_mode_leaves_the_pool_usable():
    """The measurement mode enqueues a streamed step's copies without kernels (its
    host outputs are then slot contents, not results); switched off again, the same
    pool runs a fresh state to the oracle's bits."""
    cfg = small_config(RAGGED, K=2, steps=2, units=ragged_units())
    sr = StreamedRunner(cfg, DeviceGrads(cfg))
    lema.lema_pool_copies_only(sr.pool.handle, True)
    try:
        for t in range(cfg.steps):
            sr.step(t)
        sr.pool.sync(60_000)
    finally:
        lema.lema_pool_copies_only(sr.pool.handle, False)
    fresh = StreamedRunner(cfg, DeviceGrads(cfg))
    fresh.pool.close()
    fresh.pool = sr.pool
    for t in range(cfg.steps):
        fresh.step(t)
    fresh.pool.sync(60_000)
    assert check_streamed(cfg, fresh, oracle_states(cfg), label="after copies-only") == 0
    fresh.state.close()
    sr.close()


def test_pool_slices_argument_checks():
    pool = Pool(2, 8192)
    for bad in ((0, 8192), (9, 8192), (4, 0)):
        with pytest.raises(lema.LemaError) as e:
            pool.slices(*bad)
        assert e.value.status == lema.LEMA_ERR_ARG
    pool.close()


def test_streamed_single_micro_step():
    cfg = small_config([4099, 64, 1], K=1, steps=2, units=[0, 1, 1])
    sr = run_streamed(cfg)
    assert check_streamed(cfg, sr, oracle_states(cfg)) == 0
    sr.close()


def test_resident_residency_through_stream_layers():
    cfg = small_config(RAGGED, K=2, steps=2, units=ragged_units())
    a = ResidentRunner(cfg, DeviceGrads(cfg), fused=False)
    b = ResidentRunner(cfg, DeviceGrads(cfg), fused=False)
    lay = Layers(b.state, [cfg.unit_tensors(u) for u in range(cfg.n_units)])
    hp = hparams(cfg.hyper, cfg.accum_steps)
    for t in range(cfg.steps):
        a.step(t)
        for k in range(cfg.accum_steps):
            arr, keep = lay.build([b.grads(j, t, k) for j in range(len(cfg.tensors))])
            lema.lema_stream_layers(None, arr, lema.LEMA_RESIDENT, k + 1, hp, t + 1)
    torch.cuda.synchronize()
    for ta, tb in zip(a.state.tensors, b.state.tensors):
        for f in ta:
            assert torch.equal(ta[f].view(torch.uint8), tb[f].view(torch.uint8)), f


def test_config3_full():
    """The 268M-param attention set streamed: 4 units of 4 tensors, 2 slots, K=8,
    5 steps; every element against the oracle."""
    cfg = configs.CONFIGS[3]
    sr = run_streamed(cfg)
    assert check_streamed(cfg, sr, oracle_states(cfg), label="config 3") == 0
    sr.close()


def test_config3_device_accumulators_full():
    """Config 3 with its accumulators in HBM: every element against the oracle."""
    cfg = configs.CONFIGS[3]
    sr = StreamedRunner(cfg, DeviceGrads(cfg), acc_on_device=True)
    try:
        for t in range(cfg.steps):
            sr.step(t)
        sr.pool.sync(600_000)
        assert check_streamed(cfg, sr, oracle_states(cfg), label="config 3, device acc") == 0
    finally:
        sr.close()


def test_unit_larger_than_slot_is_rejected_before_any_copy():
    cfg = small_config([5000, 5000], K=2, steps=1, units=[0, 1])
    st = HostState([inputs.w0_bf16(cfg, j) for j in range(2)])
    pool = Pool(2, 4000)
    grads = DeviceGrads(cfg)
    arr, keep = Layers(st, [[0], [1]]).build([grads(j, 0, 0) for j in range(2)])
    before = [t["acc"].clone() for t in st.tensors]
    with pytest.raises(lema.LemaError) as e:
        pool.stream_layers(arr, 1, hparams(cfg.hyper, 2), 1)
    assert e.value.status == lema.LEMA_ERR_ARG and "slot" in e.value.message
    pool.sync(10_000)
    assert all(torch.equal(a, t["acc"]) for a, t in zip(before, st.tensors))
    pool.close()


def test_packed_flag_needs_a_packed_layout():
    """A unit flagged LEMA_UNIT_PACKED whose buffers are not at the slot offsets is
    rejected before anything is copied."""
    cfg = small_config([5000, 300], K=1, steps=1, units=[0, 0])
    st = HostState([inputs.w0_bf16(cfg, j) for j in range(2)])       # per-tensor buffers
    pool = Pool(2, 8192)
    arr, keep = Layers(st, [[0, 1]], packed=True).build([DeviceGrads(cfg)(j, 0, 0) for j in range(2)])
    with pytest.raises(lema.LemaError) as e:
        pool.stream_layers(arr, 1, hparams(cfg.hyper, 1), 1)
    assert e.value.status == lema.LEMA_ERR_ARG and "packed" in e.value.message
    pool.close()
    st.close()


def test_pageable_host_states_are_rejected():
    """Pageable host states are refused; once the same buffers are registered
    (page-locked), the same pool accepts them."""
    cfg = small_config([4096], K=1, steps=1)
    st = _State([inputs.w0_bf16(cfg, 0)], "cpu", pin=False)
    pool = Pool(2, 4096)
    arr, keep = Layers(st, [[0]]).build([DeviceGrads(cfg)(0, 0, 0)])
    with pytest.raises(lema.LemaError) as e:
        pool.stream_layers(arr, 1, hparams(cfg.hyper, 1), 1)
    assert e.value.status == lema.LEMA_ERR_ARG and "pinned" in e.value.message
    cudart = torch.cuda.cudart()
    bufs = list(st.tensors[0].values())
    for t in bufs:
        assert int(cudart.cudaHostRegister(t.data_ptr(), t.numel() * t.element_size(), 0)) == 0
    try:
        pool.stream_layers(arr, 1, hparams(cfg.hyper, 1), 1)
        pool.sync(60_000)
        ref = oracle_states(cfg)
        rep = check_tensor(state_dict(st, 0), dict(oracle_dict(ref[0]), acc=last_step_acc(cfg, 0)))
        assert sum(rep.values()) == 0, rep
    finally:
        torch.cuda.synchronize()
        for t in bufs:
            cudart.cudaHostUnregister(t.data_ptr())
    pool.close()


def test_injected_copy_failure_then_recovery():
    """A copy enqueue that fails (made on the host by the test hook) is reported;
    the pool stays usable and a fresh run is correct."""
    cfg = small_config([20_000, 3000, 9], K=2, steps=2, units=[0, 1, 1])
    sr = StreamedRunner(cfg, DeviceGrads(cfg))
    lema.lema_test_fail_copy(4)
    try:
        with pytest.raises(lema.LemaError) as e:
            sr.step(0)
        assert e.value.status == lema.LEMA_ERR_CUDA and "injected" in e.value.message
    finally:
        lema.lema_test_fail_copy(0)
    sr.pool.sync(60_000)
    fresh = StreamedRunner(cfg, DeviceGrads(cfg))
    fresh.pool.close()
    fresh.pool = sr.pool                       # reuse the pool that saw the failure
    for t in range(cfg.steps):
        fresh.step(t)
    fresh.pool.sync(60_000)
    assert check_streamed(cfg, fresh, oracle_states(cfg)) == 0
    sr.close()


def test_bounded_wait_times_out_then_completes():
    """The pool waits for work on the caller's stream; while that work (a bounded
    spin of ~0.5 s) runs, a 1 ms sync returns LEMA_ERR_TIMEOUT; a long one succeeds."""
    cfg = small_config([8192], K=1, steps=1)
    sr = StreamedRunner(cfg, DeviceGrads(cfg))
    torch.cuda._sleep(int(1e9))
    sr.step(0)
    with pytest.raises(lema.LemaError) as e:
        sr.pool.sync(1)
    assert e.value.status == lema.LEMA_ERR_TIMEOUT
    sr.pool.sync(120_000)
    assert check_streamed(cfg, sr, oracle_states(cfg)) == 0
    sr.close()
