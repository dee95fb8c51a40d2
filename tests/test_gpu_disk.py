"""The disk tier (optimizer states, weights and delta in a file, accumulators in
pinned RAM; lema_stream_layers_disk) on the GPU: the file's contents and the host
accumulator equal the oracle's, element by element, and the streamed path's bits."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from adamw_step_gb300 import lema
from adamw_step_gb300.runner import DeviceGrads, DiskRunner, StreamedRunner
from adamw_step_gb300.state import DiskLayers, DiskState, Pool, hparams
from gpu_common import RAGGED, ensure_library, small_config
from oracle_cache import oracle_states
from parity import check_tensor, oracle_dict, state_dict
from test_gpu_stream import last_step_acc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    return ensure_library()


def run_disk(cfg, path, flags=lema.LEMA_DISK_DIRECT, host_grads=False, n_io_threads=8):
    r = DiskRunner(cfg, DeviceGrads(cfg, pin_host=host_grads), str(path), flags=flags,
                   n_io_threads=n_io_threads)
    for t in range(cfg.steps):
        r.step(t)
    r.sync()
    return r


@pytest.mark.parametrize("flags", [lema.LEMA_DISK_DIRECT, 0], ids=["o_direct", "buffered"])
@pytest.mark.parametrize("K", [1, 2, 3])
def test_disk_tier_matches_oracle(tmp_path, K, flags):
    # 13 ragged tensors in 5 units: the three staging buffers rotate more than once
    cfg = small_config(RAGGED, K=K, steps=3, units=[i // 3 for i in range(len(RAGGED))])
    r = run_disk(cfg, tmp_path / "states.bin", flags)
    ref = oracle_states(cfg)
    try:
        for j in ref:
            want = dict(oracle_dict(ref[j]), acc=last_step_acc(cfg, j))
            rep = check_tensor(state_dict(r.state, j), want, f"disk K={K} tensor {j}")
            assert sum(rep.values()) == 0, rep
    finally:
        r.close()


@pytest.mark.parametrize("q8", [False, True], ids=["fp32", "8-bit"])
def test_disk_tier_device_accumulators(tmp_path, q8):
    """The disk tier with its accumulators in HBM instead of pinned RAM: the file
    and the accumulators equal the oracle's."""
    from oracle.runner import run_config_q8
    from test_gpu_stream_q8 import compare
    sizes, units = (Q8_SIZES, Q8_UNITS) if q8 else (RAGGED, [i // 3 for i in range(len(RAGGED))])
    cfg = small_config(sizes, K=3, steps=2, units=units)
    r = DiskRunner(cfg, DeviceGrads(cfg), str(tmp_path / "acc_dev.bin"), q8=q8,
                   acc_on_device=True)
    for t in range(cfg.steps):
        r.step(t)
    r.sync()
    try:
        if q8:
            compare(r.state, run_config_q8(cfg, fused=True), "q8 disk, device acc")
        else:
            ref = oracle_states(cfg)
            for j in ref:
                want = dict(oracle_dict(ref[j]), acc=last_step_acc(cfg, j))
                rep = check_tensor(state_dict(r.state, j), want, f"disk device acc tensor {j}")
                assert sum(rep.values()) == 0, rep
    finally:
        r.close()


def test_disk_tier_equals_streamed_bits(tmp_path):
    """Nine units of one to three tensors, host-resident grads, two IO threads: the
    file and accumulators end bit-identical to the pinned-RAM streamed path's."""
    sizes = [70_001, 3, 8192, 40_000, 1, 17, 100_003, 64, 65, 5000, 9000, 2048, 777]
    units = [0, 1, 1, 2, 3, 3, 4, 5, 5, 6, 7, 8, 8]
    cfg = small_config(sizes, K=2, steps=3, units=units)
    d = run_disk(cfg, tmp_path / "s.bin", host_grads=True, n_io_threads=2)
    s = StreamedRunner(cfg, DeviceGrads(cfg, pin_host=True))
    for t in range(cfg.steps):
        s.step(t)
    s.pool.sync()
    try:
        for j in range(len(sizes)):
            for a, b in zip(d.state.numpy_views(j), s.state.numpy_views(j)):
                assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), j
    finally:
        d.close()
        s.close()


def test_disk_tier_rejects_state_pointers_and_wrong_units(tmp_path):
    cfg = small_config([5000, 300], K=1, steps=1, units=[0, 1])
    st = DiskState(str(tmp_path / "s.bin"), [torch.zeros(5000, dtype=torch.bfloat16),
                                             torch.zeros(300, dtype=torch.bfloat16)],
                   [[0], [1]], flags=0)
    pool = Pool(2, 8192)
    hp = hparams(cfg.hyper, 1)
    g = [DeviceGrads(cfg)(j, 0, 0) for j in range(2)]
    arr, keep = DiskLayers(st).build(g)
    arr[0].tensors[0].master = st.acc["acc"][0].data_ptr()   # states live in the file
    with pytest.raises(lema.LemaError) as e:
        lema.lema_stream_layers_disk(pool.handle, st.handle, arr, 1, hp, 1)
    assert e.value.status == lema.LEMA_ERR_ARG and "disk file" in e.value.message
    arr, keep = DiskLayers(st).build(g)
    arr[1].tensors[0].n = 400                                 # packs 448, its block 320
    with pytest.raises(lema.LemaError) as e:
        lema.lema_stream_layers_disk(pool.handle, st.handle, arr, 1, hp, 1)
    assert e.value.status == lema.LEMA_ERR_ARG and "disk block" in e.value.message
    pool.close()
    st.close()


@pytest.mark.parametrize("q8", [False, True], ids=["fp32", "8-bit"])
def test_disk_read_failure_is_reported_and_the_pool_stays_usable(tmp_path, q8):
    """A host-made fault: the state file is cut short between steps, so the next
    step's reads hit its end.  The failure comes back as LEMA_ERR_IO (from the call
    or from lema_disk_sync), the pool keeps working, and close() returns."""
    import os
    cfg = small_config([70_001, 8192, 300, 17, 50_000], K=2, steps=3, units=[0, 0, 1, 2, 2])
    path = tmp_path / "s.bin"
    r = DiskRunner(cfg, DeviceGrads(cfg), str(path), flags=0, q8=q8)
    r.step(0)
    r.sync()
    os.truncate(path, r.state.unit_offset[1] + 4096)        # units 1 and 2 now lie past the end
    status = None
    try:
        r.step(1)
    except lema.LemaError as e:
        status = e.status
    try:
        r.state.sync()
    except lema.LemaError as e:
        status = status or e.status
    assert status == lema.LEMA_ERR_IO
    r.pool.sync(60_000)                                     # the GPU side is unharmed
    # a resident step on the same device still runs and matches the oracle
    from adamw_step_gb300.runner import ResidentRunner
    small = small_config([4099, 17], K=1, steps=1)
    rr = ResidentRunner(small, DeviceGrads(small))
    rr.step(0)
    torch.cuda.synchronize()
    ref = oracle_states(small)
    for j in ref:
        assert sum(check_tensor(state_dict(rr.state, j), dict(oracle_dict(ref[j]),
                                acc=np.zeros(small.tensors[j].numel, np.float32))).values()) == 0
    r.close()


# ------------------------------------------------------------ 8-bit states on disk

Q8_SIZES = [1, 7, 0, 255, 256, 257, 1023, 1024, 1025, 8191, 8193, 16640, 100_003]
Q8_UNITS = [0, 0, 0, 1, 1, 2, 2, 2, 3, 3, 4, 4, 5]


def run_disk_q8(cfg, path, flags=lema.LEMA_DISK_DIRECT, host_grads=False, n_io_threads=8):
    r = DiskRunner(cfg, DeviceGrads(cfg, pin_host=host_grads), str(path), flags=flags,
                   n_io_threads=n_io_threads, q8=True)
    for t in range(cfg.steps):
        r.step(t)
    r.sync()
    return r


@pytest.mark.parametrize("flags", [lema.LEMA_DISK_DIRECT, 0], ids=["o_direct", "buffered"])
@pytest.mark.parametrize("K", [1, 2, 3])
def test_q8_disk_tier_matches_oracle(tmp_path, K, flags):
    """13 ragged tensors (with an empty one and sizes around the 256-element block
    and the 1024-element unit offset) in 6 units: every field in the file (master,
    codes, scales, delta, w) and the pinned 8-bit accumulator, bit for bit against
    the oracle's 8-bit form with the last grad folded in."""
    from oracle.runner import run_config_q8
    from test_gpu_stream_q8 import compare
    cfg = small_config(Q8_SIZES, K=K, steps=3, units=Q8_UNITS)
    r = run_disk_q8(cfg, tmp_path / "q8.bin", flags)
    try:
        compare(r.state, run_config_q8(cfg, fused=True), f"q8 disk K={K}")
    finally:
        r.close()


def test_q8_disk_tier_equals_streamed_bits(tmp_path):
    """Host-resident grads and two IO threads: the 8-bit file and accumulators end
    bit-identical to the pinned-RAM 8-bit streamed path's."""
    from adamw_step_gb300.runner import StreamedRunnerQ8
    from test_gpu_stream_q8 import FIELDS
    cfg = small_config(Q8_SIZES, K=2, steps=3, units=Q8_UNITS)
    d = run_disk_q8(cfg, tmp_path / "q8.bin", host_grads=True, n_io_threads=2)
    s = StreamedRunnerQ8(cfg, DeviceGrads(cfg, pin_host=True))
    for t in range(cfg.steps):
        s.step(t)
    s.pool.sync()
    try:
        for j in range(len(Q8_SIZES)):
            a, b = d.state.numpy_views(j), s.state.numpy_views(j)
            for f in FIELDS:
                assert np.array_equal(a[f].view(np.uint8), b[f].view(np.uint8)), (j, f)
    finally:
        d.close()
        s.close()


def test_q8_disk_tier_rejects_state_pointers_and_wrong_units(tmp_path):
    from adamw_step_gb300.state import DiskLayersQ8, DiskStateQ8
    cfg = small_config([5000, 300], K=1, steps=1, units=[0, 1])
    st = DiskStateQ8(str(tmp_path / "s.bin"), [torch.zeros(5000, dtype=torch.bfloat16),
                                               torch.zeros(300, dtype=torch.bfloat16)],
                     [[0], [1]], flags=0)
    pool = Pool(2, 8192)
    hp = hparams(cfg.hyper, 1)
    g = [DeviceGrads(cfg)(j, 0, 0) for j in range(2)]
    arr, keep = DiskLayersQ8(st).build(g)
    arr[0].tensors[0].m_scale = st.acc["acc_scale"][0].data_ptr()   # states live in the file
    with pytest.raises(lema.LemaError) as e:
        lema.lema_stream_layers_disk_q8(pool.handle, st.handle, arr, 1, hp, 1)
    assert e.value.status == lema.LEMA_ERR_ARG and "disk file" in e.value.message
    arr, keep = DiskLayersQ8(st).build(g)
    arr[1].tensors[0].n = 1100                                # packs 2048, its block 1024
    with pytest.raises(lema.LemaError) as e:
        lema.lema_stream_layers_disk_q8(pool.handle, st.handle, arr, 1, hp, 1)
    assert e.value.status == lema.LEMA_ERR_ARG and "disk block" in e.value.message
    pool.close()
    st.close()
