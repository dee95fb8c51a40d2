"""lema_adamw_step_noalloc: the optimizer step for callers that cannot let the
library allocate device memory (a framework that owns all free HBM through its own
allocator, or a loop that cannot afford the device-wide synchronization of
cudaMalloc/cudaFree).  Its descriptor table lives in a fixed device array inside
the library instead.

Through the C ABI, two calls in a row must give the same results as lema_adamw_step
on the same inputs, and the oracle's, within the parity tolerance (the expectation
is bit equality).  Calls after the first must leave the device's free memory and
the torch allocator's counters as they were.  Calls queued back to back on one
stream, with different tensor lists, are ordered.  The file is named to run last,
and it builds everything it needs itself, so it passes alone in a fresh process as
well as after the other tests.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from adamw_step_gb300 import configs, inputs, lema
from adamw_step_gb300.state import DeviceState
from gpu_common import RAGGED, ensure_library
from oracle.runner import run_config
from parity import check_tensor, oracle_dict, state_dict

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    return ensure_library()


def _cfg(sizes, K=2, steps=2):
    tensors = tuple(configs.TensorSpec(f"t{i}", (n,), 0) for i, n in enumerate(sizes))
    return configs.scaled(configs.CONFIGS[1], tensors, accum_steps=K, steps=steps)


def _accumulate(cfg, states, t):
    for k in range(cfg.accum_steps):
        g = [inputs.fresh_grad(cfg, j, t, k).cuda() for j in range(len(cfg.tensors))]
        for st in states:
            lema.lema_accum_grad(st.grad_descs(g))


def test_noalloc_matches_lema_adamw_step_on_two_calls():
    cfg = _cfg(RAGGED + [3 * 8192 + 77])
    w0 = [inputs.w0_bf16(cfg, j) for j in range(len(cfg.tensors))]
    a, b = DeviceState(w0), DeviceState(w0)
    hp = cfg.hyper
    for t in range(2):
        _accumulate(cfg, (a, b), t)
        lema.lema_adamw_step(a.tensor_descs(), t + 1, hp.lr, hp.beta1, hp.beta2, hp.eps,
                             hp.weight_decay, cfg.accum_steps)
        lema.lema_adamw_step_noalloc(b.tensor_descs(), t + 1, hp.lr, hp.beta1, hp.beta2,
                                     hp.eps, hp.weight_decay, cfg.accum_steps)
        torch.cuda.synchronize()
        ref = run_config(cfg, steps=t + 1)
        for j in range(len(cfg.tensors)):
            got = state_dict(b, j)
            rep = check_tensor(got, state_dict(a, j), f"call {t + 1} tensor {j} vs lema_adamw_step")
            assert sum(rep.values()) == 0, rep
            rep = check_tensor(got, oracle_dict(ref[j]), f"call {t + 1} tensor {j} vs oracle")
            assert sum(rep.values()) == 0, rep


def test_noalloc_calls_allocate_nothing():
    """After the first call (which looks up the array's device address), further
    calls change neither the device's free memory nor the torch allocator's
    counters; the descriptors and grads are built before the measurement."""
    cfg = _cfg([70_001, 8192, 5], K=1, steps=6)
    st = DeviceState([inputs.w0_bf16(cfg, j) for j in range(len(cfg.tensors))])
    hp = cfg.hyper
    g = [inputs.fresh_grad(cfg, j, 0, 0).cuda() for j in range(len(cfg.tensors))]
    grads = st.grad_descs(g)
    descs = st.tensor_descs()
    args = (hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, 1)
    lema.lema_accum_grad(grads)
    lema.lema_adamw_step_noalloc(descs, 1, *args)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    stats0 = torch.cuda.memory_stats()
    for t in range(2, 6):
        lema.lema_accum_grad(grads)
        lema.lema_adamw_step_noalloc(descs, t, *args)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    stats1 = torch.cuda.memory_stats()
    assert free1 == free0
    for key in ("allocation.all.allocated", "segment.all.allocated", "reserved_bytes.all.current",
                "allocated_bytes.all.current"):
        assert stats1.get(key, 0) == stats0.get(key, 0), key


def test_noalloc_calls_back_to_back_on_one_stream():
    """Two calls queued on one stream with no host sync between them, over different
    tensor lists (one in place with LEMA_STEP_KEEP_ACC, one out of place): the
    second call's table upload waits for the first call's kernel, so both match the
    oracle."""
    cfg_a = _cfg([100_003, 17, 8192], K=2, steps=1)
    cfg_b = _cfg([5, 3 * 8192 + 1, 4096, 999], K=3, steps=1)
    sa = DeviceState([inputs.w0_bf16(cfg_a, j) for j in range(len(cfg_a.tensors))])
    sb = DeviceState([inputs.w0_bf16(cfg_b, j) for j in range(len(cfg_b.tensors))])
    _accumulate(cfg_a, (sa,), 0)
    _accumulate(cfg_b, (sb,), 0)
    acc_a = [t["acc"].clone() for t in sa.tensors]
    acc_b = [t["acc"].clone() for t in sb.tensors]
    outs = [[torch.empty_like(t["master"]) for _ in range(3)] for t in sb.tensors]
    da = [sa.tensor_desc(j, flags=lema.LEMA_STEP_KEEP_ACC) for j in range(len(sa.tensors))]
    db = [sb.tensor_desc(j, out_of_place=outs[j]) for j in range(len(sb.tensors))]
    torch.cuda.synchronize()
    h = cfg_a.hyper
    torch.cuda._sleep(int(2e7))        # keep the stream busy while both calls are queued
    lema.lema_adamw_step_noalloc(da, 1, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay, 2)
    lema.lema_adamw_step_noalloc(db, 1, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay, 3)
    torch.cuda.synchronize()
    ref_a, ref_b = run_config(cfg_a), run_config(cfg_b)
    for j in range(len(cfg_a.tensors)):
        want = dict(oracle_dict(ref_a[j]), acc=acc_a[j].cpu().numpy())    # KEEP_ACC
        rep = check_tensor(state_dict(sa, j), want, f"first call tensor {j}")
        assert sum(rep.values()) == 0, rep
    for j in range(len(cfg_b.tensors)):
        t = sb.tensors[j]
        got = {"master": outs[j][0].cpu().numpy(), "m": outs[j][1].cpu().numpy(),
               "v": outs[j][2].cpu().numpy(), "delta": t["delta"].cpu().numpy(),
               "acc": t["acc"].cpu().numpy(),
               "w": t["w"].cpu().view(torch.int16).numpy().view(np.uint16)}
        want = dict(oracle_dict(ref_b[j]), acc=acc_b[j].cpu().numpy())    # out of place
        rep = check_tensor(got, want, f"second call tensor {j}")
        assert sum(rep.values()) == 0, rep
        # out of place leaves the inputs as they were
        assert torch.equal(t["master"], t["orig"].float())
        assert torch.all(t["m"] == 0) and torch.all(t["v"] == 0)


def test_noalloc_rejects_sizes_beyond_its_table():
    n = 8
    bufs = [torch.zeros(n * 1025, dtype=torch.float32, device="cuda") for _ in range(5)]
    bf = [torch.zeros(n * 1025, dtype=torch.int16, device="cuda") for _ in range(2)]
    descs = []
    for i in range(1025):
        p = [x[i * n:(i + 1) * n].data_ptr() for x in bufs] + \
            [x[i * n:(i + 1) * n].data_ptr() for x in bf]
        descs.append(lema.LemaTensor(master=p[0], m=p[1], v=p[2], acc=p[3], delta=p[4],
                                     orig_bf16=p[5], w_bf16=p[6], n=n))
    with pytest.raises(lema.LemaError) as e:
        lema.lema_adamw_step_noalloc(descs, 1, 1e-4, 0.9, 0.999, 1e-8, 0.01, 1)
    assert e.value.status == lema.LEMA_ERR_ARG and "1024 tensors" in e.value.message
    # More elements than its chunk map holds (2 x (2^28 + 8192) > 65536 x 8192): real
    # buffers of that size, rejected on the host before anything is copied or launched.
    big = (1 << 28) + 8192
    f32 = [torch.zeros(2 * big, dtype=torch.float32, device="cuda") for _ in range(5)]
    b16 = [torch.zeros(2 * big, dtype=torch.int16, device="cuda") for _ in range(2)]
    descs = []
    for i in range(2):
        p = [x[i * big:(i + 1) * big].data_ptr() for x in f32 + b16]
        descs.append(lema.LemaTensor(master=p[0], m=p[1], v=p[2], acc=p[3], delta=p[4],
                                     orig_bf16=p[5], w_bf16=p[6], n=big))
    before = f32[0][:16].clone()
    with pytest.raises(lema.LemaError) as e:
        lema.lema_adamw_step_noalloc(descs, 1, 1e-4, 0.9, 0.999, 1e-8, 0.01, 1)
    assert e.value.status == lema.LEMA_ERR_ARG and "elements per call" in e.value.message
    torch.cuda.synchronize()
    assert torch.equal(before, f32[0][:16])
    assert np.all(b16[1].cpu().numpy() == 0)
