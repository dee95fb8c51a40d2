"""Seeded random workloads through the C ABI against the oracle, bit for bit.

Each case draws a tensor count (on both sides of the by-value descriptor table's
64-tensor limit), ragged sizes (empty tensors included), K, the number of steps,
the hyperparameters (betas, lr, eps, weight decay inside the method's domain) and
the form (fused: last grad folded in; unfused: K accumulates, then the step), and
runs it resident and streamed (through a pool of two or three slots; every third
case with its accumulators kept in HBM), with fp32 states and with 8-bit states.  Every field must equal the oracle's bits.  The seeds
are fixed, so every run checks the same cases.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle.runner import run_config, run_config_q8
from adamw_step_gb300 import configs
from adamw_step_gb300.runner import (DeviceGrads, ResidentRunner, ResidentRunnerQ8,
                                     StreamedRunner, StreamedRunnerQ8)
from gpu_common import ensure_library
from parity import check_tensor, oracle_dict, partial_acc, state_dict

pytestmark = pytest.mark.gpu
CASES = 40


@pytest.fixture(scope="module", autouse=True)
def lib():
    return ensure_library()


def draw(seed):
    rng = np.random.default_rng(1000 + seed)
    count = int(rng.choice([1, 3, 17, 64, 65, 90]))
    sizes = []
    for _ in range(count):
        kind = rng.integers(0, 4)
        n = (0 if kind == 0 else int(rng.integers(1, 300)) if kind == 1
             else int(rng.integers(1, 9000)) if kind == 2 else int(rng.integers(8000, 70_000)))
        sizes.append(n)
    K = int(rng.integers(1, 6))
    steps = int(rng.integers(1, 4))
    b1 = float(rng.choice([0.0, 0.5, 0.9, 0.95]))
    b2 = float(rng.choice([0.9, 0.99, 0.999, 0.9999]))
    lr = float(rng.choice([0.0, 1e-5, 1e-4, 3e-3]))
    wd = float(rng.choice([0.0, 0.01, 0.1]))
    eps = float(rng.choice([1e-8, 1e-6, 1e-12]))
    units = sorted(int(u) for u in rng.integers(0, max(1, count // 4) + 1, size=count))
    units = [u - units[0] for u in units]
    remap = {u: i for i, u in enumerate(sorted(set(units)))}
    units = [remap[u] for u in units]
    tensors = tuple(configs.TensorSpec(f"f{seed}_{i}", (n,), u)
                    for i, (n, u) in enumerate(zip(sizes, units)))
    cfg = configs.scaled(configs.CONFIGS[1], tensors, accum_steps=K, steps=steps,
                         grad_mode="fresh", name=f"fuzz {seed}",
                         hyper=configs.Hyper(lr=lr, beta1=b1, beta2=b2, eps=eps, weight_decay=wd))
    fused = bool(rng.integers(0, 2))
    return cfg, fused, int(rng.integers(2, 4))


@pytest.mark.parametrize("seed", range(CASES))
def test_fuzz_resident_fp32(seed):
    cfg, fused, _ = draw(seed)
    r = ResidentRunner(cfg, DeviceGrads(cfg), fused=fused)
    for t in range(cfg.steps):
        r.step(t)
    torch.cuda.synchronize()
    ref = run_config(cfg)
    for j, st in ref.items():
        want = oracle_dict(st)
        if fused:
            want = dict(want, acc=partial_acc(cfg, j))
        rep = check_tensor(state_dict(r.state, j), want, f"seed {seed} tensor {j}")
        assert sum(rep.values()) == 0, rep


@pytest.mark.parametrize("seed", range(CASES))
def test_fuzz_resident_q8(seed):
    cfg, fused, _ = draw(seed)
    r = ResidentRunnerQ8(cfg, DeviceGrads(cfg), fused=fused)
    for t in range(cfg.steps):
        r.step(t)
    torch.cuda.synchronize()
    for j, st in run_config_q8(cfg, fused=fused).items():
        got = r.state.numpy_views(j)
        for f in ("master", "delta", "w", "m_q", "m_scale", "r_q", "r_scale", "acc_q",
                  "acc_scale"):
            same = got[f].view(np.uint8) == getattr(st, f).view(np.uint8)
            assert same.all(), f"seed {seed} tensor {j} {f}: byte {np.flatnonzero(~same)[:3]}"


@pytest.mark.parametrize("seed", range(CASES))
def test_fuzz_streamed_fp32(seed):
    cfg, _, n_slots = draw(seed)
    # every third case keeps its accumulators in HBM (only the states stream)
    sr = StreamedRunner(cfg, DeviceGrads(cfg), n_slots=n_slots, acc_on_device=seed % 3 == 1)
    try:
        for t in range(cfg.steps):
            sr.step(t)
        sr.pool.sync(120_000)
        ref = run_config(cfg)
        for j, st in ref.items():
            # the host accumulator keeps micro-steps 1..K-1 of the last step
            want = dict(oracle_dict(st), acc=partial_acc(cfg, j))
            rep = check_tensor(state_dict(sr.state, j), want, f"seed {seed} tensor {j}")
            assert sum(rep.values()) == 0, rep
    finally:
        sr.close()


@pytest.mark.parametrize("seed", range(CASES))
def test_fuzz_streamed_q8(seed):
    cfg, _, n_slots = draw(seed)
    sr = StreamedRunnerQ8(cfg, DeviceGrads(cfg), n_slots=n_slots, acc_on_device=seed % 3 == 1)
    try:
        for t in range(cfg.steps):
            sr.step(t)
        sr.pool.sync(120_000)
        for j, st in run_config_q8(cfg, fused=True).items():
            got = sr.state.numpy_views(j)
            for f in ("master", "delta", "w", "m_q", "m_scale", "r_q", "r_scale", "acc_q",
                      "acc_scale"):
                same = got[f].view(np.uint8) == getattr(st, f).view(np.uint8)
                assert same.all(), f"seed {seed} tensor {j} {f}: byte {np.flatnonzero(~same)[:3]}"
    finally:
        sr.close()


@pytest.mark.parametrize("seed", range(0, CASES, 2))
def test_fuzz_noalloc_out_of_place_and_shards(seed):
    """The same random workloads, unfused, through three other forms of the step,
    each against the oracle: lema_adamw_step_noalloc in place, lema_adamw_step out of
    place (fresh outputs every step, the inputs then copied forward), and the step
    sharded over 2-5 "ranks" (each an aligned element range of every tensor, run one
    after another)."""
    from adamw_step_gb300 import inputs, lema
    from adamw_step_gb300.shard import shard_bounds, shard_grad, shard_tensor
    from adamw_step_gb300.state import DeviceState
    cfg, _, _ = draw(seed)
    world = 2 + seed % 4
    hp, K = cfg.hyper, cfg.accum_steps
    args = lambda t: (t + 1, hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, K)  # noqa: E731
    w0 = [inputs.w0_bf16(cfg, j) for j in range(len(cfg.tensors))]
    a, b, c = DeviceState(w0), DeviceState(w0), DeviceState(w0)
    n = [x.numel for x in cfg.tensors]
    for t in range(cfg.steps):
        grads = [[inputs.fresh_grad(cfg, j, t, k).cuda() for j in range(len(n))] for k in range(K)]
        for st in (a, b, c):
            for k in range(K):
                lema.lema_accum_grad(st.grad_descs(grads[k], first=k == 0))
        lema.lema_adamw_step_noalloc(a.tensor_descs(), *args(t))
        outs = [[torch.empty_like(x["master"]) for _ in range(3)] for x in b.tensors]
        lema.lema_adamw_step([b.tensor_desc(j, out_of_place=outs[j]) for j in range(len(n))],
                             *args(t))
        for rank in range(world):
            bounds = [shard_bounds(x, rank, world) for x in n]
            d = c.tensor_descs()
            lema.lema_adamw_step([shard_tensor(d[j], *bounds[j]) for j in range(len(n))],
                                 *args(t))
        torch.cuda.synchronize()
        for j, x in enumerate(b.tensors):       # out of place: carry the outputs forward
            for f, o in zip(("master", "m", "v"), outs[j]):
                x[f].copy_(o)
            x["acc"].zero_()                    # an out-of-place step leaves acc as it was
    ref = run_config(cfg)
    for st, label in ((a, "noalloc"), (b, "out of place"), (c, f"{world} shards")):
        for j, r in ref.items():
            rep = check_tensor(state_dict(st, j), oracle_dict(r), f"seed {seed} {label} tensor {j}")
            assert sum(rep.values()) == 0, rep
