"""8-bit optimizer states on the GPU against the oracle's 8-bit form, every field
(codes, block scales, master, delta, bf16 weight) bit for bit, through the C ABI."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle.runner import run_config_q8
from adamw_step_gb300 import configs, lema
from adamw_step_gb300.runner import DeviceGrads, ResidentRunnerQ8
from gpu_common import ensure_library, small_config

pytestmark = pytest.mark.gpu
SIZES = [1, 7, 8, 9, 0, 255, 256, 257, 511, 8191, 8192, 8193, 16640, 100_003]
FIELDS = ("master", "delta", "w", "m_q", "m_scale", "r_q", "r_scale", "acc_q", "acc_scale")


@pytest.fixture(scope="module", autouse=True)
def lib():
    return ensure_library()


def run_q8(cfg, fused):
    r = ResidentRunnerQ8(cfg, DeviceGrads(cfg), fused=fused)
    for t in range(cfg.steps):
        r.step(t)
    torch.cuda.synchronize()
    return r


def compare(r, ref, label):
    for j, st in ref.items():
        got = r.state.numpy_views(j)
        want = {"master": st.master, "delta": st.delta, "w": st.w, "m_q": st.m_q,
                "m_scale": st.m_scale, "r_q": st.r_q, "r_scale": st.r_scale,
                "acc_q": st.acc_q, "acc_scale": st.acc_scale}
        for f in FIELDS:
            a, b = got[f], want[f]
            same = a.view(np.uint8) == b.view(np.uint8)
            assert same.all(), f"{label} tensor {j} {f}: first mismatch at byte {np.flatnonzero(~same)[:3]}"
        # and the stated fp32 tolerance, trivially implied by the bit equality above
        ok = np.abs(got["master"].astype(np.float64) - st.master) <= np.maximum(2e-6 * np.abs(st.master), 1e-9)
        assert ok.all()


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "unfused"])
@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_q8_ragged_bit_exact(K, fused):
    cfg = small_config(SIZES, K=K, steps=3)
    compare(run_q8(cfg, fused), run_config_q8(cfg, fused=fused), f"q8 K={K}")


@pytest.mark.parametrize("count", [16, 17, 64, 65])
def test_q8_descriptor_table_sizes(count):
    """By-value tables (up to 16, up to 64 tensors) and the uploaded one, both sides
    of each boundary, both 8-bit kernels."""
    sizes = [(i * 977) % 9000 + (8192 if i % 5 == 0 else 0) for i in range(count)]
    cfg = small_config(sizes, K=2, steps=2)
    compare(run_q8(cfg, fused=True), run_config_q8(cfg, fused=True), f"q8 {count} tensors")


def test_q8_config2_full():
    """The 268M-param workload with 8-bit states, K=8, 5 steps; every element of
    every tensor against the oracle."""
    from oracle_cache import oracle_states_q8
    cfg = configs.CONFIGS[2]
    r = run_q8(cfg, fused=True)
    compare(r, oracle_states_q8(cfg, fused=True), "q8 config 2")


def test_q8_argument_checks():
    cfg = small_config([4096], K=2, steps=1)
    r = ResidentRunnerQ8(cfg, DeviceGrads(cfg))
    hp = cfg.hyper
    args = (1, hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay)
    with pytest.raises(lema.LemaError) as e:          # no accumulator with K = 2
        lema.lema_adamw_step_q8([r.state.tensor_desc(0, grad=r.grads(0, 0, 1), with_acc=False)],
                                *args, 2)
    assert e.value.status == lema.LEMA_ERR_ARG
    d = r.state.tensor_desc(0)
    d.m_q_out = d.m_q                                 # only one of the five outputs
    with pytest.raises(lema.LemaError) as e:
        lema.lema_adamw_step_q8([d], *args, 2)
    assert e.value.status == lema.LEMA_ERR_ARG
    d = r.state.tensor_desc(0)
    d.r_q = d.m_q                                     # two code arrays on the same bytes
    with pytest.raises(lema.LemaError) as e:
        lema.lema_adamw_step_q8([d], *args, 2)
    assert e.value.status == lema.LEMA_ERR_ARG and "overlap" in e.value.message
    d = r.state.tensor_desc(0)
    d.m_scale = d.m_scale + 4                         # misaligned
    with pytest.raises(lema.LemaError) as e:
        lema.lema_adamw_step_q8([d], *args, 2)
    assert e.value.status == lema.LEMA_ERR_ALIGN


def test_q8_out_of_place_leaves_inputs():
    cfg = small_config([70_001, 300], K=2, steps=1)
    a = run_q8(cfg, fused=False)
    b = ResidentRunnerQ8(cfg, DeviceGrads(cfg), fused=False)
    b.accumulate(0)
    outs = []
    descs = []
    for j, t in enumerate(b.state.tensors):
        o = {"master": torch.empty_like(t["master"]), "m_q": torch.empty_like(t["m_q"]),
             "m_scale": torch.empty_like(t["m_scale"]), "r_q": torch.empty_like(t["r_q"]),
             "r_scale": torch.empty_like(t["r_scale"])}
        outs.append(o)
        d = b.state.tensor_desc(j)
        d.master_out, d.m_q_out, d.m_scale_out = o["master"].data_ptr(), o["m_q"].data_ptr(), o["m_scale"].data_ptr()
        d.r_q_out, d.r_scale_out = o["r_q"].data_ptr(), o["r_scale"].data_ptr()
        descs.append(d)
    acc_before = [t["acc_q"].clone() for t in b.state.tensors]
    hp = cfg.hyper
    lema.lema_adamw_step_q8(descs, 1, hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, 2)
    torch.cuda.synchronize()
    for j, t in enumerate(b.state.tensors):
        ta = a.state.tensors[j]
        for f in ("master", "m_q", "m_scale", "r_q", "r_scale"):
            assert torch.equal(outs[j][f].view(torch.uint8), ta[f].view(torch.uint8)), f
        assert torch.equal(t["acc_q"], acc_before[j])
        assert torch.all(t["m_q"] == 0) and torch.equal(t["master"], t["orig"].float())


def test_q8_tiny_blocks_match_the_oracle():
    """Blocks with magnitudes just below and just above 2^-100 (the rule that stores
    tiny blocks as zero), and subnormal grads, through the 8-bit accumulate."""
    import oracle
    from oracle import OracleStateQ8
    n = 256 * 4 + 40
    rng = np.random.default_rng(5)
    x = rng.uniform(-1, 1, n).astype(np.float32)      # |x| < 1 before scaling
    x[:256] *= np.float32(2.0 ** -101)                # every |x| < 2^-100: stored as zero
    x[256:512] *= np.float32(2.0 ** -99)
    x[300] = np.float32(2.0 ** -99)                   # a maximum above the threshold
    x[512:768] *= np.float32(2.0 ** -130)             # subnormal fp32 / bf16
    x[768:] *= np.float32(1e-3)
    g = torch.from_numpy(x).to(torch.bfloat16)
    orc = oracle.Oracle()
    st = OracleStateQ8(np.zeros(n, np.uint16), orc)
    from adamw_step_gb300.inputs import as_u16
    orc.accum_q8(st, as_u16(g), first=True)
    acc_q = torch.zeros(n, dtype=torch.int8, device="cuda")
    acc_s = torch.full(((n + 255) // 256,), 7.0, dtype=torch.float32, device="cuda")
    gd = g.cuda()
    lema.lema_accum_grad_q8([lema.LemaGradQ8(acc_q=acc_q.data_ptr(), acc_scale=acc_s.data_ptr(),
                                             grad_bf16=gd.data_ptr(), n=n,
                                             flags=lema.LEMA_GRAD_FIRST)])
    torch.cuda.synchronize()
    assert np.array_equal(acc_q.cpu().numpy(), st.acc_q)
    assert np.array_equal(acc_s.cpu().numpy().view(np.uint32), st.acc_scale.view(np.uint32))
    assert st.acc_scale[0] == 0 and st.acc_scale[1] > 0


def test_division_by_the_per_call_constant_is_exact():
    """The 8-bit step divides sqrt(v) by c = sqrt(1 - beta2^t) with a correctly
    rounded reciprocal and two fused multiply-adds (Markstein's method); for every
    x >= 0 in its domain that must equal the IEEE division: the divisors of steps
    1..200 for several beta2, the ends of the allowed range, all-ones significands
    and random divisors."""
    import math
    cs = set()
    for beta2 in (0.999, 0.99, 0.95, 0.9, 0.5, 0.9999):
        p = 1.0
        for _ in range(200):
            p *= beta2                      # fp64, one factor at a time, as the host does
            cs.add(float(np.float32(math.sqrt(1.0 - p))))
    edge = [1.0, float(np.nextafter(np.float32(2.0 ** -27), np.float32(1))),
            float(np.nextafter(np.float32(1), np.float32(0)))]
    edge += [float(np.float32((2 - 2.0 ** -23) * 2.0 ** -k)) for k in range(1, 28)]
    rng = np.random.default_rng(3)
    rand = [float(x) for x in np.float32(2.0 ** rng.uniform(-26.9, 0, 200))]
    divisors = sorted(c for c in cs | set(edge) | set(rand) if 2.0 ** -27 < c <= 1.0)
    bad, outside = lema.lema_test_divide_by_constant(divisors)
    wrong = [(c, b) for c, b in zip(divisors, bad) if b]
    assert not wrong, f"{len(wrong)} divisors with mismatches, e.g. {wrong[:3]}"
    assert len(divisors) > 900


def test_no_kernel_wait_ran_out():
    """The staged 8-bit step waits (bounded) for its shared-memory copies; no launch
    of an ordinary run gives up."""
    before = lema.lema_kernel_wait_timeouts()
    run_q8(small_config([3 * 8192, 8192 + 5], K=2, steps=2), fused=True)
    run_q8(configs.CONFIGS[1], fused=True)
    assert lema.lema_kernel_wait_timeouts() == before
