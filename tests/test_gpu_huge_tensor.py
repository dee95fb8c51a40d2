"""One tensor of more than 2^31 elements (64-bit element indexing in the chunk map,
the kernels and the launch grid), resident, two micro-steps and two steps, on the
fused and the plain form, with fp32 and with 8-bit states: sampled ranges below and
above 2^31 and the ragged tail against the oracle, which is elementwise (for 8-bit
states, blockwise over 256-element blocks, so a block-aligned slice of the inputs
gives that slice of the result).  Inputs are seeded PyTorch draws on the device
(copied to the host for the oracle); they never come from this library."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from oracle import Hyper
from adamw_step_gb300 import lema
from adamw_step_gb300.state import DeviceState, DeviceStateQ8
from gpu_common import ensure_library

pytestmark = pytest.mark.gpu
N = (1 << 31) + 1000
RANGES = [(0, 70_000), ((1 << 31) - 40_000, (1 << 31) + 40), (N - 9000, N)]


@pytest.fixture(scope="module", autouse=True)
def lib():
    ensure_library()
    free, _ = torch.cuda.mem_get_info()
    if free < 80 << 30:
        pytest.skip(f"needs 80 GiB of free device memory, {free >> 30} GiB free")


def _u16(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "plain"])
def test_tensor_beyond_2_31_elements(fused):
    g = torch.Generator(device="cuda").manual_seed(20260101)
    w0 = (torch.randn(N, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    K, steps = 2, 2
    grads = [[(torch.randn(N, device="cuda", generator=g) * 1e-3).to(torch.bfloat16)
              for _ in range(K)] for _ in range(steps)]
    st = DeviceState([w0])
    hp = Hyper(accum_steps=K)
    for t in range(steps):
        for k in range(K if not fused else K - 1):
            lema.lema_accum_grad(st.grad_descs([grads[t][k]], first=fused and k == 0))
        d = st.tensor_desc(0, grad=grads[t][K - 1] if fused else None,
                           flags=lema.LEMA_STEP_KEEP_ACC if fused else 0)
        lema.lema_adamw_step([d], t + 1, hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, K)
    torch.cuda.synchronize()

    orc = oracle.Oracle()
    for a, b in RANGES:
        ref = oracle.OracleState(_u16(w0[a:b]), orc)
        for t in range(steps):
            for k in range(K):
                orc.accum(ref.acc, _u16(grads[t][k][a:b]))
            orc.adamw_step(ref, t + 1, hp)
        for f, want in (("master", ref.master), ("m", ref.m), ("v", ref.v), ("delta", ref.delta)):
            got = st.tensors[0][f][a:b].cpu().numpy()
            assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), (f, a, b)
        assert np.array_equal(_u16(st.tensors[0]["w"][a:b]), ref.w), ("w", a, b)
    del st, grads, w0
    torch.cuda.empty_cache()


# block-aligned ranges (256 elements) for the 8-bit states; the last one ends in the
# ragged last block of the tensor
RANGES_Q8 = [(0, 70_144), ((1 << 31) - 40_960, (1 << 31) + 256), ((N - 9000) // 256 * 256, N)]


def test_q8_tensor_beyond_2_31_elements():
    """The 8-bit step and accumulate (fused form: micro-step 1 into the 8-bit
    accumulator, micro-step 2 folded into the step) on one tensor of 2^31 + 1000
    elements: every field, codes and block scales included, bit for bit."""
    g = torch.Generator(device="cuda").manual_seed(20260102)
    w0 = (torch.randn(N, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    K, steps = 2, 2
    grads = [[(torch.randn(N, device="cuda", generator=g) * 1e-3).to(torch.bfloat16)
              for _ in range(K)] for _ in range(steps)]
    st = DeviceStateQ8([w0])
    hp = Hyper(accum_steps=K)
    for t in range(steps):
        lema.lema_accum_grad_q8(st.grad_descs([grads[t][0]], first=True))
        d = st.tensor_desc(0, grad=grads[t][1], flags=lema.LEMA_STEP_KEEP_ACC)
        lema.lema_adamw_step_q8([d], t + 1, hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, K)
    torch.cuda.synchronize()

    orc = oracle.Oracle(threads=8)
    tq = st.tensors[0]
    for a, b in RANGES_Q8:
        ref = oracle.OracleStateQ8(_u16(w0[a:b]), orc)
        for t in range(steps):
            orc.accum_q8(ref, _u16(grads[t][0][a:b]), first=True)
            orc.adamw_step_q8(ref, t + 1, hp, grad_last=_u16(grads[t][1][a:b]))
        ba, bb = a // 256, (b + 255) // 256
        for f, want, lo, hi in (("master", ref.master, a, b), ("delta", ref.delta, a, b),
                                ("m_q", ref.m_q, a, b), ("r_q", ref.r_q, a, b),
                                ("acc_q", ref.acc_q, a, b), ("m_scale", ref.m_scale, ba, bb),
                                ("r_scale", ref.r_scale, ba, bb),
                                ("acc_scale", ref.acc_scale, ba, bb)):
            got = tq[f][lo:hi].cpu().numpy()
            assert np.array_equal(got.view(np.uint8), want.view(np.uint8)), (f, a, b)
        assert np.array_equal(_u16(tq["w"][a:b]), ref.w), ("w", a, b)
    del st, grads, w0
    torch.cuda.empty_cache()
