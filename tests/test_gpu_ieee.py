"""IEEE special values through the fp32 path, element by element against the oracle.

Reading of the LEMA page's section "Selective Full Fine-Tuning" (fp32 states and
accumulators) taken by both sides: every operation is an IEEE fp32 operation rounded
to nearest even with subnormals kept (no flush to zero, no denormals-are-zero), NaN
and infinities propagate, nothing is skipped or clipped.  The ordinary workloads
never leave the normal range, so these cases feed the kernels inputs that do:

* grads near 1e-20, whose squares, (1 - beta2) g^2 and v are subnormal;
* accumulators, moments and masters holding +-Inf, NaN, -0 and values near FLT_MAX,
  so that m / den, the update, the delta and the bf16 rounding overflow;
* bf16 grads and originals that are subnormal, infinite or NaN;
* beta1 = 0, lr = 0, a subnormal eps, K = 3 (divide) and K = 4 (the exact
  reciprocal multiply), steps 1 and 7.

The 8-bit path gets the finite part of this (its states must be finite) and the
serving merge bf16(base + delta) the whole of it.  Every field must equal the
oracle's bits (NaN compared as NaN).  A build that flushed subnormals
(``-ftz=true``) or contracted into FMA would fail here.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from adamw_step_gb300 import lema
from adamw_step_gb300.state import DeviceStateQ8, HostState, Layers, Pool
from adamw_step_gb300.lema import LemaHparams
from gpu_common import ensure_library
from parity import check_tensor

pytestmark = pytest.mark.gpu

N = 3 * 8192 + 5          # several chunks and a ragged tail
FMAX = np.float32(3.4028235e38)
F32_SPECIALS = np.array([
    0.0, -0.0, np.inf, -np.inf, np.nan, FMAX, -FMAX, 3.3e38, -3.3e38, 1e-20, -1e-20,
    3e-21, 1e-40, -1e-40, 1.4e-45, -1.4e-45, 1.1754944e-38, -1.1754944e-38, 1.0, -1.0,
    1e-8, 2e19, -2e19], dtype=np.float32)
# bf16 patterns: +-0, +-Inf, NaNs (one with a payload), the largest finite, the
# smallest subnormal and normal, 2^-66 (about 1.4e-20), 1e-3-ish, 2^64.
BF16_SPECIALS = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0xFFC1, 0x7F7F, 0xFF7F,
                          0x0001, 0x8001, 0x0080, 0x8080, 0x1E80, 0x9E80, 0x3A83, 0xBA83,
                          0x5F80, 0xDF80], dtype=np.uint16)

HPARAMS = {
    "default": dict(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01),
    "beta1=0": dict(lr=1e-4, beta1=0.0, beta2=0.999, eps=1e-8, weight_decay=0.01),
    "lr=0": dict(lr=0.0, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01),
    "subnormal eps": dict(lr=0.5, beta1=0.5, beta2=0.5, eps=1e-40, weight_decay=1.0),
}


@pytest.fixture(scope="module", autouse=True)
def lib():
    return ensure_library()


def _mix_f32(rng, n, scale, frac=0.5, nonneg=False):
    x = (rng.standard_normal(n) * scale).astype(np.float32)
    if nonneg:
        x = np.abs(x)
    pick = rng.random(n) < frac
    x[pick] = F32_SPECIALS[rng.integers(0, F32_SPECIALS.size, int(pick.sum()))]
    return x


def _mix_bf16(rng, n, scale, frac=0.5):
    x = torch.from_numpy((rng.standard_normal(n) * scale).astype(np.float32))
    h = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    pick = rng.random(n) < frac
    h[pick] = BF16_SPECIALS[rng.integers(0, BF16_SPECIALS.size, int(pick.sum()))]
    return h


def special_inputs(seed, n=N):
    """master, m, v, acc (fp32) and orig, grad (bf16 bit patterns)."""
    rng = np.random.default_rng(seed)
    master = _mix_f32(rng, n, 0.02)
    m = _mix_f32(rng, n, 1e-4)
    v = _mix_f32(rng, n, 1e-8, nonneg=True)
    v[rng.random(n) < 0.01] *= -1          # a few negative second moments: sqrt gives NaN
    acc = _mix_f32(rng, n, 1e-3)
    orig = _mix_bf16(rng, n, 0.02)
    grad = _mix_bf16(rng, n, 1e-3)
    return master, m, v, acc, orig, grad


def _dev_f32(a):
    return torch.from_numpy(a.copy()).cuda()


def _dev_u16(a):
    return torch.from_numpy(a.view(np.int16).copy()).cuda()


def _host(t, u16=False):
    a = t.cpu().numpy()
    return a.view(np.uint16) if u16 else a


def oracle_step(master, m, v, acc, orig, grad, step, hp, K):
    """The oracle's step on these inputs; grad (or None) is folded in with the same
    single fp32 add as an accumulate."""
    orc = oracle.Oracle()
    acc_sum = acc.copy()
    if grad is not None:
        orc.accum(acc_sum, grad)
    h = oracle.Hyper(accum_steps=K, **hp)
    mo, mm, vv, d, w = orc.adamw_step_arrays(master.copy(), m.copy(), v.copy(), acc_sum,
                                             orig.copy(), step, h)
    return {"master": mo, "m": mm, "v": vv, "delta": d, "w": w}


@pytest.mark.parametrize("hp_name", list(HPARAMS))
@pytest.mark.parametrize("K", [3, 4])
@pytest.mark.parametrize("fold", [False, True], ids=["unfused", "fused"])
@pytest.mark.parametrize("in_place", [True, False], ids=["in-place", "out-of-place"])
def test_step_special_values(hp_name, K, fold, in_place):
    hp = HPARAMS[hp_name]
    seed = 17 + 3 * K + (5 if fold else 0) + (11 if in_place else 0) + list(HPARAMS).index(hp_name)
    master, m, v, acc, orig, grad = special_inputs(seed)
    dm, dmm, dv, dacc = (_dev_f32(x) for x in (master, m, v, acc))
    dorig, dgrad = _dev_u16(orig), _dev_u16(grad)
    delta = torch.full((N,), 7.0, dtype=torch.float32, device="cuda")
    w = torch.zeros(N, dtype=torch.int16, device="cuda")
    outs = [torch.empty(N, dtype=torch.float32, device="cuda") for _ in range(3)]
    desc = lema.LemaTensor(master=dm.data_ptr(), m=dmm.data_ptr(), v=dv.data_ptr(),
                           acc=dacc.data_ptr(), delta=delta.data_ptr(),
                           orig_bf16=dorig.data_ptr(), w_bf16=w.data_ptr(),
                           grad_bf16=dgrad.data_ptr() if fold else None, n=N)
    if not in_place:
        desc.master_out, desc.m_out, desc.v_out = (o.data_ptr() for o in outs)
    for step in (1, 7):
        want = oracle_step(master, m, v, acc, orig, grad if fold else None, step, hp, K)
        # each call starts from the same inputs
        for d, h in ((dm, master), (dmm, m), (dv, v), (dacc, acc)):
            d.copy_(torch.from_numpy(h))
        lema.lema_adamw_step([desc], step, hp["lr"], hp["beta1"], hp["beta2"], hp["eps"],
                             hp["weight_decay"], K)
        torch.cuda.synchronize()
        src = (dm, dmm, dv) if in_place else outs
        got = {"master": _host(src[0]), "m": _host(src[1]), "v": _host(src[2]),
               "delta": _host(delta), "w": _host(w, u16=True)}
        # an in-place step resets the accumulator to +0; an out-of-place one leaves it
        got["acc"] = _host(dacc)
        want["acc"] = np.zeros(N, np.float32) if in_place else acc
        rep = check_tensor(got, want, f"{hp_name} K={K} step={step}")
        assert sum(rep.values()) == 0, rep
        if not in_place:
            for d, h in ((dm, master), (dmm, m), (dv, v)):
                assert np.array_equal(_host(d).view(np.uint32), h.view(np.uint32))
    # the inputs did reach the regimes this test is about
    assert np.isnan(want["master"]).any() and np.isinf(want["master"]).any()
    tiny = np.abs(want["v"]) < np.float32(1.1754944e-38)
    assert (tiny & (want["v"] != 0)).any(), "no subnormal v in the oracle's result"


def test_accumulate_special_values():
    """acc + (fp32) g with Inf, NaN, -0, subnormal and overflowing sums, and the first
    micro-step's +0 + g, against the oracle's accumulate."""
    master, m, v, acc, orig, grad = special_inputs(5)
    orc = oracle.Oracle()
    for first in (False, True):
        dacc, dgrad = _dev_f32(acc), _dev_u16(grad)
        lema.lema_accum_grad([lema.LemaGrad(acc=dacc.data_ptr(), grad_bf16=dgrad.data_ptr(), n=N,
                                            flags=lema.LEMA_GRAD_FIRST if first else 0)])
        torch.cuda.synchronize()
        want = np.zeros(N, np.float32) if first else acc.copy()
        orc.accum(want, grad)
        got = _host(dacc)
        same = (got.view(np.uint32) == want.view(np.uint32)) | (np.isnan(got) & np.isnan(want))
        assert same.all(), f"first={first}: {np.flatnonzero(~same)[:5]}"
        if first:       # +0 + g: a zero sum is +0, never -0
            assert not np.any((got == 0) & np.signbit(got))


def test_streamed_special_values():
    """The same regimes through lema_stream_layers: pinned host states, a 2-slot
    pool, K = 2 (micro-step 1 from +0, micro-step 2 folded into the step)."""
    sizes, units = [N, 8195, 77], [[0], [1, 2]]
    rng_inputs = [special_inputs(100 + j, n) for j, n in enumerate(sizes)]
    w0 = [torch.from_numpy(x[4].view(np.int16).copy()).view(torch.bfloat16) for x in rng_inputs]
    st = HostState(w0, units=units)
    for j, (master, m, v, _, _, _) in enumerate(rng_inputs):
        for f, x in (("master", master), ("m", m), ("v", v)):
            st.tensors[j][f].copy_(torch.from_numpy(x))
    # the two micro-steps' grads: the fixture's grad, then a second special mix
    g1 = [x[5] for x in rng_inputs]
    g2 = [_mix_bf16(np.random.default_rng(200 + j), n, 1e-3) for j, n in enumerate(sizes)]
    dg1 = [_dev_u16(g) for g in g1]
    dg2 = [_dev_u16(g) for g in g2]
    hp = HPARAMS["default"]
    K = 2
    pool = Pool(2, max(sum((sizes[j] + 63) // 64 * 64 for j in u) for u in units))
    lay = Layers(st, units)
    hpa = LemaHparams(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"], K)
    for k, g in ((1, dg1), (2, dg2)):
        arr, keep = lay.build(g)
        pool.stream_layers(arr, k, hpa, 3)
    pool.sync(60_000)
    orc = oracle.Oracle()
    for j, (master, m, v, _, orig, _) in enumerate(rng_inputs):
        acc1 = np.zeros(sizes[j], np.float32)
        orc.accum(acc1, g1[j])
        want = oracle_step(master, m, v, acc1, orig, g2[j], 3, hp, K)
        want["acc"] = acc1                  # the host acc keeps micro-step 1's sum
        g_master, g_m, g_v, g_acc, g_delta, _, g_w = st.numpy_views(j)
        got = {"master": g_master, "m": g_m, "v": g_v, "acc": g_acc, "delta": g_delta, "w": g_w}
        rep = check_tensor(got, want, f"streamed tensor {j}")
        assert sum(rep.values()) == 0, rep
    pool.close()
    st.close()


# 8-bit states must stay finite (a NaN or an infinity has no code), so their case
# keeps every value finite: tiny and subnormal grads and weights, signed zeros, and
# grads as large as 2^61, whose square (2^122) is still an fp32 number.
BF16_FINITE = np.array([0x0000, 0x8000, 0x0001, 0x8001, 0x007F, 0x0080, 0x8080, 0x1E80, 0x9E80,
                        0x3A83, 0xBA83, 0x5B00, 0xDB00, 0x5E00, 0xDE00], dtype=np.uint16)


def _mix_bf16_finite(rng, n, scale, frac=0.5):
    x = torch.from_numpy((rng.standard_normal(n) * scale).astype(np.float32))
    h = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    pick = rng.random(n) < frac
    h[pick] = BF16_FINITE[rng.integers(0, BF16_FINITE.size, int(pick.sum()))]
    return h


@pytest.mark.parametrize("K", [2, 3])
def test_q8_step_tiny_subnormal_and_large_values(K):
    """The 8-bit accumulate and step (fused form) on weights and grads that include
    bf16 subnormals, +-0, 2^-66 and values up to 2^61 (0x5E00: g^2 stays finite):
    codes, block scales, master, delta and bf16 weight bit for bit against the
    oracle's 8-bit form, two steps."""
    n = 5 * 2048 + 300                      # staged groups and a ragged end
    rng = np.random.default_rng(40 + K)
    w0 = _mix_bf16_finite(rng, n, 0.02)
    grads = [[_mix_bf16_finite(rng, n, 1e-3) for _ in range(K)] for _ in range(2)]
    st = DeviceStateQ8([torch.from_numpy(w0.view(np.int16).copy()).view(torch.bfloat16)])
    dg = [[_dev_u16(g) for g in row] for row in grads]
    h = oracle.Hyper(accum_steps=K)
    for t in range(2):
        for k in range(K - 1):
            lema.lema_accum_grad_q8(st.grad_descs([dg[t][k]], first=(k == 0)))
        d = st.tensor_desc(0, grad=dg[t][K - 1], flags=lema.LEMA_STEP_KEEP_ACC)
        lema.lema_adamw_step_q8([d], t + 1, h.lr, h.beta1, h.beta2, h.eps, h.weight_decay, K)
    torch.cuda.synchronize()
    orc = oracle.Oracle()
    ref = oracle.OracleStateQ8(w0, orc)
    for t in range(2):
        for k in range(K - 1):
            orc.accum_q8(ref, grads[t][k], first=(k == 0))
        orc.adamw_step_q8(ref, t + 1, h, grad_last=grads[t][K - 1])
    got = st.numpy_views(0)
    for f in ("master", "delta", "w", "m_q", "m_scale", "r_q", "r_scale", "acc_q", "acc_scale"):
        a, b = got[f], getattr(ref, f)
        same = a.view(np.uint8) == b.view(np.uint8)
        assert same.all(), f"K={K} {f}: first mismatch at byte {np.flatnonzero(~same)[:3]}"
    assert np.isfinite(ref.master).all() and np.isfinite(ref.r_scale).all()


def test_merge_special_values():
    """bf16(base + delta) with NaN, +-Inf, -0, subnormal and overflowing sums, against
    the oracle's merge bit for bit (a NaN result is the bf16 pattern 0x7FC0 on both
    sides); in place and out of place."""
    rng = np.random.default_rng(77)
    n = 3 * 8192 + 21
    base = _mix_bf16(rng, n, 0.02)
    delta = _mix_f32(rng, n, 1e-4)
    want = oracle.Oracle().merge_delta(base, delta)
    for in_place in (False, True):
        db, dd = _dev_u16(base), _dev_f32(delta)
        out = db if in_place else torch.zeros(n, dtype=torch.int16, device="cuda")
        lema.lema_merge_delta([lema.LemaMerge(base_bf16=db.data_ptr(), delta=dd.data_ptr(),
                                              merged_bf16=out.data_ptr(), n=n)])
        torch.cuda.synchronize()
        got = _host(out, u16=True)
        assert np.array_equal(got, want), f"in_place={in_place}: {np.flatnonzero(got != want)[:5]}"
    assert (want == 0x7FC0).any() and (want == 0x7F80).any() and (want == 0xFF80).any()
