"""The CPU oracle against its pins (no GPU)."""
import pytest

import oracle
from oracle.exact_trace import exact_trace
import oracle_pins as P


@pytest.fixture(scope="module")
def orc():
    return oracle.Oracle()


@pytest.mark.parametrize("pin", P.QUICK_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_bf16_exhaustive(orc):
    P.pin_bf16_exhaustive(orc)


def test_golden_file_matches_exact_trace():
    """The stored trace is what oracle.exact_trace computes from the stored inputs."""
    hyper, w0d, gd, out = P.load_golden()
    n = len(w0d)
    K, steps = int(hyper["accum_steps"]), int(hyper["steps"])
    grads = [[[gd[(t, k, i)] for i in range(n)] for k in range(1, K + 1)]
             for t in range(1, steps + 1)]
    tr = exact_trace([w0d[i] for i in range(n)], grads,
                     **{k: hyper[k] for k in ("lr", "beta1", "beta2", "eps", "weight_decay")})
    for t in range(steps):
        for f in ("w", "m", "v", "delta"):
            for i in range(n):
                a, b = tr[t][f][i], out[(t + 1, i, f)]
                assert abs(a - b) <= abs(a) * 1e-35 + 1e-45


def test_scalars_reject_out_of_domain(orc):
    for bad in [dict(step=0), dict(accum_steps=0), dict(beta1=1.0), dict(beta2=-0.1),
                dict(eps=0.0), dict(lr=-1.0), dict(weight_decay=-1.0),
                dict(lr=1.0, weight_decay=1.0)]:
        kw = dict(step=1, lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01,
                  accum_steps=1)
        kw.update(bad)
        with pytest.raises(ValueError):
            orc.scalars(**kw)


def test_threads_do_not_change_the_oracle():
    """The OpenMP loops only split independent elements (8-bit: independent blocks)
    across threads: one thread and four give the same bits, fp32 and 8-bit."""
    import numpy as np
    rng = np.random.default_rng(9)
    n = 40_000 + 77
    w0 = (rng.standard_normal(n).astype(np.float32) * 0.02).view(np.uint32)
    w0 = ((w0 + 0x7FFF + ((w0 >> 16) & 1)) >> 16).astype(np.uint16)      # bf16 of the draws
    gs = [((rng.standard_normal(n).astype(np.float32) * 1e-3).view(np.uint32) >> 16)
          .astype(np.uint16) for _ in range(3)]
    h = oracle.Hyper(accum_steps=3)
    out = []
    for th in (1, 4):
        o = oracle.Oracle(threads=th)
        st = oracle.OracleState(w0, o)
        sq = oracle.OracleStateQ8(w0, o)
        for t in range(2):
            for g in gs:
                o.accum(st.acc, g)
            o.adamw_step(st, t + 1, h)
            for k, g in enumerate(gs[:-1]):
                o.accum_q8(sq, g, first=(k == 0))
            o.adamw_step_q8(sq, t + 1, h, grad_last=gs[-1])
        out.append([st.master, st.m, st.v, st.delta, st.w, sq.master, sq.m_q, sq.m_scale,
                    sq.r_q, sq.r_scale, sq.acc_q, sq.acc_scale, sq.delta, sq.w])
    for a, b in zip(*out):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
