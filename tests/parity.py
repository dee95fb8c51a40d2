"""Element-by-element comparison of CUDA-path results with the oracle.

Tolerances (the stated bar for the optimizer step):
  acc                      bit-exact
  master, m, v, delta      |x - ref| <= max(2e-6 |ref|, 1e-9)
  w_bf16                   within 1 bf16 ulp (|bits(x) - bits(ref)| <= 1, same sign)
Bit-exactness of every field is reported separately (the design target: the CUDA
path performs the same fp32 operations in the same order as the oracle).
"""
from __future__ import annotations

import numpy as np

FIELDS_F32 = ("master", "m", "v", "delta")


def _same_bits_f32(a, b):
    ua, ub = a.view(np.uint32), b.view(np.uint32)
    return (ua == ub) | (np.isnan(a) & np.isnan(b))


def _identical(a, b) -> bool:
    """Same bytes (a quick pass that settles the common, bit-exact case)."""
    return a.shape == b.shape and np.array_equal(a.view(np.uint8), b.view(np.uint8))


def check_tensor(got: dict, ref: dict, label: str = "") -> dict:
    """got/ref: dicts with master, m, v, delta, acc (float32) and w (uint16).
    Asserts the tolerance bar; returns counts of non-bit-exact elements per field."""
    report = {}
    if not _identical(got["acc"], ref["acc"]):
        acc_same = _same_bits_f32(got["acc"], ref["acc"])
        assert acc_same.all(), f"{label} acc not bit-exact at {np.flatnonzero(~acc_same)[:5]}"
    report["acc"] = 0
    for f in FIELDS_F32:
        if _identical(got[f], ref[f]):
            report[f] = 0
            continue
        x, r = got[f].astype(np.float64), ref[f].astype(np.float64)
        tol = np.maximum(2e-6 * np.abs(r), 1e-9)
        with np.errstate(invalid="ignore"):      # an infinite ref needs the same infinity
            ok = (x == r) | (np.isfinite(r) & (np.abs(x - r) <= tol)) | (np.isnan(x) & np.isnan(r))
        assert ok.all(), (f"{label} {f} outside tolerance at {np.flatnonzero(~ok)[:5]}: "
                          f"{x[~ok][:3]} vs {r[~ok][:3]}")
        report[f] = int((~_same_bits_f32(got[f], ref[f])).sum())
    if _identical(got["w"], ref["w"]):
        report["w"] = 0
        return report
    gw, rw = got["w"].astype(np.int32), ref["w"].astype(np.int32)
    same_sign = (gw >> 15) == (rw >> 15)
    ok = (np.abs(gw - rw) <= 1) & same_sign
    assert ok.all(), f"{label} w_bf16 beyond 1 ulp at {np.flatnonzero(~ok)[:5]}"
    report["w"] = int((gw != rw).sum())
    return report


def oracle_dict(st) -> dict:
    return {"master": st.master, "m": st.m, "v": st.v, "delta": st.delta, "acc": st.acc,
            "w": st.w}


def state_dict(state, j: int) -> dict:
    master, m, v, acc, delta, orig, w = state.numpy_views(j)
    return {"master": master, "m": m, "v": v, "delta": delta, "acc": acc, "w": w}


def partial_acc(cfg, j, micro_steps=None):
    """Sum of micro-steps 1..K-1 of the last step for tensor j (what the accumulator
    holds after a step that folds the K-th grad in without writing it back)."""
    import oracle
    from adamw_step_gb300 import inputs
    orc = oracle.Oracle()
    gs = inputs.GradSource(cfg)
    acc = np.zeros(cfg.tensors[j].numel, np.float32)
    for k in range(cfg.accum_steps - 1 if micro_steps is None else micro_steps):
        orc.accum(acc, inputs.as_u16(gs(j, cfg.steps - 1, k)))
    return acc
