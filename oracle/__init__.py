"""CPU oracle for the selective-full-fine-tuning optimizer step (TEST INFRASTRUCTURE).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path never does.

Two independent references live here:
  * ``liboracle.so`` (``lema_oracle.c``): the scalar fp32 step, the 8-bit-state
    form (block encode/decode around the same fp32 update) and the delta merge,
    wrapped below with numpy arrays (bf16 data is carried as ``uint16`` bit
    patterns);
  * ``exact_trace``: the fp32 method in exact rational arithmetic, used only to pin
    the fp32 oracle on a hand-sized trace.

Page "LEMA: Layer-wise Efficient Memory Abstraction", sections "Selective Full
Fine-Tuning" (fp32 states and accumulation, per-layer AdamW, fp32 delta, base +
delta for serving), "Quick Start" (torch.optim.AdamW as the optimizer) and
"Quantization" (8-bit optimizer states and accumulators).
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import numpy as np

from . import build as _build

_lib = None


class OracleScalars(ctypes.Structure):
    _fields_ = [(name, ctypes.c_float) for name in (
        "decay", "beta1", "one_minus_beta1", "beta2", "one_minus_beta2",
        "step_size", "bc2_sqrt", "eps", "accum_steps")]


def load(path: str | None = None):
    """Load (building first if needed) the oracle library.  ``path`` selects
    another build of the same source, e.g. a deliberately mutated copy."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    lib = ctypes.CDLL(path or _build.ensure_built())
    f32p = ctypes.POINTER(ctypes.c_float)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    i64 = ctypes.c_int64
    lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f32.restype = ctypes.c_float
    lib.oracle_f32_to_bf16_rne.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_bf16_rne.restype = ctypes.c_uint16
    lib.oracle_f32_to_bf16_array.argtypes = [f32p, u16p, i64]
    lib.oracle_bf16_to_f32_array.argtypes = [u16p, f32p, i64]
    lib.oracle_accum.argtypes = [f32p, u16p, i64, ctypes.c_int]
    lib.oracle_make_scalars.argtypes = [i64, ctypes.c_double, ctypes.c_double,
                                        ctypes.c_double, ctypes.c_double,
                                        ctypes.c_double, ctypes.c_int32,
                                        ctypes.POINTER(OracleScalars)]
    lib.oracle_make_scalars.restype = ctypes.c_int
    lib.oracle_adamw_step.argtypes = [i64, f32p, f32p, f32p, f32p, u16p,
                                      f32p, f32p, f32p, f32p, u16p,
                                      ctypes.POINTER(OracleScalars), ctypes.c_int]
    lib.oracle_max_threads.restype = ctypes.c_int
    i8p = ctypes.POINTER(ctypes.c_int8)
    u8p = ctypes.POINTER(ctypes.c_uint8)
    lib.oracle_q8_encode_signed.argtypes = [f32p, i64, i8p, f32p]
    lib.oracle_q8_decode_signed.argtypes = [i8p, f32p, i64, f32p]
    lib.oracle_q8_encode_root.argtypes = [f32p, i64, u8p, f32p]
    lib.oracle_q8_decode_root.argtypes = [u8p, f32p, i64, f32p]
    lib.oracle_accum_q8.argtypes = [i8p, f32p, u16p, i64, ctypes.c_int, ctypes.c_int]
    lib.oracle_merge_delta.argtypes = [u16p, f32p, i64, u16p]
    lib.oracle_adamw_step_q8.argtypes = [i64, f32p, i8p, f32p, u8p, f32p, i8p, f32p, u16p, u16p,
                                         f32p, i8p, f32p, u8p, f32p, f32p, u16p,
                                         ctypes.POINTER(OracleScalars), ctypes.c_int]
    if path is None:
        _lib = lib
    return lib


def _f32(a: np.ndarray):
    assert a.dtype == np.float32 and a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def _u16(a: np.ndarray):
    assert a.dtype == np.uint16 and a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))


def _i8(a: np.ndarray):
    assert a.dtype == np.int8 and a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int8))


def _u8(a: np.ndarray):
    assert a.dtype == np.uint8 and a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))


Q8_BLOCK = 256


def q8_blocks(n: int) -> int:
    return (int(n) + Q8_BLOCK - 1) // Q8_BLOCK


class Oracle:
    """numpy front end over one build of ``lema_oracle.c``."""

    def __init__(self, path: str | None = None, threads: int = 1):
        self.lib = load(path)
        self.threads = threads

    # bf16 conversions -----------------------------------------------------
    def f32_to_bf16(self, x: np.ndarray, out: np.ndarray | None = None) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.float32)
        if out is None:
            out = np.empty(x.shape, dtype=np.uint16)
        assert out.shape == x.shape
        self.lib.oracle_f32_to_bf16_array(_f32(x), _u16(out), x.size)
        return out

    def bf16_to_f32(self, h: np.ndarray) -> np.ndarray:
        h = np.ascontiguousarray(h, dtype=np.uint16)
        out = np.empty(h.shape, dtype=np.float32)
        self.lib.oracle_bf16_to_f32_array(_u16(h), _f32(out), h.size)
        return out

    # hyperparameter scalars ------------------------------------------------
    def scalars(self, step, lr, beta1, beta2, eps, weight_decay, accum_steps) -> OracleScalars:
        s = OracleScalars()
        rc = self.lib.oracle_make_scalars(int(step), float(lr), float(beta1), float(beta2),
                                          float(eps), float(weight_decay), int(accum_steps),
                                          ctypes.byref(s))
        if rc != 0:
            raise ValueError("hyperparameters outside the method's domain")
        return s

    # the two operations ----------------------------------------------------
    def accum(self, acc: np.ndarray, g_bf16: np.ndarray) -> None:
        """In place: acc += (fp32) g."""
        assert acc.size == g_bf16.size
        self.lib.oracle_accum(_f32(acc), _u16(np.ascontiguousarray(g_bf16)), acc.size,
                              self.threads)

    def adamw_step(self, st: "OracleState", step: int, hp: "Hyper") -> None:
        """In place on ``st``: one AdamW step, then the accumulator is reset to +0."""
        s = self.scalars(step, hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay,
                         hp.accum_steps)
        n = st.master.size
        self.lib.oracle_adamw_step(n, _f32(st.master), _f32(st.m), _f32(st.v), _f32(st.acc),
                                   _u16(st.orig), _f32(st.master), _f32(st.m), _f32(st.v),
                                   _f32(st.delta), _u16(st.w), ctypes.byref(s), self.threads)
        st.acc[...] = 0.0

    def adamw_step_arrays(self, master, m, v, acc, orig, step, hp):
        """Out of place on plain arrays; returns (master', m', v', delta, w_bf16)."""
        s = self.scalars(step, hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay,
                         hp.accum_steps)
        n = master.size
        outs = [np.empty(n, np.float32) for _ in range(4)] + [np.empty(n, np.uint16)]
        self.lib.oracle_adamw_step(n, _f32(master), _f32(m), _f32(v), _f32(acc), _u16(orig),
                                   _f32(outs[0]), _f32(outs[1]), _f32(outs[2]), _f32(outs[3]),
                                   _u16(outs[4]), ctypes.byref(s), self.threads)
        return tuple(outs)

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())

    def merge_delta(self, base_bf16, delta):
        """bf16(base + delta): the servable weight from a base and a saved delta."""
        base = np.ascontiguousarray(base_bf16, dtype=np.uint16)
        delta = np.ascontiguousarray(delta, dtype=np.float32)
        out = np.empty(base.size, np.uint16)
        self.lib.oracle_merge_delta(_u16(base), _f32(delta), base.size, _u16(out))
        return out

    # 8-bit states ------------------------------------------------------------
    def q8_encode_signed(self, x):
        x = np.ascontiguousarray(x, dtype=np.float32)
        q = np.empty(x.size, np.int8)
        s = np.empty(q8_blocks(x.size), np.float32)
        self.lib.oracle_q8_encode_signed(_f32(x), x.size, _i8(q), _f32(s))
        return q, s

    def q8_decode_signed(self, q, s):
        x = np.empty(q.size, np.float32)
        self.lib.oracle_q8_decode_signed(_i8(q), _f32(s), q.size, _f32(x))
        return x

    def q8_encode_root(self, r):
        r = np.ascontiguousarray(r, dtype=np.float32)
        c = np.empty(r.size, np.uint8)
        s = np.empty(q8_blocks(r.size), np.float32)
        self.lib.oracle_q8_encode_root(_f32(r), r.size, _u8(c), _f32(s))
        return c, s

    def q8_decode_root(self, c, s):
        r = np.empty(c.size, np.float32)
        self.lib.oracle_q8_decode_root(_u8(c), _f32(s), c.size, _f32(r))
        return r

    def accum_q8(self, st: "OracleStateQ8", g_bf16, first: bool) -> None:
        self.lib.oracle_accum_q8(_i8(st.acc_q), _f32(st.acc_scale),
                                 _u16(np.ascontiguousarray(g_bf16)), st.acc_q.size, int(first),
                                 self.threads)

    def adamw_step_q8(self, st: "OracleStateQ8", step: int, hp: "Hyper", grad_last=None,
                      use_acc=True) -> None:
        """In place on ``st``.  grad_last: the K-th micro-batch grad folded into the
        step (the accumulator then holds micro-steps 1..K-1 and is not written);
        use_acc=False: no accumulator (K = 1 with grad_last)."""
        s = self.scalars(step, hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay,
                         hp.accum_steps)
        n = st.master.size
        m_q, m_s = np.empty_like(st.m_q), np.empty_like(st.m_scale)
        r_q, r_s = np.empty_like(st.r_q), np.empty_like(st.r_scale)
        gl = None if grad_last is None else _u16(np.ascontiguousarray(grad_last))
        self.lib.oracle_adamw_step_q8(
            n, _f32(st.master), _i8(st.m_q), _f32(st.m_scale), _u8(st.r_q), _f32(st.r_scale),
            _i8(st.acc_q) if use_acc else None, _f32(st.acc_scale) if use_acc else None, gl,
            _u16(st.orig), _f32(st.master), _i8(m_q), _f32(m_s), _u8(r_q), _f32(r_s),
            _f32(st.delta), _u16(st.w), ctypes.byref(s), self.threads)
        st.m_q, st.m_scale, st.r_q, st.r_scale = m_q, m_s, r_q, r_s


@dataclass(frozen=True)
class Hyper:
    lr: float = 1e-4
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01
    accum_steps: int = 1


class OracleStateQ8:
    """fp32 master/delta, 8-bit m, sqrt(v) and accumulator with per-block scales,
    bf16 orig/w, for one flat tensor (all moments start at 0)."""

    def __init__(self, w0_bf16: np.ndarray, oracle: Oracle):
        w0 = np.ascontiguousarray(w0_bf16, dtype=np.uint16).ravel()
        n, nb = w0.size, q8_blocks(w0.size)
        self.orig = w0.copy()
        self.master = oracle.bf16_to_f32(w0)
        self.m_q = np.zeros(n, np.int8)
        self.m_scale = np.zeros(nb, np.float32)
        self.r_q = np.zeros(n, np.uint8)
        self.r_scale = np.zeros(nb, np.float32)
        self.acc_q = np.zeros(n, np.int8)
        self.acc_scale = np.zeros(nb, np.float32)
        self.delta = np.zeros(n, np.float32)
        self.w = w0.copy()


class OracleState:
    """fp32 master/m/v/acc/delta and bf16 orig/w for one flat tensor."""

    def __init__(self, w0_bf16: np.ndarray, oracle: Oracle):
        w0 = np.ascontiguousarray(w0_bf16, dtype=np.uint16).ravel()
        self.orig = w0.copy()
        self.master = oracle.bf16_to_f32(w0)
        self.m = np.zeros_like(self.master)
        self.v = np.zeros_like(self.master)
        self.acc = np.zeros_like(self.master)
        self.delta = np.zeros_like(self.master)
        self.w = w0.copy()
