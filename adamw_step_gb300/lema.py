"""Python binding of ``liblema.so`` (include/lema.h), argument marshalling only.

Every function has the C entry point's name; each returns normally on LEMA_OK and
raises ``LemaError`` (status, message) otherwise.  ``raw()`` gives the ctypes
library itself for callers that want the status codes.  Nothing here computes any
part of the step: there is no CPU path and no fallback, and loading fails loudly
when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

import torch  # noqa: F401  (loads the CUDA runtime PyTorch uses before liblema.so)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblema.so")

LEMA_OK = 0
LEMA_ERR_ARG = -1
LEMA_ERR_ALIGN = -2
LEMA_ERR_CUDA = -3
LEMA_ERR_OOM = -4
LEMA_ERR_TIMEOUT = -5
LEMA_ERR_STATE = -6
LEMA_ERR_IO = -7
LEMA_DISK_DIRECT = 1
LEMA_DISK_Q8 = 2
LEMA_RESIDENT = 0
LEMA_STREAMED = 1
LEMA_STEP_KEEP_ACC = 1
LEMA_GRAD_FIRST = 1
LEMA_UNIT_PACKED = 1

c_void_p, c_int32, c_int64, c_double = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double


class _KeywordOnly(ctypes.Structure):
    """Descriptors are built by field name only: a positional argument would land in
    whatever field sits at that position if the layout ever changes."""

    def __init__(self, *args, **kw):
        if args:
            raise TypeError(f"{type(self).__name__} takes keyword arguments only")
        super().__init__(**kw)


class LemaTensor(_KeywordOnly):
    _fields_ = [("master", c_void_p), ("m", c_void_p), ("v", c_void_p), ("acc", c_void_p),
                ("delta", c_void_p), ("orig_bf16", c_void_p), ("w_bf16", c_void_p),
                ("master_out", c_void_p), ("m_out", c_void_p), ("v_out", c_void_p),
                ("grad_bf16", c_void_p), ("n", c_int64), ("flags", c_int32),
                ("reserved", c_int32)]


class LemaGrad(_KeywordOnly):
    _fields_ = [("acc", c_void_p), ("grad_bf16", c_void_p), ("n", c_int64), ("flags", c_int32),
                ("reserved", c_int32)]


class LemaTensorQ8(_KeywordOnly):
    _fields_ = [("master", c_void_p), ("m_q", c_void_p), ("m_scale", c_void_p),
                ("r_q", c_void_p), ("r_scale", c_void_p), ("acc_q", c_void_p),
                ("acc_scale", c_void_p), ("delta", c_void_p), ("orig_bf16", c_void_p),
                ("w_bf16", c_void_p), ("grad_bf16", c_void_p), ("master_out", c_void_p),
                ("m_q_out", c_void_p), ("m_scale_out", c_void_p), ("r_q_out", c_void_p),
                ("r_scale_out", c_void_p), ("n", c_int64), ("flags", c_int32),
                ("reserved", c_int32)]


class LemaGradQ8(_KeywordOnly):
    _fields_ = [("acc_q", c_void_p), ("acc_scale", c_void_p), ("grad_bf16", c_void_p),
                ("n", c_int64), ("flags", c_int32), ("reserved", c_int32)]


class LemaMerge(_KeywordOnly):
    _fields_ = [("base_bf16", c_void_p), ("delta", c_void_p), ("merged_bf16", c_void_p),
                ("n", c_int64)]


class LemaHparams(ctypes.Structure):
    _fields_ = [("lr", c_double), ("beta1", c_double), ("beta2", c_double), ("eps", c_double),
                ("weight_decay", c_double), ("accum_steps", c_int32)]


class LemaLayer(ctypes.Structure):
    _fields_ = [("tensors", ctypes.POINTER(LemaTensor)), ("grads", ctypes.POINTER(c_void_p)),
                ("count", c_int32), ("flags", c_int32)]


class LemaLayerQ8(ctypes.Structure):
    _fields_ = [("tensors", ctypes.POINTER(LemaTensorQ8)), ("grads", ctypes.POINTER(c_void_p)),
                ("count", c_int32), ("flags", c_int32)]


class LemaTraceEvent(ctypes.Structure):
    _fields_ = [("stage", c_int32), ("unit", c_int32), ("call", c_int32), ("reserved", c_int32),
                ("start_ms", c_double), ("end_ms", c_double)]


class LemaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_string(status)}: {message}")
        self.status = status
        self.message = message


_lib = None


def raw():
    """The ctypes handle of liblema.so, with argument types declared."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with adamw_step_gb300.build.build() "
                           "(there is no fallback path)")
    lib = ctypes.CDLL(LIB_PATH)
    lib.lema_accum_grad.argtypes = [ctypes.POINTER(LemaGrad), c_int32, c_void_p]
    lib.lema_adamw_step.argtypes = [ctypes.POINTER(LemaTensor), c_int32, c_int64, c_double,
                                    c_double, c_double, c_double, c_double, c_int32, c_void_p]
    lib.lema_adamw_step_noalloc.argtypes = lib.lema_adamw_step.argtypes
    lib.lema_accum_grad_q8.argtypes = [ctypes.POINTER(LemaGradQ8), c_int32, c_void_p]
    lib.lema_merge_delta.argtypes = [ctypes.POINTER(LemaMerge), c_int32, c_void_p]
    lib.lema_adamw_step_q8.argtypes = [ctypes.POINTER(LemaTensorQ8), c_int32, c_int64, c_double,
                                       c_double, c_double, c_double, c_double, c_int32, c_void_p]
    lib.lema_pool_create.argtypes = [c_int32, c_int64, ctypes.POINTER(c_void_p)]
    lib.lema_stream_layers.argtypes = [c_void_p, ctypes.POINTER(LemaLayer), c_int32, c_int32,
                                       c_int32, ctypes.POINTER(LemaHparams), c_int64, c_void_p]
    lib.lema_stream_layers_q8.argtypes = [c_void_p, ctypes.POINTER(LemaLayerQ8), c_int32,
                                          c_int32, ctypes.POINTER(LemaHparams), c_int64,
                                          c_void_p]
    i64p = ctypes.POINTER(c_int64)
    lib.lema_disk_layout.argtypes = [i64p, c_int32, i64p, i64p]
    lib.lema_disk_layout_q8.argtypes = [i64p, c_int32, i64p, i64p]
    lib.lema_disk_open.argtypes = [ctypes.c_char_p, i64p, c_int32, c_int32, c_int32,
                                   ctypes.POINTER(c_void_p)]
    lib.lema_disk_sync.argtypes = [c_void_p, c_int32]
    lib.lema_disk_close.argtypes = [c_void_p]
    lib.lema_stream_layers_disk.argtypes = [c_void_p, c_void_p, ctypes.POINTER(LemaLayer),
                                            c_int32, c_int32, ctypes.POINTER(LemaHparams),
                                            c_int64, c_void_p]
    lib.lema_stream_layers_disk_q8.argtypes = [c_void_p, c_void_p, ctypes.POINTER(LemaLayerQ8),
                                               c_int32, c_int32, ctypes.POINTER(LemaHparams),
                                               c_int64, c_void_p]
    dp = ctypes.POINTER(c_double)
    lib.lema_disk_probe.argtypes = [ctypes.c_char_p, c_int64, c_int32, c_int32, dp, dp, dp]
    lib.lema_kernel_wait_timeouts.argtypes = [ctypes.POINTER(c_int64)]
    lib.lema_pool_sync.argtypes = [c_void_p, c_int32]
    lib.lema_pool_wait_stream.argtypes = [c_void_p, c_void_p]
    lib.lema_pool_destroy.argtypes = [c_void_p]
    lib.lema_last_error.restype = ctypes.c_char_p
    lib.lema_status_string.argtypes = [ctypes.c_int]
    lib.lema_status_string.restype = ctypes.c_char_p
    lib.lema_pool_trace.argtypes = [c_void_p, c_int32]
    lib.lema_pool_copies_only.argtypes = [c_void_p, c_int32]
    lib.lema_pool_slices.argtypes = [c_void_p, c_int32, c_int64]
    lib.lema_pool_slice_first_unit.argtypes = [c_void_p, c_int32]
    lib.lema_pool_trace_read.argtypes = [c_void_p, ctypes.POINTER(LemaTraceEvent), c_int32,
                                         ctypes.POINTER(c_int32)]
    lib.lema_test_fail_copy.argtypes = [c_int64]
    lib.lema_test_fail_copy.restype = None
    lib.lema_test_kernel_wait_limit.argtypes = [c_int64]
    lib.lema_test_divide_by_constant.argtypes = [ctypes.POINTER(ctypes.c_float), c_int32,
                                                 ctypes.POINTER(c_int64), ctypes.POINTER(c_int64)]
    for name in ("lema_accum_grad", "lema_adamw_step", "lema_adamw_step_noalloc",
                 "lema_accum_grad_q8", "lema_adamw_step_q8", "lema_merge_delta",
                 "lema_pool_create", "lema_stream_layers", "lema_stream_layers_q8",
                 "lema_disk_layout", "lema_disk_layout_q8", "lema_disk_open",
                 "lema_disk_sync", "lema_disk_close", "lema_stream_layers_disk",
                 "lema_stream_layers_disk_q8", "lema_disk_probe", "lema_kernel_wait_timeouts",
                 "lema_pool_sync", "lema_pool_wait_stream", "lema_pool_destroy",
                 "lema_pool_trace", "lema_pool_trace_read", "lema_test_kernel_wait_limit",
                 "lema_pool_copies_only", "lema_pool_slices", "lema_pool_slice_first_unit",
                 "lema_test_divide_by_constant"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return raw().lema_status_string(int(status)).decode()


def lema_last_error() -> str:
    return raw().lema_last_error().decode()


def _check(status: int) -> None:
    if status != LEMA_OK:
        raise LemaError(status, lema_last_error())


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _array(ctype, items):
    if isinstance(items, ctypes.Array):
        return items
    return (ctype * len(items))(*items)


def lema_accum_grad(grads, stream=None) -> None:
    """acc += (fp32) grad for each LemaGrad, one launch."""
    arr = _array(LemaGrad, grads)
    _check(raw().lema_accum_grad(arr, len(arr), _stream(stream)))


def lema_adamw_step(tensors, step, lr, beta1, beta2, eps, weight_decay, accum_steps,
                    stream=None) -> None:
    """One fused AdamW step over a list of LemaTensor, one launch."""
    arr = _array(LemaTensor, tensors)
    _check(raw().lema_adamw_step(arr, len(arr), int(step), float(lr), float(beta1), float(beta2),
                                 float(eps), float(weight_decay), int(accum_steps),
                                 _stream(stream)))


def lema_adamw_step_noalloc(tensors, step, lr, beta1, beta2, eps, weight_decay, accum_steps,
                            stream=None) -> None:
    """lema_adamw_step with its table in the library's fixed device array: no
    allocation (at most 1024 tensors and 2^29 elements per call)."""
    arr = _array(LemaTensor, tensors)
    _check(raw().lema_adamw_step_noalloc(arr, len(arr), int(step), float(lr), float(beta1),
                                         float(beta2), float(eps), float(weight_decay),
                                         int(accum_steps), _stream(stream)))


def lema_accum_grad_q8(grads, stream=None) -> None:
    """8-bit accumulators: per 256-element block decode, add the grad, encode."""
    arr = _array(LemaGradQ8, grads)
    _check(raw().lema_accum_grad_q8(arr, len(arr), _stream(stream)))


def lema_adamw_step_q8(tensors, step, lr, beta1, beta2, eps, weight_decay, accum_steps,
                       stream=None) -> None:
    """The AdamW step on 8-bit moments and accumulators."""
    arr = _array(LemaTensorQ8, tensors)
    _check(raw().lema_adamw_step_q8(arr, len(arr), int(step), float(lr), float(beta1),
                                    float(beta2), float(eps), float(weight_decay),
                                    int(accum_steps), _stream(stream)))


def lema_merge_delta(items, stream=None) -> None:
    """merged = bf16(base + delta) for each LemaMerge, one launch."""
    arr = _array(LemaMerge, items)
    _check(raw().lema_merge_delta(arr, len(arr), _stream(stream)))


def lema_pool_create(n_slots: int, slot_params: int) -> int:
    out = c_void_p()
    _check(raw().lema_pool_create(int(n_slots), int(slot_params), ctypes.byref(out)))
    return out.value


def lema_stream_layers(pool, layers, residency, micro_step, hparams, step, stream=None) -> None:
    arr = _array(LemaLayer, layers)
    _check(raw().lema_stream_layers(pool, arr, len(arr), int(residency), int(micro_step),
                                    ctypes.byref(hparams), int(step), _stream(stream)))


def lema_stream_layers_q8(pool, layers, micro_step, hparams, step, stream=None) -> None:
    arr = _array(LemaLayerQ8, layers)
    _check(raw().lema_stream_layers_q8(pool, arr, len(arr), int(micro_step),
                                       ctypes.byref(hparams), int(step), _stream(stream)))


def lema_pool_sync(pool, timeout_ms: int) -> None:
    _check(raw().lema_pool_sync(pool, int(timeout_ms)))


def lema_pool_wait_stream(pool, stream=None) -> None:
    _check(raw().lema_pool_wait_stream(pool, _stream(stream)))


def lema_pool_destroy(pool) -> None:
    _check(raw().lema_pool_destroy(pool))


def lema_pool_slices(pool, max_slices: int, min_slice_params: int) -> None:
    """Split packed units into at most max_slices slices of whole chunks, each at
    least min_slice_params elements, so their copies and kernels overlap."""
    _check(raw().lema_pool_slices(pool, int(max_slices), int(min_slice_params)))


def lema_pool_slice_first_unit(pool, on: bool) -> None:
    """Slice only the first slot-using unit of each streamed call."""
    _check(raw().lema_pool_slice_first_unit(pool, 1 if on else 0))


def lema_pool_copies_only(pool, on: bool) -> None:
    """Measurement mode: streamed calls enqueue their copies but launch no kernel."""
    _check(raw().lema_pool_copies_only(pool, 1 if on else 0))


def lema_pool_trace(pool, max_events: int) -> None:
    _check(raw().lema_pool_trace(pool, int(max_events)))


def lema_pool_trace_read(pool, max_events: int = 1 << 16) -> list:
    """[(stage, unit, call, start_ms, end_ms)] of the traced stages."""
    buf = (LemaTraceEvent * max_events)()
    n = c_int32()
    _check(raw().lema_pool_trace_read(pool, buf, max_events, ctypes.byref(n)))
    return [(e.stage, e.unit, e.call, e.start_ms, e.end_ms) for e in buf[:min(n.value, max_events)]]


def lema_test_fail_copy(nth_copy: int) -> None:
    """Test hook: make the nth host<->device copy the pool enqueues fail (0 disarms)."""
    raw().lema_test_fail_copy(int(nth_copy))


def lema_test_kernel_wait_limit(limit_ns: int) -> None:
    """Test hook: the 8-bit step kernel's wait limit for its staged inputs on the
    current device (< 0: the default; 0: give up at the first poll that finds the
    copies in flight)."""
    _check(raw().lema_test_kernel_wait_limit(int(limit_ns)))


def lema_test_divide_by_constant(divisors):
    """Test hook: (mismatches, outside) per divisor of the 8-bit step's division by a
    per-call constant against the IEEE division, over every x >= 0."""
    n = len(divisors)
    d = (ctypes.c_float * max(n, 1))(*[float(x) for x in divisors])
    bad = (c_int64 * max(n, 1))()
    out = (c_int64 * max(n, 1))()
    _check(raw().lema_test_divide_by_constant(d, n, bad, out))
    return list(bad)[:n], list(out)[:n]


def lema_disk_layout(unit_params, q8: bool = False):
    """(unit_offset[n+1], padded[n]) of the disk file for units of these sizes (the
    8-bit layout with q8)."""
    n = len(unit_params)
    P = (c_int64 * max(n, 1))(*[int(x) for x in unit_params])
    off = (c_int64 * (n + 1))()
    Q = (c_int64 * max(n, 1))()
    fn = raw().lema_disk_layout_q8 if q8 else raw().lema_disk_layout
    _check(fn(P, n, off, Q))
    return list(off), list(Q)[:n]


def lema_disk_open(path: str, unit_params, flags: int = 0, n_io_threads: int = 8) -> int:
    n = len(unit_params)
    P = (c_int64 * max(n, 1))(*[int(x) for x in unit_params])
    out = c_void_p()
    _check(raw().lema_disk_open(os.fsencode(path), P, n, int(flags), int(n_io_threads),
                                ctypes.byref(out)))
    return out.value


def lema_disk_sync(disk, timeout_ms: int = 600_000) -> None:
    _check(raw().lema_disk_sync(disk, int(timeout_ms)))


def lema_disk_close(disk) -> None:
    _check(raw().lema_disk_close(disk))


def lema_stream_layers_disk(pool, disk, layers, micro_step, hparams, step, stream=None) -> None:
    arr = _array(LemaLayer, layers)
    _check(raw().lema_stream_layers_disk(pool, disk, arr, len(arr), int(micro_step),
                                         ctypes.byref(hparams), int(step), _stream(stream)))


def lema_stream_layers_disk_q8(pool, disk, layers, micro_step, hparams, step,
                               stream=None) -> None:
    arr = _array(LemaLayerQ8, layers)
    _check(raw().lema_stream_layers_disk_q8(pool, disk, arr, len(arr), int(micro_step),
                                            ctypes.byref(hparams), int(step), _stream(stream)))


def lema_disk_probe(path: str, nbytes: int, flags: int = 0, n_io_threads: int = 8) -> dict:
    """Write / read / mixed GB/s of the disk tier's IO threads on a scratch file."""
    w, r, m = c_double(), c_double(), c_double()
    _check(raw().lema_disk_probe(os.fsencode(path), int(nbytes), int(flags), int(n_io_threads),
                                 ctypes.byref(w), ctypes.byref(r), ctypes.byref(m)))
    return {"write_gbs": w.value, "read_gbs": r.value, "mixed_gbs": m.value}


def lema_kernel_wait_timeouts() -> int:
    """Bounded waits inside kernels that ran out on the current device (expected 0)."""
    n = c_int64()
    _check(raw().lema_kernel_wait_timeouts(ctypes.byref(n)))
    return n.value
