"""The C-ABI library without a GPU: it loads, exports every declared entry point,
and rejects bad arguments before it touches CUDA (no compute calls here)."""
import ctypes
import os
import re

import pytest

from adamw_step_gb300 import build as B

HEADER = os.path.join(B.ROOT, "include", "lema.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(B.LIB) or any(
            os.path.getmtime(os.path.join(B.CSRC, s)) > os.path.getmtime(B.LIB) for s in B.SOURCES):
        B.build()
    from adamw_step_gb300 import lema
    return lema.raw()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lema_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("lema_accum_grad", "lema_adamw_step", "lema_stream_layers", "lema_pool_create",
              "lema_pool_sync", "lema_pool_destroy", "lema_last_error"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    from adamw_step_gb300 import lema
    assert lema.status_string(0) == "LEMA_OK"
    assert lema.status_string(-5) == "LEMA_ERR_TIMEOUT"


def test_validation_before_cuda(lib):
    from adamw_step_gb300.lema import LemaTensor, LemaGrad, LemaHparams
    T = (LemaTensor * 1)()
    args = (1, 1e-4, 0.9, 0.999, 1e-8, 0.01, 1, None)
    assert lib.lema_adamw_step(T, -1, *args) == -1
    assert lib.lema_adamw_step(None, 1, *args) == -1
    assert lib.lema_adamw_step(T, 0, *args) == 0            # count 0: no-op
    assert lib.lema_adamw_step(T, 1, 0, 1e-4, 0.9, 0.999, 1e-8, 0.01, 1, None) == -1  # step 0
    assert lib.lema_adamw_step(T, 1, 1, 1e-4, 1.0, 0.999, 1e-8, 0.01, 1, None) == -1  # beta1
    assert lib.lema_adamw_step(T, 1, 1, 1e-4, 0.9, 0.999, 0.0, 0.01, 1, None) == -1   # eps
    assert lib.lema_adamw_step(T, 1, 1, -1.0, 0.9, 0.999, 1e-8, 0.01, 1, None) == -1  # lr
    assert lib.lema_adamw_step(T, 1, 1, 2.0, 0.9, 0.999, 1e-8, 0.5, 1, None) == -1    # lr*wd
    assert lib.lema_adamw_step(T, 1, 1, 1e-4, 0.9, 0.999, 1e-8, 0.01, 0, None) == -1  # K
    assert b"accum_steps" in lib.lema_last_error()
    T[0].n = 16                                              # NULL buffers
    assert lib.lema_adamw_step(T, 1, *args) == -1
    for f in ("master", "m", "v", "acc", "delta", "orig_bf16", "w_bf16"):
        setattr(T[0], f, 0x100000)
    T[0].delta = 0x100004                                    # misaligned
    assert lib.lema_adamw_step(T, 1, *args) == -2
    T[0].master_out = 0x200000                               # only one of the three outputs
    assert lib.lema_adamw_step(T, 1, *args) == -1
    G = (LemaGrad * 1)()
    assert lib.lema_accum_grad(G, -1, None) == -1
    assert lib.lema_accum_grad(G, 0, None) == 0
    G[0].n = 8
    assert lib.lema_accum_grad(G, 1, None) == -1
    G[0].acc, G[0].grad_bf16 = 0x100000, 0x100002
    assert lib.lema_accum_grad(G, 1, None) == -2


def test_pool_validation_before_cuda(lib):
    from adamw_step_gb300.lema import LemaHparams, LemaLayer
    out = ctypes.c_void_p()
    assert lib.lema_pool_create(1, 100, ctypes.byref(out)) == -1 and not out.value
    assert lib.lema_pool_create(2, 0, ctypes.byref(out)) == -1
    assert lib.lema_pool_sync(None, 10) == -1
    hp = LemaHparams(1e-4, 0.9, 0.999, 1e-8, 0.01, 4)
    L = (LemaLayer * 1)()
    assert lib.lema_stream_layers(None, L, 1, 1, 1, None, 1, None) == -1      # no hparams
    assert lib.lema_stream_layers(None, L, 1, 1, 5, ctypes.byref(hp), 1, None) == -1  # k > K
    assert lib.lema_stream_layers(None, L, 1, 1, 0, ctypes.byref(hp), 1, None) == -1  # k < 1
    assert lib.lema_stream_layers(None, L, 0, 1, 1, ctypes.byref(hp), 1, None) == 0   # no units
    L[0].count = 2                                           # NULL arrays
    assert lib.lema_stream_layers(None, L, 1, 1, 1, ctypes.byref(hp), 1, None) == -1
    from adamw_step_gb300.lema import LemaLayerQ8
    Q = (LemaLayerQ8 * 1)()
    assert lib.lema_stream_layers_q8(None, Q, 1, 1, None, 1, None) == -1     # no hparams
    assert lib.lema_stream_layers_q8(None, Q, 1, 5, ctypes.byref(hp), 1, None) == -1  # k > K
    assert lib.lema_stream_layers_q8(None, Q, 0, 1, ctypes.byref(hp), 1, None) == 0   # no units
    assert lib.lema_stream_layers_q8(None, Q, 1, 1, ctypes.byref(hp), 1, None) == -1  # no pool
    Q[0].count = 1
    assert lib.lema_stream_layers_q8(None, Q, 1, 1, ctypes.byref(hp), 1, None) == -1
    assert lib.lema_pool_destroy(None) == 0
    assert lib.lema_pool_slices(None, 4, 8192) == -1
    assert lib.lema_pool_slice_first_unit(None, 1) == -1
    assert lib.lema_pool_copies_only(None, 1) == -1
    # the division check takes divisors in (2^-27, 1] only (rejected before any CUDA call)
    d = (ctypes.c_float * 1)(2.0)
    bad, out = (ctypes.c_int64 * 1)(), (ctypes.c_int64 * 1)()
    assert lib.lema_test_divide_by_constant(d, 1, bad, out) == -1
    assert lib.lema_test_divide_by_constant(d, -1, bad, out) == -1


def test_struct_layouts_match_header(tmp_path):
    """sizeof/offsetof of every ABI struct, from a C program compiled against
    include/lema.h, equal the ctypes mirrors the binding uses."""
    import subprocess
    from adamw_step_gb300 import lema
    structs = {
        "lema_tensor": lema.LemaTensor, "lema_grad": lema.LemaGrad,
        "lema_adamw_hparams": lema.LemaHparams, "lema_layer": lema.LemaLayer,
        "lema_layer_q8": lema.LemaLayerQ8,
        "lema_trace_event": lema.LemaTraceEvent,
        "lema_tensor_q8": lema.LemaTensorQ8, "lema_grad_q8": lema.LemaGradQ8,
        "lema_merge": lema.LemaMerge,
    }
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "lema.h"', "int main(void){"]
    for cname, py in structs.items():
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for fname, _ in py._fields_:
            lines.append(f'printf("{cname} {fname} %zu\\n", offsetof({cname}, {fname}));')
    lines.append("return 0;}")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    got = {tuple(l.split()[:2]): int(l.split()[2]) for l in out if l.strip()}
    for cname, py in structs.items():
        assert got[(cname, "size")] == ctypes.sizeof(py), cname
        for fname, _ in py._fields_:
            assert got[(cname, fname)] == getattr(py, fname).offset, (cname, fname)


def test_binding_fails_loudly_without_the_library(tmp_path, monkeypatch):
    """No CPU fallback: with liblema.so absent the binding raises instead of running
    anything else."""
    from adamw_step_gb300 import lema
    monkeypatch.setattr(lema, "_lib", None)
    monkeypatch.setattr(lema, "LIB_PATH", str(tmp_path / "liblema.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        lema.raw()
    with pytest.raises(RuntimeError, match="no fallback"):
        lema.lema_accum_grad([])
