"""Optimizer-state containers: PyTorch allocates, the C ABI computes.

``DeviceState`` keeps every tensor's fp32 master/m/v/acc/delta and bf16 orig/w in
HBM (resident residency).  ``HostState`` keeps them in pinned host RAM (streamed
residency) and hands them to a ``Pool``.  Both only allocate memory and build the
ctypes descriptor arrays of include/lema.h; every arithmetic step runs in the CUDA
kernels of liblema.so.  Initial state (page "LEMA: Layer-wise Efficient Memory
Abstraction", section "Selective Full Fine-Tuning": the fp32 master starts as the
original weight, the delta is updated - original): master = widen(orig), m = v =
acc = delta = 0, w = orig.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import lema
from .hostmem import PinnedBuffers
from .lema import LemaGrad, LemaGradQ8, LemaHparams, LemaLayer, LemaTensor, LemaTensorQ8


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


class _State:
    fields_f32 = ("master", "m", "v", "acc", "delta")

    def __init__(self, w0_list, device, pin: bool, units=None, acc_device=None):
        """units (pinned host only): lists of tensor indices.  Each unit's fields are
        then laid out like a VRAM slot -- one block per field, tensor j at the
        64-element-aligned offset the slot uses -- so the pool moves each field of
        a unit with one copy (LEMA_UNIT_PACKED).  acc_device (pinned host only): keep
        the accumulators in that device's memory instead (same layout), where the
        pool updates them in place and never copies them."""
        self.tensors = [None] * len(w0_list)
        self.pinned = None
        self.units = [list(u) for u in units] if (pin and units is not None) else None
        if pin:
            groups = self.units or [[j] for j in range(len(w0_list))]
            sizes = []
            host_f32 = [f for f in self.fields_f32 if not (acc_device and f == "acc")]
            for u in groups:
                P = sum(_pad(w0_list[j].numel()) for j in u)
                sizes += [(P, torch.bfloat16)] * 2 + [(P, torch.float32)] * len(host_f32)
            # one registered arena for every buffer of every tensor
            self.pinned = PinnedBuffers(PinnedBuffers.arena_size(sizes))
            for u in groups:
                P = sum(_pad(w0_list[j].numel()) for j in u)
                block = {f: self.pinned.zeros(P, torch.float32) for f in host_f32}
                if acc_device:
                    block["acc"] = torch.zeros(P, dtype=torch.float32, device=acc_device)
                block["orig"] = self.pinned.zeros(P, torch.bfloat16)
                block["w"] = self.pinned.zeros(P, torch.bfloat16)
                o = 0
                for j in u:
                    n = w0_list[j].numel()
                    st = {f: b[o:o + n] for f, b in block.items()}
                    st["orig"].copy_(w0_list[j].reshape(-1))
                    st["w"].copy_(w0_list[j].reshape(-1))
                    self.tensors[j] = st
                    o += _pad(n)
        else:
            for j, w0 in enumerate(w0_list):
                orig = w0.reshape(-1).to(device) if device != "cpu" else w0.reshape(-1).clone()
                st = {"orig": orig, "w": orig.clone()}
                for f in self.fields_f32:
                    st[f] = torch.zeros(orig.numel(), dtype=torch.float32, device=device)
                self.tensors[j] = st
        for st in self.tensors:
            st["master"].copy_(st["orig"])    # exact bf16 -> fp32 widening (initial state)
        self._descs = None

    def close(self):
        """Release the page-locked registration of host states (streamed residency)."""
        if self.pinned is not None:
            self.pinned.close()

    @property
    def numel(self) -> int:
        return sum(t["orig"].numel() for t in self.tensors)

    def tensor_desc(self, j: int, out_of_place=None, grad=None, flags=0,
                    with_acc=True) -> LemaTensor:
        """Descriptor of tensor j.  grad: the last micro-batch grad to fold into the
        step; flags: LEMA_STEP_KEEP_ACC; with_acc=False passes no accumulator (only
        valid with grad and K = 1)."""
        t = self.tensors[j]
        d = LemaTensor(master=_ptr(t["master"]), m=_ptr(t["m"]), v=_ptr(t["v"]),
                       acc=_ptr(t["acc"]) if with_acc else None, delta=_ptr(t["delta"]),
                       orig_bf16=_ptr(t["orig"]), w_bf16=_ptr(t["w"]), grad_bf16=_ptr(grad),
                       n=t["orig"].numel(), flags=flags)
        if out_of_place is not None:
            d.master_out, d.m_out, d.v_out = (_ptr(x) for x in out_of_place)
        return d

    def tensor_descs(self):
        if self._descs is None:
            self._descs = (LemaTensor * len(self.tensors))(
                *[self.tensor_desc(j) for j in range(len(self.tensors))])
        return self._descs

    def grad_descs(self, grads, first: bool = False):
        """LemaGrad array for one micro-step; grads[j] is tensor j's bf16 grad.
        first: the step's first micro-step (acc = +0 + g, old contents not read)."""
        assert len(grads) == len(self.tensors)
        fl = lema.LEMA_GRAD_FIRST if first else 0
        return (LemaGrad * len(grads))(*[
            LemaGrad(acc=_ptr(self.tensors[j]["acc"]), grad_bf16=_ptr(grads[j]),
                     n=self.tensors[j]["orig"].numel(), flags=fl)
            for j in range(len(grads))])

    def numpy_views(self, j: int):
        """(master, m, v, acc, delta, orig_u16, w_u16) as numpy arrays on the host."""
        import numpy as np
        t = self.tensors[j]
        out = [t[f].cpu().numpy() for f in self.fields_f32]
        out += [t[f].cpu().view(torch.int16).numpy().view(np.uint16) for f in ("orig", "w")]
        return out


def _pad(n: int) -> int:
    """Elements a tensor occupies in a slot (and in a packed host unit)."""
    return (int(n) + 63) // 64 * 64


class DeviceState(_State):
    """All states resident in HBM."""

    def __init__(self, w0_list, device="cuda"):
        super().__init__(w0_list, device, pin=False)


class HostState(_State):
    """All states in pinned host RAM (the streamed residency); `units` packs each
    unit like a slot; acc_device keeps the accumulators in device memory."""

    def __init__(self, w0_list, units=None, acc_device=None):
        super().__init__(w0_list, "cpu", pin=True, units=units, acc_device=acc_device)


def hparams(hyper, accum_steps: int) -> LemaHparams:
    return LemaHparams(hyper.lr, hyper.beta1, hyper.beta2, hyper.eps, hyper.weight_decay,
                       int(accum_steps))


class Layers:
    """The lema_layer array of one micro-step: units of tensor indices over a state."""

    def __init__(self, state: _State, units, packed=None):
        self.state = state
        self.units = [list(u) for u in units]
        if packed is None:
            packed = getattr(state, "units", None) == self.units
        self.flags = lema.LEMA_UNIT_PACKED if packed else 0
        self._tensor_arrays = [
            (LemaTensor * len(u))(*[state.tensor_desc(j) for j in u]) for u in self.units]

    def build(self, grads):
        """grads[j]: tensor j's bf16 grad for this micro-step (device or pinned host)."""
        keep = []
        arr = (LemaLayer * len(self.units))()
        for i, u in enumerate(self.units):
            g = (ctypes.c_void_p * len(u))(*[_ptr(grads[j]) for j in u])
            keep.append(g)
            arr[i].tensors = ctypes.cast(self._tensor_arrays[i], ctypes.POINTER(LemaTensor))
            arr[i].grads = ctypes.cast(g, ctypes.POINTER(ctypes.c_void_p))
            arr[i].count = len(u)
            arr[i].flags = self.flags
        return arr, keep


class Pool:
    """Owning wrapper of a lema_pool."""

    def __init__(self, n_slots: int, slot_params: int):
        self.handle = lema.lema_pool_create(n_slots, slot_params)

    def stream_layers(self, layers_arr, micro_step, hp: LemaHparams, step, stream=None,
                      residency=lema.LEMA_STREAMED):
        lema.lema_stream_layers(self.handle, layers_arr, residency, micro_step, hp, step, stream)

    def sync(self, timeout_ms: int = 600_000):
        lema.lema_pool_sync(self.handle, timeout_ms)

    def slices(self, max_slices: int, min_slice_params: int, first_unit_only=False):
        lema.lema_pool_slices(self.handle, max_slices, min_slice_params)
        lema.lema_pool_slice_first_unit(self.handle, first_unit_only)

    def wait_stream(self, stream=None):
        lema.lema_pool_wait_stream(self.handle, stream)

    def close(self):
        if self.handle:
            lema.lema_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def slot_params_for(cfg) -> int:
    """Slot capacity (elements) that fits the largest streaming unit of cfg (at least
    one element: a pool needs a size even when every tensor is empty)."""
    return max(1, max(sum(_pad(cfg.tensors[j].numel) for j in cfg.unit_tensors(u))
                      for u in range(cfg.n_units)))


Q8_BLOCK = 256


def _pad_q8(n: int) -> int:
    """Elements a tensor occupies in an 8-bit slot (and packed host unit): whole
    groups of four 256-element blocks, so each tensor's block scales are a slice
    of their own that starts on a 16-byte boundary."""
    return (int(n) + 4 * Q8_BLOCK - 1) // (4 * Q8_BLOCK) * (4 * Q8_BLOCK)


_Q8_FIELDS = (("master", torch.float32, 1), ("delta", torch.float32, 1),
              ("m_q", torch.int8, 1), ("r_q", torch.uint8, 1), ("acc_q", torch.int8, 1),
              ("orig", torch.bfloat16, 1), ("w", torch.bfloat16, 1),
              ("m_scale", torch.float32, Q8_BLOCK), ("r_scale", torch.float32, Q8_BLOCK),
              ("acc_scale", torch.float32, Q8_BLOCK))


class DeviceStateQ8:
    """States with 8-bit moments and accumulators: per tensor fp32 master and
    delta, bf16 orig and w, int8 m and accumulator codes, uint8 codes of sqrt(v),
    and one fp32 scale per 256-element block of each 8-bit field.  Resident in HBM
    here; HostStateQ8 keeps the same fields in pinned host RAM."""

    def __init__(self, w0_list, device="cuda"):
        self.pinned = None
        self.units = None
        self.tensors = []
        for w0 in w0_list:
            orig = w0.reshape(-1).to(device)
            n = orig.numel()
            st = {f: torch.zeros((n + per - 1) // per, dtype=dt, device=device)
                  for f, dt, per in _Q8_FIELDS if f not in ("orig", "w")}
            st["orig"], st["w"] = orig, orig.clone()
            st["master"].copy_(orig)          # exact bf16 -> fp32 widening
            self.tensors.append(st)

    def close(self):
        if self.pinned is not None:
            self.pinned.close()

    @property
    def numel(self) -> int:
        return sum(t["orig"].numel() for t in self.tensors)

    def tensor_desc(self, j, grad=None, flags=0, with_acc=True) -> LemaTensorQ8:
        t = self.tensors[j]
        return LemaTensorQ8(
            master=_ptr(t["master"]), m_q=_ptr(t["m_q"]), m_scale=_ptr(t["m_scale"]),
            r_q=_ptr(t["r_q"]), r_scale=_ptr(t["r_scale"]),
            acc_q=_ptr(t["acc_q"]) if with_acc else None,
            acc_scale=_ptr(t["acc_scale"]) if with_acc else None,
            delta=_ptr(t["delta"]), orig_bf16=_ptr(t["orig"]), w_bf16=_ptr(t["w"]),
            grad_bf16=_ptr(grad), n=t["orig"].numel(), flags=flags)

    def grad_descs(self, grads, first=False):
        fl = lema.LEMA_GRAD_FIRST if first else 0
        return (LemaGradQ8 * len(grads))(*[
            LemaGradQ8(acc_q=_ptr(self.tensors[j]["acc_q"]),
                       acc_scale=_ptr(self.tensors[j]["acc_scale"]), grad_bf16=_ptr(grads[j]),
                       n=self.tensors[j]["orig"].numel(), flags=fl)
            for j in range(len(grads))])

    def numpy_views(self, j):
        """Every field of tensor j as numpy arrays (bf16 as uint16 patterns)."""
        import numpy as np
        t = self.tensors[j]
        out = {f: t[f].cpu().numpy() for f in ("master", "delta", "m_q", "r_q", "acc_q",
                                                 "m_scale", "r_scale", "acc_scale")}
        for f in ("orig", "w"):
            out[f] = t[f].cpu().view(torch.int16).numpy().view(np.uint16)
        return out


class HostStateQ8(DeviceStateQ8):
    """8-bit states in pinned host RAM (the streamed residency).  With `units`, each
    unit's fields are laid out like an 8-bit slot: one block per field, tensor j at
    its 1024-element offset o_j and its scales at o_j / 256 (LEMA_UNIT_PACKED).
    acc_device: the accumulator's codes and scales in that device's memory instead
    (same layout)."""

    def __init__(self, w0_list, units=None, acc_device=None):
        self.units = [list(u) for u in units] if units is not None else None
        groups = self.units or [[j] for j in range(len(w0_list))]
        on_device = ("acc_q", "acc_scale") if acc_device else ()
        sizes = []
        for u in groups:
            P = sum(_pad_q8(w0_list[j].numel()) for j in u)
            sizes += [(P // per, dt) for f, dt, per in _Q8_FIELDS if f not in on_device]
        self.pinned = PinnedBuffers(PinnedBuffers.arena_size(sizes))
        self.tensors = [None] * len(w0_list)
        for u in groups:
            P = sum(_pad_q8(w0_list[j].numel()) for j in u)
            block = {f: (torch.zeros(P // per, dtype=dt, device=acc_device) if f in on_device
                         else self.pinned.zeros(P // per, dt)) for f, dt, per in _Q8_FIELDS}
            o = 0
            for j in u:
                n = w0_list[j].numel()
                st = {f: block[f][o // per:o // per + (n + per - 1) // per]
                      for f, _, per in _Q8_FIELDS}
                st["orig"].copy_(w0_list[j].reshape(-1))
                st["w"].copy_(w0_list[j].reshape(-1))
                st["master"].copy_(st["orig"])
                self.tensors[j] = st
                o += _pad_q8(n)


class LayersQ8:
    """The lema_layer_q8 array of one micro-step over 8-bit states."""

    def __init__(self, state: DeviceStateQ8, units, packed=None):
        self.units = [list(u) for u in units]
        if packed is None:
            packed = state.units == self.units
        self.flags = lema.LEMA_UNIT_PACKED if packed else 0
        self._tensor_arrays = [
            (LemaTensorQ8 * len(u))(*[state.tensor_desc(j) for j in u]) for u in self.units]

    def build(self, grads):
        keep = []
        arr = (lema.LemaLayerQ8 * len(self.units))()
        for i, u in enumerate(self.units):
            g = (ctypes.c_void_p * len(u))(*[_ptr(grads[j]) for j in u])
            keep.append(g)
            arr[i].tensors = ctypes.cast(self._tensor_arrays[i], ctypes.POINTER(LemaTensorQ8))
            arr[i].grads = ctypes.cast(g, ctypes.POINTER(ctypes.c_void_p))
            arr[i].count = len(u)
            arr[i].flags = self.flags
        return arr, keep


def slot_params_for_q8(cfg) -> int:
    """Slot capacity (elements) whose 8-bit carving fits the largest unit of cfg."""
    need = max(sum(_pad_q8(cfg.tensors[j].numel) for j in cfg.unit_tensors(u))
               for u in range(cfg.n_units))
    return max(need, slot_params_for(cfg))


def _round_up(x: int, a: int) -> int:
    return (int(x) + a - 1) // a * a


class DiskState:
    """States of the disk tier: master, m, v, delta, orig and w of every unit in one
    file (the layout of lema_disk_layout), the accumulators in pinned host RAM packed
    like a slot.  The file gets the initial state (master = widen(orig), m = v =
    delta = 0, w = orig) here; the library reads and writes it from then on."""

    q8 = False
    # field -> (byte offset in a unit's block from (Q, S), dtype, elements per value)
    _FIELDS = {"master": (lambda Q, S: 0, torch.float32, 1),
               "m": (lambda Q, S: 4 * Q, torch.float32, 1),
               "v": (lambda Q, S: 8 * Q, torch.float32, 1),
               "delta": (lambda Q, S: 12 * Q, torch.float32, 1),
               "orig": (lambda Q, S: 16 * Q, torch.bfloat16, 1),
               "w": (lambda Q, S: 18 * Q, torch.bfloat16, 1)}
    _ACC = {"acc": (torch.float32, 1)}          # accumulator fields (pinned host RAM)

    @staticmethod
    def _unit_pad(n: int) -> int:
        return _pad(n)

    @staticmethod
    def _scale_bytes(Q: int) -> int:
        return 0

    def _block_bytes(self, Q: int) -> int:
        return 20 * Q

    def __init__(self, path, w0_list, units, flags=lema.LEMA_DISK_DIRECT, n_io_threads=8,
                 acc_device=None):
        """acc_device: keep the accumulators in that device's memory (same layout)
        instead of pinned host RAM."""
        import numpy as np
        self.path = path
        self.units = [list(u) for u in units]
        self.sizes = [int(w.numel()) for w in w0_list]
        self.unit_of = {}
        self.offset_in_unit = {}
        P = []
        for ui, u in enumerate(self.units):
            o = 0
            for j in u:
                self.unit_of[j], self.offset_in_unit[j] = ui, o
                o += self._unit_pad(self.sizes[j])
            P.append(o)
        self.unit_params = P
        self.unit_offset, self.padded = lema.lema_disk_layout(P, q8=self.q8)
        with open(path, "wb") as f:
            f.truncate(self.unit_offset[-1])
            for ui, u in enumerate(self.units):
                Q = self.padded[ui]
                S = self._scale_bytes(Q)
                block = np.zeros(self._block_bytes(Q), np.uint8)

                def view(name, dtype):
                    at = self._FIELDS[name][0](Q, S)
                    return block[at:].view(dtype)
                master, orig, w = view("master", np.float32), view("orig", np.uint16), view("w", np.uint16)
                for j in u:
                    o, n = self.offset_in_unit[j], self.sizes[j]
                    b = w0_list[j].reshape(-1).view(torch.int16).numpy().view(np.uint16)
                    orig[o:o + n] = b
                    w[o:o + n] = b
                    master[o:o + n] = (b.astype(np.uint32) << 16).view(np.float32)
                f.seek(self.unit_offset[ui])
                f.write(memoryview(block))
            # on disk before the library reads it with O_DIRECT (past the page cache)
            f.flush()
            os.fsync(f.fileno())
        if acc_device:
            self.pinned = None
            alloc = lambda n, dt: torch.zeros(n, dtype=dt, device=acc_device)  # noqa: E731
        else:
            self.pinned = PinnedBuffers(PinnedBuffers.arena_size(
                [(p // per, dt) for p in P for dt, per in self._ACC.values()]))
            alloc = self.pinned.zeros
        self.acc = {f: [None] * len(w0_list) for f in self._ACC}
        for ui, u in enumerate(self.units):
            for f, (dt, per) in self._ACC.items():
                block = alloc(P[ui] // per, dt)
                for j in u:
                    o = self.offset_in_unit[j] // per
                    self.acc[f][j] = block[o:o + (self.sizes[j] + per - 1) // per]
        if self.q8:
            flags |= lema.LEMA_DISK_Q8
        self.handle = lema.lema_disk_open(path, P, flags, n_io_threads)

    @property
    def numel(self) -> int:
        return sum(self.sizes)

    def tensor_desc(self, j: int) -> LemaTensor:
        return LemaTensor(acc=_ptr(self.acc["acc"][j]), n=self.sizes[j])

    def sync(self, timeout_ms: int = 600_000):
        lema.lema_disk_sync(self.handle, timeout_ms)

    def numpy_views(self, j: int):
        """(master, m, v, acc, delta, orig_u16, w_u16) of tensor j, read from the file
        (after sync())."""
        f = {name: self._read_np(j, name) for name in self._FIELDS}
        return [f["master"], f["m"], f["v"], self.acc["acc"][j].cpu().numpy().copy(),
                f["delta"], f["orig"], f["w"]]

    def _place(self, j, f):
        """(byte offset in the file, value count, torch dtype) of field f of tensor j."""
        at, dt, per = self._FIELDS[f]
        ui = self.unit_of[j]
        Q = self.padded[ui]
        size = torch.empty(0, dtype=dt).element_size()
        return (self.unit_offset[ui] + at(Q, self._scale_bytes(Q)) +
                size * (self.offset_in_unit[j] // per),
                (self.sizes[j] + per - 1) // per, dt)

    def _read(self, j, f):
        off, n, dt = self._place(j, f)
        size = torch.empty(0, dtype=dt).element_size()
        with open(self.path, "rb") as fh:
            fh.seek(off)
            raw = fh.read(n * size)
        if not n:
            return torch.empty(0, dtype=dt)
        t = torch.frombuffer(bytearray(raw), dtype=torch.uint8)
        return t.view(dt) if dt != torch.bfloat16 else t.view(torch.int16).view(dt)

    def _read_np(self, j, f):
        """Field f of tensor j as a numpy array (bf16 as uint16 patterns)."""
        import numpy as np
        t = self._read(j, f)
        return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()

    def field(self, j, f):
        """Field f of tensor j as a CPU tensor (read from the file; sync() first)."""
        if f in self._ACC:
            return self.acc[f][j].clone()
        return self._read(j, f)

    def set_field(self, j, f, value):
        """Write field f of tensor j (between steps, after sync())."""
        value = value.reshape(-1).contiguous().cpu()
        if f in self._ACC:
            self.acc[f][j].copy_(value)
            return
        off, n, dt = self._place(j, f)
        assert value.numel() == n and value.dtype == dt, (f, value.shape, value.dtype)
        if n:
            with open(self.path, "r+b") as fh:
                fh.seek(off)
                fh.write(memoryview(value.view(torch.uint8).numpy()))
                fh.flush()
                os.fsync(fh.fileno())

    def close(self):
        if self.handle:
            lema.lema_disk_close(self.handle)
            self.handle = None
        if self.pinned is not None:
            self.pinned.close()
            self.pinned = None


class DiskStateQ8(DiskState):
    """The disk tier with 8-bit states (the layout of lema_disk_layout_q8): per unit
    master, m codes, sqrt(v) codes, orig, delta, w and the two block-scale fields in
    the file; the 8-bit accumulator (codes + scales) in pinned host RAM, packed like
    an 8-bit slot.  Initial state: master = widen(orig), codes and scales 0, delta 0,
    w = orig."""

    q8 = True
    _FIELDS = {"master": (lambda Q, S: 0, torch.float32, 1),
               "m_q": (lambda Q, S: 4 * Q, torch.int8, 1),
               "r_q": (lambda Q, S: 5 * Q, torch.uint8, 1),
               "orig": (lambda Q, S: 6 * Q, torch.bfloat16, 1),
               "delta": (lambda Q, S: 8 * Q, torch.float32, 1),
               "w": (lambda Q, S: 12 * Q, torch.bfloat16, 1),
               "m_scale": (lambda Q, S: 14 * Q, torch.float32, Q8_BLOCK),
               "r_scale": (lambda Q, S: 14 * Q + S, torch.float32, Q8_BLOCK)}
    _ACC = {"acc_q": (torch.int8, 1), "acc_scale": (torch.float32, Q8_BLOCK)}

    @staticmethod
    def _unit_pad(n: int) -> int:
        return _pad_q8(n)

    @staticmethod
    def _scale_bytes(Q: int) -> int:
        return _round_up(Q // Q8_BLOCK * 4, 4096)

    def _block_bytes(self, Q: int) -> int:
        return 14 * Q + 2 * self._scale_bytes(Q)

    def tensor_desc(self, j: int) -> LemaTensorQ8:
        return LemaTensorQ8(acc_q=_ptr(self.acc["acc_q"][j]),
                            acc_scale=_ptr(self.acc["acc_scale"][j]), n=self.sizes[j])

    def numpy_views(self, j: int):
        """Every field of tensor j as numpy arrays (bf16 as uint16 patterns), the file
        fields read from the file (after sync())."""
        out = {f: self._read_np(j, f) for f in self._FIELDS}
        for f in self._ACC:
            out[f] = self.acc[f][j].cpu().numpy().copy()
        return out


class DiskLayers(Layers):
    """The lema_layer array of one micro-step over a DiskState (n and acc only)."""

    def __init__(self, state: DiskState):
        self.state = state
        self.units = state.units
        self.flags = lema.LEMA_UNIT_PACKED
        self._tensor_arrays = [
            (LemaTensor * len(u))(*[state.tensor_desc(j) for j in u]) for u in self.units]


class DiskLayersQ8(LayersQ8):
    """The lema_layer_q8 array of one micro-step over a DiskStateQ8 (n and the
    accumulator only)."""

    def __init__(self, state: DiskStateQ8):
        self.state = state
        self.units = state.units
        self.flags = lema.LEMA_UNIT_PACKED
        self._tensor_arrays = [
            (LemaTensorQ8 * len(u))(*[state.tensor_desc(j) for j in u]) for u in self.units]
