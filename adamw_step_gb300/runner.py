"""Drive whole optimizer steps through the C ABI: K micro-step accumulations, then
the fused AdamW step, with states resident in HBM or streamed from pinned host RAM.

Page "LEMA: Layer-wise Efficient Memory Abstraction", section "Selective Full
Fine-Tuning" (grad accumulation in fp32, per-layer AdamW) and section "TensorStore:
Unified Streaming Core" (residency per stream).  Steps t and micro-steps k are
0-based here and passed 1-based to the library.
"""
from __future__ import annotations

import torch

from . import inputs, lema
from .hostmem import PinnedBuffers
from .state import (Q8_BLOCK, DeviceState, DeviceStateQ8, DiskLayers, DiskLayersQ8, DiskState,
                    DiskStateQ8, HostState, HostStateQ8, Layers, LayersQ8, Pool, hparams,
                    slot_params_for, slot_params_for_q8)


class DeviceGrads:
    """The workload's micro-batch grads, resident on the device (they stand for the
    output of the backward pass): grad(j, t, k) -> bf16 device tensor."""

    def __init__(self, cfg, device="cuda", pin_host=False):
        self.cfg = cfg
        src = inputs.GradSource(cfg)
        self.pinned = None
        if pin_host:
            bufs = [b for cls in src.bank for b in cls] if src.bank is not None else \
                [src(j, t, k) for j in range(len(cfg.tensors)) for t in range(cfg.steps)
                 for k in range(cfg.accum_steps)]
            self.pinned = PinnedBuffers(PinnedBuffers.arena_size(
                [(b.numel(), b.dtype) for b in bufs]))
        move = self.pinned.copy_of if pin_host else (lambda x: x.to(device))
        if src.bank is not None:
            self.bank = [[move(b) for b in cls] for cls in src.bank]
            self.fresh = None
        else:
            self.bank = None
            self.fresh = {(j, t, k): move(src(j, t, k)) for j in range(len(cfg.tensors))
                          for t in range(cfg.steps) for k in range(cfg.accum_steps)}

    def __call__(self, j, t, k):
        if self.bank is None:
            return self.fresh[(j, t, k)]
        cfg = self.cfg
        return self.bank[cfg.shape_class(j)][inputs.bank_index(cfg, j, t % cfg.steps, k)]


def initial_weights(cfg):
    return [inputs.w0_bf16(cfg, j) for j in range(len(cfg.tensors))]


class ResidentRunner:
    """All states in HBM.

    fused=False: one step = K accumulate launches + 1 step launch (the accumulator
    starts from +0, the in-place step resets it): 10K + 40 bytes per param.
    fused=True (default): micro-step 1 writes acc = +0 + g without reading acc,
    micro-steps 2..K-1 accumulate, and micro-step K's grad is folded into the step,
    which keeps acc as it is (LEMA_STEP_KEEP_ACC): 6 + 10(K-2) + 38 bytes per param
    for K >= 2, K launches.  Same master/m/v/delta/w bits; afterwards acc holds the
    partial sum of micro-steps 1..K-1 instead of +0.
    """

    def __init__(self, cfg, grads: DeviceGrads, w0_list=None, device="cuda", fused=True):
        self.cfg = cfg
        self.grads = grads
        self.fused = fused
        self.state = DeviceState(w0_list or initial_weights(cfg), device)
        self._gd = {}
        self._sd = {}

    def grad_descs(self, t, k, first=False):
        key = (t % self.cfg.steps, k, first)
        if key not in self._gd:
            self._gd[key] = self.state.grad_descs(
                [self.grads(j, t, k) for j in range(len(self.cfg.tensors))], first=first)
        return self._gd[key]

    def fused_step_descs(self, t):
        key = t % self.cfg.steps
        if key not in self._sd:
            K = self.cfg.accum_steps
            n = len(self.cfg.tensors)
            self._sd[key] = (lema.LemaTensor * n)(*[
                self.state.tensor_desc(j, grad=self.grads(j, t, K - 1),
                                       flags=lema.LEMA_STEP_KEEP_ACC, with_acc=K > 1)
                for j in range(n)])
        return self._sd[key]

    def accumulate(self, t, stream=None):
        """The accumulate launches of step t (all K, or K-1 when fused)."""
        K = self.cfg.accum_steps
        if not self.fused:
            for k in range(K):
                lema.lema_accum_grad(self.grad_descs(t, k), stream)
            return
        for k in range(K - 1):
            lema.lema_accum_grad(self.grad_descs(t, k, first=(k == 0)), stream)

    def adamw(self, t, stream=None):
        cfg, hp = self.cfg, self.cfg.hyper
        descs = self.fused_step_descs(t) if self.fused else self.state.tensor_descs()
        lema.lema_adamw_step(descs, t + 1, hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay,
                             cfg.accum_steps, stream)

    def step(self, t, stream=None):
        """Optimizer step t (0-based)."""
        self.accumulate(t, stream)
        self.adamw(t, stream)

    @property
    def launches_per_step(self):
        return self.cfg.accum_steps + (0 if self.fused else 1)

    def bytes_per_step(self):
        """Algorithmic bytes one optimizer step moves, per launch kind (per param)."""
        K = self.cfg.accum_steps
        if not self.fused:
            return {"accum_grad": (K, 10), "adamw_fused": (1, 40)}
        if K == 1:
            return {"adamw_fused": (1, 34)}
        return {"accum_grad_first": (1, 6), "accum_grad": (K - 2, 10), "adamw_fused": (1, 38)}


class StreamedRunner:
    """States in pinned host RAM, streamed unit by unit through a slot pool."""

    def __init__(self, cfg, grads: DeviceGrads, w0_list=None, n_slots=None, packed=True,
                 acc_on_device=False):
        """packed: lay each unit's host states out like a slot (one copy per field
        per unit); False: an independent buffer per tensor (one copy per tensor).
        acc_on_device: the accumulators live in HBM (only the optimizer states and
        weights stream)."""
        self.cfg = cfg
        self.grads = grads
        self.acc_on_device = acc_on_device
        units = [cfg.unit_tensors(u) for u in range(cfg.n_units)]
        self.state = HostState(w0_list or initial_weights(cfg), units=units if packed else None,
                               acc_device="cuda" if acc_on_device else None)
        self.pool = Pool(n_slots or cfg.n_slots, slot_params_for(cfg))
        self.layers = Layers(self.state, [cfg.unit_tensors(u) for u in range(cfg.n_units)])
        self.hp = hparams(cfg.hyper, cfg.accum_steps)
        self._built = {}

    def _layers(self, t, k):
        key = (t % self.cfg.steps, k)
        if key not in self._built:
            self._built[key] = self.layers.build(
                [self.grads(j, t, k) for j in range(len(self.cfg.tensors))])
        return self._built[key][0]

    def step(self, t, stream=None):
        for k in range(self.cfg.accum_steps):
            self.pool.stream_layers(self._layers(t, k), k + 1, self.hp, t + 1, stream)

    def wait(self, stream=None):
        self.pool.wait_stream(stream)

    def link_bytes_per_step(self, host_grads=False):
        """(H2D, D2H) bytes one optimizer step moves over the host link."""
        n, K = self.state.numel, self.cfg.accum_steps
        acc = 0 if self.acc_on_device else 4 * (K - 1)
        h2d = n * (14 + acc + (2 * K if host_grads else 0))
        d2h = n * (18 + acc)
        return h2d, d2h

    def close(self):
        self.pool.close()
        self.state.close()


class ResidentRunnerQ8:
    """8-bit moments and accumulators, resident in HBM.

    fused=True (default): micro-step 1 encodes +0 + g (LEMA_GRAD_FIRST), micro-steps
    2..K-1 decode, add and re-encode, and micro-step K's grad is added to the decoded
    accumulator inside the step (not re-encoded), which keeps the accumulator
    (LEMA_STEP_KEEP_ACC).  fused=False: K accumulate launches, then a step that
    resets the accumulator.  The two forms differ by that one re-encoding of the
    final sum; each matches its own oracle form bit for bit."""

    def __init__(self, cfg, grads: DeviceGrads, w0_list=None, device="cuda", fused=True):
        self.cfg = cfg
        self.grads = grads
        self.fused = fused
        self.state = DeviceStateQ8(w0_list or initial_weights(cfg), device)
        self._gd = {}
        self._sd = {}

    def grad_descs(self, t, k, first=False):
        key = (t % self.cfg.steps, k, first)
        if key not in self._gd:
            self._gd[key] = self.state.grad_descs(
                [self.grads(j, t, k) for j in range(len(self.cfg.tensors))], first=first)
        return self._gd[key]

    def step_descs(self, t):
        key = (t % self.cfg.steps) if self.fused else -1
        if key not in self._sd:
            K, n = self.cfg.accum_steps, len(self.cfg.tensors)
            if self.fused:
                ds = [self.state.tensor_desc(j, grad=self.grads(j, t, K - 1),
                                             flags=lema.LEMA_STEP_KEEP_ACC, with_acc=K > 1)
                      for j in range(n)]
            else:
                ds = [self.state.tensor_desc(j) for j in range(n)]
            self._sd[key] = (lema.LemaTensorQ8 * n)(*ds)
        return self._sd[key]

    def accumulate(self, t, stream=None):
        K = self.cfg.accum_steps
        for k in range(K - 1 if self.fused else K):
            lema.lema_accum_grad_q8(self.grad_descs(t, k, first=(k == 0)), stream)

    def adamw(self, t, stream=None):
        cfg, hp = self.cfg, self.cfg.hyper
        lema.lema_adamw_step_q8(self.step_descs(t), t + 1, hp.lr, hp.beta1, hp.beta2, hp.eps,
                                hp.weight_decay, cfg.accum_steps, stream)

    def step(self, t, stream=None):
        self.accumulate(t, stream)
        self.adamw(t, stream)


class StreamedRunnerQ8:
    """8-bit states in pinned host RAM, streamed unit by unit through a slot pool
    (lema_stream_layers_q8).  Same arithmetic as ResidentRunnerQ8(fused=True): the
    last micro-batch grad is folded into the step and the host accumulator keeps
    micro-steps 1..K-1."""

    def __init__(self, cfg, grads: DeviceGrads, w0_list=None, n_slots=None, packed=True,
                 acc_on_device=False):
        self.cfg = cfg
        self.grads = grads
        self.acc_on_device = acc_on_device
        units = [cfg.unit_tensors(u) for u in range(cfg.n_units)]
        self.state = HostStateQ8(w0_list or initial_weights(cfg),
                                 units=units if packed else None,
                                 acc_device="cuda" if acc_on_device else None)
        self.pool = Pool(n_slots or cfg.n_slots, slot_params_for_q8(cfg))
        self.layers = LayersQ8(self.state, units)
        self.hp = hparams(cfg.hyper, cfg.accum_steps)
        self._built = {}

    def _layers(self, t, k):
        key = (t % self.cfg.steps, k)
        if key not in self._built:
            self._built[key] = self.layers.build(
                [self.grads(j, t, k) for j in range(len(self.cfg.tensors))])
        return self._built[key][0]

    def step(self, t, stream=None):
        for k in range(self.cfg.accum_steps):
            lema.lema_stream_layers_q8(self.pool.handle, self._layers(t, k), k + 1, self.hp,
                                       t + 1, stream)

    def wait(self, stream=None):
        self.pool.wait_stream(stream)

    def link_bytes_per_step(self, host_grads=False):
        """(H2D, D2H) bytes one optimizer step moves over the host link."""
        K = self.cfg.accum_steps
        n = self.state.numel
        nb = sum((t["orig"].numel() + Q8_BLOCK - 1) // Q8_BLOCK for t in self.state.tensors)
        acc = 0 if self.acc_on_device else n + 4 * nb   # codes + scales of the accumulator
        h2d = 8 * n + 8 * nb + (K - 1) * acc + (2 * K * n if host_grads else 0)
        d2h = 12 * n + 8 * nb + (K - 1) * acc
        return h2d, d2h

    def close(self):
        self.pool.close()
        self.state.close()


class DiskRunner:
    """The disk tier: optimizer states, weights and delta in a file, accumulators in
    pinned host RAM, each unit streamed file -> pinned staging -> VRAM -> staging ->
    file at the step's last micro-step (lema_stream_layers_disk).  q8: 8-bit moments
    and accumulators (lema_stream_layers_disk_q8; the arithmetic of
    StreamedRunnerQ8)."""

    def __init__(self, cfg, grads: DeviceGrads, path, w0_list=None, n_slots=None,
                 flags=lema.LEMA_DISK_DIRECT, n_io_threads=8, q8=False, acc_on_device=False):
        self.cfg = cfg
        self.grads = grads
        self.q8 = q8
        self.acc_on_device = acc_on_device
        units = [cfg.unit_tensors(u) for u in range(cfg.n_units)]
        State = DiskStateQ8 if q8 else DiskState
        self.state = State(path, w0_list or initial_weights(cfg), units, flags, n_io_threads,
                           acc_device="cuda" if acc_on_device else None)
        self.pool = Pool(n_slots or cfg.n_slots,
                         slot_params_for_q8(cfg) if q8 else slot_params_for(cfg))
        self.layers = DiskLayersQ8(self.state) if q8 else DiskLayers(self.state)
        self.hp = hparams(cfg.hyper, cfg.accum_steps)
        self._built = {}

    def _layers(self, t, k):
        key = (t % self.cfg.steps, k)
        if key not in self._built:
            self._built[key] = self.layers.build(
                [self.grads(j, t, k) for j in range(len(self.cfg.tensors))])
        return self._built[key][0]

    def step(self, t, stream=None):
        fn = lema.lema_stream_layers_disk_q8 if self.q8 else lema.lema_stream_layers_disk
        for k in range(self.cfg.accum_steps):
            fn(self.pool.handle, self.state.handle, self._layers(t, k), k + 1, self.hp, t + 1,
               stream)

    def wait(self, stream=None):
        self.pool.wait_stream(stream)

    def sync(self):
        self.pool.sync()
        self.state.sync()

    def disk_bytes_per_step(self):
        """(read, write) bytes of the file per optimizer step."""
        q = sum(self.state.padded)
        if self.q8:
            s = sum(2 * self.state._scale_bytes(Q) for Q in self.state.padded)
            return 8 * q + s, 12 * q + s
        return 14 * q, 18 * q

    def link_bytes_per_step(self):
        n, K = self.state.numel, self.cfg.accum_steps
        if self.q8:
            nb = sum((x + Q8_BLOCK - 1) // Q8_BLOCK for x in self.state.sizes)
            acc = 0 if self.acc_on_device else n + 4 * nb
            return 8 * n + 8 * nb + (K - 1) * acc, 12 * n + 8 * nb + (K - 1) * acc
        acc = 0 if self.acc_on_device else 4 * (K - 1)
        return n * (14 + acc), n * (18 + acc)

    def close(self):
        self.pool.close()
        self.state.close()


class HostGradRunner:
    """Resident states, micro-batch grads arriving from pinned host memory: the end-
    to-end form of the resident step.  Each micro-step's grads are copied into one of
    two device buffer sets on a copy stream while the kernels consume the other set
    (events order the reuse); the step folds micro-step K's grads in (as
    ResidentRunner, fused); `read_weights` copies the bf16 working weights back to
    pinned host memory, the step's result.  q8: 8-bit moments and accumulators (as
    ResidentRunnerQ8, fused)."""

    def __init__(self, cfg, host_grads: DeviceGrads, w0_list=None, device="cuda", q8=False):
        assert host_grads.pinned is not None, "host_grads must be pinned host memory"
        self.cfg = cfg
        self.host = host_grads
        self.q8 = q8
        w0 = w0_list or initial_weights(cfg)
        self.state = DeviceStateQ8(w0, device) if q8 else DeviceState(w0, device)
        n = [t.numel for t in cfg.tensors]
        self.dev = [[torch.empty(x, dtype=torch.bfloat16, device=device) for x in n]
                    for _ in range(2)]
        self.copy_stream = torch.cuda.Stream(device=device)
        self.ready = [torch.cuda.Event() for _ in range(2)]
        self.free = [torch.cuda.Event() for _ in range(2)]
        for e in self.free:
            e.record(torch.cuda.current_stream(device))
        self.pinned = PinnedBuffers(PinnedBuffers.arena_size([(x, torch.bfloat16) for x in n]))
        self.w_host = [self.pinned.empty(x, torch.bfloat16) for x in n]
        K = cfg.accum_steps
        self._acc = {(b, first): self.state.grad_descs(self.dev[b], first=first)
                     for b in range(2) for first in (False, True)}
        T = lema.LemaTensorQ8 if q8 else lema.LemaTensor
        self._step = [(T * len(n))(*[
            self.state.tensor_desc(j, grad=self.dev[b][j], flags=lema.LEMA_STEP_KEEP_ACC,
                                   with_acc=K > 1) for j in range(len(n))]) for b in range(2)]
        self._accum = lema.lema_accum_grad_q8 if q8 else lema.lema_accum_grad
        self._adamw = lema.lema_adamw_step_q8 if q8 else lema.lema_adamw_step

    def h2d_bytes_per_step(self):
        return 2 * self.cfg.accum_steps * self.state.numel

    def d2h_bytes_per_step(self):
        return 2 * self.state.numel

    def step(self, t, stream=None):
        cfg, hp = self.cfg, self.cfg.hyper
        stream = stream or torch.cuda.current_stream()
        K = cfg.accum_steps
        for k in range(K):
            b = k % 2
            with torch.cuda.stream(self.copy_stream):
                self.copy_stream.wait_event(self.free[b])
                for j in range(len(cfg.tensors)):
                    self.dev[b][j].copy_(self.host(j, t, k), non_blocking=True)
                self.ready[b].record(self.copy_stream)
            stream.wait_event(self.ready[b])
            if k < K - 1:
                self._accum(self._acc[(b, k == 0)], stream)
            else:
                self._adamw(self._step[b], t + 1, hp.lr, hp.beta1, hp.beta2, hp.eps,
                            hp.weight_decay, K, stream)
            self.free[b].record(stream)

    def read_weights(self, stream=None):
        """Copy the bf16 working weights to pinned host memory (on `stream`)."""
        stream = stream or torch.cuda.current_stream()
        with torch.cuda.stream(stream):
            for j, t in enumerate(self.state.tensors):
                self.w_host[j].copy_(t["w"], non_blocking=True)

    def close(self):
        torch.cuda.synchronize()
        self.pinned.close()
