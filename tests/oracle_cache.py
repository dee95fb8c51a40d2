"""Oracle results shared between test modules within one pytest process (the
resident and streamed forms of a workload have the same inputs and results)."""
from __future__ import annotations

import os

from oracle.runner import run_config, run_config_q8

_cache = {}
_cache_q8 = {}


def oracle_states(cfg, tensors=None):
    key = (cfg.tensors, cfg.accum_steps, cfg.steps, cfg.grad_mode, cfg.zero_frac, cfg.hyper,
           None if tensors is None else tuple(tensors))
    if key not in _cache:
        _cache.clear()
        _cache[key] = run_config(cfg, tensors=tensors, threads=os.cpu_count() or 1)
    return _cache[key]


def oracle_states_q8(cfg, fused=True):
    """The oracle's 8-bit form over every tensor (shared by the resident and streamed
    8-bit tests of one workload: same inputs, same arithmetic)."""
    key = (cfg.tensors, cfg.accum_steps, cfg.steps, cfg.grad_mode, cfg.zero_frac, cfg.hyper,
           fused)
    if key not in _cache_q8:
        _cache_q8.clear()
        _cache_q8[key] = run_config_q8(cfg, fused=fused, threads=os.cpu_count() or 1)
    return _cache_q8[key]
