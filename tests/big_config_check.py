"""Streamed run of a whole-model workload (config 4 or 5) at full size, checked
against the oracle on every element of every tensor.

Run as a script (a child process of the GPU test, so that its pinned host memory
is returned when it exits):  python tests/big_config_check.py <config>
Exit 0: checked; 3: skipped (not enough host memory); anything else: failure.
The last stdout line is a JSON summary.
"""
from __future__ import annotations

import json
import os
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from oracle.runner import run_config  # noqa: E402
from adamw_step_gb300 import configs, inputs  # noqa: E402
from adamw_step_gb300.hostmem import mem_available_bytes  # noqa: E402
from adamw_step_gb300.runner import DeviceGrads, StreamedRunner  # noqa: E402
from parity import check_tensor, oracle_dict, state_dict  # noqa: E402

# Host bytes the run holds beyond the pinned states: the oracle's per-tensor copy,
# the CPU grad bank while it is built, comparison copies, the CUDA/torch runtime.
HEADROOM = 24 << 30


def main(cid: int) -> int:
    cfg = configs.CONFIGS[cid]
    need = cfg.params * 24 + HEADROOM
    avail = mem_available_bytes()
    if avail < need:
        print(json.dumps({"skipped": True, "need_gb": need / 2 ** 30, "avail_gb": avail / 2 ** 30}))
        return 3
    t0 = time.time()
    grads = DeviceGrads(cfg)
    sr = StreamedRunner(cfg, grads)
    t_setup = time.time() - t0
    t0 = time.time()
    for t in range(cfg.steps):
        sr.step(t)
    sr.pool.sync(1_800_000)
    t_run = time.time() - t0

    # The oracle on every tensor, one at a time: its inputs regenerated from the
    # tensor's seed (never read back from the GPU side), freed after the comparison.
    t0 = time.time()
    threads = os.cpu_count() or 1
    gs = inputs.GradSource(cfg)
    orc = oracle.Oracle(threads=threads)
    bad = checked = checked_params = 0
    for j in range(len(cfg.tensors)):
        ref = run_config(cfg, tensors=[j], threads=threads, grad_source=gs)[j]
        partial = np.zeros(ref.acc.size, np.float32)
        for k in range(cfg.accum_steps - 1):
            orc.accum(partial, inputs.as_u16(gs(j, cfg.steps - 1, k)))
        rep = check_tensor(state_dict(sr.state, j), dict(oracle_dict(ref), acc=partial),
                           f"config {cid} tensor {j}")
        bad += sum(rep.values())
        checked += 1
        checked_params += cfg.tensors[j].numel
        del ref, partial
    t_check = time.time() - t0
    sr.close()
    print(json.dumps({"config": cid, "params": cfg.params, "tensors": len(cfg.tensors),
                      "tensors_checked": checked, "params_checked": checked_params,
                      "non_bit_exact": bad, "setup_s": round(t_setup, 1),
                      "run_s": round(t_run, 1), "check_s": round(t_check, 1)}))
    return 0 if (bad == 0 and checked_params == cfg.params) else 1


if __name__ == "__main__":
    sys.exit(main(int(sys.argv[1])))
