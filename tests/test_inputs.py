"""Workload definitions and the seeded input generator (no GPU)."""
import numpy as np
import torch

from adamw_step_gb300 import configs, inputs
from adamw_step_gb300.configs import CONFIGS, EXPECTED_PARAMS


def test_param_counts():
    for cid, cfg in CONFIGS.items():
        assert cfg.params == EXPECTED_PARAMS[cid], cid


def test_config_shapes():
    c1 = CONFIGS[1]
    assert [t.numel for t in c1.tensors] == [768 * 2304, 2304, 768 * 2304, 2304, 1_000_003]
    assert c1.tensors[-1].numel % 8 == 3          # ragged tail
    assert (CONFIGS[2].accum_steps, CONFIGS[2].steps) == (8, 5)
    assert CONFIGS[3].n_units == 4 and CONFIGS[3].unit_params(0) == 4 * 4096 * 4096
    c4, c5 = CONFIGS[4], CONFIGS[5]
    assert len(c4.tensors) == 201 and len(c5.tensors) == 291
    assert c4.unit_params(1) == 44_044_288 and c5.unit_params(1) == 202_383_360
    assert max(c4.unit_params(u) for u in range(c4.n_units)) == 32000 * 2048 + 2048
    assert len(c4.shape_classes) == 5 and sum(c4.shape_classes) == 81_790_976
    assert len(c5.shape_classes) == 4 and sum(c5.shape_classes) == 192_942_080


def test_generator_is_deterministic_and_shaped():
    cfg = configs.scaled(CONFIGS[2], tuple(configs.TensorSpec(f"t{i}", (64, 96), 0)
                                           for i in range(3)))
    a, b = inputs.w0_bf16(cfg, 1), inputs.w0_bf16(cfg, 1)
    assert a.dtype == torch.bfloat16 and a.numel() == 64 * 96
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert not torch.equal(a.view(torch.int16), inputs.w0_bf16(cfg, 2).view(torch.int16))
    std = a.float().std().item()
    assert 0.017 < std < 0.023


def test_zero_mask_in_every_bank_buffer():
    cfg = configs.scaled(CONFIGS[2], (configs.TensorSpec("t", (100, 100), 0),))
    mask = inputs.zero_mask(cfg, 0)
    assert mask.numel() == 100 and mask.unique().numel() == 100
    gs = inputs.GradSource(cfg)
    for t in range(2):
        for k in range(3):
            g = gs(0, t, k)
            assert torch.all(g[mask].float() == 0)
            assert (g.float() == 0).sum().item() < 200


def test_bank_rotation_avoids_reuse():
    cfg = CONFIGS[2]
    seq = [inputs.bank_index(cfg, j, t, k) for t in range(2) for k in range(8) for j in range(16)]
    assert all(seq[i] != seq[i + 1] for i in range(len(seq) - 1))


def test_fresh_grads_are_distinct():
    cfg = configs.scaled(CONFIGS[1], (configs.TensorSpec("a", (1000,), 0),), accum_steps=2)
    g = [inputs.fresh_grad(cfg, 0, t, k) for t in range(2) for k in range(2)]
    bits = {bytes(inputs.as_u16(x).tobytes()) for x in g}
    assert len(bits) == 4
    assert np.abs(g[0].float().numpy()).max() < 1e-2


def test_kernel_hash_ignores_comments_only():
    """bench.py keys its DRAM counters by a hash of the kernel code; comments and
    whitespace do not count, code does."""
    import bench
    a = 'int f(int x) { return x + 1; }  // one\n'
    assert bench._code_only(a) == bench._code_only('/* doc */ int  f(int x)\n{ return x + 1; }')
    assert bench._code_only(a) != bench._code_only(a.replace("+ 1", "+ 2"))
    assert bench._code_only('s = "a // b";') == 's="a // b";'


def test_bench_l2_label_follows_the_bytes_per_launch():
    """bench.py labels a workload by whether its launches can be served from the
    129 MB L2: every launch above it, every launch within it, or some of each."""
    import bench
    assert bench.l2_label([1.6e9, 10.2e9]).startswith("inputs larger than L2")
    assert "within the 129 MB L2" in bench.l2_label([6e6, 10e6])
    mixed = bench.l2_label([27e6, 45e6, 173e6])
    assert "partly L2-served" in mixed and "27-173 MB" in mixed


def test_bench_traffic_figures_match_the_current_kernels():
    """The committed DRAM counters are keyed by the kernel families' current code,
    so the bench line reports them (a stale key would make it report null)."""
    import bench
    for kind in ("accum_grad_first", "accum_grad", "adamw_fused", "accum_grad_first_q8",
                 "accum_grad_q8", "adamw_fused_q8"):
        t = bench.ncu_traffic(kind)
        assert t is not None, kind
        # every byte streamed once per launch: no more than 1 % above the algorithmic
        # bytes, and at most 5 % below (reads the L2 still held from the launch before)
        alg = bench.BYTES[kind]
        assert -0.05 * alg <= t - alg <= 0.01 * alg, (kind, t)


def test_bench_streamed_options_parse(monkeypatch):
    """The streamed legs' options: accumulators in HBM, slicing of every unit or only
    each call's first."""
    import sys
    import bench
    monkeypatch.setattr(sys, "argv", ["bench.py", "--config", "3", "--acc-on-device",
                                      "--slices", "2", "--slice-first", "--q8"])
    a = bench.parse()
    assert a.config == 3 and a.acc_on_device and a.slices == 2 and a.slice_first and a.q8
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    a = bench.parse()
    assert a.config == 2 and not a.acc_on_device and a.slices == 0 and not a.slice_first


def test_link_floor_uses_the_better_probe_per_direction():
    """A probe that met a slow moment of the shared host must not lower the link
    peaks the floor divides by."""
    import bench
    from adamw_step_gb300.probes import link_time_floor
    slow = {"h2d_gbs": 88.1, "d2h_gbs": 192.2, "bidir_gbs": 91.1}
    fast = {"h2d_gbs": 210.0, "d2h_gbs": 190.0, "bidir_gbs": 339.0}
    best = bench.best_link_peaks(slow, fast)
    assert best == {"h2d_gbs": 210.0, "d2h_gbs": 192.2, "bidir_gbs": 339.0}
    assert bench.best_link_peaks(fast, slow) == best
    h2d, d2h = 28.6e9, 33.0e9
    assert link_time_floor(h2d, d2h, best) <= min(link_time_floor(h2d, d2h, slow),
                                                   link_time_floor(h2d, d2h, fast))
    rec = bench.probes_record(slow, fast)
    assert rec["before"]["h2d_gbs"] == 88.1 and rec["after"]["h2d_gbs"] == 210.0
