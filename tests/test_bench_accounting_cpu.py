"""bench.py's workload accounting on CPU: FLOP and byte counts in closed form,
the training-mode workload charged like the eval block, the oracle samplers'
units, and the recorded DRAM counters."""
import os

import pytest

import bench
from normalization_convolution_blocks_gb300 import synthetic as syn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_flops_in_closed_form():
    assert bench.workload_info("prenorm_block_f32")["flops"] == 2 * 32 * 4096 * 256 * 256 * 3
    assert bench.workload_info("conv1d_groupnorm_f32")["flops"] == 2 * 16 * 1024 * 256 * 128 * 3
    assert bench.workload_info("linear_bn_swish_f32")["flops"] == 2 * 1024 * 8192 * 8192
    assert bench.workload_info("prenorm_block_bf16_C512_d8")["flops"] == \
        2 * 8 * 16384 * 512 * 512 * 3


def test_block_min_bytes():
    # x read once, out written once, weights, bias, four BN vectors
    info = bench.workload_info("prenorm_block_f32")
    N, C, L = 32, 256, 4096
    assert info["min_bytes"] == 4 * (2 * N * C * L + 3 * C * C + C) + 16 * C
    bf = bench.workload_info("prenorm_block_bf16_C256_d1")
    assert bf["min_bytes"] == 2 * (2 * 8 * 256 * 16384 + 3 * 256 * 256 + 256) + 16 * 256
    assert bf["dtype"] == "bf16" and info["dtype"] == "f32"


def test_training_workload_is_charged_like_the_eval_block():
    ev, tr = bench.workload_info("prenorm_block_f32"), bench.workload_info(
        "prenorm_block_train_f32")
    assert tr["flops"] == ev["flops"] and tr["min_bytes"] == ev["min_bytes"]
    assert tr["main_kernel"] == ev["main_kernel"] == "prenorm_block_gemm"
    assert tr["config"]["bn"] == "training" and tr["config"]["momentum"] == bench.TRAIN_MOMENTUM


def test_every_workload_kind_has_a_source_and_a_sampler_unit():
    for name, wl in syn.WORKLOADS.items():
        assert wl.kind in bench.KERNEL_TU, name
        assert os.path.exists(os.path.join(ROOT, "normalization_convolution_blocks_gb300", "csrc",
                                           bench.KERNEL_TU[wl.kind]))


@pytest.mark.parametrize("name", ["prenorm_block_tiny_f32"])
def test_block_sampler_counts_flops_per_row(name):
    run, unit, total = bench.oracle_sampler(name)
    assert total == 2 * 32 and "rows" in unit
    assert run(2) == 2 * (2 * 32 * 3 * 512)       # two rows of C*3 MACs per position


def test_recorded_dram_counters_are_well_formed():
    for name, rec in bench.NCU_TRAFFIC.items():
        assert name in syn.WORKLOADS
        assert rec["bytes"] > 0 and len(rec["src_hash"]) == 16


def test_l2_note_tells_apart_workloads_that_exceed_l2():
    assert "exceeds L2" in bench.l2_note(bench.workload_info("prenorm_block_f32"))
    assert "exceeds L2" in bench.l2_note(bench.workload_info("linear_bn_swish_f32"))
    assert "fits in L2" in bench.l2_note(bench.workload_info("conv1d_groupnorm_f32"))


def test_json_line_assembly_with_a_stubbed_gpu_arm(monkeypatch, capsys):
    """main() on one rank with the GPU arm replaced by fixed numbers: the line
    carries the contract's keys, and value/bandwidth follow from them."""
    import json
    import sys
    info = bench.workload_info("prenorm_block_f32")
    fake = dict(value=430.0, ms_per_step=0.12, steps=100, launches=200,
                roofline=dict(bound="tensor", achieved=430.0, peak=963.2, unit="TFLOP/s",
                              frac=0.446, traffic=None),
                kernels={}, clocks=dict(sm_mhz=2070.0, sm_max_mhz=2070.0, reasons=[]),
                info=info, step_ms_p10=0.119, step_ms_p90=0.121, step_ms_median=0.12,
                e2e=dict(value=50.0, unit="TFLOP/s", h2d_bytes_per_step=1,
                         d2h_bytes_per_step=1),
                graph=dict(ms_per_call_median=0.118, ms_per_call_p10=0.117, replays=100,
                           host_us_per_call_eager=30.0, host_us_per_call_graph=4.0))
    monkeypatch.setattr(bench, "gpu_arm", lambda args, world, rank, local: fake)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--no-cpu-baseline", "--steps", "100"])
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    bench.main()
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "clocks", "bandwidth",
                "ms_per_call_median", "graph"):
        assert key in line, key
    assert line["n_gpus"] == 1 and line["value"] == 430.0 and line["warmup"] >= 3
    assert line["config"]["workload"] == "prenorm_block_f32"
    assert line["bandwidth"]["value"] == pytest.approx(info["min_bytes"] / 0.12e-3 / 1e9, abs=0.1)


def test_roofline_of_picks_the_longer_bound_and_scales_the_fraction():
    """Tensor-bound fp32 workload: strict fraction against the TF32 peak, and
    the effective one against three TF32 products per term; an HBM-bound one
    against the copy bandwidth, with effective = strict."""
    peaks = dict(bf16_tflops=2250.0, hbm_gbs=8000.0)
    tf32 = 2250.0 * bench.TF32_PER_BF16
    f32 = dict(flops=1e12, min_bytes=1e6, dtype="f32")
    ms = 2.0 * 1e12 / (tf32 * 1e12) * 1e3          # twice the strict roofline time
    roof, _ = bench.roofline_of(f32, ms, peaks)
    assert roof["bound"] == "tensor" and roof["frac"] == pytest.approx(0.5, abs=1e-4)
    assert roof["frac_effective"] == pytest.approx(1.5, abs=1e-4)
    hbm = dict(flops=1e6, min_bytes=8e9, dtype="bf16")
    roof, _ = bench.roofline_of(hbm, 4.0, peaks)      # 8 GB at 8 TB/s is 1 ms
    assert roof["bound"] == "hbm" and roof["frac"] == pytest.approx(0.25, abs=1e-4)
    assert roof["frac_effective"] == roof["frac"]
