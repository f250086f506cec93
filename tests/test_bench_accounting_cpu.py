"""bench.py's workload accounting on CPU: FLOP and byte counts in closed form,
the training-mode workload charged like the eval block, the oracle samplers'
units, and the recorded DRAM counters pointing at committed profiles."""
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


def test_recorded_dram_counters_name_committed_profiles():
    for name, rec in bench.NCU_TRAFFIC.items():
        assert name in syn.WORKLOADS
        assert os.path.exists(os.path.join(ROOT, rec["profile"])), rec["profile"]
        assert rec["bytes"] > 0 and len(rec["src_hash"]) == 16
