"""Host-side arithmetic of bench.py (CPU only): the algorithmic byte and FLOP counts per unit follow
from the block's shapes, and the layer roofline reproduces hand-computed figures for the decode
and prefill workloads against the measured and the nominal peaks."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

H, E, K, I, D = 2816, 128, 8, 704, 2112
EXPERT_BYTES = 3 * I * H * 2            # gate, up and down of one expert, bf16: 11,894,784
DENSE_BYTES = 3 * D * H * 2             # the shared MLP's three matrices: 35,684,352


def test_unit_counts_follow_from_the_shapes():
    assert bench.GATE_UP_BYTES_PER_EXPERT + bench.DOWN_BYTES_PER_EXPERT == EXPERT_BYTES == 11_894_784
    assert bench.DENSE_GATE_UP_BYTES + bench.DENSE_DOWN_BYTES == DENSE_BYTES == 35_684_352
    assert bench.ROUTER_BYTES == E * H * 4
    # Two FLOPs per multiply-add: per token, K experts of gate+up (2I x H) and down (H x I), and the
    # shared MLP's gate+up (2D x H) and down (H x D).
    assert bench.FLOPS_PER_TOKEN_EXPERTS + bench.FLOPS_PER_TOKEN_DENSE == 130_842_624


def _layer(T, experts_hit, step_us):
    b = experts_hit * EXPERT_BYTES + DENSE_BYTES + E * H * 4 + T * H * 2 * 2
    f = T * 130_842_624
    return bench.layer_roofline(b, f, step_us * 1e-6, 6794.5, 1916.3, experts_hit, 1)


def test_decode_roofline_is_the_weight_stream():
    # T=64 with 127 experts hit: 1,548,484,608 bytes, 227.9 us at 6794.5 GB/s, 193.6 us at 8 TB/s.
    r = _layer(64, 127, 253.1)
    assert r["bytes"] == 1_548_484_608 and r["bound"] == "hbm"
    assert r["roofline_us"] == pytest.approx(1_548_484_608 / 6794.5e3, rel=1e-12)
    assert r["roofline_us"] == pytest.approx(227.9, abs=0.05)
    assert r["roofline_nominal_us"] == pytest.approx(193.56, abs=0.01)
    assert r["frac"] == pytest.approx(227.9 / 253.1, abs=1e-3)
    assert r["frac_nominal"] == pytest.approx(193.56 / 253.1, abs=1e-3)


def test_prefill_roofline_is_the_tensor_rate():
    # T=4096: 535.9 GFLOP, 279.7 us at 1916.3 TFLOP/s, 238.2 us at 2.25 PFLOP/s; the bytes (88
    # experts hit) take far less.
    r = _layer(4096, 88, 592.7)
    assert r["flops"] == 4096 * 130_842_624 and r["bound"] == "tensor"
    assert r["roofline_us"] == pytest.approx(279.7, abs=0.05)
    assert r["roofline_nominal_us"] == pytest.approx(238.19, abs=0.01)
    assert r["frac"] == pytest.approx(279.7 / 592.7, abs=1e-3)


def test_job_throughput_counts_every_rank():
    assert bench.job_throughput(64, 10, 1, 0.5) == pytest.approx(1280.0)
    assert bench.job_throughput(64, 10, 4, 0.5) == pytest.approx(5120.0)


def test_default_run_follows_the_contract():
    # No flags: one GPU, at least three warm-up steps, the decode workload the metric is quoted on,
    # and the same arm the driver compares against the reference.
    a = bench.parse_args([])
    assert a.gpus == 1 and a.warmup >= 3 and a.steps >= 1
    assert a.impl == "ours" and a.workload == "decode64"
    wl = bench.workload_of(a)
    assert wl["T"] == 64 and wl["full"] and not wl["skew"]
    assert bench.workload_of(bench.parse_args(["--workload", "prefill4096"]))["skew"]


def test_reference_and_gpu_arms_print_the_same_config():
    # The driver compares the two arms' lines; both build `config` from one function.
    for name in ("decode64", "prefill4096", "moe8"):
        wl = bench.workload_of(bench.parse_args(["--workload", name]))
        assert bench.config_of(wl, 1) == bench.config_of(dict(wl), 1)
        assert bench.config_of(wl, 1)["T"] == wl["T"]
    src = open(os.path.join(ROOT, "bench.py")).read()
    assert src.count('"config": config_of(wl, world)') == 2


def test_default_run_adds_the_prefill_leg():
    # The metric is quoted at T=64 and at T=4096: the default run measures both.
    a = bench.parse_args([])
    assert not a.no_prefill
    wl = bench.workload_of(bench.argparse.Namespace(workload="prefill4096", T=None))
    assert wl["T"] == 4096 and wl["skew"] and wl["full"]


def test_clock_summary_names_its_window():
    c = bench.ClockSampler(uuid=None)
    row = ["0", "GPU-x", "2070", "2070", "500", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"]
    c.rows = [(10.0, row), (10.5, row), (11.2, row)]
    inside = c.summary(9.9, 10.6)
    assert inside["in_timed_region"] and inside["samples"] == 2 and inside["window"] == "timed region"
    after = c.summary(10.6, 10.61, 11.0, 11.5)
    assert not after["in_timed_region"] and after["samples"] == 1 and "right after" in after["window"]
    none = c.summary(10.6, 10.61)
    assert none["samples"] == 0 and not none["in_timed_region"]


def test_default_run_covers_every_configuration():
    # Beside the decode value and the prefill leg, the default run measures the experts-only block
    # at T=8, the sweep's other sizes and the 30-layer stack, so each configuration the metric is
    # reported on gets a number from the same run.
    a = bench.parse_args([])
    assert not a.no_configs
    assert set(bench.SWEEP_T) | {64} == {1, 16, 64, 256, 1024, 4096, 16384}
    assert bench.WORKLOADS["moe8"]["T"] == 8 and not bench.WORKLOADS["moe8"]["full"]
    assert bench.WORKLOADS["stack30"]["layers"] == 30 and bench.WORKLOADS["stack30"]["T"] == 256
    res = {"value": 1.0, "ms_per_step": 0.5,
           "layer_roofline": {"frac": 0.9, "bound": "hbm", "roofline_us": 200.0, "step_us": 222.0, "experts_hit": 8,
                              "bytes": 1, "flops": 2},
           "roofline": {"kernel": "gate_up_gemm", "bound": "hbm", "achieved": 6000.0, "peak": 6794.5,
                        "unit": "GB/s", "frac": 0.88, "traffic": None, "kernel_us": 1.0},
           "e2e": {"value": 0.9}, "gpu_launches": 80, "clocks": {"sm_mhz": 2070.0, "reasons": []},
           "kernels_us": {"combine": 1.0}}
    c = bench.compact_result(res, bench.WORKLOADS["moe8"], a)
    assert c["T"] == 8 and c["value"] == 1.0 and c["warmup"] >= 3 and c["e2e"] == 0.9
    assert c["layer_roofline"]["frac"] == 0.9 and c["roofline"]["kernel"] == "gate_up_gemm"
