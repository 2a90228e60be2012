"""bench.py's roofline arithmetic on made-up kernel times (host-only): achieved = the algorithmic work of
one launch of the dominant kernel / its mean launch time, frac = achieved / the measured peak, with the
expert GEMM taken as HBM-bound when the layer has few rows per expert."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402
from mixture_experts_sparse_03_b300.inputs import WORKLOADS  # noqa: E402


def test_tensor_bound_headline():
    wl = WORKLOADS["bf16_noisy_e64"]
    kern = {"gate_logits_gemm": 0.05, "gate_topk": 0.03, "gate_rescore": 0.02, "dispatch_rank_scan": 0.02,
            "dispatch_gather": 0.04, "expert_up_gelu": 1.0, "expert_down_combine": 0.9}
    kept, used = 32768, 64
    roof, gemm_flops, gate_flops, wbytes = bench.roofline(wl, kern, list(kern), kept, used)
    assert gemm_flops == 2.0 * kept * wl.d * wl.h
    assert gate_flops == 4.0 * wl.T * wl.d * wl.E  # clean and noise logits
    assert roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s"
    mean_ms = (1.0 + 0.9) / 2
    assert roof["kernel_ms"] == pytest.approx(mean_ms)
    assert roof["achieved"] == pytest.approx(gemm_flops / (mean_ms * 1e-3) / 1e12)
    pk = bench.peaks()
    assert roof["frac"] == pytest.approx(roof["achieved"] / pk["bf16"])
    assert roof["frac_of_sustained"] == pytest.approx(roof["achieved"] / pk["bf16_sustained"])
    assert roof["kernel"].startswith("expert_gemm")


def test_hbm_bound_decode():
    wl = WORKLOADS["bf16_decode_e256"]
    kern = {"gate_logits_gemm": 0.016, "gate_topk": 0.018, "gate_rescore": 0.022, "dispatch_rank_scan": 0.014,
            "dispatch_gather": 0.008, "expert_up_gelu": 1.0, "expert_down": 0.95, "combine_gather": 0.014}
    kept, used = 512, 214
    roof, _, _, wbytes = bench.roofline(wl, kern, list(kern), kept, used)
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s"
    assert wbytes == used * (wl.expert_weight_bytes() // wl.E)
    # one expert GEMM streams one of the two weight matrices of every used expert
    assert roof["algorithmic_per_launch"] == pytest.approx(wbytes / 2)
    assert roof["achieved"] == pytest.approx((wbytes / 2) / (0.975e-3) / 1e9)
    assert roof["frac"] == pytest.approx(roof["achieved"] / bench.peaks()["hbm"])


def test_gate_dominant_reports_no_gemm_fraction():
    wl = WORKLOADS["bf16_recsys_e8"]
    kern = {"gate_logits_gemm": 0.01, "gate_topk": 0.2, "gate_cos_fold": 0.01, "gate_rescore": 0.01,
            "dispatch_rank_scan": 0.01, "dispatch_gather": 0.01, "expert_up_gelu": 0.02,
            "expert_down_combine": 0.015}
    roof, _, _, _ = bench.roofline(wl, kern, list(kern), 16384, 8)
    assert roof["kernel"] == "gate_topk" and roof["achieved"] is None and roof["frac"] is None


def test_job_throughput_counts_every_rank():
    # two replicas, 10 steps of 16384 tokens each in 20 ms (the slowest rank's total)
    assert bench.job_throughput(2, 10, 16384, 20.0) == pytest.approx(2 * 10 * 16384 / 0.02)
