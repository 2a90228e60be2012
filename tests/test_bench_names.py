"""bench.py's per-kernel names must match the launches moe_forward makes for every workload (host-only:
moe_forward_launches plans the call without touching a GPU)."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402
from mixture_experts_sparse_03_b300 import binding as b  # noqa: E402
from mixture_experts_sparse_03_b300.inputs import WORKLOADS, small_workload  # noqa: E402


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_kernel_names_match_launch_count(name):
    wl = WORKLOADS[name]
    names = bench.kernel_names(wl, b.moe_forward_launches(b.config(wl)))
    assert len(set(names)) == len(names)
    assert names[-1] in ("expert_down_combine", "combine_gather")


def test_scan_in_gather_naming_follows_the_histogram_size():
    """The fused softmax gate leaves the dispatch scan to the gather while ceil(T/32)*E <= 2048 ints."""
    small = small_workload(T=4096, d=1024, h=64, E=8, k=2)     # 128 blocks x 8 experts
    large = small_workload(T=16384, d=1024, h=64, E=8, k=2)    # 512 blocks x 8 experts
    assert bench.kernel_names(small, 4)[:2] == ["gate_fused_gemm_topk", "dispatch_scan_gather"]
    assert bench.kernel_names(large, 4)[:2] == ["gate_fused_gemm_topk_scan", "dispatch_gather"]
    with pytest.raises(RuntimeError):
        bench.kernel_names(small, 5)
