"""The C ABI without a GPU: the library loads, exports every function include/moe_b300.h declares,
its struct layout matches the C compiler's, and host-side validation and sizing behave as documented
(no call here launches a kernel)."""
import ctypes
import math
import os
import subprocess

import pytest

import oracle
from mixture_experts_sparse_03_b300 import binding as b
from mixture_experts_sparse_03_b300.inputs import WORKLOADS, small_workload

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_exports_every_declared_function():
    names = b.declared_functions()
    assert len(names) >= 13
    lib = ctypes.CDLL(b.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    for n in ("moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine", "moe_forward"):
        assert n in names


def test_config_layout_matches_c(tmp_path):
    src = os.path.join(tmp_path, "layout.c")
    open(src, "w").write(
        '#include <stdio.h>\n#include <stddef.h>\n#include "moe_b300.h"\n'
        'int main(void){printf("%zu %zu %zu %zu %zu %zu\\n", sizeof(moe_config), offsetof(moe_config, capacity),'
        ' offsetof(moe_config, capacity_factor), offsetof(moe_config, cos_dim), offsetof(moe_config, cos_temperature),'
        ' offsetof(moe_config, reserved)); return 0;}\n')
    exe = os.path.join(tmp_path, "layout")
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-o", exe, src], check=True)
    got = [int(v) for v in subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split()]
    C = b.MoEConfig
    assert got == [ctypes.sizeof(C), C.capacity.offset, C.capacity_factor.offset, C.cos_dim.offset,
                   C.cos_temperature.offset, C.reserved.offset]


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_capacity_matches_oracle(name):
    wl = WORKLOADS[name]
    c = b.config(wl)
    assert b.moe_capacity(c) == oracle.capacity(wl.T, wl.E, wl.k, wl.capacity_factor, wl.capacity)


def test_capacity_values_and_rows_bound():
    want = {"tiny_fp32": 77, "bf16_e8_k2": 1229, "bf16_noisy_e64": 768, "bf16_cosine_skew": 615, "bf16_decode_e256": 64}
    for name, C in want.items():
        wl = WORKLOADS[name]
        c = b.config(wl)
        assert b.moe_capacity(c) == C
        Ceff = min(C, wl.T)
        rows = min(wl.T * wl.k + 127 * wl.E, wl.E * math.ceil(Ceff / 128) * 128)
        assert b.moe_dispatch_rows(c) == rows
        assert b.moe_workspace_size(c) > rows * wl.d * (2 if wl.dtype == "bf16" else 4)


def _bad(**kw):
    c = b.config(small_workload())
    for k_, v in kw.items():
        setattr(c, k_, v)
    return c


@pytest.mark.parametrize("field,value,status", [
    ("model_dim", 96, 1), ("model_dim", 0, 1), ("hidden_size_per_expert", 100, 1), ("num_experts", 0, 1),
    ("num_experts", 2000, 1), ("top_k", 0, 1), ("top_k", 6, 1), ("top_k", 17, 1), ("tokens", -1, 1),
    ("gate_type", 3, 1), ("gate_norm", 2, 1), ("dtype", 2, 1), ("flags", 64, 1), ("reserved", 1, 1),
    ("capacity_factor", 0.0, 1), ("capacity_factor", float("nan"), 1), ("capacity_factor", float("inf"), 1),
])
def test_invalid_config_rejected(field, value, status):
    c = _bad(**{field: value})
    assert b.moe_workspace_size(c) == 0
    assert b.moe_capacity(c) == -1
    assert b.lib.moe_route(ctypes.byref(c), None, None, None, None, None, None, None, None, None, 0, None) == status


def test_cosine_and_noisy_limits():
    wl = small_workload(gate="cosine", cos_dim=12)
    assert b.moe_workspace_size(b.config(wl)) == 0  # cos_dim must be a multiple of 8
    c = b.config(small_workload(gate="cosine", cos_dim=16))
    c.cos_temperature = 0.0
    assert b.moe_workspace_size(c) == 0
    c = b.config(small_workload(gate="noisy", E=600, k=2))
    assert b.lib.moe_route(ctypes.byref(c), None, None, None, None, None, None, None, None, None, 0, None) == 2


def test_null_and_misaligned_pointers_rejected_before_launch():
    c = b.config(small_workload())
    lib = b.lib
    P = 0x10000
    W = 0x100000
    n = b.moe_workspace_size(c)
    # missing x / outputs
    assert lib.moe_route(ctypes.byref(c), None, P, None, None, None, None, P, P, W, n, None) == 1
    assert lib.moe_route(ctypes.byref(c), P, P, None, None, None, None, None, P, W, n, None) == 1
    # misaligned
    assert lib.moe_route(ctypes.byref(c), P + 2, P, None, None, None, None, P, P, W, n, None) == 1
    # noisy needs w_noise and eps
    cn = b.config(small_workload(gate="noisy"))
    nn = b.moe_workspace_size(cn)
    assert lib.moe_route(ctypes.byref(cn), P, P, None, None, None, None, P, P, W, nn, None) == 1
    # cosine needs proj and emb
    cc = b.config(small_workload(gate="cosine", cos_dim=16))
    nc = b.moe_workspace_size(cc)
    assert lib.moe_route(ctypes.byref(cc), P, P, None, None, None, None, P, P, W, nc, None) == 1
    # the gate's partial logits live in the workspace
    assert lib.moe_route(ctypes.byref(c), P, P, None, None, None, None, P, P, None, n, None) == 3
    assert lib.moe_route(ctypes.byref(c), P, P, None, None, None, None, P, P, W, n - 1, None) == 3
    # the logits GEMM alone: bf16 only, needs its weights
    L = 0x20000
    assert lib.moe_gate_logits(ctypes.byref(c), P, None, None, None, L, W, n, None) == 1
    assert lib.moe_gate_logits(ctypes.byref(cn), P, P, None, None, L, W, nn, None) == 1
    assert lib.moe_gate_logits(ctypes.byref(cc), P, P, None, None, L, W, nc, None) == 1
    cf = b.config(small_workload(dtype="f32"))
    assert lib.moe_gate_logits(ctypes.byref(cf), P, P, None, None, L, W, b.moe_workspace_size(cf), None) == 2
    # workspace missing / too small / misaligned
    args = [P] * 9
    assert lib.moe_dispatch(ctypes.byref(c), *args, None, n, None) == 3
    assert lib.moe_dispatch(ctypes.byref(c), *args, 0x100000, n - 1, None) == 3
    assert lib.moe_dispatch(ctypes.byref(c), *args, 0x100010, n, None) == 3
    assert lib.moe_forward(ctypes.byref(c), P, P, None, None, None, None, P, None, P, None, P, None, None, n, None) == 3
    assert lib.moe_forward(ctypes.byref(c), P, P, None, None, None, None, None, None, P, None, P, None, 0x100000, n,
                           None) == 1


def test_empty_input_is_a_no_op():
    c = b.config(small_workload(), tokens=0)
    assert b.moe_capacity(c) == 0
    assert b.moe_dispatch_rows(c) == 0
    assert b.moe_forward_launches(c) == 0
    lib = b.lib
    assert lib.moe_route(ctypes.byref(c), None, None, None, None, None, None, None, None, None, 0, None) == 0
    assert lib.moe_gate_logits(ctypes.byref(c), *([None] * 6), 0, None) == 0
    assert lib.moe_dispatch(ctypes.byref(c), *([None] * 10), 0, None) == 0
    assert lib.moe_expert_ffn(ctypes.byref(c), *([None] * 11), 0, None) == 0
    assert lib.moe_combine(ctypes.byref(c), *([None] * 7)) == 0
    assert lib.moe_forward(ctypes.byref(c), *([None] * 13), 0, None) == 0


def test_launch_counts():
    # bf16 softmax gate with E <= 64: one fused gate launch (logits, top-k, dispatch ranks and scan),
    # dispatch gather, up, down (+ combine when k > 2 or unfused)
    assert b.moe_forward_launches(b.config(small_workload(k=2))) == 4
    assert b.moe_forward_launches(b.config(small_workload(k=3))) == 5
    assert b.moe_forward_launches(b.config(small_workload(k=2), flags=b.FLAG_UNFUSED_COMBINE)) == 5
    # other bf16 gates: logits GEMM, selection, grid-wide re-scoring, rank step with the scan
    assert b.moe_forward_launches(b.config(small_workload(k=2, gate="noisy"))) == 7
    assert b.moe_forward_launches(b.config(small_workload(k=2, E=65))) == 7
    # the cosine gate adds the fold of the projection into the expert embeddings
    assert b.moe_forward_launches(b.config(small_workload(k=2, gate="cosine"))) == 8
    # fp32: the gate computes its logits itself
    assert b.moe_forward_launches(b.config(small_workload(k=2, dtype="f32"))) == 4
    assert b.moe_forward_launches(b.config(small_workload(k=3, dtype="f32"))) == 5


def test_status_strings():
    for s in range(7):
        assert b.moe_status_string(s) != "unknown status"
    assert b.moe_status_string(99) == "unknown status"


def test_router_stats_host_validation():
    """moe_router_stats refuses a short workspace, missing outputs and a misaligned drop counter on the
    host, before any CUDA call (the pointers below are never dereferenced)."""
    c = b.config(small_workload(k=2))
    nbytes = b.lib.moe_workspace_size(ctypes.byref(c))
    fake = ctypes.c_void_p(1 << 20)
    st = b.lib.moe_router_stats(ctypes.byref(c), fake, fake, None, fake, fake, None, fake, 0, None)
    assert st == 3  # MOE_ERR_WORKSPACE
    st = b.lib.moe_router_stats(ctypes.byref(c), fake, fake, None, None, fake, None, fake, nbytes, None)
    assert st == 1  # importance missing
    st = b.lib.moe_router_stats(ctypes.byref(c), fake, fake, None, fake, fake, ctypes.c_void_p((1 << 20) + 4), fake,
                                nbytes, None)
    assert st == 1  # dropped not 8-byte aligned



@pytest.mark.parametrize("field,value,status", [("model_dim", 1 << 17, 2), ("hidden_size_per_expert", 1 << 17, 2),
                                                ("model_dim", 96, 1), ("top_k", 0, 1)])
def test_static_scratch_dispatch_rejects_configs_like_moe_dispatch(field, value, status):
    """The dispatch without a caller workspace validates the config with the same planner as
    moe_dispatch and returns the same status (unsupported sizes included), before any CUDA call."""
    c = _bad(**{field: value})
    nulls = [None] * 9
    assert b.lib.moe_dispatch(ctypes.byref(c), *nulls, None, 0, None) == status
    assert b.lib.moe_dispatch_static_scratch(ctypes.byref(c), *nulls, None) == status
