"""GPU parity of the layer's backward (moe_backward) against the fp64 oracle's backward, itself pinned by
central differences of the oracle's forward.  Gradients of sum(dout * out) for x, the gate weights, both
expert weights and both biases; the comparison is normwise per tensor, max |GPU - oracle| / max |oracle|,
because the GPU rounds the intermediate gradients (dY = g dout, dZ, the scores' gradient) to bf16 for its
tensor-core GEMMs."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_sparse_03_b300 import binding as b
from mixture_experts_sparse_03_b300.inputs import make_inputs, small_workload
from tests import parity as P

pytestmark = pytest.mark.gpu

TOL = 2e-2  # normwise, per gradient tensor (bf16 operands and intermediate gradients)

CASES = [
    small_workload(T=300, d=128, h=256, E=6, k=2, capacity_factor=1.0, bias="normal"),
    small_workload(T=257, d=64, h=320, E=3, k=1, norm="all", capacity_factor=1.3, bias="normal"),
    small_workload(T=200, d=192, h=128, E=8, k=2, gate="noisy", capacity_factor=0.7, bias="none"),
    small_workload(T=150, d=128, h=128, E=5, k=3, capacity_factor=0.8, priority="rank", bias="normal"),
    small_workload(T=512, d=256, h=512, E=8, k=2, gate="noisy", capacity_factor=1.2, bias="normal"),
    # several 128-row tiles per expert and several 256-wide column tiles in every GEMM
    small_workload(T=1024, d=256, h=1024, E=4, k=2, capacity_factor=1.1, bias="none"),
]


def _id(wl):
    return "%s_%s_T%d_d%d_h%d_E%d_k%d%s" % (wl.gate, wl.norm, wl.T, wl.d, wl.h, wl.E, wl.k,
                                          "_rank" if wl.priority == "rank" else "")


def run_backward(wl, tg, dout):
    c = b.config(wl)
    n = b.moe_backward_workspace_size(c)
    assert n > 0
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    T, d, h, E = wl.T, wl.d, wl.h, wl.E
    f = lambda *s: torch.full(s, float("nan"), dtype=torch.float32, device="cuda")  # noqa: E731
    g = dict(dx=f(T, d), dw_gate=f(E, d), dw_noise=f(E, d) if wl.gate == "noisy" else None, dw1=f(E, h, d),
             db1=f(E, h), dw2=f(E, d, h), db2=f(E, d))
    b.check(b.moe_backward(c, tg["x"], tg["w_gate"], tg.get("w_noise"), tg.get("eps"), tg["w1"], tg.get("b1"),
                           tg["w2"], tg.get("b2"), dout.cuda(), g["dx"], g["dw_gate"], g["dw_noise"], g["dw1"],
                           g["db1"], g["dw2"], g["db2"], ws, n), "moe_backward")
    st, info = b.moe_device_status(ws, n)
    assert st == 0, (b.STATUS[st], info)
    return {k: (v.cpu().numpy().astype(np.float64) if v is not None else None) for k, v in g.items()}


@pytest.mark.parametrize("wl", CASES, ids=_id)
def test_backward_matches_oracle(wl):
    tc = make_inputs(wl)
    tg = {k: (v.cuda() if v is not None else None) for k, v in tc.items()}
    scores = oracle.gate_scores(wl.gate, tc["x"], tc["w_gate"], tc["w_noise"], tc["eps"], None, None, 1.0)
    assert not P.near_ties(scores, wl.k).any()  # the GPU's exact routing is then the oracle's
    dout = torch.randn(wl.T, wl.d, generator=torch.Generator().manual_seed(wl.seed + 100))
    got = run_backward(wl, tg, dout)
    want = oracle.backward(wl.spec(), tc, dout.double())
    report = {}
    for k, ref in want.items():
        if ref is None:
            continue
        g = got[k]
        assert np.isfinite(g).all(), k
        err = np.abs(g - ref).max() / max(np.abs(ref).max(), 1e-30)
        report[k] = err
    print(" ".join("%s %.2e" % kv for kv in sorted(report.items())))
    for k, err in report.items():
        assert err <= TOL, (k, err, report)


def test_backward_rejects_cosine_and_fp32():
    wl = small_workload(T=16, d=64, h=64, E=4, k=2, gate="cosine", cos_dim=32)
    assert b.moe_backward_workspace_size(b.config(wl)) == 0
    wl32 = small_workload(T=16, d=64, h=64, E=4, k=2, dtype="f32")
    assert b.moe_backward_workspace_size(b.config(wl32)) == 0
    assert b.lib.moe_backward(ctypes.byref(b.config(wl32)), *([None] * 17), 0, None) == 2


def test_backward_full_size_sampled():
    """moe_backward on the E = 64 noisy layer at full size (T = 16384, d = 2048, h = 8192, top-2) against the
    oracle's single-output backward (pinned against its whole backward): the dx rows of 6 tokens, 16 entries
    each of dW1 / db1 and dW2 / db2 in experts with rows, normwise per group as above."""
    from mixture_experts_sparse_03_b300.inputs import WORKLOADS

    wl = WORKLOADS["bf16_noisy_e64"]
    tg = make_inputs(wl, device="cuda", expert_device="cuda")
    tc = {k: (v.cpu() if v is not None else None) for k, v in tg.items()}
    dout = torch.randn(wl.T, wl.d, generator=torch.Generator().manual_seed(wl.seed + 100))
    c = b.config(wl)
    n = b.moe_backward_workspace_size(c)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    T, d, h, E = wl.T, wl.d, wl.h, wl.E
    f = lambda *s: torch.full(s, float("nan"), dtype=torch.float32, device="cuda")  # noqa: E731
    g = dict(dx=f(T, d), dw_gate=f(E, d), dw_noise=f(E, d), dw1=f(E, h, d), db1=f(E, h), dw2=f(E, d, h), db2=f(E, d))
    b.check(b.moe_backward(c, tg["x"], tg["w_gate"], tg["w_noise"], tg["eps"], tg["w1"], tg.get("b1"), tg["w2"],
                           tg.get("b2"), dout.cuda(), g["dx"], g["dw_gate"], g["dw_noise"], g["dw1"], g["db1"],
                           g["dw2"], g["db2"], ws, n), "moe_backward")
    st, info = b.moe_device_status(ws, n)
    assert st == 0, (b.STATUS[st], info)
    rng = np.random.default_rng(17)
    toks = rng.choice(T, size=6, replace=False)
    s1 = [(int(rng.integers(E)), int(rng.integers(h)), int(rng.integers(d))) for _ in range(16)]
    s2 = [(int(rng.integers(E)), int(rng.integers(d)), int(rng.integers(h))) for _ in range(16)]
    want = oracle.backward_sampled(wl.spec(), tc, dout.double(), toks, s1, s2)
    assert (want["slot"] >= 0).sum() > 0
    ix = lambda t, idx: t[tuple(torch.as_tensor(list(a), device="cuda") for a in zip(*idx))].cpu().numpy()  # noqa
    got = dict(dx=g["dx"][torch.as_tensor(toks, device="cuda")].cpu().numpy(),
               dw1=ix(g["dw1"], s1), db1=ix(g["db1"], [(e, n_) for e, n_, _ in s1]),
               dw2=ix(g["dw2"], s2), db2=ix(g["db2"], [(e, m) for e, m, _ in s2]))
    report = {}
    for k, gv in got.items():
        ref = want[k]
        assert np.isfinite(gv).all(), k
        report[k] = np.abs(gv.astype(np.float64) - ref).max() / max(np.abs(ref).max(), 1e-30)
    print(" ".join("%s %.2e" % kv for kv in sorted(report.items())))
    for k, err in report.items():
        assert err <= TOL, (k, err, report)
