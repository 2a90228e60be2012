"""moe_router_stats on the GPU against the oracle's router statistics, on the GPU's own routing and
dispatch (the statistics are a function of those; their parity is tested elsewhere).  Importance may
differ from the oracle's fp64 sums only by the documented fixed-point rounding (each gate to a multiple
of 2^-32, at most 2^-33 per pair) plus the final rounding to fp32; the losses are computed in fp64 from
the same sums and rounded to fp32; the drop count is exact.  The result is identical on every run."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_sparse_03_b300 import binding as b
from mixture_experts_sparse_03_b300.inputs import WORKLOADS, small_workload
from tests import parity as P

pytestmark = pytest.mark.gpu

CASES = [
    small_workload(T=300, d=128, h=256, E=8, k=2, capacity_factor=0.7),                 # drops
    small_workload(T=129, d=128, h=128, E=12, k=2, gate="noisy", capacity_factor=1.1),
    small_workload(T=180, d=128, h=256, E=10, k=2, gate="cosine", cos_dim=64, capacity_factor=1.0),
    small_workload(T=257, d=64, h=320, E=3, k=1, norm="all", capacity_factor=1.3),      # full-softmax gates
    small_workload(T=211, d=128, h=128, E=7, k=2, dtype="f32", capacity_factor=0.9),
    small_workload(T=33, d=64, h=64, E=1, k=1, norm="all", capacity_factor=1.0),        # one expert: NaN loss
    WORKLOADS["bf16_e8_k2"],
]


def _stats(wl, g, use_slot=True):
    c = b.config(wl)
    dev = torch.device("cuda", 0)
    ws = b.workspace(c, dev)
    idx = torch.from_numpy(g["idx"]).to(dev)
    gate = torch.from_numpy(g["gate"]).to(dev)
    slot = torch.from_numpy(g["slot"]).to(dev) if use_slot else None
    imp = torch.full((wl.E,), float("nan"), dtype=torch.float32, device=dev)
    losses = torch.full((2,), -1.0, dtype=torch.float32, device=dev)
    dropped = torch.full((1,), -7, dtype=torch.int64, device=dev)
    b.check(b.moe_router_stats(c, idx, gate, slot, imp, losses, dropped, ws, ws.numel()), "moe_router_stats")
    st, info = b.moe_device_status(ws, ws.numel())
    assert st == 0, (b.STATUS[st], info)
    return imp.cpu().numpy(), losses.cpu().numpy(), int(dropped.cpu()[0])


@pytest.mark.parametrize("wl", CASES, ids=lambda w: "%s_%s_T%d_E%d_k%d" % (w.gate, w.dtype, w.T, w.E, w.k))
def test_router_stats_match_oracle(wl):
    _, tg = P.inputs(wl)
    g = P.run_steps(wl, tg)
    imp, losses, dropped = _stats(wl, g)
    oimp, oil, olb, odrop = oracle.router_stats(g["idx"], g["gate"].astype(np.float64), wl.E, g["slot"])
    n_e = np.bincount(g["idx"].ravel(), minlength=wl.E)
    tol = n_e * 2.0 ** -33 + np.abs(oimp) * 2.0 ** -24 + 1e-30
    assert np.all(np.abs(imp.astype(np.float64) - oimp) <= tol), np.abs(imp - oimp).max()
    if wl.E > 1:
        assert abs(losses[0] - oil) <= 1e-5 * abs(oil) + 1e-7
    else:
        assert np.isnan(losses[0])
    assert abs(losses[1] - olb) <= 1e-5 * abs(olb) + 1e-7
    assert dropped == odrop == int((g["slot"] < 0).sum())
    # deterministic: a second call gives the same bits; without slot the drop count reads 0
    imp2, losses2, _ = _stats(wl, g)
    assert np.array_equal(imp.view(np.int32), imp2.view(np.int32))
    assert np.array_equal(losses.view(np.int32), losses2.view(np.int32))
    _, _, d0 = _stats(wl, g, use_slot=False)
    assert d0 == 0


def test_router_stats_flags_bad_gates():
    """A gate outside [0, 1] and an expert id outside [0, E) are skipped and recorded (no fault)."""
    wl = small_workload(T=64, d=64, h=64, E=4, k=2)
    c = b.config(wl)
    dev = torch.device("cuda", 0)
    ws = b.workspace(c, dev)
    idx = torch.zeros((64, 2), dtype=torch.int32, device=dev)
    idx[:, 1] = 1
    gate = torch.full((64, 2), 0.5, dtype=torch.float32, device=dev)
    gate[3, 0] = 1.5
    idx[5, 1] = 9
    imp = torch.empty((4,), dtype=torch.float32, device=dev)
    losses = torch.empty((2,), dtype=torch.float32, device=dev)
    b.check(b.moe_router_stats(c, idx, gate, None, imp, losses, None, ws, ws.numel()), "moe_router_stats")
    st, _ = b.moe_device_status(ws, ws.numel())
    assert b.STATUS[st] == "MOE_ERR_DEVICE_CHECK"
    assert np.allclose(imp.cpu().numpy(), [63 * 0.5, 63 * 0.5, 0.0, 0.0])


FUSED_CASES = CASES[:5] + [small_workload(T=300, d=128, h=256, E=8, k=2, capacity_factor=0.7, priority="rank"),
                           WORKLOADS["bf16_e8_k2"], WORKLOADS["bf16_noisy_e64"]]


@pytest.mark.parametrize("wl", FUSED_CASES, ids=lambda w: "%s_%s_T%d_E%d_k%d_%s" % (w.gate, w.dtype, w.T, w.E, w.k,
                                                                                    w.priority))
def test_router_stats_fused_into_forward(wl):
    """moe_forward with MOE_FLAG_ROUTER_STATS: the statistics come out of the forward's own dispatch kernel
    (the launch count does not change), equal bit for bit to the standalone moe_router_stats on the same
    routing (both sum the gates exactly in fixed point), on two calls in a row (the last CTA resets the
    accumulators); the layer output is the same bits as without the flag."""
    _, tg = P.inputs(wl)
    c0 = b.config(wl)
    c = b.config(wl, flags=b.FLAG_ROUTER_STATS)
    assert b.moe_forward_launches(c) == b.moe_forward_launches(c0)
    dev = torch.device("cuda", 0)
    ws = b.workspace(c, dev)
    plain, _ = P.run_forward(wl, tg)
    for call in range(2):
        out = torch.full((wl.T, wl.d), float("nan"), dtype=torch.float32, device=dev)
        b.forward(c, tg, out=out, ws=ws)
        imp = torch.full((wl.E,), float("nan"), dtype=torch.float32, device=dev)
        losses = torch.full((2,), -1.0, dtype=torch.float32, device=dev)
        dropped = torch.full((1,), -7, dtype=torch.int64, device=dev)
        b.check(b.moe_router_stats_result(c, ws, ws.numel(), imp, losses, dropped), "moe_router_stats_result")
        st, info = b.moe_device_status(ws, ws.numel())
        assert st == 0, (b.STATUS[st], info)
        assert np.array_equal(out.cpu().numpy().view(np.int32), plain.view(np.int32))
        if call == 0:
            g = P.run_steps(wl, tg)
            simp, slosses, sdrop = _stats(wl, g)
        assert np.array_equal(imp.cpu().numpy().view(np.int32), simp.view(np.int32)), call
        assert np.array_equal(losses.cpu().numpy().view(np.int32), slosses.view(np.int32)), call
        assert int(dropped.cpu()[0]) == sdrop
    # a config without the flag has nothing to read
    assert b.moe_router_stats_result(c0, ws, ws.numel(), imp, losses, dropped) == 1
