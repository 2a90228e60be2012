"""GPU parity of the layer with block-FP8 expert weights (moe_forward_fp8, moe_expert_ffn_fp8) against the
fp64 oracle on the dequantised weights: E4M3 codes times a fp32 scale per 128 x 128 block, the reading of
"Block FP8" the library documents.  Routing and dispatch are those of the bf16 layer (the gate is not
quantised); outputs are compared per token at the bf16 tolerance."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_sparse_03_b300 import binding as b
from mixture_experts_sparse_03_b300.inputs import WORKLOADS, make_inputs, small_workload
from tests import parity as P

pytestmark = pytest.mark.gpu

SMALL = [
    small_workload(T=200, d=256, h=384, E=6, k=2, capacity_factor=1.0, weights="fp8_block"),           # fused combine
    small_workload(T=150, d=128, h=256, E=5, k=3, capacity_factor=0.8, weights="fp8_block"),           # gather combine
    small_workload(T=97, d=384, h=128, E=4, k=1, norm="all", capacity_factor=1.2, bias="none", weights="fp8_block"),
    small_workload(T=300, d=256, h=256, E=8, k=2, gate="noisy", capacity_factor=0.7, weights="fp8_block"),
]


def _id(wl):
    return "%s_T%d_d%d_h%d_E%d_k%d" % (wl.gate, wl.T, wl.d, wl.h, wl.E, wl.k)


def oracle_out_fp8(wl, tc, tg, scores, idx, slot, tokens, chunk=4):
    """Oracle output for `tokens` with dequantised FP8 weights, a few experts at a time (their fp64 copies
    of big layers would not fit at once): each chunk's pairs through the oracle's combine, summed."""
    gate = P.gates_for(scores, idx, wl.norm)
    used = sorted({int(e) for t in tokens for e, s in zip(idx[t], slot[t]) if s >= 0})
    out = np.zeros((len(tokens), wl.d))
    src = tg if tc.get("w1") is None else tc
    for c0 in range(0, len(used), chunk):
        ids = used[c0:c0 + chunk]
        remap = {e: i for i, e in enumerate(ids)}
        sel = torch.as_tensor(ids, dtype=torch.long, device=src["w1"].device)
        w1 = oracle.dequant_block_fp8(src["w1"].index_select(0, sel).cpu(), src["w1_scale"].index_select(0, sel).cpu())
        w2 = oracle.dequant_block_fp8(src["w2"].index_select(0, sel).cpu(), src["w2_scale"].index_select(0, sel).cpu())
        b1 = None if src.get("b1") is None else src["b1"].index_select(0, sel).cpu()
        b2 = None if src.get("b2") is None else src["b2"].index_select(0, sel).cpu()
        idx2 = np.array([[remap.get(int(e), 0) for e in row] for row in idx], dtype=np.int32)
        slot2 = np.where(np.isin(idx, ids), slot, -1).astype(np.int32)
        out += oracle.combine_tokens(tokens, tc["x"], idx2, gate, slot2, w1, b1, w2, b2)
    return out


def _forward_fp8(wl, tg):
    c = b.config(wl)
    ws = b.workspace(c, "cuda")
    count = torch.full((wl.E,), -7, dtype=torch.int32, device="cuda")
    out = torch.full((wl.T, wl.d), float("nan"), dtype=torch.float32, device="cuda")
    b.forward(c, tg, out=out, expert_count=count, ws=ws)
    st, info = b.moe_device_status(ws, ws.numel())
    assert st == 0, (b.STATUS[st], info)
    return out.cpu().numpy(), count.cpu().numpy()


@pytest.mark.parametrize("wl", SMALL, ids=_id)
def test_small_fp8_layer(wl):
    tc = make_inputs(wl)
    tg = {k: (v.cuda() if v is not None else None) for k, v in tc.items()}
    scores = oracle.gate_scores(wl.gate, tc["x"], tc["w_gate"], tc["w_noise"], tc["eps"], tc["proj"], tc["emb"],
                                wl.temperature)
    assert not P.near_ties(scores, wl.k).any()  # so the GPU's exact routing is the oracle's
    out, count = _forward_fp8(wl, tg)
    idx, _ = oracle.topk(scores, wl.k, wl.norm)
    C = oracle.capacity(wl.T, wl.E, wl.k, wl.capacity_factor, wl.capacity)
    slot, ocount = oracle.dispatch(idx, wl.E, C, wl.priority)
    assert np.array_equal(count, ocount)
    toks = np.arange(wl.T, dtype=np.int32)
    ref = oracle_out_fp8(wl, tc, tg, scores, idx, slot, toks)
    P.check_output(wl, out, ref, toks)


def test_fp8_ffn_step_matches_forward():
    """moe_expert_ffn_fp8 on moe_dispatch's rows, with per-row outputs and the gather combine, equals the
    whole-layer call (fused combine, k = 2) within fp32 rounding of the additions."""
    wl = SMALL[0]
    tc = make_inputs(wl)
    tg = {k: (v.cuda() if v is not None else None) for k, v in tc.items()}
    c = b.config(wl)
    ws = b.workspace(c, "cuda")
    T, k, E, d = wl.T, wl.k, wl.E, wl.d
    rows = b.moe_dispatch_rows(c)
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gate = torch.empty((T, k), dtype=torch.float32, device="cuda")
    b.check(b.moe_route(c, tg["x"], tg["w_gate"], None, None, None, None, idx, gate, ws, ws.numel()), "moe_route")
    slot = torch.empty((T, k), dtype=torch.int32, device="cuda")
    cnt = torch.empty((E,), dtype=torch.int32, device="cuda")
    off = torch.empty((E + 1,), dtype=torch.int32, device="cuda")
    rtok = torch.empty((rows,), dtype=torch.int32, device="cuda")
    rgate = torch.empty((rows,), dtype=torch.float32, device="cuda")
    xd = torch.zeros((rows, d), dtype=torch.bfloat16, device="cuda")
    b.check(b.moe_dispatch(c, tg["x"], idx, gate, slot, cnt, off, rtok, rgate, xd, ws, ws.numel()), "moe_dispatch")
    y = torch.full((rows, d), float("nan"), dtype=torch.float32, device="cuda")
    b.check(b.moe_expert_ffn_fp8(c, xd, off, rtok, rgate, tg["w1"], tg["w1_scale"], tg["b1"], tg["w2"],
                                 tg["w2_scale"], tg["b2"], y, None, ws, ws.numel()), "moe_expert_ffn_fp8")
    out = torch.full((T, d), float("nan"), dtype=torch.float32, device="cuda")
    b.check(b.moe_combine(c, y, slot, off, idx, gate, out), "moe_combine")
    st, info = b.moe_device_status(ws, ws.numel())
    assert st == 0, (b.STATUS[st], info)
    whole, _ = _forward_fp8(wl, tg)
    assert np.allclose(out.cpu().numpy(), whole, rtol=1e-5, atol=1e-6)


def test_fp8_rejects_unsupported_configs():
    """Host-side checks: an fp32 layer, d not a multiple of 128, or missing scales launch nothing."""
    wl = small_workload(T=8, d=192, h=256, E=2, k=1, weights="fp8_block")
    c = b.config(wl)
    ws = b.workspace(c, "cuda")
    dummy = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    st = b.moe_forward_fp8(c, dummy, dummy, None, None, None, None, dummy, dummy, None, dummy, dummy, None,
                           dummy, None, ws, ws.numel())
    assert st == 2  # d = 192 is not a multiple of the 128-wide scale blocks
    wl32 = small_workload(T=8, d=128, h=256, E=2, k=1, dtype="f32", weights="fp8_block")
    c32 = b.config(wl32)
    ws32 = b.workspace(c32, "cuda")
    assert b.moe_forward_fp8(c32, dummy, dummy, None, None, None, None, dummy, dummy, None, dummy, dummy, None,
                             dummy, None, ws32, ws32.numel()) == 2
    assert b.moe_forward_fp8(b.config(small_workload(T=8, d=128, h=256, E=2, k=1)), dummy, dummy, None, None, None,
                             None, dummy, None, None, dummy, dummy, None, dummy, None, ws, ws.numel()) == 1


def test_full_size_decode_fp8():
    """The decode-shaped layer (T = 64, d = 7168, E = 256, k = 8, dropless) with block-FP8 weights: the
    routing equals the bf16 layer's oracle routing, and every token's output matches the oracle on the
    dequantised weights."""
    wl = WORKLOADS["bf16_decode_e256_fp8"]
    tg = make_inputs(wl, device="cuda", expert_device="cuda")
    tc = {k: (None if k in ("w1", "w2", "w1_scale", "w2_scale") else (v.cpu() if v is not None else None))
          for k, v in tg.items()}
    out, count = _forward_fp8(wl, tg)
    scores = oracle.gate_scores(wl.gate, tc["x"], tc["w_gate"], None, None, None, None, 1.0)
    assert not P.near_ties(scores, wl.k).any()
    idx, _ = oracle.topk(scores, wl.k, wl.norm)
    slot, ocount = oracle.dispatch(idx, wl.E, wl.capacity)
    assert np.array_equal(count, ocount)
    toks = np.arange(wl.T, dtype=np.int32)
    ref = oracle_out_fp8(wl, tc, tg, scores, idx, slot, toks)
    err = P.check_output(wl, out, ref, toks)
    print("decode fp8: max per-token relative error %.3e over %d tokens" % (err, wl.T))


def _one_hot_fp8_layer(T, cap, rows_per_expert, seed):
    """An FFN step whose every output is one dequantised W2 code times 8, so that the widening of the
    codes is checked bit for bit.  Row r of expert e (local index i) holds the unit vector x = e_i; W1[e]
    has the code of 8.0 (0x50, scale 1) at (j_i, i) and zeros elsewhere, so W1 x = 8 e_j and GELU(8)
    rounds to 8 in bf16; then y = 8 * W2[e][:, j] exactly (one product per output, no bias).  W2's
    columns cycle through all 254 non-NaN E4M3 codes (zeros, subnormals, both signs) and its 128 x 128
    blocks carry different power-of-two scales."""
    d, h, E = 128, 256, len(rows_per_expert)
    wl = small_workload(T=T, d=d, h=h, E=E, k=1, capacity=cap, bias="none", weights="fp8_block")
    c = b.config(wl)
    rows = b.moe_dispatch_rows(c)
    rng = np.random.default_rng(seed)
    valid = np.array([v for v in range(256) if v not in (0x7F, 0xFF)], dtype=np.uint8)
    off = np.zeros(E + 1, dtype=np.int32)
    for e, n in enumerate(rows_per_expert):
        off[e + 1] = off[e] + -(-n // 128) * 128
    assert off[E] <= rows
    xd = np.zeros((rows, d), dtype=np.float32)
    rtok = np.full(rows, -1, dtype=np.int32)
    w1 = np.zeros((E, h, d), dtype=np.uint8)
    w2 = np.zeros((E, d, h), dtype=np.uint8)
    jsel = {}
    for e, n in enumerate(rows_per_expert):
        js = rng.permutation(h)[:n]
        for i in range(n):
            r = off[e] + i
            xd[r, i] = 1.0
            rtok[r] = (e * 131 + i) % T
            w1[e, js[i], i] = 0x50  # 8.0
            jsel[r] = (e, js[i])
        w2[e] = valid[(np.arange(d)[:, None] * 7 + np.arange(h)[None, :] * 3 + 17 * e) % len(valid)]
    s1 = np.ones((E, h // 128, d // 128), dtype=np.float32)
    s2 = np.ldexp(1.0, rng.integers(-12, 4, size=(E, d // 128, h // 128))).astype(np.float32)
    w2dq = oracle.dequant_block_fp8(w2, s2)
    expect = {r: 8.0 * w2dq[e, :, j] for r, (e, j) in jsel.items()}
    ws = b.workspace(c, "cuda")
    t = lambda a, dt=None: torch.as_tensor(a).to("cuda") if dt is None else torch.as_tensor(a).to("cuda", dt)  # noqa
    y = torch.full((rows, d), float("nan"), dtype=torch.float32, device="cuda")
    b.check(b.moe_expert_ffn_fp8(c, t(xd, torch.bfloat16), t(off), t(rtok), t(np.ones(rows, np.float32)), t(w1),
                                 t(s1), None, t(w2), t(s2), None, y, None, ws, ws.numel()), "moe_expert_ffn_fp8")
    st, info = b.moe_device_status(ws, ws.numel())
    assert st == 0, (b.STATUS[st], info)
    yh = y.cpu().numpy()
    for r, ref in expect.items():
        assert np.array_equal(yh[r], ref.astype(np.float32)), (r, np.flatnonzero(yh[r] != ref.astype(np.float32))[:8])


@pytest.mark.parametrize("case", [
    (64, 64, [64, 37, 1]),     # at most 64 rows per expert: the swapped kernel (64-row chunks)
    (256, 128, [128, 100]),    # 128-row tiles
    (256, 128, [65, 3, 128]),  # 128-row tiles, ragged
], ids=["swapped", "tiles", "ragged"])
def test_fp8_every_code_exact(case):
    T, cap, rows_per_expert = case
    _one_hot_fp8_layer(T, cap, rows_per_expert, seed=len(rows_per_expert))
