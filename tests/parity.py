"""Shared helpers of the GPU parity tests: run the library's steps on a workload, run the oracle, and
compare (routing bit-exact outside near ties, dispatch bit-exact, outputs within tolerance)."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from mixture_experts_sparse_03_b300 import binding as b
from mixture_experts_sparse_03_b300.inputs import Workload, make_inputs

# output tolerance: max over tokens of |out_t - ref_t|_inf / |ref_t|_inf
TOL = {"bf16": 2e-2, "f32": 1e-4}
NEAR_TIE = 1e-6  # selection-score margin below which a token's routing may legitimately differ


def inputs(wl: Workload):
    """(cpu tensors for the oracle, cuda tensors for the library) of a workload.  Expert weights of big
    workloads are drawn on the GPU; the CPU dict then holds None for w1/w2 and the oracle reads only
    the experts it needs (see expert_subset)."""
    big = wl.expert_weight_bytes() > (1 << 30)
    if big:
        tg = make_inputs(wl, device="cuda", expert_device="cuda")
        tc = {k: (None if k in ("w1", "w2") else (v.cpu() if v is not None else None)) for k, v in tg.items()}
    else:
        tc = make_inputs(wl, device="cpu")
        tg = {k: (v.cuda() if v is not None else None) for k, v in tc.items()}
    return tc, tg


def expert_subset(tg, tc, experts):
    """Host copies of the listed experts' weights (stacked in that order)."""
    sel = torch.as_tensor(experts, dtype=torch.long, device="cuda")
    out = {}
    for n in ("w1", "w2", "b1", "b2"):
        src = tg[n]
        out[n] = None if src is None else src.index_select(0, sel).cpu()
    return out


def near_ties(scores: np.ndarray, k: int) -> np.ndarray:
    """Tokens whose top-(k+1) scores have an adjacent gap below NEAR_TIE."""
    s = -np.sort(-scores, axis=1)
    m = min(k + 1, scores.shape[1])
    gaps = s[:, : m - 1] - s[:, 1:m]
    return (gaps < NEAR_TIE).any(axis=1) if m > 1 else np.zeros(len(scores), bool)


def gates_for(scores: np.ndarray, idx: np.ndarray, norm: str) -> np.ndarray:
    """Gate weights of a given choice of experts, from fp64 scores (for re-running the oracle's later
    steps on the GPU's routing)."""
    chosen = np.take_along_axis(scores, idx.astype(np.int64), axis=1)
    if norm == "all":
        return np.take_along_axis(torch.softmax(torch.from_numpy(scores), 1).numpy(), idx.astype(np.int64), 1)
    return torch.softmax(torch.from_numpy(chosen), 1).numpy()


def run_steps(wl: Workload, tg: dict, flags: int = 0):
    """route -> dispatch -> expert_ffn (y) -> combine through the step entry points; CPU copies."""
    c = b.config(wl, flags=flags)
    T, k, E, d = wl.T, wl.k, wl.E, wl.d
    dev = tg["x"].device
    rows = b.moe_dispatch_rows(c)
    ws = b.workspace(c, dev)
    idx = torch.full((T, k), -7, dtype=torch.int32, device=dev)
    gate = torch.full((T, k), float("nan"), dtype=torch.float32, device=dev)
    b.check(b.moe_route(c, tg["x"], tg["w_gate"], tg["w_noise"], tg["eps"], tg["proj"], tg["emb"], idx, gate, ws,
                        ws.numel()), "moe_route")
    slot = torch.full((T, k), -7, dtype=torch.int32, device=dev)
    count = torch.full((E,), -7, dtype=torch.int32, device=dev)
    off = torch.full((E + 1,), -7, dtype=torch.int32, device=dev)
    rtok = torch.full((max(rows, 1),), -7, dtype=torch.int32, device=dev)
    rgate = torch.full((max(rows, 1),), float("nan"), dtype=torch.float32, device=dev)
    xd = torch.zeros((max(rows, 1), d), dtype=tg["x"].dtype, device=dev)
    b.check(b.moe_dispatch(c, tg["x"], idx, gate, slot, count, off, rtok, rgate, xd, ws, ws.numel()), "moe_dispatch")
    y = torch.full((max(rows, 1), d), float("nan"), dtype=torch.float32, device=dev)
    b.check(b.moe_expert_ffn(c, xd, off, rtok, rgate, tg["w1"], tg["b1"], tg["w2"], tg["b2"], y, None, ws,
                             ws.numel()), "moe_expert_ffn")
    out = torch.full((T, d), float("nan"), dtype=torch.float32, device=dev)
    b.check(b.moe_combine(c, y, slot, off, idx, gate, out), "moe_combine")
    st, info = b.moe_device_status(ws, ws.numel())
    assert st == 0, (b.STATUS[st], info)
    return dict(idx=idx.cpu().numpy(), gate=gate.cpu().numpy(), slot=slot.cpu().numpy(), count=count.cpu().numpy(),
                off=off.cpu().numpy(), rtok=rtok.cpu().numpy()[:rows], rgate=rgate.cpu().numpy()[:rows],
                xd=xd[:rows].cpu(), out=out.cpu().numpy(), rows=rows)


def run_forward(wl: Workload, tg: dict, flags: int = 0):
    c = b.config(wl, flags=flags)
    dev = tg["x"].device
    ws = b.workspace(c, dev)
    count = torch.full((wl.E,), -7, dtype=torch.int32, device=dev)
    out = torch.full((wl.T, wl.d), float("nan"), dtype=torch.float32, device=dev)
    b.forward(c, tg, out=out, expert_count=count, ws=ws)
    st, info = b.moe_device_status(ws, ws.numel())
    assert st == 0, (b.STATUS[st], info)
    return out.cpu().numpy(), count.cpu().numpy()


def check_routing(wl, tc, g, scores=None):
    """GPU routing vs the oracle: bit-exact except tokens with a near tie (returned count)."""
    if scores is None:
        scores = oracle.gate_scores(wl.gate, tc["x"], tc["w_gate"], tc["w_noise"], tc["eps"], tc["proj"], tc["emb"],
                                    wl.temperature)
    oidx, ogate = oracle.topk(scores, wl.k, wl.norm)
    ties = near_ties(scores, wl.k)
    diff = (g["idx"] != oidx).any(axis=1)
    assert not (diff & ~ties).any(), "routing differs outside near ties at tokens %s" % np.nonzero(diff & ~ties)[0][:10]
    same = ~diff
    assert np.allclose(g["gate"][same], ogate[same], rtol=1e-4, atol=1e-6), \
        np.abs(g["gate"][same] - ogate[same]).max()
    return scores, int(ties.sum()), int(diff.sum())


def check_dispatch(wl, tc_x, g):
    """Dispatch outputs vs the oracle's dispatch run on the GPU's own routing; bit-exact."""
    C = oracle.capacity(wl.T, wl.E, wl.k, wl.capacity_factor, wl.capacity)
    oslot, ocount = oracle.dispatch(g["idx"], wl.E, C, wl.priority)
    assert np.array_equal(g["slot"], oslot)
    assert np.array_equal(g["count"], ocount)
    kept = np.minimum(ocount, C)
    pad = (kept + 127) // 128 * 128
    off = np.concatenate([[0], np.cumsum(pad)])
    assert np.array_equal(g["off"], off)
    assert g["rows"] >= off[-1]
    rtok = g["rtok"][: off[-1]]
    want_tok = np.full(off[-1], -1, np.int64)
    want_gate = np.zeros(off[-1], np.float32)
    t_idx, j_idx = np.nonzero(oslot >= 0)
    r = off[g["idx"][t_idx, j_idx]] + oslot[t_idx, j_idx]
    want_tok[r] = t_idx
    want_gate[r] = g["gate"][t_idx, j_idx]
    assert np.array_equal(rtok, want_tok)
    assert np.array_equal(g["rgate"][: off[-1]].view(np.int32), want_gate.view(np.int32))
    if len(r):
        xd = g["xd"][torch.from_numpy(r)]
        assert torch.equal(xd, tc_x[torch.from_numpy(t_idx)])
    return C, oslot


def oracle_out(wl, tc, tg, scores, idx, slot, tokens):
    """The oracle's output for `tokens`, given a routing (idx, slot); gates from the fp64 scores."""
    gate = gates_for(scores, idx, wl.norm)
    if tc.get("w1") is not None:
        return oracle.combine_tokens(tokens, tc["x"], idx, gate, slot, tc["w1"], tc["b1"], tc["w2"], tc["b2"])
    # weights live on the GPU only: hand the oracle the experts these tokens use, renumbered
    used = sorted({int(e) for t in tokens for e, s in zip(idx[t], slot[t]) if s >= 0}) or [0]
    remap = {e: i for i, e in enumerate(used)}
    sub = expert_subset(tg, tc, used)
    idx2 = np.array([[remap.get(int(e), 0) for e in row] for row in idx], dtype=np.int32)
    return oracle.combine_tokens(tokens, tc["x"], idx2, gate, slot, sub["w1"], sub["b1"], sub["w2"], sub["b2"])


def check_output(wl, out, ref, tokens):
    """Per-token relative error <= TOL[dtype]; tokens whose reference is exactly 0 must be exactly 0."""
    got = out[tokens].astype(np.float64)
    zero = np.all(ref == 0.0, axis=1)
    assert np.all(got[zero] == 0.0), "dropped tokens must output exactly 0"
    nz = ~zero
    if nz.any():
        err = np.abs(got[nz] - ref[nz]).max(1) / np.abs(ref[nz]).max(1)
        assert err.max() <= TOL[wl.dtype], "max per-token relative error %.3e" % err.max()
        return float(err.max())
    return 0.0


def sample_tokens(T: int, n: int, seed: int = 0) -> np.ndarray:
    if n >= T:
        return np.arange(T, dtype=np.int32)
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(T, size=n, replace=False)).astype(np.int32)


def segment_edge_tokens(idx: np.ndarray, slot: np.ndarray, E: int, C: int) -> np.ndarray:
    """Tokens that own the rows at the edges of every expert's segment of the dispatched rows: slots 0,
    127, 128 (either side of the first 128-row tile boundary) and the last kept slot (the expert's
    last, usually partial, tile).  Checking their outputs reaches every expert's tile edges."""
    T, k = idx.shape
    counts = np.zeros(E, np.int64)
    np.add.at(counts, idx[slot >= 0], 1)
    kept = np.minimum(counts, C)
    want = {}
    for e in range(E):
        for sl in (0, 127, 128, int(kept[e]) - 1):
            if 0 <= sl < kept[e]:
                want[(e, sl)] = None
    toks = set()
    t_idx, j_idx = np.nonzero(slot >= 0)
    for t, j in zip(t_idx.tolist(), j_idx.tolist()):
        if (int(idx[t, j]), int(slot[t, j])) in want:
            toks.add(t)
    return np.array(sorted(toks), dtype=np.int32)
