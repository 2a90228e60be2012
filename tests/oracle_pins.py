"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError if the oracle disagrees
with: a hand-worked case (tests/golden/hand_worked.json), a library routine applied to a special case
(torch / numpy / scipy in float64), an invariant the definition implies, or a second, dense
formulation of the whole layer (``dense_layer`` below: every expert on every token, masked).

They are run against the real oracle (test_oracle_pins.py) and against deliberately broken copies of
its source (test_oracle_mutants.py), where at least one pin must fail for every planted mistake.
"""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np
import torch
import torch.nn.functional as F

from mixture_experts_sparse_03_b300.inputs import make_inputs, small_workload

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")))


def _t(a, dtype=torch.float32):
    return torch.tensor(a, dtype=dtype)


def _f64(t):
    return None if t is None else t.detach().cpu().to(torch.float64)


# ---------------------------------------------------------------- a second formulation of the layer
def dense_layer(wl, t):
    """The whole layer written differently from the oracle: scores by matrix products, top-k by a
    stable sort, capacity by a cumulative count per expert, every expert evaluated on every token with
    torch's own Linear and exact GELU, and the result masked.  float64 throughout."""
    X = _f64(t["x"])
    T = X.shape[0]
    if wl.gate == "softmax":
        S = X @ _f64(t["w_gate"]).T
    elif wl.gate == "noisy":
        S = X @ _f64(t["w_gate"]).T + t["eps"].to(torch.float64) * torch.from_numpy(
            np.logaddexp(0.0, (X @ _f64(t["w_noise"]).T).numpy()))
    else:
        U = X @ _f64(t["proj"]).T
        S = F.cosine_similarity(U[:, None, :], _f64(t["emb"])[None, :, :], dim=-1, eps=1e-12) / wl.temperature
    S = S.numpy()
    E, k = wl.E, wl.k
    # stable sort on -score keeps the lower expert id first among equal scores
    order = np.argsort(-S, axis=1, kind="stable")[:, :k].astype(np.int32)
    if wl.norm == "all":
        P = torch.softmax(torch.from_numpy(S), dim=1).numpy()
        gate = np.take_along_axis(P, order, axis=1)
    else:
        chosen = np.take_along_axis(S, order, axis=1)
        gate = torch.softmax(torch.from_numpy(chosen), dim=1).numpy()
    C = wl.capacity if wl.capacity >= 0 else math.ceil(wl.capacity_factor * T * k / E)
    # position of pair (t, j) in its expert's queue = pairs of earlier tokens with that expert
    onehot = np.zeros((T, E), dtype=np.int64)
    for j in range(k):
        onehot[np.arange(T), order[:, j]] += 1
    before = np.cumsum(onehot, axis=0) - onehot
    pos = np.take_along_axis(before, order, axis=1)
    slot = np.where(pos < C, pos, -1).astype(np.int32)
    count = onehot.sum(axis=0).astype(np.int32)
    W1, W2 = _f64(t["w1"]), _f64(t["w2"])
    b1 = _f64(t["b1"]) if t.get("b1") is not None else torch.zeros(E, W1.shape[1], dtype=torch.float64)
    b2 = _f64(t["b2"]) if t.get("b2") is not None else torch.zeros(E, W2.shape[1], dtype=torch.float64)
    Y = torch.stack([F.linear(F.gelu(F.linear(X, W1[e], b1[e]), approximate="none"), W2[e], b2[e])
                     for e in range(E)])  # [E, T, d]
    out = torch.zeros_like(X)
    for j in range(k):
        keep = torch.from_numpy(slot[:, j] >= 0)
        ye = Y[torch.from_numpy(order[:, j]).long(), torch.arange(T)]
        out += torch.where(keep[:, None], torch.from_numpy(gate[:, j])[:, None] * ye, torch.zeros_like(ye))
    return dict(scores=S, idx=order, gate=gate, C=C, slot=slot, count=count, out=out.numpy())


# ------------------------------------------------------------------------------------------- pins
def pin_softmax_gate_hand(o):
    g = GOLDEN["softmax_gate"]
    s, idx, gate = o.route("softmax", 2, "topk", _t(g["x"]), _t(g["w_gate"]))
    assert np.array_equal(s, np.array(g["scores"]))
    assert np.array_equal(idx, np.array(g["top2_idx"]))
    assert np.allclose(gate, np.array(g["top2_gate"]), rtol=1e-15, atol=0)
    # the same data in bf16 (every value is exact in bf16)
    s2 = o.gate_scores("softmax", _t(g["x"], torch.bfloat16), _t(g["w_gate"], torch.bfloat16))
    assert np.array_equal(s2, s)


def pin_full_softmax_top1_hand(o):
    g = GOLDEN["full_softmax_top1"]
    idx, gate = o.topk(np.array(g["scores"]), 1, "all")
    assert np.array_equal(idx, np.array(g["idx"]))
    assert abs(gate[0, 0] - 0.75) < 1e-15


def pin_cosine_gate_hand(o):
    g = GOLDEN["cosine_gate"]
    s = o.gate_scores("cosine", _t(g["x"]), proj=_t(g["proj"]), emb=_t(g["emb"]), temperature=g["temperature"])
    want = np.array(g["cosines"]) / g["temperature"]
    assert np.allclose(s, want, rtol=1e-14, atol=1e-14)


def pin_noisy_gate_hand(o):
    g = GOLDEN["noisy_gate_zero_noise_weights"]
    s = o.gate_scores("noisy", _t(g["x"]), _t(g["w_gate"]), _t(g["w_noise"]), eps=np.array(g["eps"], np.float32))
    assert np.allclose(s, np.array(g["scores"]), rtol=1e-15, atol=0)


def pin_capacity_values(o):
    for c in GOLDEN["capacity"]["cases"]:
        assert o.capacity(c["T"], c["E"], c["k"], c["cf"], c["capacity"]) == c["C"], c


def pin_dispatch_hand(o):
    for c in GOLDEN["dispatch"]["cases"]:
        slot, count = o.dispatch(np.array(c["idx"], np.int32), c["E"], c["C"])
        assert np.array_equal(slot, np.array(c["slot"])), (slot, c)
        assert np.array_equal(count, np.array(c["count"])), (count, c)


def pin_dispatch_rank_priority_hand(o):
    """Hand-worked rank-priority dispatch; the same routings in token order differ as worked out too."""
    for c in GOLDEN["dispatch_rank_priority"]["cases"]:
        idx = np.array(c["idx"], np.int32)
        slot, count = o.dispatch(idx, c["E"], c["C"], priority="rank")
        assert np.array_equal(slot, np.array(c["slot"])), (slot, c)
        assert np.array_equal(count, np.array(c["count"])), (count, c)
        tslot, _ = o.dispatch(idx, c["E"], c["C"])
        assert np.array_equal(tslot, np.array(c["token_order_slot"])), (tslot, c)


def pin_dispatch_rank_priority_properties(o):
    """Random routings in rank priority: with k = 1 it is token order; each expert keeps exactly the first
    C of its pairs ordered by (rank, token) with slots 0..kept-1 in that order, so every kept pair of a
    lower rank has a lower slot than every pair of a higher rank; counts are the routing histogram."""
    rng = np.random.default_rng(7)
    for (T, E, k, C) in [(50, 4, 1, 9), (64, 6, 2, 15), (33, 5, 3, 20), (40, 8, 2, 1), (30, 4, 4, 30)]:
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        slot, count = o.dispatch(idx, E, C, priority="rank")
        assert np.array_equal(count, np.bincount(idx.ravel(), minlength=E))
        if k == 1:
            assert np.array_equal(slot, o.dispatch(idx, E, C)[0])
        for e in range(E):
            order = sorted((j, t) for t in range(T) for j in range(k) if idx[t, j] == e)
            got = [slot[t, j] for j, t in order]
            n = min(C, len(order))
            assert got == list(range(n)) + [-1] * (len(order) - n)


def pin_fp8_codes_hand(o):
    """Hand-decoded E4M3 codes (normal, subnormal, signed, zero) and a hand-worked block-scaled matrix."""
    g = GOLDEN["fp8_e4m3_codes"]
    q = np.array([g["codes"]], np.uint8)
    got = o.dequant_block_fp8(q, np.ones((1, 1), np.float32), block=128)[0]
    assert np.array_equal(got, np.array(g["values"])), got
    assert np.array_equal(np.signbit(got), np.signbit(np.array(g["values"])))
    b = GOLDEN["fp8_block_scale"]
    got = o.dequant_block_fp8(np.array(b["codes"], np.uint8), np.array(b["scale"], np.float32), block=b["block"])
    assert np.array_equal(got, np.array(b["values"])), got


def pin_fp8_dequant_vs_torch(o):
    """Every non-NaN E4M3 code against torch's float8_e4m3fn conversion (a library routine), and random
    block-scaled matrices (ragged edge blocks, power-of-two and other scales) against numpy."""
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = o.dequant_block_fp8(codes.reshape(1, -1), np.ones((1, 1), np.float32), block=256)[0]
    assert np.array_equal(got, want)
    assert np.isnan(o.dequant_block_fp8(np.array([[0x7F, 0xFF]], np.uint8), np.ones((1, 1), np.float32))).all()
    rng = np.random.default_rng(11)
    for rows, cols, blk in [(5, 7, 2), (130, 260, 128), (64, 64, 32)]:
        q = rng.choice(codes, size=(rows, cols)).astype(np.uint8)
        sc = (np.exp2(rng.integers(-12, 4, size=(-(-rows // blk), -(-cols // blk)))) *
              rng.choice([1.0, 1.25, -0.75], size=(-(-rows // blk), -(-cols // blk)))).astype(np.float32)
        val = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        full = np.repeat(np.repeat(sc.astype(np.float64), blk, 0), blk, 1)[:rows, :cols]
        assert np.array_equal(o.dequant_block_fp8(q, sc, block=blk), val * full)


def pin_fp8_expert_with_dequantised_weights(o):
    """The expert on float64 (dequantised) weights with a bf16 token: against torch fp64 Linear-GELU-Linear
    on the same values, and against the same expert with the weights given as bf16 when they are
    exactly representable in bf16 (E4M3 values times power-of-two scales)."""
    rng = np.random.default_rng(12)
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    d, h = 24, 40
    x = torch.randn(d, generator=torch.Generator().manual_seed(13)).to(torch.bfloat16)
    w1 = o.dequant_block_fp8(rng.choice(codes, size=(h, d)).astype(np.uint8),
                             np.exp2(rng.integers(-9, -5, size=(1, 1))).astype(np.float32), block=128)
    w2 = o.dequant_block_fp8(rng.choice(codes, size=(d, h)).astype(np.uint8),
                             np.exp2(rng.integers(-9, -5, size=(1, 1))).astype(np.float32), block=128)
    b1 = torch.randn(h, generator=torch.Generator().manual_seed(14)).to(torch.bfloat16)
    b2 = torch.randn(d, generator=torch.Generator().manual_seed(15)).to(torch.bfloat16)
    y = o.expert(x, w1, b1, w2, b2)
    xt, t1, t2 = x.double(), torch.from_numpy(w1), torch.from_numpy(w2)
    want = F.linear(F.gelu(F.linear(xt, t1, b1.double()), approximate="none"), t2, b2.double()).numpy()
    assert np.allclose(y, want, rtol=1e-12, atol=1e-12)
    yb = o.expert(x, torch.from_numpy(w1).to(torch.bfloat16), b1, torch.from_numpy(w2).to(torch.bfloat16), b2)
    assert np.array_equal(y, yb)


def _fd_layer(seed, gate, E=4):
    g = torch.Generator().manual_seed(seed)
    T, d, h = 6, 8, 12
    t = {"x": torch.randn(T, d, generator=g), "w_gate": torch.randn(E, d, generator=g) * 0.6,
         "w1": torch.randn(E, h, d, generator=g) * 0.4, "b1": torch.randn(E, h, generator=g) * 0.3,
         "w2": torch.randn(E, d, h, generator=g) * 0.3, "b2": torch.randn(E, d, generator=g) * 0.3}
    if gate == "noisy":
        t["w_noise"] = torch.randn(E, d, generator=g) * 0.6
        t["eps"] = torch.randn(T, E, generator=g)
    dout = torch.randn(T, d, generator=g, dtype=torch.float64)
    return t, dout


def pin_backward_finite_differences(o):
    """The backward against central differences of the oracle's own forward (loss = sum(dout * out)) on tiny
    fp32 layers: every gradient tensor (x, both gate weights, both expert weights and biases) at sampled
    entries, for the softmax and noisy gates, both gate normalisations, with and without capacity drops,
    token and rank priority.  The step is a power of two, each perturbed value is exact in fp32, and the
    routing must not change under the step (else the case would not be differentiable there)."""
    cases = [("softmax", "topk", 2, 6, "token", 21), ("softmax", "all", 1, 6, "token", 22),
             ("noisy", "topk", 2, 2, "token", 23), ("softmax", "topk", 3, 3, "rank", 24), ("noisy", "topk", 1, 2, "token", 25)]
    rng = np.random.default_rng(9)
    dropped_somewhere = False
    for gate, norm, k, cap, prio, seed in cases:
        t, dout = _fd_layer(seed, gate)
        spec = dict(gate=gate, norm=norm, k=k, E=4, capacity=cap, capacity_factor=1.0, temperature=1.0,
                    priority=prio)
        grads = o.backward(spec, t, dout)
        base = o.forward(spec, t)
        dropped_somewhere = dropped_somewhere or bool((base["slot"] < 0).any())

        def loss(tt):
            f = o.forward(spec, tt)
            assert np.array_equal(f["idx"], base["idx"]) and np.array_equal(f["slot"], base["slot"])
            return float((f["out"] * dout.numpy()).sum())

        names = [("x", "dx"), ("w_gate", "dw_gate"), ("w1", "dw1"), ("b1", "db1"), ("w2", "dw2"), ("b2", "db2")]
        if gate == "noisy":
            names.append(("w_noise", "dw_noise"))
        for name, key in names:
            flat = t[name].reshape(-1)
            for i in rng.choice(flat.numel(), size=6, replace=False):
                step = 2.0 ** -12
                plus, minus = dict(t), dict(t)
                vp, vm = t[name].clone(), t[name].clone()
                vp.view(-1)[i] += step
                vm.view(-1)[i] -= step
                plus[name], minus[name] = vp, vm
                width = float(vp.view(-1)[i]) - float(vm.view(-1)[i])
                fd = (loss(plus) - loss(minus)) / width
                an = grads[key].reshape(-1)[i]
                assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (gate, norm, name, int(i), fd, an)
    assert dropped_somewhere  # the capacity cases do drop pairs


def pin_backward_sampled_equals_whole(o):
    """The single-output backward (for layers too large for the whole one) against the whole backward, which
    the finite differences above pin: dx rows and dW1 / db1 / dW2 / db2 entries agree to rounding, for both
    gates and normalisations, with capacity drops, on bf16 layers."""
    rng = np.random.default_rng(13)
    dropped = False
    for gate, norm, k, cap, seed in (("softmax", "topk", 2, 2, 31), ("noisy", "topk", 2, 2, 32),
                                     ("softmax", "all", 1, 8, 33)):
        t, dout = _fd_layer(seed, gate)
        tb = {n: (v.to(torch.bfloat16) if n != "eps" and v is not None else v) for n, v in t.items()}
        spec = dict(gate=gate, norm=norm, k=k, E=4, capacity=cap, capacity_factor=1.0, temperature=1.0,
                    priority="token")
        whole = o.backward(spec, tb, dout)
        T, d = tb["x"].shape
        E, h, _ = tb["w1"].shape
        toks = rng.choice(T, size=4, replace=False)
        s1 = [(int(rng.integers(E)), int(rng.integers(h)), int(rng.integers(d))) for _ in range(10)]
        s2 = [(int(rng.integers(E)), int(rng.integers(d)), int(rng.integers(h))) for _ in range(10)]
        part = o.backward_sampled(spec, tb, dout, toks, s1, s2)
        assert np.allclose(part["dx"], whole["dx"][toks], rtol=1e-12, atol=1e-14)
        assert np.allclose(part["dw1"], [whole["dw1"][e, n, m] for e, n, m in s1], rtol=1e-12, atol=1e-14)
        assert np.allclose(part["db1"], [whole["db1"][e, n] for e, n, _ in s1], rtol=1e-12, atol=1e-14)
        assert np.allclose(part["dw2"], [whole["dw2"][e, m, n] for e, m, n in s2], rtol=1e-12, atol=1e-14)
        assert np.allclose(part["db2"], [whole["db2"][e, m] for e, m, _ in s2], rtol=1e-12, atol=1e-14)
        dropped = dropped or bool((part["slot"] < 0).any())
    assert dropped  # some case drops pairs


def pin_gelu_normal_cdf(o):
    """Identity weights make the expert return GELU(x) itself; GELU(z) = z Phi(z) with Phi from a table."""
    g = GOLDEN["gelu_normal_cdf"]
    z = np.array(g["z"])
    n = len(z)
    I = torch.eye(n, dtype=torch.float32)
    y = o.expert(_t(z.tolist()), I, None, I, None)
    assert np.allclose(y, z * np.array(g["phi"]), rtol=1e-14, atol=1e-300)
    big = o.expert(_t([10.0, -10.0]), torch.eye(2), None, torch.eye(2), None)
    assert abs(big[0] - 10.0) < 1e-20 and abs(big[1]) < 1e-20


def pin_topk_bruteforce(o):
    """Every k on small E, against a stable sort by (-score, id); scores quantised to force ties."""
    rng = np.random.default_rng(5)
    for E in range(1, 7):
        S = np.round(rng.normal(size=(40, E)) * 2) / 2  # many exact ties
        for k in range(1, E + 1):
            for norm in ("all", "topk"):
                idx, gate = o.topk(S, k, norm)
                want = np.array([sorted(range(E), key=lambda e: (-S[t, e], e))[:k] for t in range(40)])
                assert np.array_equal(idx, want), (E, k)
                assert np.all(gate > 0)
                if norm == "topk" or k == E:
                    assert np.allclose(gate.sum(1), 1.0, rtol=0, atol=1e-12)
                if norm == "all":
                    full = torch.softmax(torch.from_numpy(S), dim=1).numpy()
                    assert np.allclose(gate, np.take_along_axis(full, want, axis=1), rtol=1e-13, atol=0)


def pin_duplicate_rows_tie(o):
    """Experts with identical gate rows tie exactly: the lower id is chosen first."""
    x = torch.randn(16, 8, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    w = torch.randn(3, 8, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    w = torch.stack([w[0], w[1], w[1], w[2], w[0]])  # 1 == 2 and 0 == 4
    s, idx, _ = o.route("softmax", 5, "topk", x, w)
    for t in range(16):
        r = list(idx[t])
        assert r.index(1) < r.index(2) and r.index(0) < r.index(4)
        assert s[t, 1] == s[t, 2] and s[t, 0] == s[t, 4]


def pin_noisy_reductions(o):
    """eps = 0 gives the clean logits; W_n = 0 adds exactly eps ln 2; random case vs numpy logaddexp."""
    g = torch.Generator().manual_seed(7)
    x = torch.randn(12, 16, generator=g).to(torch.bfloat16)
    wg = (torch.randn(5, 16, generator=g) / 4).to(torch.bfloat16)
    wn = (torch.randn(5, 16, generator=g) / 4).to(torch.bfloat16)
    eps = torch.randn(12, 5, generator=g)
    clean = o.gate_scores("softmax", x, wg)
    assert np.array_equal(o.gate_scores("noisy", x, wg, wn, eps=torch.zeros(12, 5)), clean)
    s0 = o.gate_scores("noisy", x, wg, torch.zeros_like(wn), eps=eps)
    assert np.allclose(s0, clean + eps.double().numpy() * math.log(2.0), rtol=1e-15, atol=1e-15)
    s = o.gate_scores("noisy", x, wg, wn, eps=eps)
    want = clean + eps.double().numpy() * np.logaddexp(0.0, (_f64(x) @ _f64(wn).T).numpy())
    assert np.allclose(s, want, rtol=1e-13, atol=1e-14)


def pin_cosine_invariants(o):
    """Scaling P and the embeddings by powers of two changes nothing (exactly); random case vs torch's
    cosine_similarity; orthogonal and opposite embeddings give 0 and -1/temperature."""
    g = torch.Generator().manual_seed(9)
    x = torch.randn(10, 32, generator=g).to(torch.bfloat16)
    P = (torch.randn(8, 32, generator=g) / 6).to(torch.bfloat16)
    em = (torch.randn(6, 8, generator=g) / 3).to(torch.bfloat16)
    s = o.gate_scores("cosine", x, proj=P, emb=em, temperature=0.07)
    s2 = o.gate_scores("cosine", x, proj=P * 2, emb=em * 4, temperature=0.07)
    assert np.array_equal(s, s2)
    U = _f64(x) @ _f64(P).T
    want = F.cosine_similarity(U[:, None, :], _f64(em)[None], dim=-1).numpy() / 0.07
    assert np.allclose(s, want, rtol=1e-12, atol=1e-12)
    assert np.all(np.abs(s) <= 1 / 0.07 + 1e-12)


def pin_dispatch_properties(o):
    """Random routings: counts are the routing histogram; each expert keeps exactly its first C tokens
    in token order, with slots 0..kept-1 in that order; kept + dropped = T k; reversing the token order
    keeps each expert's last C tokens instead."""
    rng = np.random.default_rng(3)
    for (T, E, k, C) in [(50, 4, 1, 9), (64, 6, 2, 15), (33, 5, 3, 20), (20, 3, 3, 20), (40, 8, 2, 1)]:
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        slot, count = o.dispatch(idx, E, C)
        assert np.array_equal(count, np.bincount(idx.ravel(), minlength=E))
        assert (slot >= 0).sum() + (slot < 0).sum() == T * k
        for e in range(E):
            toks = np.nonzero((idx == e).any(1))[0]  # ascending token order
            kept = toks[:C]
            got = [(t, slot[t][list(idx[t]).index(e)]) for t in toks]
            assert [t for t, s_ in got if s_ >= 0] == list(kept)
            assert [s_ for t, s_ in got if s_ >= 0] == list(range(len(kept)))
        rslot, _ = o.dispatch(idx[::-1].copy(), E, C)
        for e in range(E):
            toks = np.nonzero((idx == e).any(1))[0]
            want_kept = set(toks[::-1][:C])
            got_kept = {T - 1 - r for r in range(T) for j in range(k) if idx[::-1][r][j] == e and rslot[r][j] >= 0}
            assert got_kept == want_kept


def pin_expert_vs_torch(o):
    g = torch.Generator().manual_seed(4)
    for dt in (torch.float32, torch.bfloat16):
        x = torch.randn(24, generator=g).to(dt)
        w1 = (torch.randn(40, 24, generator=g) / 5).to(dt)
        b1 = torch.randn(40, generator=g).to(dt)
        w2 = (torch.randn(24, 40, generator=g) / 6).to(dt)
        b2 = torch.randn(24, generator=g).to(dt)
        y = o.expert(x, w1, b1, w2, b2)
        want = F.linear(F.gelu(F.linear(_f64(x), _f64(w1), _f64(b1)), approximate="none"), _f64(w2), _f64(b2))
        assert np.allclose(y, want.numpy(), rtol=1e-13, atol=1e-13)
        y0 = o.expert(x, w1, None, w2, None)
        want0 = F.linear(F.gelu(F.linear(_f64(x), _f64(w1)), approximate="none"), _f64(w2))
        assert np.allclose(y0, want0.numpy(), rtol=1e-13, atol=1e-13)


def pin_single_expert_is_dense_ffn(o):
    """E = 1, k = 1, capacity >= T: the layer is the dense Linear-GELU-Linear (gate weight 1)."""
    wl = small_workload(T=9, d=16, h=24, E=1, k=1, norm="all", capacity_factor=1.0, dtype="f32", bias="normal")
    t = make_inputs(wl)
    r = o.forward(wl.spec(), t)
    want = F.linear(F.gelu(F.linear(_f64(t["x"]), _f64(t["w1"][0]), _f64(t["b1"][0])), approximate="none"),
                    _f64(t["w2"][0]), _f64(t["b2"][0]))
    assert np.allclose(r["gate"], 1.0, rtol=0, atol=1e-15)
    assert np.allclose(r["out"], want.numpy(), rtol=1e-13, atol=1e-13)


def pin_naive_top1_layer(o):
    """The top-1 layer as the 'PyTorch-CUDA-v2.6' page writes it (gate Linear without bias here,
    softmax, max -> weight and index, each expert on its masked tokens, output times the weight), in
    torch float64, equals the oracle with a capacity that drops nothing."""
    wl = small_workload(T=40, d=16, h=32, E=4, k=1, norm="all", capacity=40, dtype="f32", bias="normal")
    t = make_inputs(wl)
    X = _f64(t["x"])
    weights = torch.softmax(X @ _f64(t["w_gate"]).T, dim=-1)
    top1_w, top1_i = weights.max(dim=-1)
    final = torch.zeros_like(X)
    for i in range(wl.E):
        mask = top1_i == i
        if mask.any():
            final[mask] = F.linear(F.gelu(F.linear(X[mask], _f64(t["w1"][i]), _f64(t["b1"][i])), approximate="none"),
                                   _f64(t["w2"][i]), _f64(t["b2"][i]))
    final = final * top1_w.unsqueeze(-1)
    r = o.forward(wl.spec(), t)
    assert np.allclose(r["out"], final.numpy(), rtol=1e-12, atol=1e-13)


def pin_layer_vs_dense_formulation(o):
    """Whole layer on small workloads of every gate type, both dtypes, several k, with and without
    drops, against ``dense_layer``."""
    cases = [
        small_workload(T=37, d=16, h=32, E=4, k=1, norm="all", dtype="f32", capacity_factor=1.0),
        small_workload(T=41, d=32, h=16, E=5, k=2, dtype="bf16", capacity_factor=0.8),
        small_workload(T=30, d=16, h=16, E=6, k=3, dtype="bf16", capacity_factor=2.0, bias="none"),
        small_workload(T=33, d=16, h=32, E=5, k=2, gate="noisy", dtype="bf16", capacity_factor=0.9),
        small_workload(T=29, d=32, h=16, E=4, k=2, gate="cosine", cos_dim=8, dtype="bf16", capacity_factor=1.0,
                       x_dist="clusters"),
        small_workload(T=25, d=16, h=16, E=3, k=3, dtype="f32", capacity=25, norm="all"),
    ]
    for wl in cases:
        t = make_inputs(wl)
        r = o.forward(wl.spec(), t)
        ref = dense_layer(wl, t)
        assert r["C"] == ref["C"]
        assert np.allclose(r["scores"], ref["scores"], rtol=1e-12, atol=1e-12), wl
        assert np.array_equal(r["idx"], ref["idx"]), wl
        assert np.allclose(r["gate"], ref["gate"], rtol=1e-12, atol=1e-15), wl
        assert np.array_equal(r["slot"], ref["slot"]), wl
        assert np.array_equal(r["count"], ref["count"]), wl
        scale = np.abs(ref["out"]).max()
        assert np.allclose(r["out"], ref["out"], rtol=1e-11, atol=1e-12 * scale), wl


def pin_drops_zero_output(o):
    """A token whose pairs are all dropped outputs exactly 0; with C = 0 every token does."""
    wl = small_workload(T=20, d=16, h=16, E=2, k=1, capacity=0, dtype="f32")
    r = o.forward(wl.spec(), make_inputs(wl))
    assert np.all(r["slot"] == -1) and np.all(r["out"] == 0.0)


def pin_router_stats_hand(o):
    """Router statistics worked by hand from their definitions: three tokens, top-2 over three experts.
    Importance = gate column sums: e0 = 0.6 + 0.9 = 1.5, e1 = 0.4 + 0.5 = 0.9, e2 = 0.5 + 0.1 = 0.6;
    mean 1.0, so load_balance_loss = 0.25 + 0.01 + 0.16 = 0.42 and expert_importance_loss =
    0.1 * sqrt(0.42 / (3 - 1)); one pair has slot -1."""
    idx = np.array([[0, 1], [1, 2], [0, 2]], dtype=np.int32)
    gate = np.array([[0.6, 0.4], [0.5, 0.5], [0.9, 0.1]])
    slot = np.array([[0, 0], [1, -1], [1, 0]], dtype=np.int32)
    imp, il, lb, dropped = o.router_stats(idx, gate, 3, slot)
    assert np.allclose(imp, [1.5, 0.9, 0.6], rtol=0, atol=1e-15)
    assert abs(lb - 0.42) < 1e-15 and abs(il - 0.1 * (0.21 ** 0.5)) < 1e-15
    assert dropped == 1


def pin_router_stats_invariants(o):
    """Balanced routing gives zero losses; relabelling the experts permutes the importance and leaves the
    losses alone; importance sums to the gates' total; one expert has no standard deviation (NaN)."""
    T, k, E = 40, 2, 4
    idx = np.array([[(2 * t) % E, (2 * t + 1) % E] for t in range(T)], dtype=np.int32)
    gate = np.full((T, k), 0.5)
    imp, il, lb, dropped = o.router_stats(idx, gate, E)
    assert np.allclose(imp, T * k * 0.5 / E) and il == 0.0 and lb == 0.0 and dropped == 0
    rng = np.random.default_rng(5)
    idx2 = rng.integers(0, E, size=(T, k)).astype(np.int32)
    idx2[:, 1] = (idx2[:, 0] + 1 + rng.integers(0, E - 1, size=T)) % E
    g2 = rng.random((T, k))
    imp2, il2, lb2, _ = o.router_stats(idx2, g2, E)
    perm = np.array([2, 0, 3, 1], dtype=np.int32)  # expert e becomes perm[e]
    imp3, il3, lb3, _ = o.router_stats(perm[idx2], g2, E)
    assert np.allclose(imp3[perm], imp2, rtol=1e-14) and abs(il3 - il2) < 1e-14 and abs(lb3 - lb2) < 1e-12
    assert abs(imp2.sum() - g2.sum()) < 1e-12
    assert abs(lb2 - (E - 1) * (il2 / 0.1) ** 2) < 1e-10
    _, il1, lb1, _ = o.router_stats(np.zeros((T, 1), dtype=np.int32), np.ones((T, 1)), 1)
    assert np.isnan(il1) and lb1 == 0.0


ALL_PINS = [v for k_, v in sorted(globals().items()) if k_.startswith("pin_") and callable(v)]
