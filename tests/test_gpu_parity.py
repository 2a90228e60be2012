"""GPU parity of the CUDA path against the fp64 oracle, through the C ABI.

Small workloads (several tiles and a ragged tail, every gate type, both dtypes, k from 1 to 4, with
and without drops) compare every token; the five full-size workloads compare routing and dispatch on
every token and the layer output on sampled tokens, in the launch configuration the benchmark uses."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_sparse_03_b300 import binding as b
from mixture_experts_sparse_03_b300.inputs import WORKLOADS, small_workload
from tests import parity as P

pytestmark = pytest.mark.gpu

SMALL = [
    small_workload(T=97, d=64, h=128, E=5, k=2, capacity_factor=1.0),
    small_workload(T=300, d=128, h=256, E=8, k=2, capacity_factor=0.7),          # drops
    small_workload(T=257, d=64, h=320, E=3, k=1, norm="all", capacity_factor=1.3),  # h not a multiple of 256
    small_workload(T=200, d=192, h=192, E=6, k=3, capacity_factor=1.0),          # k > 2: gather combine
    small_workload(T=150, d=64, h=128, E=16, k=4, capacity=150, bias="none"),     # dropless
    small_workload(T=129, d=128, h=128, E=12, k=2, gate="noisy", capacity_factor=1.1),
    small_workload(T=180, d=128, h=256, E=10, k=2, gate="cosine", cos_dim=64, capacity_factor=1.0,
                   x_dist="clusters"),
    small_workload(T=75, d=64, h=64, E=4, k=1, norm="all", dtype="f32", capacity_factor=1.2, bias="zero"),
    small_workload(T=211, d=128, h=128, E=7, k=2, dtype="f32", capacity_factor=0.9),
    small_workload(T=64, d=64, h=128, E=40, k=3, gate="noisy", dtype="f32", capacity_factor=1.5),
    small_workload(T=1, d=64, h=64, E=2, k=1, capacity_factor=1.0),
    small_workload(T=33, d=64, h=64, E=1, k=1, norm="all", capacity_factor=1.0),  # one expert: dense FFN
    # fused softmax gate with 32- and 64-wide logit tiles (clusters of 4 and 2 CTAs over K)
    small_workload(T=300, d=256, h=128, E=24, k=2, capacity_factor=1.0),
    small_workload(T=200, d=192, h=128, E=48, k=2, norm="all", capacity_factor=1.1),
    small_workload(T=520, d=128, h=128, E=64, k=4, capacity_factor=0.8),        # 64 experts, k > 2, drops
    # capacity slots in rank order (first choices first), with drops: the fused softmax gate, the
    # unfused noisy and cosine gates, the fp32 gate, and k > 2
    small_workload(T=300, d=128, h=256, E=8, k=2, capacity_factor=0.7, priority="rank"),
    small_workload(T=129, d=128, h=128, E=12, k=2, gate="noisy", capacity_factor=0.8, priority="rank"),
    small_workload(T=180, d=128, h=256, E=10, k=2, gate="cosine", cos_dim=64, capacity_factor=0.9,
                   x_dist="clusters", priority="rank"),
    small_workload(T=211, d=128, h=128, E=7, k=2, dtype="f32", capacity_factor=0.6, priority="rank"),
    small_workload(T=200, d=192, h=192, E=6, k=3, capacity_factor=0.8, priority="rank"),
    small_workload(T=2000, d=128, h=128, E=16, k=4, capacity_factor=0.9, priority="rank"),  # 250 pair blocks
]


def _id(wl):
    return "%s_%s_T%d_d%d_h%d_E%d_k%d%s" % (wl.gate, wl.dtype, wl.T, wl.d, wl.h, wl.E, wl.k,
                                           "_rank" if wl.priority == "rank" else "")


def _full_check(wl, flags=0):
    tc, tg = P.inputs(wl)
    g = P.run_steps(wl, tg, flags)
    scores, nties, ndiff = P.check_routing(wl, tc, g)
    C, slot = P.check_dispatch(wl, tc["x"], g)
    toks = np.arange(wl.T, dtype=np.int32)
    ref = P.oracle_out(wl, tc, tg, scores, g["idx"], slot, toks)
    P.check_output(wl, g["out"], ref, toks)
    out, count = P.run_forward(wl, tg, flags)
    assert np.array_equal(count, g["count"])
    P.check_output(wl, out, ref, toks)
    return out


@pytest.mark.parametrize("wl", SMALL, ids=_id)
def test_small_parity(wl):
    _full_check(wl)


@pytest.mark.parametrize("wl", [SMALL[0], SMALL[3], SMALL[5], SMALL[6]], ids=_id)
def test_small_parity_simt_ffn(wl):
    """The CUDA-core FFN path of a bf16 layer agrees with the oracle too."""
    _full_check(wl, flags=b.FLAG_SIMT_FFN)


def test_unfused_combine_matches_fused():
    wl = SMALL[1]
    _, tg = P.inputs(wl)
    fused, _ = P.run_forward(wl, tg)
    unfused, _ = P.run_forward(wl, tg, flags=b.FLAG_UNFUSED_COMBINE)
    assert np.allclose(fused, unfused, rtol=1e-6, atol=1e-6)


def test_deterministic():
    for wl in (SMALL[1], SMALL[3]):
        _, tg = P.inputs(wl)
        a, _ = P.run_forward(wl, tg)
        b2, _ = P.run_forward(wl, tg)
        assert np.array_equal(a.view(np.int32), b2.view(np.int32))


def test_exact_ties_go_to_lower_expert():
    wl = small_workload(T=64, d=64, h=64, E=6, k=3, capacity=64)
    tc, tg = P.inputs(wl)
    wg = tc["w_gate"].clone()
    wg[3] = wg[1]
    wg[5] = wg[0]
    tc["w_gate"] = wg
    tg["w_gate"] = wg.cuda()
    g = P.run_steps(wl, tg)
    P.check_routing(wl, tc, g)
    for t in range(wl.T):
        r = list(g["idx"][t])
        if 1 in r and 3 in r:
            assert r.index(1) < r.index(3)
        if 0 in r and 5 in r:
            assert r.index(0) < r.index(5)


def _ulp_step(w: torch.Tensor, up: bool) -> torch.Tensor:
    """The next bf16 value above (or below) each element of a bf16 tensor."""
    bits = w.view(torch.int16).to(torch.int32)
    away = (bits >= 0) == up  # moving away from zero increments the magnitude bits
    nb = torch.where(away, bits + 1, bits - 1)
    return nb.to(torch.int16).view(torch.bfloat16)


@pytest.mark.parametrize("gate,E,p", [("softmax", 6, 0), ("softmax", 72, 0), ("noisy", 6, 0), ("cosine", 6, 64),
                                       ("cosine", 40, 512)])
def test_near_ties_resolved_exactly(gate, E, p):
    """Gate rows (cosine gate: expert embeddings) that differ from another row by one bf16 ulp in one
    element: their scores differ by 1e-7 to 1e-3, often inside the fp32 error bound, so the kernel must
    settle the order with its float-float re-scoring (inside the fused gate for softmax with E <= 64,
    else the grid-wide re-scoring kernel; for the cosine gate through v_e = P^T e_e, folded in chunks of
    256 components when p = 512).  The choice must equal the oracle's on every token."""
    wl = small_workload(T=256, d=256, h=64, E=E, k=2, gate=gate, capacity=256, cos_dim=p or 32)
    tc, tg = P.inputs(wl)
    name = "emb" if gate == "cosine" else "w_gate"
    col = (5, 17) if gate != "cosine" else (5, 40)
    wg = tc[name].clone()
    wg[2] = wg[0]
    wg[2, col[0]] = _ulp_step(wg[0, col[0]:col[0] + 1], True)[0]
    wg[4] = wg[1]
    wg[4, col[1]] = _ulp_step(wg[1, col[1]:col[1] + 1], False)[0]
    tc[name] = wg
    tg[name] = wg.cuda()
    if gate == "noisy":
        wn = tc["w_noise"].clone()
        wn[2] = wn[0]
        wn[4] = wn[1]
        tc["w_noise"] = wn
        tg["w_noise"] = wn.cuda()
        # the noise term of a copied row must match too, so its draws are copied as well
        ep = tc["eps"].clone()
        ep[:, 2] = ep[:, 0]
        ep[:, 4] = ep[:, 1]
        tc["eps"] = ep
        tg["eps"] = ep.cuda()
    g = P.run_steps(wl, tg)
    scores, nties, ndiff = P.check_routing(wl, tc, g)
    assert ndiff == 0
    gaps = np.abs(scores[:, 2] - scores[:, 0])
    assert gaps.max() > 0 and np.median(gaps) < 1e-3  # the pairs really are near ties


def test_all_dropped_outputs_zero():
    wl = small_workload(T=50, d=64, h=64, E=4, k=2, capacity=0)
    _, tg = P.inputs(wl)
    out, count = P.run_forward(wl, tg)
    assert np.all(out == 0.0) and count.sum() == 100


@pytest.mark.parametrize("gate,E", [("softmax", 100), ("noisy", 64)])
def test_wide_gate_tiles_full_layer(gate, E):
    """Enough tokens that the gate GEMM takes its one-wave tiles (100 softmax logits in a 112-wide tile;
    the noisy gate's 64 + 64 rows in one tile): routing, dispatch and outputs against the oracle."""
    wl = small_workload(T=9500, d=256, h=64, E=E, k=2, gate=gate, capacity_factor=1.2)
    _full_check(wl)


@pytest.mark.parametrize("cf", [1.2, 0.3])
def test_output_cleared_by_the_up_projection(cf):
    """A layer whose up projection is long enough (rows x h >= 8192 per token) clears the fused combine's
    output inside the up projection's kernel instead of the gather: every token's output, dropped ones
    included (exactly zero), still matches the oracle after a call that leaves `out` dirty."""
    wl = small_workload(T=256, d=128, h=4096, E=4, k=2, capacity_factor=cf)
    _full_check(wl)


def test_heavy_drops_and_bias():
    wl = small_workload(T=400, d=64, h=128, E=4, k=2, capacity_factor=0.25, bias="normal")
    _full_check(wl)


def test_rank_priority_differs_from_token_order():
    """With drops, rank order keeps a different set of pairs than token order (the flag reaches the
    kernels): every first choice that fits is kept before any second choice."""
    wl = small_workload(T=300, d=128, h=256, E=8, k=2, capacity_factor=0.7, priority="rank")
    _, tg = P.inputs(wl)
    g_rank = P.run_steps(wl, tg)
    g_tok = P.run_steps(wl.with_(priority="token"), tg)
    assert np.array_equal(g_rank["idx"], g_tok["idx"])
    assert not np.array_equal(g_rank["slot"], g_tok["slot"])
    assert (g_rank["slot"][:, 0] >= 0).sum() >= (g_tok["slot"][:, 0] >= 0).sum()


@pytest.mark.parametrize("name", ["tiny_fp32", "bf16_e8_k2", "bf16_cosine_skew", "bf16_noisy_e64", "bf16_decode_e256",
                                  "bf16_recsys_e8"])
def test_full_size_workload(name):
    """Full sizes, launch configuration of the benchmark: routing and dispatch on every token, the
    output on sampled tokens (all tokens for the tiny layer)."""
    wl = WORKLOADS[name]
    tc, tg = P.inputs(wl)
    g = P.run_steps(wl, tg)
    scores, nties, ndiff = P.check_routing(wl, tc, g)
    C, slot = P.check_dispatch(wl, tc["x"], g)
    # random tokens plus the owners of every expert segment's edge rows (first row, either side of the
    # first 128-row tile boundary, last kept row), so that every expert's last partial tile is checked
    n = {"tiny_fp32": wl.T, "bf16_e8_k2": 64, "bf16_cosine_skew": 64, "bf16_noisy_e64": 128,
         "bf16_decode_e256": wl.T, "bf16_recsys_e8": 512}[name]
    edges = P.segment_edge_tokens(g["idx"], slot, wl.E, C)
    toks = np.union1d(P.sample_tokens(wl.T, n, seed=wl.seed), edges).astype(np.int32)
    ref = P.oracle_out(wl, tc, tg, scores, g["idx"], slot, toks)
    P.check_output(wl, g["out"], ref, toks)
    out, count = P.run_forward(wl, tg)
    assert np.array_equal(count, g["count"])
    P.check_output(wl, out, ref, toks)
    print("%s: near-tie tokens %d, routing differences %d, drops %d, output checked on %d tokens (%d edge owners)"
          % (name, nties, ndiff, int((slot < 0).sum()), len(toks), len(edges)))


def _logits_error_ratio(wl, tc, tg):
    """max over logits of |GPU - exact| / (2^-23 sum_i |x_i w_i|) for moe_gate_logits."""
    c = b.config(wl)
    ws = b.workspace(c, "cuda")
    rows = {"softmax": [tc["w_gate"]], "noisy": [tc["w_gate"], tc["w_noise"]], "cosine": [tc["proj"]]}[wl.gate]
    N = sum(r.shape[0] for r in rows)
    got = torch.full((wl.T, N), float("nan"), dtype=torch.float32, device="cuda")
    b.check(b.moe_gate_logits(c, tg["x"], tg.get("w_gate"), tg.get("w_noise"), tg.get("proj"), got, ws, ws.numel()),
            "moe_gate_logits")
    got = got.cpu().numpy().astype(np.float64)
    # the exact logits are the oracle's softmax-gate scores x W^T of each weight tensor
    want = np.concatenate([oracle.gate_scores("softmax", tc["x"], w_gate=w) for w in rows], axis=1)
    xa = np.abs(tc["x"].double().numpy())
    wa = np.abs(torch.cat(rows).double().numpy())
    scale = 2.0 ** -23 * (xa @ wa.T)
    return np.max(np.abs(got - want) / np.maximum(scale, 1e-300))


@pytest.mark.parametrize("gate,E,p,d,T", [("softmax", 8, 0, 1024, 300), ("noisy", 37, 0, 256, 200),
                                          ("cosine", 10, 256, 512, 129), ("softmax", 256, 0, 7168, 64),
                                          ("noisy", 64, 0, 320, 9733), ("cosine", 32, 256, 256, 4900),
                                          ("softmax", 100, 0, 256, 9500)])
def test_gate_logits_within_assumed_tensor_core_bound(gate, E, p, d, T):
    """The tensor-core logits GEMM against the exact products' sum: the routing step assumes
    |error| <= 64 * 2^-23 * sum |x_i w_i| and re-scores near ties inside twice that, so the observed
    error must sit well inside it (here: below an eighth of it).  The last two cases need more than one
    wave of 64-logit tiles, so the GEMM takes 128-logit tiles (the noisy gate's two weight tensors in one
    tile; the cosine projection in two; 100 softmax logits in one 112-wide tile, whose second column half
    is partly empty), with a ragged last token tile and an odd number of K blocks (d = 320: two two-block
    accumulator chunks and a one-block chunk)."""
    wl = small_workload(T=T, d=d, h=64, E=E, k=2, gate=gate, cos_dim=p or 32, capacity_factor=1.0)
    tc, tg = P.inputs(wl)
    ratio = _logits_error_ratio(wl, tc, tg)
    print("observed error / (2^-23 sum|x w|) = %.3e" % ratio)
    assert ratio < 8.0


def test_gate_logits_bound_under_cancellation():
    """Rows built so that the products cancel: each weight row is +-x of one token with signs chosen
    to keep the running sum near zero, the dot product is tiny next to sum |x_i w_i| and rounding in
    the accumulator shows at full strength."""
    wl = small_workload(T=128, d=1024, h=64, E=16, k=2, capacity_factor=1.0)
    tc, tg = P.inputs(wl)
    x = tc["x"].float()
    scale = torch.exp2(torch.randint(-6, 7, x.shape, generator=torch.Generator().manual_seed(5)).float())
    x = (x * scale).to(torch.bfloat16)
    w = torch.empty((wl.E, wl.d), dtype=torch.bfloat16)
    for e in range(wl.E):
        xr = x[e].double()
        run, signs = 0.0, []
        for v in (xr * xr).tolist():
            sg = -1.0 if run > 0 else 1.0
            run += sg * v
            signs.append(sg)
        w[e] = (xr * torch.tensor(signs, dtype=torch.float64)).to(torch.bfloat16)
    tc["x"], tc["w_gate"] = x, w
    tg["x"], tg["w_gate"] = x.cuda(), w.cuda()
    ratio = _logits_error_ratio(wl, tc, tg)
    print("cancellation: observed error / (2^-23 sum|x w|) = %.3e" % ratio)
    assert ratio < 8.0


PAIR_CASES = [wl for wl in SMALL if wl.dtype == "bf16"] + [
    small_workload(T=1500, d=128, h=512, E=3, k=2, capacity_factor=1.0),   # several 256-row tiles per expert
    small_workload(T=700, d=256, h=256, E=5, k=1, capacity_factor=2.0, bias="none"),
]


@pytest.mark.parametrize("wl", PAIR_CASES, ids=_id)
def test_expert_ffn_on_sm_pairs(wl):
    """The expert GEMMs on pairs of SMs (tcgen05 cta_group::2, 256 x 256 tiles), forced on small layers
    whose experts end in odd 128-row blocks (the upper half of their last tile is discarded)."""
    _full_check(wl, flags=b.FLAG_FFN_SM_PAIR)


def test_expert_ffn_single_sm_on_large_experts():
    """The single-SM expert GEMMs, forced on a layer that would use pairs by default."""
    _full_check(small_workload(T=2048, d=128, h=256, E=2, k=2, capacity_factor=1.0), flags=b.FLAG_FFN_ONE_SM)


def test_gelu_against_exact_erf():
    """The expert's GELU (erf via Abramowitz & Stegun 7.1.26 in the GEMM epilogue) against the exact
    erf GELU: a one-expert layer with x = 0, W1 = 0, b1 = z and W2 = I outputs bf16(GELU(z)) for every
    token, which must equal the exact value rounded to bf16 within one bf16 step (ties of the
    rounding), and lie within half a step plus 1e-6 of the exact value."""
    d = 2048
    wl = small_workload(T=64, d=d, h=d, E=1, k=1, norm="topk", capacity=64, bias="zero")
    tc, tg = P.inputs(wl)
    z = torch.linspace(-9.0, 9.0, d, dtype=torch.float64).to(torch.bfloat16)
    tg["x"] = torch.zeros_like(tg["x"])
    tg["w1"] = torch.zeros_like(tg["w1"])
    tg["b1"] = z.reshape(1, d).cuda()
    tg["w2"] = torch.eye(d, dtype=torch.bfloat16).reshape(1, d, d).cuda()
    tg["b2"] = torch.zeros_like(tg["b2"])
    out, _ = P.run_forward(wl, tg)
    zz = z.double()
    exact = (torch.nn.functional.gelu(zz, approximate="none")).numpy()
    want = torch.from_numpy(exact).to(torch.bfloat16).double().numpy()
    got = out[0]
    assert np.all(out == got[None, :])  # every token the same
    step = np.abs(np.spacing(want.astype(np.float32))) * 2 ** 16  # one bf16 step at each value
    step = np.maximum(step, 2.0 ** -133)
    assert np.all(np.abs(got - want) <= step + 1e-6)
    assert np.all(np.abs(got - exact) <= 0.5 * step + 1e-6)
    big = np.abs(exact) > 1e-3  # where the value is not lost in the absolute error bound
    assert np.mean(got[big] == want[big]) > 0.99  # rounds like the exact value almost everywhere
