"""Seeded synthetic inputs for the sparse MoE layer forward pass.

This module holds no arithmetic of the method.  It defines the workloads (shapes, seeds, value
distributions) and draws their tensors; both the CUDA path's tests and benchmark and the oracle's
tests take their inputs from here.

Distributions (the workloads' own recipe): x ~ N(0, 1); every weight ~ N(0, 1/fan_in) (std
fan_in^-1/2; fan_in = d for W_g, W_n, P and W1, h for W2, cos_dim for the expert embeddings); biases 0
where a workload has them; eps ~ N(0, 1) fp32 [T, E] for the noisy gate; for the skewed cosine workload
x is drawn from 4 Gaussian clusters with means ~ N(0, 4 I), mixing weights 0.55 / 0.25 / 0.15 / 0.05
and unit within-cluster covariance.  Values are drawn in fp32 and rounded to bf16 (round to nearest
even) for bf16 workloads.

Every tensor has its own generator, seeded from (workload seed, tensor tag, expert id), so any one
expert's weights can be re-drawn alone.  Tensors are drawn on the CPU generator, except expert weights
of workloads whose expert weights exceed 1 GiB, which are drawn by torch's seeded CUDA generator on
the GPU (the oracle then reads host copies of those exact values).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

# tags: one per tensor, fixed forever (changing one changes every input of every workload)
_TAG = {"x": 1, "w_gate": 2, "w_noise": 3, "eps": 4, "proj": 5, "emb": 6, "w1": 7, "b1": 8, "w2": 9,
        "b2": 10, "cluster_mean": 11, "cluster_id": 12}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    h: int
    E: int
    k: int
    gate: str = "softmax"       # softmax | noisy | cosine
    norm: str = "topk"          # all | topk
    capacity_factor: float = 1.2
    capacity: int = -1          # -1: from capacity_factor; T: dropless
    dtype: str = "bf16"         # bf16 | f32
    cos_dim: int = 0
    temperature: float = 1.0
    bias: str = "none"          # none | zero | normal
    x_dist: str = "normal"      # normal | clusters
    seed: int = 0
    priority: str = "token"     # capacity slots in token order | rank order (first choices first)
    weights: str = "dense"      # dense (the workload dtype) | fp8_block (E4M3 codes + 128 x 128 fp32 scales)

    def spec(self) -> dict:
        """The plain parameters the oracle and the C-ABI config need."""
        return dict(T=self.T, d=self.d, h=self.h, E=self.E, k=self.k, gate=self.gate, norm=self.norm,
                    capacity_factor=self.capacity_factor, capacity=self.capacity, dtype=self.dtype,
                    cos_dim=self.cos_dim, temperature=self.temperature, priority=self.priority)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def expert_weight_bytes(self) -> int:
        """Bytes of the expert weights as the layer reads them."""
        if self.weights == "fp8_block":
            return 2 * self.E * self.h * self.d + 2 * self.E * (self.h // 128) * (self.d // 128) * 4
        return 2 * self.E * self.h * self.d * (2 if self.dtype == "bf16" else 4)


# The workloads: a tiny fp32 parity layer, a bf16 top-2 layer, noisy gating at scale, cosine gating with
# skewed load, a decode-shaped fine-grained layer (bf16 and block-FP8 weights), and a small-d recommender
# layer.
WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", T=256, d=64, h=256, E=4, k=1, gate="softmax", norm="all",
                          capacity_factor=1.2, dtype="f32", bias="zero", seed=0),
    "bf16_e8_k2": Workload("bf16_e8_k2", T=4096, d=1024, h=2048, E=8, k=2, gate="softmax", norm="topk",
                           capacity_factor=1.2, seed=1),
    "bf16_noisy_e64": Workload("bf16_noisy_e64", T=16384, d=2048, h=8192, E=64, k=2, gate="noisy",
                               norm="topk", capacity_factor=1.5, seed=2),
    "bf16_cosine_skew": Workload("bf16_cosine_skew", T=8192, d=1024, h=2048, E=32, k=2, gate="cosine",
                                 norm="topk", capacity_factor=1.2, cos_dim=256, temperature=0.07,
                                 x_dist="clusters", seed=3),
    "bf16_decode_e256": Workload("bf16_decode_e256", T=64, d=7168, h=2048, E=256, k=8, gate="softmax",
                                 norm="topk", capacity=64, seed=4),
    # the recommender layer of the "Tutel MoE guide" (cosine_top gate over 128-wide user embeddings,
    # 8 experts, top-2, capacity_factor 1.5 from its tips), expert FFN 128 -> 512 -> 128 (4x, as in
    # CANN's MOELayer example); x ~ N(0, 1) like a freshly initialised embedding table; capacity slots
    # in rank order (first choices first)
    "bf16_recsys_e8": Workload("bf16_recsys_e8", T=8192, d=128, h=512, E=8, k=2, gate="cosine", norm="topk",
                               capacity_factor=1.5, cos_dim=256, temperature=0.07, seed=5, priority="rank"),
    # the decode-shaped layer with block-FP8 expert weights (the same draws, rounded to E4M3 with a
    # power-of-two scale per 128 x 128 block): half the bytes of the HBM-bound expert GEMMs
    "bf16_decode_e256_fp8": Workload("bf16_decode_e256_fp8", T=64, d=7168, h=2048, E=256, k=8, gate="softmax",
                                     norm="topk", capacity=64, seed=4, weights="fp8_block"),
}
WORKLOAD_ORDER = ["tiny_fp32", "bf16_e8_k2", "bf16_noisy_e64", "bf16_cosine_skew", "bf16_decode_e256",
                  "bf16_recsys_e8", "bf16_decode_e256_fp8"]

CLUSTER_WEIGHTS = (0.55, 0.25, 0.15, 0.05)


def _seed(seed: int, tag: str, sub: int = 0) -> int:
    return ((seed & 0xFFFF) << 40) | (_TAG[tag] << 24) | (sub & 0xFFFFFF)


def _gen(device: str, seed: int, tag: str, sub: int = 0) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_seed(seed, tag, sub))
    return g


def _normal(shape, std: float, seed: int, tag: str, sub: int = 0, device: str = "cpu") -> torch.Tensor:
    g = _gen(device, seed, tag, sub)
    v = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        v.mul_(std)
    return v


def draw_x(wl: Workload) -> torch.Tensor:
    """Token activations [T, d] in the workload dtype (CPU)."""
    if wl.x_dist == "normal":
        x = _normal((wl.T, wl.d), 1.0, wl.seed, "x")
    elif wl.x_dist == "clusters":
        means = _normal((len(CLUSTER_WEIGHTS), wl.d), 2.0, wl.seed, "cluster_mean")
        g = _gen("cpu", wl.seed, "cluster_id")
        cid = torch.multinomial(torch.tensor(CLUSTER_WEIGHTS, dtype=torch.float64), wl.T,
                                replacement=True, generator=g)
        x = means[cid] + _normal((wl.T, wl.d), 1.0, wl.seed, "x")
    else:
        raise ValueError(wl.x_dist)
    return x.to(wl.torch_dtype)


def _expert_stack(wl: Workload, tag: str, rows: int, cols: int, std: float, device: str) -> torch.Tensor:
    """[E, rows, cols] with each expert drawn from its own generator."""
    out = torch.empty((wl.E, rows, cols), dtype=wl.torch_dtype, device=device)
    for e in range(wl.E):
        out[e] = _normal((rows, cols), std, wl.seed, tag, e, device=device).to(wl.torch_dtype)
    return out


def quantize_block_fp8(w: torch.Tensor, block: int = 128):
    """Block-FP8 form of weights w [..., rows, cols] (rows, cols multiples of `block`): every block x
    block tile gets the power-of-two scale 2^ceil(log2(amax / 448)) (448 = the largest E4M3 value; 1 for
    an all-zero tile) and its elements become E4M3 codes of w / scale, rounded to nearest even.  Returns
    (codes as torch.float8_e4m3fn, scales fp32 [..., rows/block, cols/block]).  This prepares the
    workload's weights; the layer itself only ever dequantises."""
    *lead, R, C = w.shape
    wf = w.float().reshape(-1, R // block, block, C // block, block)
    amax = wf.abs().amax(dim=(2, 4))
    mant, ex = torch.frexp(amax / 448.0)  # amax / 448 = mant * 2^ex, mant in [0.5, 1)
    ex = torch.where(mant == 0.5, ex - 1, ex)  # an exact power of two needs no extra factor
    scale = torch.where(amax > 0, torch.ldexp(torch.ones_like(amax), ex), torch.ones_like(amax))
    q = (wf / scale[:, :, None, :, None]).to(torch.float8_e4m3fn)
    return q.reshape(w.shape), scale.reshape(*lead, R // block, C // block).contiguous()


def make_inputs(wl: Workload, device: Optional[str] = None, expert_device: Optional[str] = None) -> dict:
    """All tensors of a workload.  Non-expert tensors are drawn on the CPU and moved to ``device``;
    expert weights are drawn on ``expert_device`` (default: the GPU when the workload's expert weights
    exceed 1 GiB and a GPU is present, else the CPU) and placed on ``device``."""
    device = device or "cpu"
    if expert_device is None:
        big = wl.expert_weight_bytes() > (1 << 30)
        expert_device = "cuda" if (big and torch.cuda.is_available()) else "cpu"
    dt = wl.torch_dtype
    t = {"x": draw_x(wl)}
    if wl.gate in ("softmax", "noisy"):
        t["w_gate"] = _normal((wl.E, wl.d), wl.d ** -0.5, wl.seed, "w_gate").to(dt)
    if wl.gate == "noisy":
        t["w_noise"] = _normal((wl.E, wl.d), wl.d ** -0.5, wl.seed, "w_noise").to(dt)
        t["eps"] = _normal((wl.T, wl.E), 1.0, wl.seed, "eps")
    if wl.gate == "cosine":
        t["proj"] = _normal((wl.cos_dim, wl.d), wl.d ** -0.5, wl.seed, "proj").to(dt)
        t["emb"] = _normal((wl.E, wl.cos_dim), wl.cos_dim ** -0.5, wl.seed, "emb").to(dt)
    t = {n: v.to(device) for n, v in t.items()}
    if wl.weights == "fp8_block":  # the dense draws, quantised one expert at a time
        for n, rows, cols, fan in (("w1", wl.h, wl.d, wl.d), ("w2", wl.d, wl.h, wl.h)):
            q = torch.empty((wl.E, rows, cols), dtype=torch.float8_e4m3fn, device=expert_device)
            sc = torch.empty((wl.E, rows // 128, cols // 128), dtype=torch.float32, device=expert_device)
            for e in range(wl.E):
                w = _normal((rows, cols), fan ** -0.5, wl.seed, n, e, device=expert_device).to(wl.torch_dtype)
                q[e], sc[e] = quantize_block_fp8(w)
            t[n], t[n + "_scale"] = q.to(device), sc.to(device)
    else:
        t["w1"] = _expert_stack(wl, "w1", wl.h, wl.d, wl.d ** -0.5, expert_device).to(device)
        t["w2"] = _expert_stack(wl, "w2", wl.d, wl.h, wl.h ** -0.5, expert_device).to(device)
    if wl.bias == "zero":
        t["b1"] = torch.zeros((wl.E, wl.h), dtype=dt, device=device)
        t["b2"] = torch.zeros((wl.E, wl.d), dtype=dt, device=device)
    elif wl.bias == "normal":
        t["b1"] = _normal((wl.E, wl.h), 0.5, wl.seed, "b1").to(dt).to(device)
        t["b2"] = _normal((wl.E, wl.d), 0.5, wl.seed, "b2").to(dt).to(device)
    else:
        t["b1"] = None
        t["b2"] = None
    for n in ("w_gate", "w_noise", "eps", "proj", "emb", "w1_scale", "w2_scale"):
        t.setdefault(n, None)
    return t


def small_workload(T=97, d=64, h=128, E=5, k=2, gate="softmax", norm="topk", capacity_factor=1.0,
                   capacity=-1, dtype="bf16", cos_dim=32, temperature=0.07, bias="normal",
                   x_dist="normal", seed=11, priority="token", weights="dense") -> Workload:
    """A small workload for parity tests that span a few tiles and a ragged tail."""
    return Workload("small", T=T, d=d, h=h, E=E, k=k, gate=gate, norm=norm, capacity_factor=capacity_factor,
                    capacity=capacity, dtype=dtype, cos_dim=cos_dim if gate == "cosine" else 0,
                    temperature=temperature if gate == "cosine" else 1.0, bias=bias, x_dist=x_dist,
                    seed=seed, priority=priority, weights=weights)
