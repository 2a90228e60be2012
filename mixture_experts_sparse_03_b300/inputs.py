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

    def spec(self) -> dict:
        """The plain parameters the oracle and the C-ABI config need."""
        return dict(T=self.T, d=self.d, h=self.h, E=self.E, k=self.k, gate=self.gate, norm=self.norm,
                    capacity_factor=self.capacity_factor, capacity=self.capacity, dtype=self.dtype,
                    cos_dim=self.cos_dim, temperature=self.temperature)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def expert_weight_bytes(self) -> int:
        return 2 * self.E * self.h * self.d * (2 if self.dtype == "bf16" else 4)


# The five workloads: a tiny fp32 parity layer, the headline bf16 layer, noisy gating at scale,
# cosine gating with skewed load, and a decode-shaped fine-grained layer.
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
}
WORKLOAD_ORDER = ["tiny_fp32", "bf16_e8_k2", "bf16_noisy_e64", "bf16_cosine_skew", "bf16_decode_e256"]

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
    for n in ("w_gate", "w_noise", "eps", "proj", "emb"):
        t.setdefault(n, None)
    return t


def small_workload(T=97, d=64, h=128, E=5, k=2, gate="softmax", norm="topk", capacity_factor=1.0,
                   capacity=-1, dtype="bf16", cos_dim=32, temperature=0.07, bias="normal",
                   x_dist="normal", seed=11) -> Workload:
    """A small workload for parity tests that span a few tiles and a ragged tail."""
    return Workload("small", T=T, d=d, h=h, E=E, k=k, gate=gate, norm=norm, capacity_factor=capacity_factor,
                    capacity=capacity, dtype=dtype, cos_dim=cos_dim if gate == "cosine" else 0,
                    temperature=temperature if gate == "cosine" else 1.0, bias=bias, x_dist=x_dist,
                    seed=seed)
