"""The re-scoring of the cosine gate orders a token's experts by x . (P^T e_j) / |e_j| instead of by
cos(u, e_j) / temperature with u = x P^T.  Since u . e_j = x . (P^T e_j) and |u| and the temperature are
common to all experts of a token, both orders are the same; this pins that reading on the CPU against
the oracle's fp64 cosine scores (no GPU)."""
import numpy as np
import torch

import oracle


def test_folded_projection_orders_experts_like_the_cosine_scores():
    g = torch.Generator().manual_seed(1234)
    T, d, p, E = 64, 96, 40, 12
    x = torch.randn(T, d, generator=g)
    proj = torch.randn(p, d, generator=g) / d ** 0.5
    emb = torch.randn(E, p, generator=g) / p ** 0.5
    emb[3] *= 7.0  # a long embedding: the norm division must be per expert
    scores = oracle.gate_scores("cosine", x, proj=proj, emb=emb, temperature=0.07)
    x64, p64, e64 = x.double(), proj.double(), emb.double()
    v = e64 @ p64                                           # [E, d]: v_j = P^T e_j
    folded = (x64 @ v.T) / e64.norm(dim=1).clamp_min(1e-12)  # [T, E]
    # same order on every token: the ratio to the oracle's score is one positive constant per token
    ratio = folded.numpy() / scores
    assert np.all(ratio > 0)
    assert np.allclose(ratio, ratio[:, :1], rtol=1e-10)
    assert np.array_equal(np.argsort(-folded.numpy(), axis=1, kind="stable"),
                          np.argsort(-scores, axis=1, kind="stable"))
