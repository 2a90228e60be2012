"""The tensor cores' fp32 accumulation, as the routing step's error bound assumes it.

moe_route re-scores a token exactly when two of its scores lie within twice a bound on the logits'
error, and that bound rests on how tcgen05.mma (kind::f16, fp32 accumulator) adds exact bf16 products:
  - one MMA step adds 16 consecutive products of the reduction to the accumulator;
  - within a step every addend is aligned to the largest one's exponent e on a grid no coarser than
    2^(e-25), the aligned addends are summed exactly, and the sum is truncated to fp32 (error below
    one ulp of the result).
A step then errs by at most 17 * 2^-25 * max|addend| + 2^-23 |result|; the library starts a fresh
accumulator every 128-wide chunk of K (8 steps) and adds the chunks with compensated (Kahan) sums, which
bounds a logit's error by 44.5 * 2^-23 * sum|x_i w_i| (it assumes 64 * 2^-23).  These probes, dot products of exactly representable bf16
values through moe_gate_logits, check each part of that description on the GPU at hand."""
import pytest
import torch

from mixture_experts_sparse_03_b300 import binding as b
from mixture_experts_sparse_03_b300.inputs import small_workload

pytestmark = pytest.mark.gpu

D = 256  # two 128-wide accumulator chunks, sixteen MMA steps of 16


def _dots(rows):
    """x = all ones, so each logit is the plain sum of its weight row; rows: lists of (position, value)."""
    E = len(rows)
    wl = small_workload(T=1, d=D, h=64, E=E, k=1, capacity_factor=1.0)
    c = b.config(wl)
    ws = b.workspace(c, "cuda")
    w = torch.zeros((E, D), dtype=torch.float64)
    for e, r in enumerate(rows):
        for p, v in r:
            w[e, p] += v
    wb = w.to(torch.bfloat16)
    assert torch.equal(wb.double(), w), "probe values must be exact in bf16"
    x = torch.ones((1, D), dtype=torch.bfloat16, device="cuda")
    out = torch.full((1, E), float("nan"), device="cuda")
    b.check(b.moe_gate_logits(c, x, wb.cuda(), None, None, out, ws, ws.numel()), "moe_gate_logits")
    torch.cuda.synchronize()
    return out.cpu().double()[0].tolist()


def test_one_mma_step_adds_16_products():
    """Within one 128-wide chunk of K (one accumulator): 2^24 first, 1 at j, -2^24 last: the 1 survives
    only when it is added in the same step as -2^24 (else 2^24 + 1 is truncated to 2^24 first)."""
    for first, last in ((0, 63), (64, 127), (0, 127), (128, 255)):
        got = _dots([[(first, 2.0 ** 24), (j, 1.0), (last, -2.0 ** 24)] for j in range(first + 1, last)])
        first_same_step = last - last % 16
        assert got == [1.0 if j >= first_same_step else 0.0 for j in range(first + 1, last)]


def test_k_chunks_are_added_compensated():
    """Across 128-wide chunks of K the library adds the chunks' fp32 results with compensated sums: 2^24
    in the first chunk and 1 - 2^24 in the second sum to 1 exactly, wherever the 1 sits in the second
    chunk; in the first chunk the 1 is lost to the accumulator's truncation (2^24 + 1 -> 2^24)."""
    got = _dots([[(0, 2.0 ** 24), (j, 1.0), (255, -2.0 ** 24)] for j in range(1, 255)])
    assert got == [1.0 if j >= 128 else 0.0 for j in range(1, 255)]


def test_alignment_grid_within_a_step():
    """Inside one step, an addend 2^-24 or 2^-25 times the largest is kept exactly; one 2^-26 times it
    is lost.  So the grid is 2^(e-25)."""
    got = _dots([[(0, 2.0 ** 24), (5, 1.0), (10, -2.0 ** 24)],
                 [(0, 2.0 ** 25), (5, 1.0), (10, -2.0 ** 25)],
                 [(0, 2.0 ** 26), (5, 1.0), (10, -2.0 ** 26)],
                 [(0, 1.0)] + [(p, 2.0 ** -25) for p in range(1, 15)] + [(15, -1.0)]])
    assert got[0] == 1.0 and got[1] == 1.0 and got[2] == 0.0
    assert got[3] == 14 * 2.0 ** -25  # all fourteen small addends kept, summed exactly


def test_step_result_truncated_to_fp32():
    """1 + 0.75 ulp and 1 + 0.47 ulp (one step) become 1 and 1 + 0 ulp: truncation, error below one ulp;
    across steps the same."""
    u = 2.0 ** -23
    got = _dots([[(0, 1.0), (1, 0.75 * u)],
                 [(0, 1.0)] + [(p, 2.0 ** -25) for p in range(1, 16)],
                 [(0, 1.0), (16, 0.75 * u)],
                 [(0, 1.0), (16, 1.5 * u)]])
    assert got[0] == 1.0
    assert got[1] == 1.0 + 3 * u  # exact 1 + 3.75 ulp
    assert got[2] == 1.0
    assert got[3] == 1.0 + u
    for g, exact in zip(got, [1 + 0.75 * u, 1 + 3.75 * u, 1 + 0.75 * u, 1 + 1.5 * u]):
        assert 0 <= exact - g < u
