"""moe_dispatch_static_scratch: the dispatch for callers that cannot allocate device memory.

Such callers (code inside another framework's memory pool or a plugin host, programs that must not
allocate after start-up) pass only inputs and outputs; the scratch lives in a fixed array inside the
library.  These tests call it through the C ABI and require the same results as moe_dispatch with a
caller workspace, on consecutive calls that reuse the shared array.  The file sorts last so that a run
stopping at its first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from mixture_experts_sparse_03_b300 import binding as b
from mixture_experts_sparse_03_b300.inputs import make_inputs, small_workload

MAX_HIST = 262080  # MOE_DISPATCH_STATIC_MAX_HIST


def test_rejects_sizes_beyond_the_static_scratch():
    """ceil(T/32) * E above the array's capacity is refused on the host, before any CUDA call."""
    wl = small_workload(T=65536, d=64, h=64, E=128, k=2)
    c = b.config(wl)
    assert (65536 // 32) * 128 > MAX_HIST
    st = b.lib.moe_dispatch_static_scratch(ctypes.byref(c), None, None, None, None, None, None, None, None, None,
                                           None)
    assert st == 2  # MOE_ERR_UNSUPPORTED
    wl_ok = small_workload(T=65536, d=64, h=64, E=127, k=2)
    assert (65536 // 32) * 127 <= MAX_HIST
    st = b.lib.moe_dispatch_static_scratch(ctypes.byref(b.config(wl_ok)), None, None, None, None, None, None, None,
                                           None, None, None)
    assert st == 1  # within the limit: now the NULL pointers are the error


def _dispatch_outputs(c, x, rows, dev):
    T, k, E, d = c.tokens, c.top_k, c.num_experts, c.model_dim
    return dict(
        slot=torch.full((T, k), -7, dtype=torch.int32, device=dev),
        count=torch.full((E,), -7, dtype=torch.int32, device=dev),
        off=torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
        rtok=torch.full((rows,), -7, dtype=torch.int32, device=dev),
        rgate=torch.full((rows,), -3.0, dtype=torch.float32, device=dev),
        xd=torch.zeros((rows, d), dtype=x.dtype, device=dev),
    )


def _route(c, t, ws, dev):
    T, k = c.tokens, c.top_k
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    gate = torch.empty((T, k), dtype=torch.float32, device=dev)
    b.check(b.moe_route(c, t["x"], t.get("w_gate"), t.get("w_noise"), t.get("eps"), t.get("proj"), t.get("emb"),
                        idx, gate, ws, ws.numel()), "moe_route")
    return idx, gate


@pytest.mark.gpu
def test_static_scratch_dispatch_matches_workspace_dispatch():
    dev = torch.device("cuda", 0)
    cases = [
        small_workload(T=1000, d=128, h=64, E=6, k=2, capacity_factor=1.0),          # drops, ragged last block
        small_workload(T=777, d=192, h=64, E=37, k=3, gate="noisy", capacity_factor=0.8),
        small_workload(T=500, d=128, h=64, E=9, k=2, capacity_factor=0.8, priority="rank"),  # slots in rank order
    ]
    for i, wl in enumerate(cases):  # two calls in a row: the second reuses the array the first left dirty
        tg = {n: (v.to(dev) if v is not None else None) for n, v in make_inputs(wl, device="cpu").items()}
        c = b.config(wl)
        rows = b.moe_dispatch_rows(c)
        ws = b.workspace(c, dev)
        idx, gate = _route(c, tg, ws, dev)
        want = _dispatch_outputs(c, tg["x"], rows, dev)
        b.check(b.moe_dispatch(c, tg["x"], idx, gate, want["slot"], want["count"], want["off"], want["rtok"],
                               want["rgate"], want["xd"], ws, ws.numel()), "moe_dispatch")
        got = _dispatch_outputs(c, tg["x"], rows, dev)
        b.check(b.moe_dispatch_static_scratch(c, tg["x"], idx, gate, got["slot"], got["count"], got["off"],
                                              got["rtok"], got["rgate"], got["xd"]), "moe_dispatch_static_scratch")
        torch.cuda.synchronize()
        st, _ = b.moe_device_status(ws, ws.numel())
        assert st == b.MOE_OK
        for n in ("slot", "count", "off", "rtok", "rgate", "xd"):
            assert torch.equal(got[n], want[n]), "case %d: %s differs" % (i, n)
        assert int((got["slot"] < 0).sum()) > 0, "case %d should drop some pairs" % i
        assert np.array_equal(got["count"].cpu().numpy(),
                              np.bincount(idx.cpu().numpy().ravel(), minlength=wl.E))
