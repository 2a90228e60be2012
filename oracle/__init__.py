"""fp64 CPU oracle of the sparse MoE layer forward pass (ctypes wrapper around ``moe_oracle.c``).

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
import this package.  It shares no code with ``mixture_experts_sparse_03_b300`` and imports nothing
from it; the product path never calls it.

The C file holds the arithmetic (one function per step, each citing the page it follows); this module
only compiles it with gcc, marshals arrays and strings the steps together.  Tensors may be numpy
float32 arrays or CPU torch tensors of dtype float32 or bfloat16 (bf16 is passed as its raw 16-bit
pattern and widened exactly in C).

Module-level functions use the oracle built from ``moe_oracle.c``; ``Oracle(path)`` binds another
build of the same source (the mutation tests compile deliberately broken copies to check that the
pins catch them).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_moe_oracle.so")

GATE_SOFTMAX, GATE_NOISY, GATE_COSINE = 0, 1, 2
NORM_ALL, NORM_TOPK = 0, 1
F32, BF16, F64 = 0, 1, 2
_GATE_CODES = {"softmax": GATE_SOFTMAX, "noisy": GATE_NOISY, "cosine": GATE_COSINE}
_NORM_CODES = {"all": NORM_ALL, "topk": NORM_TOPK}
_PRIORITY_CODES = {"token": 0, "rank": 1}


def compile_source(src: str, out: str) -> str:
    """gcc -O2 (no fast-math, no FMA contraction) a copy of the oracle source into a shared object."""
    tmp = out + ".tmp%d" % os.getpid()
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, src, "-lm"],
                   check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into _moe_oracle.so beside it (if missing or older than the source)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(SOURCE):
        compile_source(SOURCE, _LIB_PATH)
    return _LIB_PATH


def _raw(t):
    """(numpy array holding the exact bits, dtype code) for a float32 / bfloat16 tensor or array."""
    if t is None:
        return None, None
    if hasattr(t, "detach"):  # torch tensor
        import torch

        t = t.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy(), BF16
        if t.dtype == torch.float32:
            return t.numpy(), F32
        raise TypeError("oracle tensors must be float32 or bfloat16, got %s" % t.dtype)
    a = np.ascontiguousarray(t)
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.float64:  # dequantised weights
        return a, F64
    raise TypeError("oracle numpy arrays must be float32 or float64 (pass bf16 as a torch tensor), got %s" % a.dtype)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _same_dtype(*pairs):
    codes = {c for _, c in pairs if c is not None}
    if len(codes) != 1:
        raise TypeError("x and all weights must share one dtype")
    return codes.pop()


def _x_and_weight_dtypes(xs, b1, b2, w1, w2):
    """(dtype of x and the biases, dtype of the two weight tensors): the same, or float64 weights
    (dequantised block-FP8) with any x dtype."""
    dt = _same_dtype(xs, b1, b2)
    wdt = _same_dtype(w1, w2)
    if wdt != dt and wdt != F64:
        raise TypeError("x and all weights must share one dtype")
    return dt, wdt


class Oracle:
    """The oracle's steps, bound to one compiled copy of moe_oracle.c."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        P, I, D, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_size_t
        sigs = {
            "oracle_gate_scores": ([I, I, I, I, I, D, I, P, P, P, P, P, P, P], None),
            "oracle_topk": ([I, I, I, I, P, P, P], None),
            "oracle_capacity": ([I, I, I, D, I], I),
            "oracle_dispatch": ([I, I, I, I, I, P, P, P], None),
            "oracle_expert": ([I, I, I, I, P, S, P, S, P, S, P, S, P, S, P], None),
            "oracle_combine_tokens": ([I, I, I, I, I, P, I, P, P, P, P, P, P, P, P, P], None),
            "oracle_dequant_block_fp8": ([I, I, I, P, P, P], None),
            "oracle_backward": ([I, I, I, I, I, I, I, I, I, I] + [P] * 16, None),
            "oracle_router_stats": ([I, I, I, P, P, P, P, P, P, P], None),
            "oracle_backward_sampled": ([I] * 8 + [P] * 13 + [I, P, P, I, P, P, P, I, P, P, P], None),
        }
        for name, (args, res) in sigs.items():
            fn = getattr(lib, name)
            fn.argtypes, fn.restype = args, res
        self.lib = lib
        self.path = path

    def gate_scores(self, gate, x, w_gate=None, w_noise=None, eps=None, proj=None, emb=None, temperature=1.0):
        """Step 1: selection scores [T, E] in float64."""
        g = _GATE_CODES[gate]
        xs = _raw(x)
        wg, wn, pj, em = _raw(w_gate), _raw(w_noise), _raw(proj), _raw(emb)
        dt = _same_dtype(xs, wg, wn, pj, em)
        T, d = xs[0].shape
        if g == GATE_COSINE:
            p, E = pj[0].shape[0], em[0].shape[0]
        else:
            p, E = 0, wg[0].shape[0]
        ep = None
        if g == GATE_NOISY:
            ep = eps.detach().cpu().numpy() if hasattr(eps, "detach") else eps
            ep = np.ascontiguousarray(ep, dtype=np.float32)
            assert ep.shape == (T, E)
        out = np.empty((T, E), dtype=np.float64)
        self.lib.oracle_gate_scores(g, T, d, E, p, float(temperature), dt, _ptr(xs[0]), _ptr(wg[0]),
                                    _ptr(wn[0]), _ptr(ep), _ptr(pj[0]), _ptr(em[0]), _ptr(out))
        return out

    def topk(self, scores, k, norm):
        """Step 2: (idx int32 [T, k] best first, gate float64 [T, k])."""
        s = np.ascontiguousarray(scores, dtype=np.float64)
        T, E = s.shape
        idx = np.empty((T, k), dtype=np.int32)
        gate = np.empty((T, k), dtype=np.float64)
        self.lib.oracle_topk(T, E, k, _NORM_CODES[norm], _ptr(s), _ptr(idx), _ptr(gate))
        return idx, gate

    def capacity(self, T, E, k, capacity_factor, capacity=-1):
        """Step 3a: the per-expert capacity C."""
        return int(self.lib.oracle_capacity(T, E, k, float(capacity_factor), int(capacity)))

    def dispatch(self, idx, E, C, priority="token"):
        """Step 3b: (slot int32 [T, k] or -1 if dropped, count int32 [E] before the limit).  priority:
        "token" (slots in token order) or "rank" (every token's first choice before any second choice)."""
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        T, k = idx.shape
        slot = np.empty((T, k), dtype=np.int32)
        count = np.empty((E,), dtype=np.int32)
        self.lib.oracle_dispatch(T, E, k, int(C), _PRIORITY_CODES[priority], _ptr(idx), _ptr(slot), _ptr(count))
        return slot, count

    def expert(self, x_row, w1_e, b1_e, w2_e, b2_e):
        """Step 4 for one token and one expert: float64 [d].  w1_e [h, d], w2_e [d, h]; the weights may
        be float64 (dequantised) while x and the biases keep their own dtype."""
        xs, a1, c1, a2, c2 = _raw(x_row), _raw(w1_e), _raw(b1_e), _raw(w2_e), _raw(b2_e)
        dt, wdt = _x_and_weight_dtypes(xs, c1, c2, a1, a2)
        h, d = a1[0].shape
        y = np.empty((d,), dtype=np.float64)
        self.lib.oracle_expert(d, h, dt, wdt, _ptr(xs[0]), 0, _ptr(a1[0]), 0, _ptr(c1[0]), 0, _ptr(a2[0]), 0,
                               _ptr(c2[0]), 0, _ptr(y))
        return y

    def combine_tokens(self, tokens, x, idx, gate, slot, w1, b1, w2, b2):
        """Steps 4+5 for the listed tokens: float64 [len(tokens), d]."""
        xs, a1, c1, a2, c2 = _raw(x), _raw(w1), _raw(b1), _raw(w2), _raw(b2)
        dt, wdt = _x_and_weight_dtypes(xs, c1, c2, a1, a2)
        E, h, d = a1[0].shape
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        gate = np.ascontiguousarray(gate, dtype=np.float64)
        slot = np.ascontiguousarray(slot, dtype=np.int32)
        k = idx.shape[1]
        out = np.empty((len(toks), d), dtype=np.float64)
        self.lib.oracle_combine_tokens(d, h, k, dt, wdt, _ptr(toks), len(toks), _ptr(xs[0]), _ptr(idx),
                                       _ptr(gate), _ptr(slot), _ptr(a1[0]), _ptr(c1[0]), _ptr(a2[0]),
                                       _ptr(c2[0]), _ptr(out))
        return out

    def dequant_block_fp8(self, q, scale, block=128):
        """Block-FP8 weights to float64: q holds E4M3 codes [..., rows, cols] (uint8 numpy array or a
        torch float8_e4m3fn / uint8 tensor), scale fp32 [..., ceil(rows/block), ceil(cols/block)]."""
        if hasattr(q, "detach"):
            import torch

            q = q.detach().cpu().contiguous()
            q = q.view(torch.uint8).numpy() if q.dtype != torch.uint8 else q.numpy()
        if hasattr(scale, "detach"):
            scale = scale.detach().cpu().numpy()
        q = np.ascontiguousarray(q, dtype=np.uint8)
        scale = np.ascontiguousarray(scale, dtype=np.float32)
        rows, cols = q.shape[-2:]
        lead = q.shape[:-2]
        qq = q.reshape((-1, rows, cols))
        ss = scale.reshape((qq.shape[0],) + scale.shape[-2:])
        assert ss.shape[1:] == (-(-rows // block), -(-cols // block)), (ss.shape, rows, cols, block)
        out = np.empty(qq.shape, dtype=np.float64)
        for i in range(qq.shape[0]):
            self.lib.oracle_dequant_block_fp8(rows, cols, block, _ptr(qq[i]), _ptr(ss[i]), _ptr(out[i]))
        return out.reshape(lead + (rows, cols))

    def backward(self, spec, t, dout):
        """Gradients of sum(dout * out) for the whole layer (softmax or noisy gate): a dict with dx [T, d],
        dw_gate [E, d], dw_noise [E, d] (noisy gate), dw1 [E, h, d], db1 [E, h], dw2 [E, d, h], db2 [E, d],
        all float64.  ``spec`` and ``t`` as for forward(); dout [T, d]."""
        gate = _GATE_CODES[spec["gate"]]
        if gate == GATE_COSINE:
            raise NotImplementedError("the oracle's backward covers the softmax and noisy gates")
        xs, wg, wn, a1, c1, a2, c2 = (_raw(t.get(n)) for n in ("x", "w_gate", "w_noise", "w1", "b1", "w2", "b2"))
        dt = _same_dtype(xs, wg, wn, a1, c1, a2, c2)
        T, d = xs[0].shape
        E, h, _ = a1[0].shape
        k = spec["k"]
        C = self.capacity(T, E, k, spec.get("capacity_factor", 1.0), spec.get("capacity", -1))
        ep = None
        if gate == GATE_NOISY:
            ep = t["eps"].detach().cpu().numpy() if hasattr(t["eps"], "detach") else t["eps"]
            ep = np.ascontiguousarray(ep, dtype=np.float32)
        go = dout.detach().cpu().numpy() if hasattr(dout, "detach") else dout
        go = np.ascontiguousarray(go, dtype=np.float64)
        out = dict(dx=np.empty((T, d)), dw_gate=np.empty((E, d)), dw1=np.empty((E, h, d)), db1=np.empty((E, h)),
                   dw2=np.empty((E, d, h)), db2=np.empty((E, d)))
        out["dw_noise"] = np.empty((E, d)) if gate == GATE_NOISY else None
        self.lib.oracle_backward(gate, _NORM_CODES[spec["norm"]], T, d, h, E, k, C,
                                 _PRIORITY_CODES[spec.get("priority", "token")], dt, _ptr(xs[0]), _ptr(wg[0]),
                                 _ptr(wn[0]), _ptr(ep), _ptr(a1[0]), _ptr(c1[0]), _ptr(a2[0]), _ptr(c2[0]), _ptr(go),
                                 _ptr(out["dx"]), _ptr(out["dw_gate"]), _ptr(out["dw_noise"]), _ptr(out["dw1"]),
                                 _ptr(out["db1"]), _ptr(out["dw2"]), _ptr(out["db2"]))
        return out

    def backward_sampled(self, spec, t, dout, tokens, s1, s2):
        """Single outputs of backward() for layers too large for the whole of it: dx rows of `tokens`,
        (dW1[e][n][m], db1[e][n]) for each (e, n, m) of s1 and (dW2[e][m][n], db2[e][m]) for each (e, m, n) of
        s2, all float64, from the whole layer's routing (scores, top-k, capacity dispatch).  Returns a dict
        with dx [len(tokens), d], dw1, db1 [len(s1)], dw2, db2 [len(s2)]."""
        gate = _GATE_CODES[spec["gate"]]
        if gate == GATE_COSINE:
            raise NotImplementedError("the oracle's backward covers the softmax and noisy gates")
        xs, wg, wn, a1, c1, a2, c2 = (_raw(t.get(n)) for n in ("x", "w_gate", "w_noise", "w1", "b1", "w2", "b2"))
        dt = _same_dtype(xs, wg, wn, a1, c1, a2, c2)
        T, d = xs[0].shape
        E, h, _ = a1[0].shape
        k = spec["k"]
        scores = self.gate_scores(spec["gate"], t["x"], t.get("w_gate"), t.get("w_noise"), t.get("eps"))
        idx, gw = self.topk(scores, k, spec["norm"])
        C = self.capacity(T, E, k, spec.get("capacity_factor", 1.0), spec.get("capacity", -1))
        slot, _ = self.dispatch(idx, E, C, spec.get("priority", "token"))
        ep = None
        if gate == GATE_NOISY:
            ep = t["eps"].detach().cpu().numpy() if hasattr(t["eps"], "detach") else t["eps"]
            ep = np.ascontiguousarray(ep, dtype=np.float32)
        go = dout.detach().cpu().numpy() if hasattr(dout, "detach") else dout
        go = np.ascontiguousarray(go, dtype=np.float64)
        tok = np.ascontiguousarray(tokens, dtype=np.int32)
        q1 = np.ascontiguousarray(np.asarray(s1, dtype=np.int32).reshape(-1, 3))
        q2 = np.ascontiguousarray(np.asarray(s2, dtype=np.int32).reshape(-1, 3))
        out = dict(dx=np.empty((len(tok), d)), dw1=np.empty(len(q1)), db1=np.empty(len(q1)), dw2=np.empty(len(q2)),
                   db2=np.empty(len(q2)))
        self.lib.oracle_backward_sampled(gate, _NORM_CODES[spec["norm"]], T, d, h, E, k, dt, _ptr(xs[0]), _ptr(wg[0]),
                                         _ptr(wn[0]), _ptr(ep), _ptr(a1[0]), _ptr(c1[0]), _ptr(a2[0]), _ptr(c2[0]),
                                         _ptr(go), _ptr(scores), _ptr(idx), _ptr(gw), _ptr(slot), len(tok), _ptr(tok),
                                         _ptr(out["dx"]), len(q1), _ptr(q1), _ptr(out["dw1"]), _ptr(out["db1"]),
                                         len(q2), _ptr(q2), _ptr(out["dw2"]), _ptr(out["db2"]))
        out.update(idx=idx, slot=slot)
        return out

    def router_stats(self, idx, gate, E, slot=None):
        """Router statistics: (importance float64 [E], expert_importance_loss, load_balance_loss, dropped)."""
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        gate = np.ascontiguousarray(gate, dtype=np.float64)
        T, k = idx.shape
        imp = np.empty((E,), dtype=np.float64)
        il, lb = ctypes.c_double(), ctypes.c_double()
        dropped = ctypes.c_int64()
        sl = None if slot is None else np.ascontiguousarray(slot, dtype=np.int32)
        self.lib.oracle_router_stats(T, E, k, _ptr(idx), _ptr(gate), _ptr(sl) if sl is not None else None,
                                     _ptr(imp), ctypes.byref(il), ctypes.byref(lb), ctypes.byref(dropped))
        return imp, il.value, lb.value, int(dropped.value)

    def route(self, gate, k, norm, x, w_gate=None, w_noise=None, eps=None, proj=None, emb=None,
              temperature=1.0):
        """Steps 1+2: (scores, idx, gate)."""
        s = self.gate_scores(gate, x, w_gate, w_noise, eps, proj, emb, temperature)
        idx, g = self.topk(s, k, norm)
        return s, idx, g

    def forward(self, spec, t, tokens=None):
        """Whole layer.  ``spec``: mapping with gate, norm, k, E, capacity_factor, capacity,
        temperature and optionally priority ("token" or "rank"); ``t``: mapping of tensors x, w_gate, w_noise, eps, proj, emb, w1, b1, w2, b2
        (absent -> None).  Returns a dict with scores, idx, gate, C, slot, count, tokens and out
        ([len(tokens), d])."""
        s, idx, g = self.route(spec["gate"], spec["k"], spec["norm"], t.get("x"), t.get("w_gate"),
                               t.get("w_noise"), t.get("eps"), t.get("proj"), t.get("emb"),
                               spec.get("temperature", 1.0))
        T = s.shape[0]
        C = self.capacity(T, spec["E"], spec["k"], spec.get("capacity_factor", 1.0), spec.get("capacity", -1))
        slot, count = self.dispatch(idx, spec["E"], C, spec.get("priority", "token"))
        if tokens is None:
            tokens = np.arange(T, dtype=np.int32)
        out = self.combine_tokens(tokens, t.get("x"), idx, g, slot, t.get("w1"), t.get("b1"), t.get("w2"),
                                  t.get("b2"))
        return dict(scores=s, idx=idx, gate=g, C=C, slot=slot, count=count, tokens=np.asarray(tokens), out=out)


_lock = threading.Lock()
_default = None


def default() -> Oracle:
    """The oracle compiled from moe_oracle.c (built on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def gate_scores(*a, **kw):
    return default().gate_scores(*a, **kw)


def topk(*a, **kw):
    return default().topk(*a, **kw)


def capacity(*a, **kw):
    return default().capacity(*a, **kw)


def dispatch(*a, **kw):
    return default().dispatch(*a, **kw)


def expert(*a, **kw):
    return default().expert(*a, **kw)


def combine_tokens(*a, **kw):
    return default().combine_tokens(*a, **kw)


def router_stats(*a, **kw):
    return default().router_stats(*a, **kw)


def dequant_block_fp8(*a, **kw):
    return default().dequant_block_fp8(*a, **kw)


def backward(*a, **kw):
    return default().backward(*a, **kw)


def backward_sampled(*a, **kw):
    return default().backward_sampled(*a, **kw)


def route(*a, **kw):
    return default().route(*a, **kw)


def forward(*a, **kw):
    return default().forward(*a, **kw)
