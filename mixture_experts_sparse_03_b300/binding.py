"""Thin ctypes binding of libmoe_b300 (include/moe_b300.h), with the same function names.

Argument marshalling only: every step of the layer runs in the library's CUDA kernels.  Tensors are
torch CUDA tensors (their data pointers are passed); PyTorch provides device memory and streams.  The
library must have been built (``python -m mixture_experts_sparse_03_b300.build``); importing this
module without it raises immediately -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

from .inputs import Workload

_HERE = os.path.dirname(os.path.abspath(__file__))
# MOE_B300_LIB names another build of the same library (e.g. one compiled with different tuning macros)
LIB_PATH = os.environ.get("MOE_B300_LIB") or os.path.join(_HERE, "libmoe_b300.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "moe_b300.h")

MOE_OK = 0
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
          4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE_CHECK", 6: "MOE_ERR_DEVICE_TIMEOUT"}
GATE = {"softmax": 0, "noisy": 1, "cosine": 2}
NORM = {"all": 0, "topk": 1}
DTYPE = {"f32": 0, "bf16": 1}
FLAG_SIMT_FFN = 1
FLAG_UNFUSED_COMBINE = 2
FLAG_FFN_ONE_SM = 4
FLAG_FFN_SM_PAIR = 8
FLAG_RANK_MAJOR = 16
FLAG_ROUTER_STATS = 32


class MoEConfig(ctypes.Structure):
    """Mirror of ``moe_config``."""
    _fields_ = [
        ("tokens", ctypes.c_int32),
        ("model_dim", ctypes.c_int32),
        ("hidden_size_per_expert", ctypes.c_int32),
        ("num_experts", ctypes.c_int32),
        ("top_k", ctypes.c_int32),
        ("capacity", ctypes.c_int32),
        ("capacity_factor", ctypes.c_double),
        ("gate_type", ctypes.c_int32),
        ("gate_norm", ctypes.c_int32),
        ("cos_dim", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("cos_temperature", ctypes.c_double),
        ("flags", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        super().__init__("%s failed: %s (%d)" % (where or "moe call", STATUS.get(status, "?"), status))


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("libmoe_b300.so is not built at %s; run python -m mixture_experts_sparse_03_b300.build"
                          % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    C = ctypes.POINTER(MoEConfig)
    sigs = {
        "moe_capacity": ([C], I32),
        "moe_dispatch_rows": ([C], I64),
        "moe_workspace_size": ([C], SZ),
        "moe_forward_launches": ([C], I32),
        "moe_route": ([C, P, P, P, P, P, P, P, P, P, SZ, P], I32),
        "moe_gate_logits": ([C, P, P, P, P, P, P, SZ, P], I32),
        "moe_dispatch": ([C, P, P, P, P, P, P, P, P, P, P, SZ, P], I32),
        "moe_dispatch_static_scratch": ([C, P, P, P, P, P, P, P, P, P, P], I32),
        "moe_expert_ffn": ([C, P, P, P, P, P, P, P, P, P, P, P, SZ, P], I32),
        "moe_combine": ([C, P, P, P, P, P, P, P], I32),
        "moe_router_stats": ([C, P, P, P, P, P, P, P, SZ, P], I32),
        "moe_forward": ([C, P, P, P, P, P, P, P, P, P, P, P, P, P, SZ, P], I32),
        "moe_expert_ffn_fp8": ([C, P, P, P, P, P, P, P, P, P, P, P, P, P, SZ, P], I32),
        "moe_backward_workspace_size": ([C], SZ),
        "moe_router_stats_result": ([C, P, SZ, P, P, P, P], I32),
        "moe_backward": ([C] + [P] * 17 + [SZ, P], I32),
        "moe_forward_fp8": ([C, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, SZ, P], I32),
        "moe_device_status": ([P, SZ, ctypes.POINTER(I32), P], I32),
        "moe_trace_events": ([ctypes.POINTER(P), I32], None),
        "moe_trace_count": ([], I32),
        "moe_status_string": ([I32], ctypes.c_char_p),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes, fn.restype = args, res
    return lib


lib = _load()


def declared_functions():
    """Names of the functions include/moe_b300.h declares."""
    return re.findall(r"^MOE_API[^(]*?\b(moe_\w+)\s*\(", open(HEADER).read(), flags=re.M)


def config(wl: Workload, flags: int = 0, tokens: int | None = None) -> MoEConfig:
    """moe_config of a workload (optionally with another token count)."""
    c = MoEConfig()
    c.tokens = wl.T if tokens is None else tokens
    c.model_dim = wl.d
    c.hidden_size_per_expert = wl.h
    c.num_experts = wl.E
    c.top_k = wl.k
    c.capacity = wl.capacity
    c.capacity_factor = wl.capacity_factor
    c.gate_type = GATE[wl.gate]
    c.gate_norm = NORM[wl.norm]
    c.cos_dim = wl.cos_dim
    c.dtype = DTYPE[wl.dtype]
    c.cos_temperature = wl.temperature
    c.flags = flags | (FLAG_RANK_MAJOR if wl.priority == "rank" else 0)
    c.reserved = 0
    return c


def ptr(t):
    """Data pointer of a tensor (None -> NULL); an int is passed through as a raw address."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def stream_handle(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def check(status: int, where: str = "") -> None:
    if status != MOE_OK:
        raise MoEError(status, where)


# ---- the C functions, same names, tensors in ------------------------------------------------------
def moe_capacity(cfg: MoEConfig) -> int:
    return lib.moe_capacity(ctypes.byref(cfg))


def moe_dispatch_rows(cfg: MoEConfig) -> int:
    return lib.moe_dispatch_rows(ctypes.byref(cfg))


def moe_workspace_size(cfg: MoEConfig) -> int:
    return lib.moe_workspace_size(ctypes.byref(cfg))


def moe_forward_launches(cfg: MoEConfig) -> int:
    return lib.moe_forward_launches(ctypes.byref(cfg))


def moe_route(cfg, x, w_gate, w_noise, noise_eps, proj, expert_emb, topk_idx, topk_gate, workspace, workspace_bytes,
              stream=None) -> int:
    return lib.moe_route(ctypes.byref(cfg), ptr(x), ptr(w_gate), ptr(w_noise), ptr(noise_eps), ptr(proj),
                         ptr(expert_emb), ptr(topk_idx), ptr(topk_gate), ptr(workspace), workspace_bytes,
                         stream_handle(stream))


def moe_gate_logits(cfg, x, w_gate, w_noise, proj, logits, workspace, workspace_bytes, stream=None) -> int:
    return lib.moe_gate_logits(ctypes.byref(cfg), ptr(x), ptr(w_gate), ptr(w_noise), ptr(proj), ptr(logits),
                               ptr(workspace), workspace_bytes, stream_handle(stream))


def moe_dispatch(cfg, x, topk_idx, topk_gate, slot, expert_count, expert_offset, row_token, row_gate, x_dispatched,
                 workspace, workspace_bytes, stream=None) -> int:
    return lib.moe_dispatch(ctypes.byref(cfg), ptr(x), ptr(topk_idx), ptr(topk_gate), ptr(slot), ptr(expert_count),
                            ptr(expert_offset), ptr(row_token), ptr(row_gate), ptr(x_dispatched), ptr(workspace),
                            workspace_bytes, stream_handle(stream))


def moe_dispatch_static_scratch(cfg, x, topk_idx, topk_gate, slot, expert_count, expert_offset, row_token, row_gate,
                                x_dispatched, stream=None) -> int:
    return lib.moe_dispatch_static_scratch(ctypes.byref(cfg), ptr(x), ptr(topk_idx), ptr(topk_gate), ptr(slot),
                                           ptr(expert_count), ptr(expert_offset), ptr(row_token), ptr(row_gate),
                                           ptr(x_dispatched), stream_handle(stream))


def moe_expert_ffn(cfg, x_dispatched, expert_offset, row_token, row_gate, w1, b1, w2, b2, y_dispatched, out,
                   workspace, workspace_bytes, stream=None) -> int:
    return lib.moe_expert_ffn(ctypes.byref(cfg), ptr(x_dispatched), ptr(expert_offset), ptr(row_token),
                              ptr(row_gate), ptr(w1), ptr(b1), ptr(w2), ptr(b2), ptr(y_dispatched), ptr(out),
                              ptr(workspace), workspace_bytes, stream_handle(stream))


def moe_combine(cfg, y_dispatched, slot, expert_offset, topk_idx, topk_gate, out, stream=None) -> int:
    return lib.moe_combine(ctypes.byref(cfg), ptr(y_dispatched), ptr(slot), ptr(expert_offset), ptr(topk_idx),
                           ptr(topk_gate), ptr(out), stream_handle(stream))


def moe_router_stats(cfg, topk_idx, topk_gate, slot, importance, losses, dropped, workspace, workspace_bytes,
                     stream=None) -> int:
    return lib.moe_router_stats(ctypes.byref(cfg), ptr(topk_idx), ptr(topk_gate), ptr(slot), ptr(importance),
                                ptr(losses), ptr(dropped), ptr(workspace), workspace_bytes, stream_handle(stream))


def moe_forward(cfg, x, w_gate, w_noise, noise_eps, proj, expert_emb, w1, b1, w2, b2, out, expert_count, workspace,
                workspace_bytes, stream=None) -> int:
    return lib.moe_forward(ctypes.byref(cfg), ptr(x), ptr(w_gate), ptr(w_noise), ptr(noise_eps), ptr(proj),
                           ptr(expert_emb), ptr(w1), ptr(b1), ptr(w2), ptr(b2), ptr(out), ptr(expert_count),
                           ptr(workspace), workspace_bytes, stream_handle(stream))


def moe_expert_ffn_fp8(cfg, x_dispatched, expert_offset, row_token, row_gate, w1_q, w1_scale, b1, w2_q, w2_scale,
                       b2, y_dispatched, out, workspace, workspace_bytes, stream=None) -> int:
    return lib.moe_expert_ffn_fp8(ctypes.byref(cfg), ptr(x_dispatched), ptr(expert_offset), ptr(row_token),
                                  ptr(row_gate), ptr(w1_q), ptr(w1_scale), ptr(b1), ptr(w2_q), ptr(w2_scale), ptr(b2),
                                  ptr(y_dispatched), ptr(out), ptr(workspace), workspace_bytes, stream_handle(stream))


def moe_forward_fp8(cfg, x, w_gate, w_noise, noise_eps, proj, expert_emb, w1_q, w1_scale, b1, w2_q, w2_scale, b2,
                    out, expert_count, workspace, workspace_bytes, stream=None) -> int:
    return lib.moe_forward_fp8(ctypes.byref(cfg), ptr(x), ptr(w_gate), ptr(w_noise), ptr(noise_eps), ptr(proj),
                               ptr(expert_emb), ptr(w1_q), ptr(w1_scale), ptr(b1), ptr(w2_q), ptr(w2_scale), ptr(b2),
                               ptr(out), ptr(expert_count), ptr(workspace), workspace_bytes, stream_handle(stream))


def moe_router_stats_result(cfg, workspace, workspace_bytes, importance, losses, dropped, stream=None) -> int:
    return lib.moe_router_stats_result(ctypes.byref(cfg), ptr(workspace), workspace_bytes, ptr(importance), ptr(losses),
                                       ptr(dropped), stream_handle(stream))


def moe_backward_workspace_size(cfg: MoEConfig) -> int:
    return lib.moe_backward_workspace_size(ctypes.byref(cfg))


def moe_backward(cfg, x, w_gate, w_noise, noise_eps, w1, b1, w2, b2, dout, dx, dw_gate, dw_noise, dw1, db1, dw2, db2,
                 workspace, workspace_bytes, stream=None) -> int:
    return lib.moe_backward(ctypes.byref(cfg), ptr(x), ptr(w_gate), ptr(w_noise), ptr(noise_eps), ptr(w1), ptr(b1),
                            ptr(w2), ptr(b2), ptr(dout), ptr(dx), ptr(dw_gate), ptr(dw_noise), ptr(dw1), ptr(db1),
                            ptr(dw2), ptr(db2), ptr(workspace), workspace_bytes, stream_handle(stream))


def moe_device_status(workspace, workspace_bytes, stream=None):
    info = ctypes.c_int32(0)
    st = lib.moe_device_status(ptr(workspace), workspace_bytes, ctypes.byref(info), stream_handle(stream))
    return st, info.value


def moe_trace_events(events, capacity: int):
    """events: a list of torch.cuda.Event (or None to turn the hook off)."""
    if events is None:
        lib.moe_trace_events(None, 0)
        return None
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    lib.moe_trace_events(arr, capacity)
    return arr  # keep alive while tracing


def moe_trace_count() -> int:
    return lib.moe_trace_count()


def moe_status_string(status: int) -> str:
    return lib.moe_status_string(status).decode()


# ---- conveniences for tests and the benchmark (device memory via torch) ---------------------------
def workspace(cfg: MoEConfig, device="cuda") -> torch.Tensor:
    n = moe_workspace_size(cfg)
    if n == 0:
        raise MoEError(1, "moe_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def forward(cfg: MoEConfig, t: dict, out=None, expert_count=None, ws=None, stream=None) -> torch.Tensor:
    """moe_forward on the tensors of ``t`` (names as in inputs.make_inputs); returns out [T, d] fp32."""
    x = t["x"]
    if out is None:
        out = torch.empty((cfg.tokens, cfg.model_dim), dtype=torch.float32, device=x.device)
    if ws is None:
        ws = workspace(cfg, x.device)
    if t.get("w1_scale") is not None:  # block-FP8 expert weights
        check(moe_forward_fp8(cfg, x, t.get("w_gate"), t.get("w_noise"), t.get("eps"), t.get("proj"), t.get("emb"),
                              t["w1"], t["w1_scale"], t.get("b1"), t["w2"], t["w2_scale"], t.get("b2"), out,
                              expert_count, ws, ws.numel(), stream), "moe_forward_fp8")
        return out
    check(moe_forward(cfg, x, t.get("w_gate"), t.get("w_noise"), t.get("eps"), t.get("proj"), t.get("emb"), t["w1"],
                      t.get("b1"), t["w2"], t.get("b2"), out, expert_count, ws, ws.numel(), stream), "moe_forward")
    return out
