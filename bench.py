"""Benchmark of the sparse MoE layer forward pass on B300 (one JSON line on rank 0).

A step is one moe_forward (gate -> top-k -> capacity dispatch -> grouped Linear-GELU-Linear -> combine)
over one batch of synthetic tokens already resident in HBM, replayed from a CUDA graph.  Between timed
steps a 256 MiB buffer is written to flush the 126 MB L2.  Each step is timed with CUDA events on the
launching stream; `value` = tokens processed by all ranks / the slowest rank's summed step time.

The default workload is the largest layer that fits one GPU (noisy top-2 gating over 64 experts,
T = 16384, d = 2048, h = 8192).  Per-kernel durations come from a second graph of the same step whose
launches are separated by event-record nodes (the library's trace hook under stream capture), so they
hold no host launch gaps.  The other four workloads are measured the same way (graph-timed step and
per-kernel split, no end-to-end leg) and reported under "workloads" unless --only is given.

  --impl ours (default)   the CUDA library through its C ABI
  --impl reference        the fp64 CPU oracle on the host cores (bounded samples; rank 0 only)

With torchrun (--gpus N > 1) every rank runs an independent replica of the layer on its own GPU
(the layer's one-GPU path has no exchange step); the ranks only meet for a barrier and the max-time
reduction.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mixture_experts_sparse_03_b300.inputs import WORKLOAD_ORDER, WORKLOADS, make_inputs  # noqa: E402

METRIC = "MoE layer fwd tokens/s on 1 B300; % of bf16 TC peak or HBM roofline"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "bf16_noisy_e64"
FLUSH_BYTES = 256 << 20
RIDGE_ROWS = 268  # bf16: FLOP per expert-weight byte = rows per expert; ridge = peak FLOP/s / HBM B/s


def kernel_names(wl, launches: int):
    """Names of the kernels moe_forward launches, in launch order (the softmax gate of a bf16 layer with
    E <= 64 runs as one fused launch)."""
    rank = getattr(wl, "priority", "token") == "rank"  # slots in rank order: a separate rank kernel
    if wl.dtype == "bf16" and wl.gate == "softmax" and wl.E <= 64:
        if rank:
            names = ["gate_fused_gemm_topk", "dispatch_rank_scan", "dispatch_gather", "expert_up_gelu"]
        elif -(-wl.T // 32) * wl.E <= 2048:  # a small histogram: the gather scans it (per CTA)
            names = ["gate_fused_gemm_topk", "dispatch_scan_gather", "expert_up_gelu"]
        else:
            names = ["gate_fused_gemm_topk_scan", "dispatch_gather", "expert_up_gelu"]
    elif wl.dtype == "bf16":
        names = ["gate_logits_gemm", "gate_topk"] + (["gate_cos_fold"] if wl.gate == "cosine" else [])
        names += ["gate_rescore", "dispatch_rank_scan", "dispatch_gather", "expert_up_gelu"]
    elif rank:
        names = ["gate_topk", "dispatch_rank_scan", "dispatch_gather", "expert_up_gelu"]
    else:
        names = ["gate_topk_scan", "dispatch_gather", "expert_up_gelu"]
    names += ["expert_down_combine"] if wl.k <= 2 else ["expert_down", "combine_gather"]
    if len(names) != launches:
        raise RuntimeError("moe_forward launches %d kernels, expected %d" % (launches, len(names)))
    return names


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-graph", action="store_true", help="time eager launches instead of a CUDA graph")
    ap.add_argument("--ffn", choices=["auto", "one-sm", "sm-pair"], default="auto",
                    help="expert GEMMs on single SMs or on pairs of SMs (default: the library's choice)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="target CPU time of the oracle sample")
    ap.add_argument("--only", action="store_true", help="measure the chosen workload only (no 'workloads' key)")
    ap.add_argument("--skip-backward", action="store_true",
                    help="profiling aid: leave out the backward timing (its CUDA-graph replay)")
    ap.add_argument("--experts", type=int, default=0,
                    help="profiling aid: the chosen workload with this many experts and T scaled to keep the rows "
                         "per expert (the same per-expert GEMM shapes on a smaller device footprint); implies --only")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sustained=d["bf16_tflops_sustained"],
                    source="measured")
    return dict(hbm=6400.0, bf16=1800.0, bf16_sustained=1400.0, source="fallback")


def layer_work(wl, kept_pairs: int, experts_used: int):
    """Algorithmic work of one forward: FLOPs of the kept (token, expert) pairs through both expert
    GEMMs plus the gate GEMM, and the expert-weight bytes the used experts occupy."""
    gemm = 2.0 * kept_pairs * wl.d * wl.h  # one of the two expert GEMMs
    if wl.gate == "softmax":
        gate = 2.0 * wl.T * wl.d * wl.E
    elif wl.gate == "noisy":
        gate = 4.0 * wl.T * wl.d * wl.E
    else:
        gate = 2.0 * wl.T * wl.d * wl.cos_dim + 2.0 * wl.T * wl.cos_dim * wl.E
    wbytes = experts_used * (wl.expert_weight_bytes() // wl.E)  # both matrices (block-FP8: codes + scales)
    return gemm, gate, wbytes


# ----------------------------------------------------------------------------------- replicas (N > 1)
def max_over_ranks(value: float, device=None) -> float:
    """The largest `value` over all ranks of the default process group (the value itself when no group
    is initialised).  Each rank runs an independent replica of the layer; the slowest one sets the time."""
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, steps: int, tokens: int, max_total_ms: float) -> float:
    """Whole-job tokens/s: the tokens every rank processed over the slowest rank's summed step time."""
    return world * steps * tokens / (max_total_ms / 1e3)


# ------------------------------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.out = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            sel = []
        # a 20 ms period: a timed region of a few tens of milliseconds still gets a handful of samples
        self.cmd = ["nvidia-smi", *sel, "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits", "-lms", "20"]

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------------- CPU oracle
def cpu_model() -> str:
    """The host CPU's model name (from /proc/cpuinfo)."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


class OneCore:
    """Pin the calling thread to one host core for the length of the block (the oracle is single-threaded
    C called from this thread), then restore the previous affinity mask."""

    def __init__(self):
        self.old = None
        self.core = None

    def __enter__(self):
        try:
            self.old = os.sched_getaffinity(0)
            self.core = min(self.old)
            os.sched_setaffinity(0, {self.core})
        except (AttributeError, OSError):
            self.old, self.core = None, None
        return self

    def __exit__(self, *exc):
        if self.old is not None:
            os.sched_setaffinity(0, self.old)
        return False


def oracle_prefix(wl, tc, n: int):
    """The oracle's whole layer (scores, top-k, capacity dispatch, expert FFN, combine) on the first n
    tokens of the workload, with the full workload's capacity.  With slots in token order a prefix's
    slots and outputs are exactly the full layer's for those tokens; in rank order they are a sample of
    the same work."""
    import oracle

    sl = (lambda t: None if t is None else t[:n])
    scores = oracle.gate_scores(wl.gate, tc["x"][:n], tc["w_gate"], tc["w_noise"], sl(tc["eps"]), tc["proj"],
                                tc["emb"], wl.temperature)
    idx, gate = oracle.topk(scores, wl.k, wl.norm)
    C = oracle.capacity(wl.T, wl.E, wl.k, wl.capacity_factor, wl.capacity)
    slot, _ = oracle.dispatch(idx, wl.E, C, wl.priority)
    return oracle.combine_tokens(np.arange(n, dtype=np.int32), tc["x"], idx, gate, slot, tc["w1"], tc["b1"],
                                 tc["w2"], tc["b2"])


def cpu_oracle_sample(wl, tc, seconds: float):
    """Time the oracle (as it stands: single-threaded C, fp64) on one host core over a bounded sample
    of the workload: the whole layer for the first n tokens, n sized to about `seconds` of CPU work from
    a 2-token calibration.  Returns (tokens/s, description, cores used, seconds spent, core)."""
    with OneCore() as pin:
        t0 = time.perf_counter()
        oracle_prefix(wl, tc, 2)
        per_tok = max((time.perf_counter() - t0) / 2, 1e-6)
        n = int(min(wl.T, max(2, seconds / per_tok)))
        t1 = time.perf_counter()
        oracle_prefix(wl, tc, n)
        dt = time.perf_counter() - t1
    desc = ("the whole layer (gate scores, top-k, capacity dispatch with the full workload's capacity, "
            "expert FFN, combine) for the first %d of %d tokens in %.2f s on one core; tokens/s = n / time"
            % (n, wl.T, dt))
    return n / dt, desc, 1, dt, pin.core


def host_inputs(wl):
    """The workload's tensors on the host, with the same values the GPU arm uses (expert weights larger
    than 1 GiB are drawn by the seeded CUDA generator when a GPU is present, then copied back)."""
    big = wl.expert_weight_bytes() > (1 << 30)
    if big and not torch.cuda.is_available():
        return None
    t = make_inputs(wl, device="cpu", expert_device="cuda" if big else "cpu")
    return {n: (v.cpu() if v is not None else None) for n, v in t.items()}


def run_reference(args, rank):
    wl = WORKLOADS[args.workload]
    if rank != 0:
        return
    if wl.expert_weight_bytes() > (4 << 30):
        print(json.dumps({"impl": "reference", "unavailable": "expert weights of this workload exceed the host "
                          "sample budget (4 GiB)"}))
        return
    tc = host_inputs(wl)
    if tc is None:
        print(json.dumps({"impl": "reference", "unavailable": "this workload's expert weights are drawn by the "
                          "CUDA generator and no GPU is present"}))
        return
    # each step is a bounded sample sized so that warm-up + steps take about two minutes in all
    per_step = min(10.0, max(0.3, 120.0 / max(1, args.steps + args.warmup)))
    vals, descs, total, core = [], [], 0.0, None
    for i in range(args.warmup + args.steps):
        v, desc, cores, dt, core = cpu_oracle_sample(wl, tc, per_step)
        if i >= args.warmup:
            vals.append(v)
            descs.append(desc)
            total += dt
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(vals),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "T": wl.T, "d_model": wl.d, "d_hidden": wl.h, "experts": wl.E,
                   "top_k": wl.k, "gate": wl.gate},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": descs[-1],
                         "pinned_core": core, "host_cores": os.cpu_count(), "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------------------- our path
def source_sha():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mixture_experts_sparse_03_b300", "csrc")
    for f in sorted(os.listdir(csrc)):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def file_sha(name: str) -> str:
    """sha256 (first 16 hex digits) of one file under csrc/."""
    path = os.path.join(ROOT, "mixture_experts_sparse_03_b300", "csrc", name)
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16] if os.path.exists(path) else ""


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summaries of `workload`, if they were
    taken on the kernel's current source (else None).  A summary states
    `traffic_bytes_per_launch <kernel>: <bytes>` and either `kernel_source_sha256 <file>: <hash>` (the
    .cu file that holds the kernel) or `source_sha256: <hash>` (all of csrc/)."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    for f in sorted(os.listdir(pdir)):
        if not f.endswith(".md") or workload not in f:
            continue
        txt = open(os.path.join(pdir, f)).read()
        m = re.search(r"traffic_bytes_per_launch %s:\s*([0-9.eE+]+)" % re.escape(kernel), txt)
        if not m:
            continue
        ks = re.findall(r"kernel_source_sha256 (\S+):\s*`?([0-9a-f]+)", txt)
        if ks and all(file_sha(name) == h for name, h in ks):
            return float(m.group(1))
        s = re.search(r"source_sha256:\s*`?([0-9a-f]+)", txt)
        if s and s.group(1) == source_sha():
            return float(m.group(1))
    return None


def roofline(wl, kern_ms, names, kept, used):
    """Roofline of the dominant kernel (the one whose launches take the largest share of a step).  The
    expert GEMM kernel runs twice per step (up-projection with GELU, down-projection) with equal work
    per launch; for it, achieved = algorithmic work of one launch / its mean launch duration."""
    gemm_flops, gate_flops, wbytes = layer_work(wl, kept, used)
    gemm_names = [n for n in names if n.startswith("expert_")]
    gemm_launch_ms = sum(kern_ms[n] for n in gemm_names) / len(gemm_names)
    rest = {n: v for n, v in kern_ms.items() if n not in gemm_names}
    top_rest = max(rest, key=rest.get)
    gemm_dominant = sum(kern_ms[n] for n in gemm_names) >= rest[top_rest]
    pk = peaks()
    hbm_bound = kept < RIDGE_ROWS * max(used, 1)  # few rows per expert: the weights' bytes bound the FFN
    if gemm_dominant and hbm_bound:
        # one expert GEMM streams one of the two weight matrices of every used expert
        achieved = (wbytes / 2) / (gemm_launch_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm"], "unit": "GB/s",
                "frac": achieved / pk["hbm"], "algorithmic_per_launch": wbytes / 2}
    elif gemm_dominant:
        achieved = gemm_flops / (gemm_launch_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": pk["bf16"], "unit": "TFLOP/s",
                "frac": achieved / pk["bf16"], "frac_of_sustained": achieved / pk["bf16_sustained"],
                "algorithmic_per_launch": gemm_flops}
    else:
        roof = {"bound": "hbm", "achieved": None, "peak": pk["hbm"], "unit": "GB/s", "frac": None}
    if gemm_dominant:
        dominant = "expert_gemm (%s)" % " + ".join(gemm_names)
        tr = [recorded_traffic(n, wl.name) for n in gemm_names]
        traffic = sum(tr) / len(tr) if all(v is not None for v in tr) else None
        dom_ms = gemm_launch_ms
    else:
        dominant, traffic, dom_ms = top_rest, recorded_traffic(top_rest, wl.name), rest[top_rest]
    roof.update({"traffic": traffic, "kernel": dominant, "peak_source": pk["source"] + " (burst)",
                 "kernel_ms": dom_ms})
    if wl.dtype != "bf16":
        roof["note"] = "fp32 CUDA-core path; bf16 tensor peak shown for reference only"
    return roof, gemm_flops, gate_flops, wbytes


class Layer:
    """One workload's inputs, workspace and output on the device, and its moe_forward step."""

    def __init__(self, wl, dev, stream, ffn="auto"):
        from mixture_experts_sparse_03_b300 import binding as b

        self.b, self.wl, self.dev, self.stream = b, wl, dev, stream
        self.cfg = b.config(wl, flags={"auto": 0, "one-sm": b.FLAG_FFN_ONE_SM, "sm-pair": b.FLAG_FFN_SM_PAIR}[ffn])
        self.tg = make_inputs(wl, device=dev,
                              expert_device="cuda" if wl.expert_weight_bytes() > (1 << 30) else "cpu")
        self.ws = b.workspace(self.cfg, dev)
        self.out = torch.empty((wl.T, wl.d), dtype=torch.float32, device=dev)
        self.count = torch.empty((wl.E,), dtype=torch.int32, device=dev)
        self.launches = b.moe_forward_launches(self.cfg)
        self.names = kernel_names(wl, self.launches)

    def step(self, x=None, eps=None, out=None, count="default"):
        b, t = self.b, self.tg
        xx = t["x"] if x is None else x
        ee = t.get("eps") if eps is None else eps
        oo = self.out if out is None else out
        cc = self.count if count == "default" else count
        if t.get("w1_scale") is not None:  # block-FP8 expert weights
            b.check(b.moe_forward_fp8(self.cfg, xx, t.get("w_gate"), t.get("w_noise"), ee, t.get("proj"), t.get("emb"),
                                      t["w1"], t["w1_scale"], t.get("b1"), t["w2"], t["w2_scale"], t.get("b2"), oo, cc,
                                      self.ws, self.ws.numel(), self.stream), "moe_forward_fp8")
            return
        b.check(b.moe_forward(self.cfg, xx, t.get("w_gate"), t.get("w_noise"), ee, t.get("proj"), t.get("emb"),
                              t["w1"], t.get("b1"), t["w2"], t.get("b2"), oo, cc, self.ws, self.ws.numel(),
                              self.stream), "moe_forward")

    def capture(self, traced_events=None):
        """A CUDA graph of one step; with events, the library's trace hook puts an event-record node
        before the first launch and after every launch."""
        b = self.b
        g = torch.cuda.CUDAGraph()
        keep = None
        with torch.cuda.graph(g, stream=self.stream):
            if traced_events is not None:
                keep = b.moe_trace_events(traced_events, len(traced_events))
            self.step()
            if traced_events is not None:
                recorded = b.moe_trace_count()
                b.moe_trace_events(None, 0)
        if traced_events is not None and recorded != len(traced_events):
            raise RuntimeError("trace hook recorded %d of %d events" % (recorded, len(traced_events)))
        del keep
        return g


def measure(wl, args, dev, stream, flush, world):
    """Graph-timed steps and the per-kernel split of one workload.  Returns (result dict, Layer)."""
    L = Layer(wl, dev, stream, args.ffn)
    b = L.b
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            L.step()
    stream.synchronize()
    st, info = b.moe_device_status(L.ws, L.ws.numel(), stream)
    b.check(st, "device status after warm-up")
    C = b.moe_capacity(L.cfg)
    cnt = L.count.cpu().numpy()
    kept = int(np.minimum(cnt, min(C, wl.T)).sum())
    used = int((np.minimum(cnt, C) > 0).sum())

    graph = None if args.no_graph else L.capture()
    run_step = graph.replay if graph is not None else L.step

    # ---- timed region: K steps, L2 flushed before each, events around each step
    K = args.steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.fill_(1)
            run_step()
    stream.synchronize()
    sampler = ClockSampler(dev.index)
    sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        for i in range(K):
            flush.fill_(i & 0xFF)
            evs[i][0].record(stream)
            run_step()
            evs[i][1].record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    times = [a.elapsed_time(z) for a, z in evs]  # ms
    total_ms = max_over_ranks(sum(times), dev)

    # ---- per-kernel durations: a graph of the same step with event-record nodes between its launches
    tev = [torch.cuda.Event(enable_timing=True) for _ in range(L.launches + 1)]
    for e in tev:  # torch creates the CUDA event at its first record; the library needs real handles
        e.record(stream)
    stream.synchronize()
    per = {n: [] for n in L.names}
    traced_steps = []
    tgraph = L.capture(tev)
    with torch.cuda.stream(stream):
        for i in range(max(5, min(K, 20))):
            flush.fill_(1)
            tgraph.replay()
            stream.synchronize()
            for j, n in enumerate(L.names):
                per[n].append(tev[j].elapsed_time(tev[j + 1]))
            traced_steps.append(tev[0].elapsed_time(tev[-1]))
    del tgraph
    kern_ms = {n: statistics.median(v) for n, v in per.items()}
    roof, gemm_flops, gate_flops, wbytes = roofline(wl, kern_ms, L.names, kept, used)
    ms_per_step = total_ms / K
    roof.update({"layer_tflops": (2 * gemm_flops + gate_flops) / (ms_per_step * 1e-3) / 1e12,
                 "layer_weight_gbs": wbytes / (ms_per_step * 1e-3) / 1e9})
    res = {"value": job_throughput(world, K, wl.T, total_ms), "ms_per_step": ms_per_step,
           "step_ms_median": statistics.median(times), "traced_step_ms_median": statistics.median(traced_steps),
           "kernel_ms": kern_ms, "capacity": C, "kept_pairs": kept, "experts_used": used,
           "graph": graph is not None, "roofline": roof, "clocks": clocks, "gpu_launches": L.launches * K}
    del graph
    return res, L


BWD_TAIL = ["fwd_up_keep_z", "fwd_down_y", "logits_gemm", "bwd_dy", "bwd_gate_grad", "bwd_dz_gemm",
            "bwd_dx_gemm", "iota_rows", "gate_weights_t", "bwd_dx_gate_gemm", "zero_pad_rows", "wgrad_w2",
            "wgrad_w1", "wgrad_gate", "colsum_db2", "colsum_db1"]


def backward_timing(L, flush, steps):
    """moe_backward (forward recomputed, then every gradient) on the layer's inputs with a seeded dout:
    graph-replayed calls, L2 flushed before each, event-timed; the per-kernel split from a graph with
    event-record nodes.  Reports ms per call and the tensor-core work of its expert GEMMs (six of them:
    the recomputed up and down projections, dZ, dX and the two weight gradients, each 2 kept-pairs d h)."""
    b, wl, dev, stream, tg = L.b, L.wl, L.dev, L.stream, L.tg
    n = b.moe_backward_workspace_size(L.cfg)
    if n == 0 or tg.get("w1_scale") is not None:
        return None
    ws = torch.empty(n, dtype=torch.uint8, device=dev)
    T, d, h, E = wl.T, wl.d, wl.h, wl.E
    gen = torch.Generator(device="cpu").manual_seed(wl.seed + 7)
    dout = torch.randn(T, d, generator=gen).to(dev)
    z = lambda *sh: torch.empty(sh, dtype=torch.float32, device=dev)  # noqa: E731
    g = dict(dx=z(T, d), dw_gate=z(E, d), dw_noise=z(E, d) if wl.gate == "noisy" else None, dw1=z(E, h, d),
             db1=z(E, h), dw2=z(E, d, h), db2=z(E, d))

    def call():
        b.check(b.moe_backward(L.cfg, tg["x"], tg.get("w_gate"), tg.get("w_noise"), tg.get("eps"), tg["w1"], tg.get("b1"),
                               tg["w2"], tg.get("b2"), dout, g["dx"], g["dw_gate"], g["dw_noise"], g["dw1"], g["db1"],
                               g["dw2"], g["db2"], ws, n, stream), "moe_backward")

    with torch.cuda.stream(stream):
        call()
    stream.synchronize()
    cap = [torch.cuda.Event(enable_timing=True) for _ in range(64)]
    for e in cap:
        e.record(stream)
    stream.synchronize()
    with torch.cuda.stream(stream):
        keep = b.moe_trace_events(cap, len(cap))
        call()
        launches = b.moe_trace_count() - 1
        b.moe_trace_events(None, 0)
    stream.synchronize()
    del keep
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        call()
    times = []
    with torch.cuda.stream(stream):
        for i in range(3 + steps):
            flush.fill_(1)
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            graph.replay()
            a1.record(stream)
            a1.synchronize()
            if i >= 3:
                times.append(a0.elapsed_time(a1))
    st, info = b.moe_device_status(ws, n, stream)
    b.check(st, "device status after moe_backward")
    tev = cap[:launches + 1]
    tgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(tgraph, stream=stream):
        keep = b.moe_trace_events(tev, len(tev))
        call()
        b.moe_trace_events(None, 0)
    per = [[] for _ in range(launches)]
    with torch.cuda.stream(stream):
        for i in range(5):
            flush.fill_(1)
            tgraph.replay()
            stream.synchronize()
            for j in range(launches):
                per[j].append(tev[j].elapsed_time(tev[j + 1]))
    route = launches - len(BWD_TAIL)
    names = L.names[:route] + BWD_TAIL if route >= 0 else ["k%d" % j for j in range(launches)]
    kern = {names[j]: statistics.median(per[j]) for j in range(launches)}
    C = b.moe_capacity(L.cfg)
    kept = int(np.minimum(L.count.cpu().numpy(), min(C, wl.T)).sum())
    flops = 6 * 2.0 * kept * d * h
    ms = statistics.median(times)
    return {"ms_per_call": ms, "launches": launches, "expert_gemm_tflop": flops / 1e12,
            "tflops_whole_call": flops / (ms * 1e-3) / 1e12, "kernel_ms": kern,
            "timing": "CUDA graph replay, L2 flushed before each call; kernel_ms from event-record nodes"}


def router_stats_timing(L, stream):
    """moe_router_stats on the layer's routing and dispatch: 20 calls captured in one CUDA graph, the
    replay event-timed, per call."""
    b, wl, dev, tg = L.b, L.wl, L.dev, L.tg
    T_, k_, E_ = wl.T, wl.k, wl.E
    r_idx = torch.empty((T_, k_), dtype=torch.int32, device=dev)
    r_gate = torch.empty((T_, k_), dtype=torch.float32, device=dev)
    r_slot = torch.empty((T_, k_), dtype=torch.int32, device=dev)
    rows_ = max(b.moe_dispatch_rows(L.cfg), 1)
    r_cnt = torch.empty((E_,), dtype=torch.int32, device=dev)
    r_off = torch.empty((E_ + 1,), dtype=torch.int32, device=dev)
    r_rtok = torch.empty((rows_,), dtype=torch.int32, device=dev)
    r_rgate = torch.empty((rows_,), dtype=torch.float32, device=dev)
    r_xd = torch.empty((rows_, wl.d), dtype=tg["x"].dtype, device=dev)
    r_imp = torch.empty((E_,), dtype=torch.float32, device=dev)
    r_loss = torch.empty((2,), dtype=torch.float32, device=dev)
    r_drop = torch.empty((1,), dtype=torch.int64, device=dev)
    ws = L.ws
    with torch.cuda.stream(stream):
        b.check(b.moe_route(L.cfg, tg["x"], tg.get("w_gate"), tg.get("w_noise"), tg.get("eps"), tg.get("proj"),
                            tg.get("emb"), r_idx, r_gate, ws, ws.numel(), stream), "moe_route")
        b.check(b.moe_dispatch(L.cfg, tg["x"], r_idx, r_gate, r_slot, r_cnt, r_off, r_rtok, r_rgate, r_xd, ws,
                               ws.numel(), stream), "moe_dispatch")

    def call():
        b.check(b.moe_router_stats(L.cfg, r_idx, r_gate, r_slot, r_imp, r_loss, r_drop, ws, ws.numel(), stream),
                "moe_router_stats")

    with torch.cuda.stream(stream):
        call()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(20):
            call()
    us = []
    with torch.cuda.stream(stream):
        for i in range(6):
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            g.replay()
            a1.record(stream)
            a1.synchronize()
            if i >= 1:
                us.append(a0.elapsed_time(a1) * 1000.0 / 20)
    rs_bytes = T_ * k_ * 12 + E_ * 4 + 16  # ids, gates, slots in; importance, losses, drops out
    return {"us": statistics.median(us), "bytes": rs_bytes, "bound": "latency", "timing": "20 calls in one graph",
            "importance_loss": float(r_loss[0]), "load_balance_loss": float(r_loss[1]), "dropped": int(r_drop[0])}


def e2e_timing(L, flush, K, world):
    """End to end through the C ABI with pinned host buffers: every step copies x (and eps) in, flushes
    L2, runs moe_forward and copies `out` back.  Steps are pipelined the way a serving loop runs them:
    step i's host-to-device copy (its own stream), its moe_forward (compute stream) and its
    device-to-host copy of `out` (a third stream) overlap the neighbouring steps' work; two device
    buffer sets alternate.  Returns (tokens/s, h2d bytes per step, d2h bytes per step)."""
    wl, dev, stream, tg = L.wl, L.dev, L.stream, L.tg
    x_host = tg["x"].cpu().pin_memory()
    eps_host = tg["eps"].cpu().pin_memory() if tg.get("eps") is not None else None
    out_host = [torch.empty((wl.T, wl.d), dtype=torch.float32).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(tg["x"]) for _ in range(2)]
    eps_dev = [torch.empty_like(tg["eps"]) for _ in range(2)] if eps_host is not None else [None, None]
    out_dev = [L.out, torch.empty_like(L.out)]
    h2d = x_host.numel() * x_host.element_size() + (eps_host.numel() * 4 if eps_host is not None else 0)
    d2h = out_host[0].numel() * 4
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def run(n):
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_fw = [torch.cuda.Event() for _ in range(n)]
        ev_out = [torch.cuda.Event() for _ in range(n)]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        s_in.wait_event(start)
        s_out.wait_event(start)
        for i in range(n):
            j = i & 1
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_fw[i - 2])  # buffer set j is free once step i-2 has run
                x_dev[j].copy_(x_host, non_blocking=True)
                if eps_host is not None:
                    eps_dev[j].copy_(eps_host, non_blocking=True)
                ev_in[i].record(s_in)
            with torch.cuda.stream(stream):
                stream.wait_event(ev_in[i])
                if i >= 2:
                    stream.wait_event(ev_out[i - 2])  # out[j] has been read back
                flush.fill_(i & 0xFF)
                L.step(x=x_dev[j], eps=eps_dev[j], out=out_dev[j], count=None)
                ev_fw[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_fw[i])
                out_host[j].copy_(out_dev[j], non_blocking=True)
                ev_out[i].record(s_out)
        stream.wait_event(ev_out[n - 1])
        stream.wait_event(ev_in[n - 1])
        end.record(stream)
        return start, end

    run(3)
    torch.cuda.synchronize(dev)
    start, end = run(K)
    end.synchronize()
    e_ms = start.elapsed_time(end)
    torch.cuda.synchronize(dev)
    return job_throughput(world, K, wl.T, max_over_ranks(e_ms, dev)), h2d, d2h


def config_of(wl, res, world):
    return {"workload": wl.name, "T": wl.T, "d_model": wl.d, "d_hidden": wl.h, "experts": wl.E, "top_k": wl.k,
            "gate": wl.gate, "capacity": res["capacity"], "kept_pairs": res["kept_pairs"],
            "experts_used": res["experts_used"], "parallelism": "replicas" if world > 1 else "single",
            "l2": "flushed between steps (256 MiB write)", "graph": res["graph"],
            "step_ms_median": res["step_ms_median"], "traced_step_ms_median": res["traced_step_ms_median"],
            "kernel_ms": res["kernel_ms"],
            "kernel_timing": "graph replay with event-record nodes between launches (no host gaps); their "
                             "sum is traced_step_ms, which lacks the overlap of programmatic dependent "
                             "launch that the timed step has"}


def scaled_workload(wl, experts: int):
    """The workload with `experts` experts and its token count scaled by experts / E (same expected rows
    per expert, same capacity when the capacity comes from the capacity factor)."""
    if not experts or experts == wl.E:
        return wl
    if wl.T * experts % wl.E or experts < wl.k:
        raise SystemExit("--experts %d does not scale T = %d evenly (E = %d, k = %d)" % (experts, wl.T, wl.E, wl.k))
    T = wl.T * experts // wl.E
    return wl.with_(name="%s_E%d" % (wl.name, experts), E=experts, T=T,
                    capacity=(T if wl.capacity == wl.T else wl.capacity))


def run_ours(args, rank, world, local):
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    wl = scaled_workload(WORKLOADS[args.workload], args.experts)
    if args.experts:
        args.only = True
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    res, L = measure(wl, args, dev, stream, flush, world)
    router_stats = router_stats_timing(L, stream)
    backward = None if args.skip_backward else backward_timing(L, flush, min(args.steps, 10))
    e2e_value, h2d, d2h = e2e_timing(L, flush, args.steps, world)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        tc = {n: (v.cpu() if v is not None else None) for n, v in L.tg.items()}
        v, desc, cores, _, core = cpu_oracle_sample(wl, tc, args.cpu_seconds)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc, "pinned_core": core,
               "host_cores": os.cpu_count(), "cpu_model": cpu_model()}
        del tc
    del L
    torch.cuda.empty_cache()

    others = {}
    if not args.only:
        for name in WORKLOAD_ORDER:
            if name == wl.name:
                continue
            o_args = argparse.Namespace(**{**vars(args), "steps": min(args.steps, 20), "warmup": 3})
            r, Lo = measure(WORKLOADS[name], o_args, dev, stream, flush, world)
            del Lo
            torch.cuda.empty_cache()
            others[name] = {"tokens_per_s": r["value"], "ms_per_step": r["ms_per_step"],
                            "config": config_of(WORKLOADS[name], r, world), "roofline": r["roofline"],
                            "clocks": r["clocks"], "steps": o_args.steps}

    if rank == 0:
        line = {
            "metric": METRIC, "value": res["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": wl.dtype,
            "data": "synthetic (seeded; shapes and distributions of the workload)",
            "config": config_of(wl, res, world),
            "roofline": res["roofline"],
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "pipelined": "2 buffer sets; H2D, compute and D2H on three streams"},
            "gpu_launches": res["gpu_launches"],
            "router_stats": router_stats,
            "backward": backward,
            "clocks": res["clocks"],
            "workloads": others,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py --impl ours needs a CUDA device")
    run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
