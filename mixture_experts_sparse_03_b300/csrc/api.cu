// api.cu -- the C ABI of libmoe_b300 (declared in include/moe_b300.h): argument validation, workspace
// planning, the launch sequence of the layer and the profiling hook.  Every argument is checked on the
// host before anything is enqueued; a failed check returns a status and launches nothing.
#include <cuda_runtime.h>
#include <math.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include <algorithm>

#include "kernels.h"
#include "moe_b300.h"

namespace {

using namespace moe;

constexpr size_t kAlign = 256;
constexpr int kMaxSmem = 227 * 1024;

size_t up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Plan {
    int T, d, h, E, k, C, Ceff, p, nblk, gate, norm, bf16, esize, fused;
    int rank_major;     // capacity slots in (rank, token) order
    int stats;          // router statistics fused into the forward's gather
    size_t o_fstats;    // their accumulators (in the zeroed header) and o_fstats_out their results
    int nblk_hist;      // blocks of the dispatch histogram: of 32 tokens, or of 32 (rank, token) pairs
    int N0, N1;         // gate logits from the first / second weight tensor
    int pair;           // expert GEMMs on pairs of SMs
    int pair_down;      // the down projection (K = h) on pairs of SMs
    GateGemmPlan gg;    // tensor-core logits GEMM (bf16 layers)
    int64_t rows;
    size_t o_err, o_idx, o_gate, o_slot, o_hist, o_count, o_off, o_rtok, o_rgate, o_xd, o_h, o_y, o_part, o_xn2,
        o_wn2, o_rq, o_cosv, o_fstats_out, total;
    size_t hdr_bytes;  // error word, its info, tickets and the cosine gate's expert flags: zeroed per call
};

// Bound on the error of the tensor-core logits: |logit - exact| <= kTcErr * 2^-23 * sum_i |x_i w_i|.
// Measured behaviour of the B300 (pinned by tests/test_gpu_tc_model.py): each MMA step adds 16 bf16
// products to the fp32 accumulator after aligning all 17 addends to the largest one's exponent e on a
// grid of 2^(e-25), sums them exactly and truncates the result to fp32, so a step errs by at most
// 17 * 2^-25 * max|addend| + 2^-23 * |result| <= 5.25 * 2^-23 * (sum of |x_i w_i| so far in the
// accumulator).  The logits GEMM starts a fresh accumulator every 128-wide chunk of K (8 steps), so each
// chunk errs by at most 42 * 2^-23 * (its sum of |x_i w_i|), and adds the chunks with compensated (Kahan)
// summation, which errs by at most 2u * sum |chunk| (u = 2^-24), its correction term by no more, and the
// final rounding by u: the whole dot product errs by at most 44.5 * 2^-23 * sum |x_i w_i|; the constant
// leaves a 1.44x margin.  Summing S fp32 split partials adds S * 2^-24 * sum |x_i w_i|.
constexpr double kTcErr = 64.0;

// expected rows per expert (T * k / E) from which the expert GEMMs run on pairs of SMs by default
constexpr int kPairMinRows = 2048;

// byte offset of the int64 drop count in the fused statistics' results (after E + 2 floats)
size_t fstats_drop_at(int E) { return (4 * (size_t)E + 8 + 7) / 8 * 8; }

moe_status make_plan(const moe_config* c, Plan* pl) {
    if (c == nullptr) return MOE_ERR_INVALID_ARG;
    Plan P{};
    P.T = c->tokens;
    P.d = c->model_dim;
    P.h = c->hidden_size_per_expert;
    P.E = c->num_experts;
    P.k = c->top_k;
    P.gate = c->gate_type;
    P.norm = c->gate_norm;
    P.bf16 = c->dtype == MOE_BF16;
    P.esize = P.bf16 ? 2 : 4;
    if (P.T < 0 || P.d < 64 || P.d % 64 || P.h < 64 || P.h % 64) return MOE_ERR_INVALID_ARG;
    if (P.d > (1 << 16) || P.h > (1 << 16)) return MOE_ERR_UNSUPPORTED;
    if (P.E < 1 || P.E > kMaxExperts || P.k < 1 || P.k > P.E || P.k > kMaxTopK) return MOE_ERR_INVALID_ARG;
    if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
    if (P.gate < MOE_GATE_SOFTMAX || P.gate > MOE_GATE_COSINE) return MOE_ERR_INVALID_ARG;
    if (P.norm != MOE_GATE_NORM_ALL && P.norm != MOE_GATE_NORM_TOPK) return MOE_ERR_INVALID_ARG;
    if (c->flags & ~(MOE_FLAG_SIMT_FFN | MOE_FLAG_UNFUSED_COMBINE | MOE_FLAG_FFN_ONE_SM | MOE_FLAG_FFN_SM_PAIR |
                     MOE_FLAG_RANK_MAJOR | MOE_FLAG_ROUTER_STATS))
        return MOE_ERR_INVALID_ARG;
    if ((c->flags & MOE_FLAG_FFN_ONE_SM) && (c->flags & MOE_FLAG_FFN_SM_PAIR)) return MOE_ERR_INVALID_ARG;
    if (c->reserved != 0) return MOE_ERR_INVALID_ARG;
    if (P.gate == MOE_GATE_NOISY && P.E > 512) return MOE_ERR_UNSUPPORTED;
    P.p = 0;
    if (P.gate == MOE_GATE_COSINE) {
        P.p = c->cos_dim;
        if (P.p < 8 || P.p > 1024 || P.p % 8) return MOE_ERR_INVALID_ARG;
        if (!(c->cos_temperature > 0.0) || !isfinite(c->cos_temperature)) return MOE_ERR_INVALID_ARG;
    }
    if (c->capacity >= 0) {
        P.C = c->capacity;
    } else {
        if (!(c->capacity_factor > 0.0) || !isfinite(c->capacity_factor)) return MOE_ERR_INVALID_ARG;
        const double v = ceil(c->capacity_factor * (double)P.T * (double)P.k / (double)P.E);
        if (!(v >= 0.0) || v > 2147483647.0) return MOE_ERR_INVALID_ARG;
        P.C = (int)v;
    }
    const size_t gsm = P.bf16 ? gate_select_smem_bytes(P.gate, P.E, P.p) : gate_smem_bytes(P.gate, P.E, P.p, P.d);
    if (gsm > (size_t)kMaxSmem) return MOE_ERR_UNSUPPORTED;
    P.N0 = P.gate == MOE_GATE_COSINE ? P.p : P.E;
    P.N1 = P.gate == MOE_GATE_NOISY ? P.E : 0;
    P.gg = gate_gemm_plan(P.T, P.d, P.N0, P.N1, kPlanSms, P.gate == MOE_GATE_SOFTMAX);
    P.Ceff = std::min(P.C, P.T);  // a token takes an expert at most once, so C >= T drops nothing
    const int64_t cpad = ((int64_t)P.Ceff + kRowAlign - 1) / kRowAlign * kRowAlign;
    P.rows = std::min<int64_t>((int64_t)P.T * P.k + (int64_t)(kRowAlign - 1) * P.E, (int64_t)P.E * cpad);
    if (P.rows > (int64_t)1 << 30) return MOE_ERR_UNSUPPORTED;
    P.nblk = (P.T + kTokensPerBlock - 1) / kTokensPerBlock;
    P.rank_major = (c->flags & MOE_FLAG_RANK_MAJOR) != 0;
    P.nblk_hist = dispatch_hist_blocks(P.T, P.k, P.rank_major);
    P.fused = P.k <= 2 && !(c->flags & MOE_FLAG_UNFUSED_COMBINE);
    // pairs of SMs pay off when experts get many rows: their 256-row tiles waste at most 128 rows per
    // expert, against 2x the rows each weight byte serves
    // (measured: with d <= 1024 and 1024 rows per expert both GEMMs gain on pairs, the step 4 %; with 512
    // rows per expert only the down projection, where K = h is long and N = d short)
    const bool auto_ok = !(c->flags & MOE_FLAG_FFN_ONE_SM);
    const int64_t pairs_tk = (int64_t)P.T * P.k;
    P.pair = (c->flags & MOE_FLAG_FFN_SM_PAIR) ||
             (auto_ok && (pairs_tk >= (int64_t)kPairMinRows * P.E || (P.d <= 1024 && pairs_tk >= 1024 * (int64_t)P.E)));
    P.pair_down = P.pair || (auto_ok && P.d >= 512 && P.d <= 1024 && pairs_tk >= 512 * (int64_t)P.E);
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t r = o; o = up(o + bytes); return r; };
    const size_t tk = (size_t)P.T * P.k;
    const bool cos_tc = P.bf16 && P.gate == MOE_GATE_COSINE;  // cosine gates never take the fused path
    P.stats = (c->flags & MOE_FLAG_ROUTER_STATS) != 0;
    const size_t cos_flags = cos_tc ? 4 * (size_t)P.E : 0;
    // the router statistics' accumulators (E + 1 uint64) and ticket sit in the header, zeroed with it by
    // one memset per call (moe_router_stats, and moe_forward with the statistics fused in)
    const size_t fstats_at = (16 + cos_flags + 7) / 8 * 8;
    P.hdr_bytes = fstats_at + 8 * (size_t)(P.E + 1) + 8;
    P.o_err = take(P.hdr_bytes);
    P.o_fstats = P.o_err + fstats_at;
    P.o_idx = take(4 * tk);
    P.o_gate = take(4 * tk);
    P.o_slot = take(4 * tk);
    P.o_hist = take(4 * (size_t)P.nblk_hist * P.E);
    P.o_count = take(4 * (size_t)P.E);
    P.o_off = take(4 * (size_t)(P.E + 1));
    P.o_rtok = take(4 * (size_t)P.rows);
    P.o_rgate = take(4 * (size_t)P.rows);
    P.o_xd = take((size_t)P.rows * P.d * P.esize);
    P.o_h = take((size_t)P.rows * P.h * P.esize);
    P.o_y = take((size_t)P.rows * P.d * 4);
    const size_t np = (size_t)P.N0 + P.N1;
    P.o_part = take(P.bf16 ? 4 * (size_t)P.gg.S * P.T * np : 0);
    P.o_xn2 = take(P.bf16 ? 4 * (size_t)P.gg.S * P.T : 0);
    P.o_wn2 = take(P.bf16 ? 4 * (size_t)P.gg.S * np : 0);
    P.o_rq = take(P.bf16 && !P.gg.fused ? 4 * (size_t)P.T * kRescoreInts : 0);
    P.o_cosv = take(cos_tc ? 8 * (size_t)P.E * P.d : 0);
    // fused statistics: importance [E] and losses [2] fp32, then the drop count (int64, 8-byte aligned)
    P.o_fstats_out = take(P.stats ? fstats_drop_at(P.E) + 8 : 0);
    P.total = o;
    *pl = P;
    return MOE_OK;
}

moe_status check_ws(const Plan& P, void* ws, size_t bytes) {
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) || bytes < P.total) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

template <typename Tp>
Tp* at(void* ws, size_t off) { return reinterpret_cast<Tp*>(static_cast<char*>(ws) + off); }

// ---- profiling hook -------------------------------------------------------------------------------
void** g_events = nullptr;
int g_capacity = 0;
int g_recorded = 0;

// A failed record (e.g. an event that was never created) turns the hook off and clears the error, so
// tracing can never change the status of a launch; moe_trace_count() then shows the shortfall.  Under
// stream capture the records are external, so each becomes an event-record node of the graph and a
// replayed graph times its kernels without host gaps between them.
void trace_record(int i, cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) cs = cudaStreamCaptureStatusNone;
    const unsigned flags = cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault;
    if (cudaEventRecordWithFlags(static_cast<cudaEvent_t>(g_events[i]), s, flags) != cudaSuccess) {
        cudaGetLastError();
        g_events = nullptr;
        return;
    }
    g_recorded = i + 1;
}
void trace_pre(cudaStream_t s) {
    if (g_events != nullptr && g_recorded == 0 && g_capacity > 0) trace_record(0, s);
}
void trace_post(cudaStream_t s) {
    if (g_events != nullptr && g_recorded > 0 && g_recorded < g_capacity) trace_record(g_recorded, s);
}

// wrap one kernel launch: trace events around it, CUDA errors mapped to a status
template <typename F>
moe_status launch(cudaStream_t s, F&& f) {
    trace_pre(s);
    cudaError_t e = f();
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    trace_post(s);
    return MOE_OK;
}
// One NVTX range per C-ABI call (visible to nsys / ncu's NVTX filters; a no-op without a tool attached).
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

#define MOE_TRY(expr)                      \
    do {                                   \
        moe_status st_ = (expr);           \
        if (st_ != MOE_OK) return st_;     \
    } while (0)

moe_status check_route_args(const Plan& P, const void* x, const void* w_gate, const void* w_noise,
                            const float* eps, const void* proj, const void* emb, const void* idx, const void* gate) {
    if (!x || !idx || !gate || !aligned16(x) || !aligned16(idx) || !aligned16(gate)) return MOE_ERR_INVALID_ARG;
    if (P.gate == MOE_GATE_COSINE) {
        if (!proj || !emb || !aligned16(proj) || !aligned16(emb)) return MOE_ERR_INVALID_ARG;
    } else {
        if (!w_gate || !aligned16(w_gate)) return MOE_ERR_INVALID_ARG;
        if (P.gate == MOE_GATE_NOISY && (!w_noise || !eps || !aligned16(w_noise) || !aligned16(eps)))
            return MOE_ERR_INVALID_ARG;
    }
    return MOE_OK;
}

GateParams gate_params(const Plan& P, const moe_config* c, const void* x, const void* w_gate, const void* w_noise,
                       const float* eps, const void* proj, const void* emb, int32_t* idx, float* gate) {
    GateParams g{};
    g.x = x;
    g.w_gate = w_gate;
    g.w_noise = w_noise;
    g.eps = eps;
    g.proj = proj;
    g.emb = emb;
    g.T = P.T;
    g.d = P.d;
    g.E = P.E;
    g.k = P.k;
    g.p = P.p;
    g.gate = P.gate;
    g.norm = P.norm;
    g.bf16 = P.bf16;
    g.temp = P.gate == MOE_GATE_COSINE ? c->cos_temperature : 1.0;
    g.inv_temp = (float)(1.0 / g.temp);
    g.topk_idx = idx;
    g.topk_gate = gate;
    g.cb = (float)(33.0 * 5.9604644775390625e-08);  // CUDA-core logits: chunked, compensated fp32 sums
    return g;
}

// bf16 layers: run the tensor-core logits GEMM into the workspace and point the gate kernel at it
moe_status gate_logits_tc(const Plan& P, GateParams& g, void* ws, cudaStream_t s) {
    const void* w0 = P.gate == MOE_GATE_COSINE ? g.proj : g.w_gate;
    const void* w1 = P.gate == MOE_GATE_NOISY ? g.w_noise : nullptr;
    float* part = at<float>(ws, P.o_part);
    float* xn2 = at<float>(ws, P.o_xn2);
    float* wn2 = at<float>(ws, P.o_wn2);
    g.part = part;
    g.xn2p = xn2;
    g.wn2p = wn2;
    g.S = P.gg.S;
    g.Np = P.gg.Np;
    g.cb = (float)(kTcErr * 1.1920928955078125e-07 + (P.gg.S + 1) * 5.9604644775390625e-08);
    return launch(s, [&] {
        return launch_gate_gemm(P.gg, g.x, w0, w1, P.T, P.d, P.N0, P.N1, part, xn2, wn2, at<int>(ws, P.o_err), &g, s);
    });
}

// the whole gate (and, with g.blk_hist set, the dispatch's rank step and scan):
//   bf16, softmax, E <= 64: one fused launch;
//   other bf16 gates: logits GEMM, selection (tokens with near ties queued), for the cosine gate the fold
//   v_e = P^T e_e of the contending experts, grid-wide re-scoring of the queue, then the rank step with
//   the scan in its last block;
//   fp32: the CUDA-core gate kernel, which does all of it
moe_status run_gate(const Plan& P, GateParams& g, void* ws, cudaStream_t s) {
    if (!P.bf16) return launch(s, [&] { return launch_gate(g, s); });
    MOE_TRY(gate_logits_tc(P, g, ws, s));
    if (P.gg.fused) return MOE_OK;
    GateParams sel = g;
    sel.blk_hist = nullptr;
    sel.ticket = nullptr;
    sel.rq_count = at<int>(ws, P.o_err) + 3;  // zeroed with the error word
    sel.rq = at<int>(ws, P.o_rq);
    if (P.gate == MOE_GATE_COSINE) {
        sel.need = at<int>(ws, P.o_err) + 4;  // zeroed with the error word
        sel.cosv = at<float2>(ws, P.o_cosv);
    }
    MOE_TRY(launch(s, [&] { return launch_gate(sel, s); }));
    if (P.gate == MOE_GATE_COSINE) MOE_TRY(launch(s, [&] { return launch_gate_cos_fold(sel, s); }));
    MOE_TRY(launch(s, [&] { return launch_gate_rescore(sel, s); }));
    if (g.blk_hist == nullptr) return MOE_OK;
    return launch(s, [&] {
        return launch_dispatch_rank(g.topk_idx, P.T, P.k, P.E, g.blk_hist, g.slot, g.err, g.ticket, g.C, g.count,
                                    g.offset, g.row_token, g.row_gate, P.rank_major, s);
    });
}

// the gate kernel itself ranks the pairs (in token order) and scans: the fused bf16 gate and the fp32 gate
bool gate_ranks_in_kernel(const Plan& P) { return !P.bf16 || P.gg.fused; }

FfnParams ffn_params(const Plan& P, int mode, const void* A, const void* W, const float* w_scale, const void* bias,
                     const int* off, const int* rtok, const float* rgate, void* C, float* out, int* err) {
    FfnParams f{};
    f.A = A;
    f.W = W;
    f.w_scale = w_scale;
    f.bias = bias;
    f.offset = off;
    f.row_token = rtok;
    f.row_gate = rgate;
    f.C = C;
    f.out = out;
    f.E = P.E;
    const bool up_proj = mode == 0 || mode == 4;  // x_d [rows, d] -> [rows, h]
    f.K = up_proj ? P.d : P.h;
    f.N = up_proj ? P.h : P.d;
    f.bf16 = P.bf16;
    f.mode = mode;
    f.rows_cap = P.rows;
    f.err = err;
    // block-FP8 weights and the backward run on single SMs
    f.pair = (w_scale || mode >= 3) ? 0 : (up_proj ? P.pair : P.pair_down);
    f.max_rows = P.C < P.T ? P.C : P.T;
    return f;
}

moe_status run_ffn(const Plan& P, const moe_config* c, const FfnParams& f, cudaStream_t s) {
    const bool tc = P.bf16 && !(c->flags & MOE_FLAG_SIMT_FFN);
    return launch(s, [&] { return tc ? launch_ffn_tc(f, s) : launch_ffn_simt(f, s); });
}

// expert FFN + (fused or separate) combine, shared by moe_expert_ffn(_fp8) and moe_forward(_fp8); s1 / s2
// are the block scales of FP8 weights (nullptr: bf16 / fp32 weights)
// whether the up projection's kernel clears `out` for the fused combine while it runs: the single-SM
// tensor-core kernel (bf16 weights, not on pairs of SMs), and only where its work hides the 4 d bytes per
// token (rows x h at least 8192 per token: the headline layer's up projection runs ~40x longer than the
// clearing, `bf16_cosine_skew`'s ~5x, where it measured +4 us against the gather's -4 us); otherwise the
// gather clears it
bool up_clears_out(const Plan& P, const moe_config* c, const float* s1) {
    return P.fused && P.bf16 && !(c->flags & MOE_FLAG_SIMT_FFN) && s1 == nullptr && !P.pair &&
           (int64_t)P.rows * P.h >= (int64_t)8192 * P.T;
}

moe_status ffn_and_combine(const Plan& P, const moe_config* c, const void* xd, const int* off, const int* rtok,
                           const float* rgate, const void* w1, const float* s1, const void* b1, const void* w2,
                           const float* s2, const void* b2, float* y, float* out, bool fused, void* ws,
                           cudaStream_t s, bool clear_out = false) {
    int* err = at<int>(ws, P.o_err);
    void* hbuf = at<void>(ws, P.o_h);
    FfnParams up = ffn_params(P, 0, xd, w1, s1, b1, off, rtok, rgate, hbuf, nullptr, err);
    if (clear_out) {
        up.zero = out;
        up.zero_n = (int64_t)P.T * P.d;
    }
    MOE_TRY(run_ffn(P, c, up, s));
    if (fused) return run_ffn(P, c, ffn_params(P, 2, hbuf, w2, s2, b2, off, rtok, rgate, nullptr, out, err), s);
    return run_ffn(P, c, ffn_params(P, 1, hbuf, w2, s2, b2, off, rtok, rgate, y, nullptr, err), s);
}

// block-FP8 weights: bf16 activations on the tensor cores, d and h multiples of the 128-wide scale blocks
moe_status check_fp8_weights(const Plan& P, const moe_config* c, const void* w1, const float* s1, const void* w2,
                             const float* s2) {
    if (!P.bf16 || (c->flags & MOE_FLAG_SIMT_FFN)) return MOE_ERR_UNSUPPORTED;
    if (P.d % 128 || P.h % 128) return MOE_ERR_UNSUPPORTED;
    if (!w1 || !w2 || !s1 || !s2 || !aligned16(w1) || !aligned16(w2)) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(s1) & 3) || (reinterpret_cast<uintptr_t>(s2) & 3)) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

}  // namespace

namespace {

moe_status expert_ffn_impl(const moe_config* cfg, const void* x_dispatched, const int32_t* expert_offset,
                           const int32_t* row_token, const float* row_gate, const void* w1, const float* s1,
                           const void* b1, const void* w2, const float* s2, const void* b2, float* y_dispatched,
                           float* out, void* workspace, size_t workspace_bytes, void* stream) {
    Plan P;
    MOE_TRY(make_plan(cfg, &P));
    if (s1 || s2) MOE_TRY(check_fp8_weights(P, cfg, w1, s1, w2, s2));
    if (P.T == 0) return MOE_OK;
    MOE_TRY(check_ws(P, workspace, workspace_bytes));
    const void* ptrs[] = {x_dispatched, expert_offset, row_token, row_gate, w1, w2};
    for (const void* q : ptrs)
        if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
    if ((b1 && !aligned16(b1)) || (b2 && !aligned16(b2))) return MOE_ERR_INVALID_ARG;
    const bool fused = y_dispatched == nullptr;
    if (fused ? (!out || !aligned16(out)) : !aligned16(y_dispatched)) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(at<int>(workspace, P.o_err), 0, 8, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (fused) MOE_TRY(launch(s, [&] { return launch_zero(out, (size_t)P.T * P.d, s); }));
    return ffn_and_combine(P, cfg, x_dispatched, expert_offset, row_token, row_gate, w1, s1, b1, w2, s2, b2,
                           y_dispatched, out, fused, workspace, s);
}
}  // namespace

namespace {

// gate, dispatch ranks and scan, row gather of moe_forward, intermediates in the workspace (the error
// header must be zeroed first); `zero` [T, d] is cleared by the gather when not null
moe_status route_and_dispatch(const Plan& P, const moe_config* cfg, const void* x, const void* w_gate,
                              const void* w_noise, const float* noise_eps, const void* proj, const void* expert_emb,
                              int* count, float* zero, void* workspace, cudaStream_t s, bool with_stats = true) {
    int32_t* idx = at<int32_t>(workspace, P.o_idx);
    float* gate = at<float>(workspace, P.o_gate);
    int* err = at<int>(workspace, P.o_err);
    int* hist = at<int>(workspace, P.o_hist);
    int* off = at<int>(workspace, P.o_off);
    int* slot = at<int>(workspace, P.o_slot);
    int* rtok = at<int>(workspace, P.o_rtok);
    float* rgate = at<float>(workspace, P.o_rgate);
    void* xd = at<void>(workspace, P.o_xd);
    GateParams g = gate_params(P, cfg, x, w_gate, w_noise, noise_eps, proj, expert_emb, idx, gate);
    // with rank priority a gate kernel that ranks in token order leaves the ranking to the rank kernel
    const bool rank_after_gate = P.rank_major && gate_ranks_in_kernel(P);
    g.blk_hist = rank_after_gate ? nullptr : hist;
    g.slot = slot;
    g.err = err;
    // a small histogram (fused softmax gate) is scanned by the gather itself, every CTA for its own
    // blocks: the gate then skips its ticket and last-CTA scan
    const bool gather_scan = !P.rank_major && P.bf16 && P.gg.fused && P.E <= kGatherScanMaxE &&
                             (int64_t)P.nblk * P.E <= kGatherScanMaxHist;
    g.ticket = gather_scan ? nullptr : err + 2;
    g.C = P.Ceff;
    g.count = count;
    g.offset = off;
    g.row_token = rtok;
    g.row_gate = rgate;
    MOE_TRY(run_gate(P, g, workspace, s));
    if (rank_after_gate)
        MOE_TRY(launch(s, [&] {
            return launch_dispatch_rank(idx, P.T, P.k, P.E, hist, slot, err, err + 2, P.Ceff, count, off, rtok, rgate,
                                        1, s);
        }));
    GatherStats st{};
    if (P.stats && with_stats) {
        st.acc = at<unsigned long long>(workspace, P.o_fstats);
        st.ticket = reinterpret_cast<int*>(st.acc + P.E + 1);
        st.importance = at<float>(workspace, P.o_fstats_out);
        st.losses = st.importance + P.E;
        st.dropped = reinterpret_cast<long long*>(at<char>(workspace, P.o_fstats_out) + fstats_drop_at(P.E));
    }
    return launch(s, [&] {
        return launch_dispatch_gather(x, P.bf16, idx, gate, hist, off, count, gather_scan, P.T, P.k, P.E, P.d, P.Ceff,
                                      slot, rtok, rgate, xd, zero, P.rank_major, st, s);
    });
}

moe_status forward_impl(const moe_config* cfg, const void* x, const void* w_gate, const void* w_noise,
                        const float* noise_eps, const void* proj, const void* expert_emb, const void* w1,
                        const float* s1, const void* b1, const void* w2, const float* s2, const void* b2, float* out,
                        int32_t* expert_count, void* workspace, size_t workspace_bytes, void* stream) {
    Plan P;
    MOE_TRY(make_plan(cfg, &P));
    if (s1 || s2) MOE_TRY(check_fp8_weights(P, cfg, w1, s1, w2, s2));
    if (P.T == 0) return MOE_OK;
    MOE_TRY(check_ws(P, workspace, workspace_bytes));
    int32_t* idx = at<int32_t>(workspace, P.o_idx);
    float* gate = at<float>(workspace, P.o_gate);
    MOE_TRY(check_route_args(P, x, w_gate, w_noise, noise_eps, proj, expert_emb, idx, gate));
    if (!w1 || !w2 || !out || !aligned16(w1) || !aligned16(w2) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
    if ((b1 && !aligned16(b1)) || (b2 && !aligned16(b2)) || (expert_count && !aligned16(expert_count)))
        return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int* err = at<int>(workspace, P.o_err);
    int* count = expert_count ? expert_count : at<int>(workspace, P.o_count);
    int* off = at<int>(workspace, P.o_off);
    int* slot = at<int>(workspace, P.o_slot);
    int* rtok = at<int>(workspace, P.o_rtok);
    float* rgate = at<float>(workspace, P.o_rgate);
    void* xd = at<void>(workspace, P.o_xd);
    float* y = at<float>(workspace, P.o_y);
    // error word, its info, the block tickets and the cosine gate's expert flags start at zero
    if (cudaMemsetAsync(err, 0, P.hdr_bytes, s) != cudaSuccess) return MOE_ERR_CUDA;
    // the fused combine adds into `out`, cleared first: by the up projection's kernel when it can (in the
    // GEMM's shadow), else by the gather
    const bool clear_in_up = up_clears_out(P, cfg, s1);
    MOE_TRY(route_and_dispatch(P, cfg, x, w_gate, w_noise, noise_eps, proj, expert_emb, count,
                               P.fused && !clear_in_up ? out : nullptr, workspace, s));
    MOE_TRY(ffn_and_combine(P, cfg, xd, off, rtok, rgate, w1, s1, b1, w2, s2, b2, y, out, P.fused != 0, workspace, s,
                            clear_in_up));
    if (!P.fused) MOE_TRY(launch(s, [&] { return launch_combine(y, slot, off, idx, gate, P.T, P.k, P.d, out, s); }));
    return MOE_OK;
}

// ---- backward: its workspace after the forward's ------------------------------------------------------
struct BwdPlan {
    int Tp, Np, NpP;  // tokens rounded to 128, gate logits per token (and rounded to 64)
    size_t o_z, o_dy, o_dz, o_logits, o_dS, o_wcatT, o_dwcat, o_rows, o_off2, total;
};

moe_status make_bwd_plan(const Plan& P, const moe_config* c, BwdPlan* B) {
    if (!P.bf16 || P.gate == MOE_GATE_COSINE || (c->flags & MOE_FLAG_SIMT_FFN)) return MOE_ERR_UNSUPPORTED;
    BwdPlan b{};
    b.Tp = (P.T + 127) / 128 * 128;
    b.Np = P.gate == MOE_GATE_NOISY ? 2 * P.E : P.E;
    b.NpP = (b.Np + 63) / 64 * 64;
    size_t o = P.total;
    auto take = [&](size_t bytes) { size_t r = o; o = up(o + bytes); return r; };
    const size_t R = (size_t)P.rows;
    b.o_z = take(R * P.h * 2);
    b.o_dy = take(R * P.d * 2);
    b.o_dz = take(R * P.h * 2);
    b.o_logits = take((size_t)P.T * b.Np * 4);
    b.o_dS = take((size_t)b.Tp * b.NpP * 2);
    b.o_wcatT = take((size_t)P.d * b.NpP * 2);
    b.o_dwcat = take((size_t)b.Np * P.d * 4);
    b.o_rows = take((size_t)b.Tp * 4);
    b.o_off2 = take(8);
    b.total = o;
    *B = b;
    return MOE_OK;
}

moe_status backward_impl(const moe_config* cfg, const void* x, const void* w_gate, const void* w_noise,
                         const float* noise_eps, const void* w1, const void* b1, const void* w2, const void* b2,
                         const float* dout, float* dx, float* dw_gate, float* dw_noise, float* dw1, float* db1,
                         float* dw2, float* db2, void* ws, size_t ws_bytes, cudaStream_t s) {
    Plan P;
    MOE_TRY(make_plan(cfg, &P));
    BwdPlan B;
    MOE_TRY(make_bwd_plan(P, cfg, &B));
    if (P.T == 0) return MOE_OK;
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) || ws_bytes < B.total) return MOE_ERR_WORKSPACE;
    int32_t* idx = at<int32_t>(ws, P.o_idx);
    float* gate = at<float>(ws, P.o_gate);
    MOE_TRY(check_route_args(P, x, w_gate, w_noise, noise_eps, nullptr, nullptr, idx, gate));
    const void* need[] = {w1, w2, dout, dx, dw_gate, dw1, dw2};
    for (const void* q : need)
        if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
    if (P.gate == MOE_GATE_NOISY && (!dw_noise || !aligned16(dw_noise))) return MOE_ERR_INVALID_ARG;
    const void* opt[] = {b1, b2, db1, db2};
    for (const void* q : opt)
        if (q && !aligned16(q)) return MOE_ERR_INVALID_ARG;
    int* err = at<int>(ws, P.o_err);
    int* off = at<int>(ws, P.o_off);
    int* slot = at<int>(ws, P.o_slot);
    int* rtok = at<int>(ws, P.o_rtok);
    float* rgate = at<float>(ws, P.o_rgate);
    void* xd = at<void>(ws, P.o_xd);
    void* hb = at<void>(ws, P.o_h);
    float* y = at<float>(ws, P.o_y);
    const int T = P.T, d = P.d, h = P.h, E = P.E, R = (int)P.rows;
    if (cudaMemsetAsync(err, 0, P.hdr_bytes, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemsetAsync(dx, 0, (size_t)T * d * 4, s) != cudaSuccess) return MOE_ERR_CUDA;
    // 1. the forward again: routing and dispatch, Z and H = GELU(Z), y per dispatched row, and the gate logits
    MOE_TRY(route_and_dispatch(P, cfg, x, w_gate, w_noise, noise_eps, nullptr, nullptr, at<int>(ws, P.o_count),
                               nullptr, ws, s, false));
    FfnParams up = ffn_params(P, 4, xd, w1, nullptr, b1, off, rtok, rgate, hb, nullptr, err);
    up.aux = at<void>(ws, B.o_z);
    MOE_TRY(run_ffn(P, cfg, up, s));
    MOE_TRY(run_ffn(P, cfg, ffn_params(P, 1, hb, w2, nullptr, b2, off, rtok, rgate, y, nullptr, err), s));
    const GateGemmPlan one = gate_gemm_plan(T, d, P.N0, P.N1, 1, false);
    float* logits = at<float>(ws, B.o_logits);
    MOE_TRY(launch(s, [&] {
        return launch_gate_gemm(one, x, w_gate, P.gate == MOE_GATE_NOISY ? w_noise : nullptr, T, d, P.N0, P.N1,
                                logits, nullptr, nullptr, err, nullptr, s);
    }));
    // 2. dY = gate * dout per row; the gates' and scores' gradient per token
    void* dy = at<void>(ws, B.o_dy);
    void* dS = at<void>(ws, B.o_dS);
    const int* rows_used = off + E;  // offset[E]: rows past it were never dispatched
    MOE_TRY(launch(s, [&] { return launch_bwd_dy(dout, rtok, rgate, R, d, rows_used, dy, s); }));
    MOE_TRY(launch(s, [&] {
        return launch_bwd_gate(dout, y, idx, gate, slot, off, logits, noise_eps, T, B.Tp, d, E, P.k,
                               P.gate == MOE_GATE_NOISY, P.norm == MOE_GATE_NORM_ALL, B.NpP, dS, s);
    }));
    // 3. data gradients through the experts: dZ = (dY W2) * GELU'(Z), dx += dZ W1 (scattered to tokens); the
    //    GEMMs read W2 [E, d, h] and W1 [E, h, d] as they are, [E, K, N], MN-major
    void* dz = at<void>(ws, B.o_dz);
    FfnParams da{};
    da.A = dy; da.W = w2; da.w_kn = 1; da.offset = off; da.row_token = rtok; da.row_gate = rgate; da.C = dz;
    da.aux = at<void>(ws, B.o_z); da.E = E; da.K = d; da.N = h; da.bf16 = 1; da.mode = 3; da.rows_cap = P.rows;
    da.err = err;
    MOE_TRY(run_ffn(P, cfg, da, s));
    FfnParams dxe{};
    dxe.A = dz; dxe.W = w1; dxe.w_kn = 1; dxe.offset = off; dxe.row_token = rtok; dxe.row_gate = rgate; dxe.out = dx;
    dxe.E = E; dxe.K = h; dxe.N = d; dxe.bf16 = 1; dxe.mode = 5; dxe.rows_cap = P.rows; dxe.err = err;
    MOE_TRY(run_ffn(P, cfg, dxe, s));
    // 4. data gradient through the gate: dx += dS [W_g ; W_n]
    int* rows_id = at<int>(ws, B.o_rows);
    int* off2 = at<int>(ws, B.o_off2);
    void* wcatT = at<void>(ws, B.o_wcatT);
    MOE_TRY(launch(s, [&] { return launch_iota_rows(rows_id, T, B.Tp, off2, s); }));
    MOE_TRY(launch(s, [&] {
        return launch_gate_weights_t(w_gate, P.gate == MOE_GATE_NOISY ? w_noise : nullptr, E, d, B.NpP, wcatT, s);
    }));
    FfnParams dxg{};
    dxg.A = dS; dxg.W = wcatT; dxg.offset = off2; dxg.row_token = rows_id; dxg.out = dx;
    dxg.E = 1; dxg.K = B.NpP; dxg.N = d; dxg.bf16 = 1; dxg.mode = 5; dxg.rows_cap = B.Tp; dxg.err = err;
    MOE_TRY(run_ffn(P, cfg, dxg, s));
    // 5. weight gradients, contracting over each expert's rows: dW2 = dY^T H, dW1 = dZ^T X_d, with the
    //    operands read as stored ([rows, d] or [rows, h], MN-major); their padding rows are zeroed first (dY's
    //    already are)
    MOE_TRY(launch(s, [&] { return launch_zero_pad_rows(xd, d, hb, h, dz, h, R, rtok, rows_used, s); }));
    MOE_TRY(launch(s, [&] {
        return launch_wgrad_tc(WgradParams{dy, hb, off, dw2, E, d, h, (int64_t)R, (int64_t)R, err}, s);
    }));
    MOE_TRY(launch(s, [&] {
        return launch_wgrad_tc(WgradParams{dz, xd, off, dw1, E, h, d, (int64_t)R, (int64_t)R, err}, s);
    }));
    // 6. gate weight gradients: [dW_g ; dW_n] = dS^T x, contracting over the tokens (x's rows past T read as 0)
    float* dwcat = at<float>(ws, B.o_dwcat);
    MOE_TRY(launch(s, [&] {
        return launch_wgrad_tc(WgradParams{dS, x, off2, dwcat, 1, B.Np, d, (int64_t)B.Tp, (int64_t)T, err, B.NpP}, s);
    }));
    if (cudaMemcpyAsync(dw_gate, dwcat, (size_t)E * d * 4, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (P.gate == MOE_GATE_NOISY &&
        cudaMemcpyAsync(dw_noise, dwcat + (size_t)E * d, (size_t)E * d * 4, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    // 7. bias gradients: column sums over each expert's rows
    if (db2) MOE_TRY(launch(s, [&] { return launch_segment_colsum(dy, off, E, d, db2, s); }));
    if (db1) MOE_TRY(launch(s, [&] { return launch_segment_colsum(dz, off, E, h, db1, s); }));
    return MOE_OK;
}

}  // namespace

namespace moe {
int32_t config_status(const void* cfg) {
    Plan P;
    return make_plan(static_cast<const moe_config*>(cfg), &P);
}
}  // namespace moe

extern "C" {

int32_t moe_capacity(const moe_config* cfg) {
    Plan P;
    return make_plan(cfg, &P) == MOE_OK ? P.C : -1;
}

int64_t moe_dispatch_rows(const moe_config* cfg) {
    Plan P;
    return make_plan(cfg, &P) == MOE_OK ? P.rows : -1;
}

size_t moe_workspace_size(const moe_config* cfg) {
    Plan P;
    return make_plan(cfg, &P) == MOE_OK ? P.total : 0;
}

int32_t moe_forward_launches(const moe_config* cfg) {
    Plan P;
    if (make_plan(cfg, &P) != MOE_OK) return -1;
    if (P.T == 0) return 0;
    const int gate_extra = P.bf16 && !P.gg.fused ? 3 + (P.gate == MOE_GATE_COSINE ? 1 : 0) : 0;
    const int rank_extra = P.rank_major && gate_ranks_in_kernel(P) ? 1 : 0;  // a separate rank kernel
    return (P.fused ? 4 : 5) + gate_extra + rank_extra;
}

moe_status moe_route(const moe_config* cfg, const void* x, const void* w_gate, const void* w_noise,
                     const float* noise_eps, const void* proj, const void* expert_emb, int32_t* topk_idx,
                     float* topk_gate, void* workspace, size_t workspace_bytes, void* stream) {
    NvtxRange nvtx_("moe_route");
    Plan P;
    MOE_TRY(make_plan(cfg, &P));
    if (P.T == 0) return MOE_OK;
    MOE_TRY(check_ws(P, workspace, workspace_bytes));
    MOE_TRY(check_route_args(P, x, w_gate, w_noise, noise_eps, proj, expert_emb, topk_idx, topk_gate));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int* err = at<int>(workspace, P.o_err);
    if (cudaMemsetAsync(err, 0, P.hdr_bytes, s) != cudaSuccess) return MOE_ERR_CUDA;
    GateParams g = gate_params(P, cfg, x, w_gate, w_noise, noise_eps, proj, expert_emb, topk_idx, topk_gate);
    g.err = err;
    return run_gate(P, g, workspace, s);
}

moe_status moe_gate_logits(const moe_config* cfg, const void* x, const void* w_gate, const void* w_noise,
                           const void* proj, float* logits, void* workspace, size_t workspace_bytes, void* stream) {
    NvtxRange nvtx_("moe_gate_logits");
    Plan P;
    MOE_TRY(make_plan(cfg, &P));
    if (!P.bf16) return MOE_ERR_UNSUPPORTED;
    if (P.T == 0) return MOE_OK;
    MOE_TRY(check_ws(P, workspace, workspace_bytes));
    const void* w0 = P.gate == MOE_GATE_COSINE ? proj : w_gate;
    const void* w1 = P.gate == MOE_GATE_NOISY ? w_noise : nullptr;
    if (!x || !logits || !w0 || !aligned16(x) || !aligned16(logits) || !aligned16(w0)) return MOE_ERR_INVALID_ARG;
    if (P.gate == MOE_GATE_NOISY && (!w1 || !aligned16(w1))) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int* err = at<int>(workspace, P.o_err);
    if (cudaMemsetAsync(err, 0, 8, s) != cudaSuccess) return MOE_ERR_CUDA;
    const GateGemmPlan one = gate_gemm_plan(P.T, P.d, P.N0, P.N1, 1, false);  // one split, logits out
    return launch(s, [&] {
        return launch_gate_gemm(one, x, w0, w1, P.T, P.d, P.N0, P.N1, logits, nullptr, nullptr, err, nullptr, s);
    });
}

moe_status moe_dispatch(const moe_config* cfg, const void* x, const int32_t* topk_idx, const float* topk_gate,
                        int32_t* slot, int32_t* expert_count, int32_t* expert_offset, int32_t* row_token,
                        float* row_gate, void* x_dispatched, void* workspace, size_t workspace_bytes, void* stream) {
    NvtxRange nvtx_("moe_dispatch");
    Plan P;
    MOE_TRY(make_plan(cfg, &P));
    if (P.T == 0) return MOE_OK;
    MOE_TRY(check_ws(P, workspace, workspace_bytes));
    const void* ptrs[] = {x, topk_idx, topk_gate, slot, expert_count, expert_offset, row_token, row_gate, x_dispatched};
    for (const void* q : ptrs)
        if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int* err = at<int>(workspace, P.o_err);
    int* hist = at<int>(workspace, P.o_hist);
    // error word, its info and the rank step's CTA ticket start at zero
    if (cudaMemsetAsync(err, 0, 16, s) != cudaSuccess) return MOE_ERR_CUDA;
    MOE_TRY(launch(s, [&] {
        return launch_dispatch_rank(topk_idx, P.T, P.k, P.E, hist, slot, err, err + 2, P.Ceff, expert_count,
                                    expert_offset, row_token, row_gate, P.rank_major, s);
    }));
    return launch(s, [&] {
        return launch_dispatch_gather(x, P.bf16, topk_idx, topk_gate, hist, expert_offset, nullptr, false, P.T, P.k,
                                      P.E, P.d, P.Ceff,
                                      slot, row_token, row_gate, x_dispatched, nullptr, P.rank_major, GatherStats{}, s);
    });
}


moe_status moe_expert_ffn(const moe_config* cfg, const void* x_dispatched, const int32_t* expert_offset,
                          const int32_t* row_token, const float* row_gate, const void* w1, const void* b1,
                          const void* w2, const void* b2, float* y_dispatched, float* out, void* workspace,
                          size_t workspace_bytes, void* stream) {
    NvtxRange nvtx_("moe_expert_ffn");
    return expert_ffn_impl(cfg, x_dispatched, expert_offset, row_token, row_gate, w1, nullptr, b1, w2, nullptr, b2,
                           y_dispatched, out, workspace, workspace_bytes, stream);
}

moe_status moe_expert_ffn_fp8(const moe_config* cfg, const void* x_dispatched, const int32_t* expert_offset,
                              const int32_t* row_token, const float* row_gate, const uint8_t* w1_q,
                              const float* w1_scale, const void* b1, const uint8_t* w2_q, const float* w2_scale,
                              const void* b2, float* y_dispatched, float* out, void* workspace,
                              size_t workspace_bytes, void* stream) {
    NvtxRange nvtx_("moe_expert_ffn_fp8");
    if (!w1_scale || !w2_scale) return MOE_ERR_INVALID_ARG;
    return expert_ffn_impl(cfg, x_dispatched, expert_offset, row_token, row_gate, w1_q, w1_scale, b1, w2_q, w2_scale,
                           b2, y_dispatched, out, workspace, workspace_bytes, stream);
}

moe_status moe_combine(const moe_config* cfg, const float* y_dispatched, const int32_t* slot,
                       const int32_t* expert_offset, const int32_t* topk_idx, const float* topk_gate, float* out,
                       void* stream) {
    NvtxRange nvtx_("moe_combine");
    Plan P;
    MOE_TRY(make_plan(cfg, &P));
    if (P.T == 0) return MOE_OK;
    const void* ptrs[] = {y_dispatched, slot, expert_offset, topk_idx, topk_gate, out};
    for (const void* q : ptrs)
        if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return launch(s, [&] {
        return launch_combine(y_dispatched, slot, expert_offset, topk_idx, topk_gate, P.T, P.k, P.d, out, s);
    });
}


moe_status moe_forward(const moe_config* cfg, const void* x, const void* w_gate, const void* w_noise,
                       const float* noise_eps, const void* proj, const void* expert_emb, const void* w1,
                       const void* b1, const void* w2, const void* b2, float* out, int32_t* expert_count,
                       void* workspace, size_t workspace_bytes, void* stream) {
    NvtxRange nvtx_("moe_forward");
    return forward_impl(cfg, x, w_gate, w_noise, noise_eps, proj, expert_emb, w1, nullptr, b1, w2, nullptr, b2, out,
                        expert_count, workspace, workspace_bytes, stream);
}

moe_status moe_forward_fp8(const moe_config* cfg, const void* x, const void* w_gate, const void* w_noise,
                           const float* noise_eps, const void* proj, const void* expert_emb, const uint8_t* w1_q,
                           const float* w1_scale, const void* b1, const uint8_t* w2_q, const float* w2_scale,
                           const void* b2, float* out, int32_t* expert_count, void* workspace, size_t workspace_bytes,
                           void* stream) {
    NvtxRange nvtx_("moe_forward_fp8");
    if (!w1_scale || !w2_scale) return MOE_ERR_INVALID_ARG;
    return forward_impl(cfg, x, w_gate, w_noise, noise_eps, proj, expert_emb, w1_q, w1_scale, b1, w2_q, w2_scale, b2,
                        out, expert_count, workspace, workspace_bytes, stream);
}

size_t moe_backward_workspace_size(const moe_config* cfg) {
    Plan P;
    BwdPlan B;
    if (make_plan(cfg, &P) != MOE_OK || make_bwd_plan(P, cfg, &B) != MOE_OK) return 0;
    return B.total;
}

moe_status moe_backward(const moe_config* cfg, const void* x, const void* w_gate, const void* w_noise,
                        const float* noise_eps, const void* w1, const void* b1, const void* w2, const void* b2,
                        const float* dout, float* dx, float* dw_gate, float* dw_noise, float* dw1, float* db1,
                        float* dw2, float* db2, void* workspace, size_t workspace_bytes, void* stream) {
    NvtxRange nvtx_("moe_backward");
    return backward_impl(cfg, x, w_gate, w_noise, noise_eps, w1, b1, w2, b2, dout, dx, dw_gate, dw_noise, dw1, db1,
                         dw2, db2, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

moe_status moe_router_stats(const moe_config* cfg, const int32_t* topk_idx, const float* topk_gate,
                            const int32_t* slot, float* importance, float* losses, int64_t* dropped,
                            void* workspace, size_t workspace_bytes, void* stream) {
    NvtxRange nvtx_("moe_router_stats");
    Plan P;
    MOE_TRY(make_plan(cfg, &P));
    MOE_TRY(check_ws(P, workspace, workspace_bytes));
    if (!importance || !losses || !aligned16(importance) || !aligned16(losses)) return MOE_ERR_INVALID_ARG;
    if (P.T > 0 && (!topk_idx || !topk_gate || !aligned16(topk_idx) || !aligned16(topk_gate)))
        return MOE_ERR_INVALID_ARG;
    if ((slot && !aligned16(slot)) || (dropped && (reinterpret_cast<uintptr_t>(dropped) & 7))) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int* err = at<int>(workspace, P.o_err);
    void* scratch = at<void>(workspace, P.o_fstats);  // in the header: one memset clears both
    if (cudaMemsetAsync(err, 0, P.hdr_bytes, s) != cudaSuccess) return MOE_ERR_CUDA;
    return launch(s, [&] {
        return launch_router_stats(topk_idx, topk_gate, slot, P.T, P.k, P.E, scratch, err, importance, losses,
                                   reinterpret_cast<long long*>(dropped), s);
    });
}

moe_status moe_router_stats_result(const moe_config* cfg, const void* workspace, size_t workspace_bytes,
                                   float* importance, float* losses, int64_t* dropped, void* stream) {
    Plan P;
    MOE_TRY(make_plan(cfg, &P));
    if (!P.stats) return MOE_ERR_INVALID_ARG;
    MOE_TRY(check_ws(P, const_cast<void*>(workspace), workspace_bytes));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const char* res = static_cast<const char*>(workspace) + P.o_fstats_out;
    if (importance && cudaMemcpyAsync(importance, res, 4 * (size_t)P.E, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (losses && cudaMemcpyAsync(losses, res + 4 * (size_t)P.E, 8, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (dropped && cudaMemcpyAsync(dropped, res + fstats_drop_at(P.E), 8, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

moe_status moe_device_status(void* workspace, size_t workspace_bytes, int32_t* info, void* stream) {
    if (workspace == nullptr || workspace_bytes < 16) return MOE_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t w[2] = {0, 0};
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemcpy(w, workspace, sizeof w, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemset(workspace, 0, sizeof w) != cudaSuccess) return MOE_ERR_CUDA;
    if (info) *info = w[1];
    if (w[0] == 0) return MOE_OK;
    return w[0] == MOE_ERR_DEVICE_TIMEOUT ? MOE_ERR_DEVICE_TIMEOUT : MOE_ERR_DEVICE_CHECK;
}

void moe_trace_events(void** events, int32_t capacity) {
    if (events == nullptr || capacity <= 0) {  // off; the count of the last trace stays readable
        g_events = nullptr;
        g_capacity = 0;
        return;
    }
    g_events = events;
    g_capacity = capacity;
    g_recorded = 0;
}

int32_t moe_trace_count(void) { return g_recorded; }

const char* moe_status_string(moe_status status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
        case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case MOE_ERR_CUDA: return "CUDA runtime error";
        case MOE_ERR_DEVICE_CHECK: return "device-side check failed";
        case MOE_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
        default: return "unknown status";
    }
}

}  // extern "C"
