// kernels.h -- host-side launchers of the kernels in this directory (internal to libmoe_b300).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

constexpr int kMaxTopK = 16;
constexpr int kMaxExperts = 1024;
constexpr int kRowAlign = 128;       // each expert's dispatched rows start on a multiple of this
constexpr int kTokensPerBlock = 32;  // gate and dispatch both cut the tokens into blocks of this size

// ---- gate -------------------------------------------------------------------------------------
struct GateParams {
    const void* x;
    const void* w_gate;
    const void* w_noise;
    const float* eps;
    const void* proj;
    const void* emb;
    int T, d, E, k, p;      // p = cosine projection width (0 otherwise)
    int gate, norm, bf16;
    float inv_temp;         // 1 / cos_temperature in fp32
    double temp;            // cos_temperature
    int* topk_idx;          // [T, k]
    float* topk_gate;       // [T, k]
    int* blk_hist;          // [ceil(T/32), E] per-block expert histogram, or nullptr
    int* slot;              // [T, k] receives each pair's rank within its block (with blk_hist)
    int* err;               // error word or nullptr
    // dispatch scan fused into the gate's last block (when ticket != nullptr; needs blk_hist)
    int* ticket;            // zero-initialised counter of finished blocks (reset by the last block)
    int C;                  // capacity
    int* count;             // [E]
    int* offset;            // [E+1]
    int* row_token;         // padding rows get -1
    float* row_gate;        // padding rows get 0
    // logits precomputed by the tensor-core GEMM (bf16 layers): partials [S][T][Np], summed in split
    // order, with the squared norms of the x rows [S][T] and weight rows [S][Np]; nullptr -> the gate
    // kernel computes the logits itself on CUDA cores
    const float* part;
    const float* xn2p;
    const float* wn2p;
    int S, Np;
    float cb;               // logit error bound = cb * |x_t| * |w_n| (+ 4u |logit|)
    // re-scoring of near ties (selection from precomputed logits): tokens with near ties go to a global
    // queue of kRescoreInts-int entries that the rescore kernel works through with every SM
    int* rq_count;          // zero-initialised entry counter
    int* rq;                // [T][kRescoreInts]
    int* need;              // cosine: [E] zero-initialised flags, set for experts that contend somewhere
    float2* cosv;           // cosine: [E][d] v_e = P^T e_e as float-float (hi, lo), flagged experts only
};
constexpr int kMaxCandidates = 64;                          // contenders re-scored per token
constexpr int kRescoreInts = 4 + 2 * kMaxCandidates;       // token, count, m, den, ids, fp32 scores
size_t gate_smem_bytes(int gate, int E, int p, int d);  // CUDA-core gate (fp32 layers)
size_t gate_select_smem_bytes(int gate, int E, int p);  // selection from precomputed logits
cudaError_t launch_gate_select(const GateParams& p, cudaStream_t s);
cudaError_t launch_gate_cos_fold(const GateParams& p, cudaStream_t s);  // cosine: p.cosv for p.need
cudaError_t launch_gate_rescore(const GateParams& p, cudaStream_t s);   // works through p.rq

// ---- gate logits GEMM on the tensor cores (gate_tc.cu) ------------------------------------------
constexpr int kGateMaxSplits = 8;
constexpr int kPlanSms = 148;  // SM count the split-K plan (and so the workspace size) assumes
struct GateGemmPlan {
    int BN;        // logits per n-tile (multiple of 16, <= 128)
    bool both;     // one n-tile holds both weight tensors' rows (N0 == N1, a multiple of 8, 2 N0 <= 128)
    int nch;       // TMEM accumulators the MMAs rotate through
    int nt0, nt1;  // n-tiles over the first / second weight tensor
    int mt;        // 128-token tiles
    int kb;        // 64-wide K blocks
    int per;       // K blocks per split
    int S;         // splits of K
    int Np;        // logits per token (N0 + N1)
    bool fused;    // selection fused into the GEMM's epilogue (no partials, no selection kernel)
    int cs;        // fused: CTAs per 128-token tile, a cluster splitting K (partials added in shared memory)
    int stages;    // TMA ring depth
    size_t smem;   // dynamic shared memory per CTA
};
GateGemmPlan gate_gemm_plan(int T, int d, int N0, int N1, int sms, bool fuse_select);
// part [S][T][Np] (S = plan.S) receives the partial logits; xn2_part [S][T] and wn2_part [S][Np]
// the partial squared norms (either may be nullptr to skip)
// sel: the selection's parameters (ids, gates, dispatch outputs; cb set) when g.fused, else ignored
cudaError_t launch_gate_gemm(const GateGemmPlan& g, const void* x, const void* w0, const void* w1, int T, int d,
                             int N0, int N1, float* part, float* xn2_part, float* wn2_part, int* err,
                             const GateParams* sel, cudaStream_t s);
cudaError_t launch_gate(const GateParams& p, cudaStream_t s);

// ---- dispatch ---------------------------------------------------------------------------------
// rank step over all tokens; the last CTA to finish (counted on `ticket`, a zero-initialised int that
// it resets) runs the scan: count[E], offset[E+1] and the padding rows of row_token / row_gate, with
// capacity C
// rank_major: pairs numbered in (rank, token) order, blocks of 32 such pairs (blk_hist [ceil(T k/32), E])
cudaError_t launch_dispatch_rank(const int* topk_idx, int T, int k, int E, int* blk_hist, int* rank, int* err,
                                 int* ticket, int C, int* count, int* offset, int* row_token, float* row_gate,
                                 int rank_major, cudaStream_t s);
inline int dispatch_hist_blocks(int T, int k, int rank_major) {
    return rank_major ? (int)(((long)T * k + kTokensPerBlock - 1) / kTokensPerBlock)
                      : (T + kTokensPerBlock - 1) / kTokensPerBlock;
}
// slot [T, k] holds the block ranks on entry (from the rank step or the gate kernel) and the slots on exit
// scan = false: blk_hist holds the scanned block prefixes and offset the segment offsets (from the rank
// step's scan, in (rank, token) order when rank_major); scan = true (token order only) (E <= kGatherScanMaxE): blk_hist holds the raw block histograms and the
// gather does the scan's work itself -- it writes count (if not null), offset and the padding rows
// router statistics fused into the gather: acc [E + 1] (expert sums as multiples of 2^-32, then the drop
// count) and ticket zero on entry (reset by the last CTA); results: importance [E], losses [2], dropped
struct GatherStats {
    unsigned long long* acc;  // nullptr: no statistics
    int* ticket;
    float* importance;
    float* losses;
    long long* dropped;
};
constexpr int kGatherScanMaxE = 64;
constexpr int kGatherScanMaxHist = 2048;  // ints of histogram every gather CTA reads
cudaError_t launch_dispatch_gather(const void* x, int bf16, const int* topk_idx, const float* topk_gate,
                                   const int* blk_hist, int* offset, int* count, bool scan, int T, int k, int E,
                                   int d, int C, int* slot, int* row_token, float* row_gate, void* x_dispatched,
                                   float* out_to_zero, int rank_major, const GatherStats& stats, cudaStream_t s);

// ---- expert FFN -------------------------------------------------------------------------------
// mode: 0 = up projection (+b1, GELU, store hidden), 1 = down projection to y (fp32),
//       2 = down projection with the combine fused (atomic fp32 add of gate * y into out),
//       3 = (backward) times GELU'(aux) into bf16, 4 = up projection storing Z (aux) and GELU(Z),
//       5 = (backward) atomic fp32 add into out[row_token] with gate 1
struct FfnParams {
    const void* A;            // [rows, K] dispatched activations (x_dispatched or hidden)
    const void* W;            // [E, N, K]
    const void* bias;         // [E, N] or nullptr
    const int* offset;        // [E+1]
    const int* row_token;     // [rows]
    const float* row_gate;    // [rows]
    void* C;                  // mode 0: hidden [rows, N] (dtype); mode 1: y [rows, N] fp32
    float* out;               // mode 2: [T, N] fp32
    int E, K, N, bf16, mode;
    int pair;                 // tensor-core kernel on pairs of SMs (256 x 256 tiles)
    int64_t rows_cap;
    int* err;
    const float* w_scale;     // block-FP8 weights: W holds E4M3 codes, w_scale [E, N/128, K/128]; else nullptr
    void* aux;                // modes 3 / 4 (backward): pre-activations Z [rows, N] bf16
    int max_rows;             // most rows any expert holds (its capacity, at most the token count); 0: unknown
    int w_kn;                 // W is [E, K, N] instead (bf16, single-SM tensor-core kernel): read MN-major
    float* zero;              // mode 0, single-SM tensor-core kernel: an fp32 buffer of zero_n floats (a multiple
    int64_t zero_n;           // of 4, 16-byte aligned) that one extra warp per CTA clears meanwhile, or nullptr
};
size_t ffn_fp8_smem_bytes(int E, bool bias, int ring, bool swap);
// weight gradients grouped along K (ffn_tc.cu): dW[e] [M, N] fp32 = sum over the rows r of expert e
// (offset[e] <= r < offset[e+1], multiples of 64) of A[r][m] B[r][n], both operands read MN-major
struct WgradParams {
    const void* A;      // [rows, M] bf16, row-major (M contiguous)
    const void* B;      // [rows_b, N] bf16, row-major (N contiguous); rows_b <= rows: the rest reads as 0
    const int* offset;  // [E+1]
    float* dW;          // [E, M, N]
    int E, M, N;
    int64_t rows;       // rows of A (segments of offset lie below it; multiples of 64)
    int64_t rows_b;     // rows of B
    int* err;
    int a_ld;           // elements per row of A (>= M, a multiple of 8); 0: M
};
cudaError_t launch_wgrad_tc(const WgradParams& p, cudaStream_t s);
cudaError_t launch_ffn_simt(const FfnParams& p, cudaStream_t s);
cudaError_t launch_ffn_tc(const FfnParams& p, cudaStream_t s);  // bf16 only; tcgen05 + TMA

// ---- combine / misc ---------------------------------------------------------------------------
// router statistics: scratch holds E + 1 uint64 and an int, zero on entry (router_stats.cu)
cudaError_t launch_router_stats(const int* topk_idx, const float* topk_gate, const int* slot, int T, int k, int E,
                                void* scratch, int* err, float* importance, float* losses, long long* dropped,
                                cudaStream_t s);
cudaError_t launch_combine(const float* y, const int* slot, const int* offset, const int* topk_idx,
                           const float* topk_gate, int T, int k, int d, float* out, cudaStream_t s);
cudaError_t launch_zero(float* p, size_t n, cudaStream_t s);

// ---- backward (bwd.cu) ------------------------------------------------------------------------------
// dst[b][c][r] = src[b][r][c] (bf16) for r < R, zero for R <= r < Rp; with row_mask, zero where
// row_mask[r] < 0 and from row *row_limit on (device int: the dispatched rows in use, offset[E])
// padding rows (row_token < 0, below *row_limit) of up to three bf16 row-major buffers [rows, width_i] set
// to zero, so that contractions over whole row segments see exact zeros there
cudaError_t launch_zero_pad_rows(void* p0, int w0, void* p1, int w1, void* p2, int w2, int rows,
                                 const int* row_token, const int* row_limit, cudaStream_t s);
// dY[r] = row_gate[r] * dout[row_token[r]] in bf16 (zero for padding rows and from row *row_limit on)
cudaError_t launch_bwd_dy(const float* dout, const int* row_token, const float* row_gate, int rows, int d,
                          const int* row_limit, void* dY, cudaStream_t s);
// per token: the gates' and scores' gradient, dS [Tp, Np] bf16 = [ds | dn (noisy) | 0]
cudaError_t launch_bwd_gate(const float* dout, const float* y, const int* topk_idx, const float* topk_gate,
                            const int* slot, const int* offset, const float* logits, const float* eps, int T, int Tp,
                            int d, int E, int k, int noisy, int norm_all, int Np, void* dS, cudaStream_t s);
// db[e][c] = column sums of src [rows, C] (bf16) over expert e's row segment (its padding rows hold zeros)
cudaError_t launch_segment_colsum(const void* src, const int* offset, int E, int C, float* db, cudaStream_t s);
// out [d][Np] = [W_g ; W_n ; 0]^T
cudaError_t launch_gate_weights_t(const void* wg, const void* wn, int E, int d, int Np, void* out, cudaStream_t s);
// rows[i] = i for i < T, -1 up to Tp; off2 = {0, Tp}
cudaError_t launch_iota_rows(int* rows, int T, int Tp, int* off2, cudaStream_t s);

// ---- configuration ------------------------------------------------------------------------------
// The status the library's own planner gives a config (MOE_OK, MOE_ERR_INVALID_ARG or
// MOE_ERR_UNSUPPORTED), so that every entry point reports a bad config the same way.
int32_t config_status(const void* cfg);

}  // namespace moe
