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
    int* err;               // error word or nullptr
    // dispatch scan fused into the gate's last block (when ticket != nullptr; needs blk_hist)
    int* ticket;            // zero-initialised counter of finished blocks (reset by the last block)
    int C;                  // capacity
    int* count;             // [E]
    int* offset;            // [E+1]
    int* row_token;         // padding rows get -1
    float* row_gate;        // padding rows get 0
};
size_t gate_smem_bytes(int gate, int E, int p, int d);
cudaError_t launch_gate(const GateParams& p, cudaStream_t s);

// ---- dispatch ---------------------------------------------------------------------------------
cudaError_t launch_dispatch_count(const int* topk_idx, int T, int k, int E, int* blk_hist, int* err,
                                  cudaStream_t s);
cudaError_t launch_dispatch_scan(int* blk_hist, int T, int k, int E, int C, int* count, int* offset,
                                 int* row_token, float* row_gate, cudaStream_t s);
cudaError_t launch_dispatch_assign(const void* x, int bf16, const int* topk_idx, const float* topk_gate,
                                   const int* blk_hist, const int* offset, int T, int k, int E, int d, int C,
                                   int* slot, int* row_token, float* row_gate, void* x_dispatched,
                                   float* out_to_zero, int* err, cudaStream_t s);

// ---- expert FFN -------------------------------------------------------------------------------
// mode: 0 = up projection (+b1, GELU, store hidden), 1 = down projection to y (fp32),
//       2 = down projection with the combine fused (atomic fp32 add of gate * y into out)
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
    int64_t rows_cap;
    int* err;
};
cudaError_t launch_ffn_simt(const FfnParams& p, cudaStream_t s);
cudaError_t launch_ffn_tc(const FfnParams& p, cudaStream_t s);  // bf16 only; tcgen05 + TMA

// ---- combine / misc ---------------------------------------------------------------------------
cudaError_t launch_combine(const float* y, const int* slot, const int* offset, const int* topk_idx,
                           const float* topk_gate, int T, int k, int d, float* out, cudaStream_t s);
cudaError_t launch_zero(float* p, size_t n, cudaStream_t s);

}  // namespace moe
