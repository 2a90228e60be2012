// combine.cu -- gate-weighted combine back into token order, Output = sum_i g_i(x) E_i(x) (the layer
// formula of "MoE on a single card", section 1.2), and a zero fill.
//
// One warp per token, 16-byte loads: out[t] = sum over ranks j = 0..k-1 (in that order) of the kept
// pairs of gate[t, j] * y[off[e] + slot[t, j]]; a token with every pair dropped gets 0.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y, const int* __restrict__ slot,
                                                      const int* __restrict__ offset, const int* __restrict__ topk_idx,
                                                      const float* __restrict__ topk_gate, int T, int k, int d,
                                                      float* __restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (t >= T) return;
    int rows[kMaxTopK];
    float g[kMaxTopK];
    for (int j = 0; j < k; ++j) {
        const int s = slot[(size_t)t * k + j];
        rows[j] = s >= 0 ? offset[topk_idx[(size_t)t * k + j]] + s : -1;
        g[j] = topk_gate[(size_t)t * k + j];
    }
    const int n4 = d / 4;
    float4* o = reinterpret_cast<float4*>(out + (size_t)t * d);
    for (int i = lane; i < n4; i += 32) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {
            if (rows[j] < 0) continue;
            const float4 v = reinterpret_cast<const float4*>(y + (size_t)rows[j] * d)[i];
            acc.x = fmaf(g[j], v.x, acc.x);
            acc.y = fmaf(g[j], v.y, acc.y);
            acc.z = fmaf(g[j], v.z, acc.z);
            acc.w = fmaf(g[j], v.w, acc.w);
        }
        o[i] = acc;
    }
}

__global__ void zero_kernel(float4* __restrict__ p, size_t n4) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x)
        p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

}  // namespace

cudaError_t launch_combine(const float* y, const int* slot, const int* offset, const int* topk_idx,
                           const float* topk_gate, int T, int k, int d, float* out, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    combine_kernel<<<(T + 7) / 8, 256, 0, s>>>(y, slot, offset, topk_idx, topk_gate, T, k, d, out);
    return cudaGetLastError();
}

cudaError_t launch_zero(float* p, size_t n, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    const size_t n4 = n / 4;  // n is a multiple of 4 (d is a multiple of 64)
    unsigned blocks = (unsigned)((n4 + 255) / 256);
    if (blocks > 148u * 16u) blocks = 148u * 16u;
    zero_kernel<<<blocks, 256, 0, s>>>(reinterpret_cast<float4*>(p), n4);
    return cudaGetLastError();
}

}  // namespace moe
