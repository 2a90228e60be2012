// combine.cu -- gate-weighted combine back into token order, Output = sum_i g_i(x) E_i(x) (the layer
// formula of "MoE on a single card", section 1.2), and a zero fill.
//
// One thread per 4 consecutive outputs: out[t] = sum over ranks j = 0..k-1 (in that order) of the kept
// pairs of gate[t, j] * y[off[e] + slot[t, j]], all k rows loaded before the sum; a token with every
// pair dropped gets 0.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y, const int* __restrict__ slot,
                                                      const int* __restrict__ offset, const int* __restrict__ topk_idx,
                                                      const float* __restrict__ topk_gate, int T, int k, int d,
                                                      float* __restrict__ out) {
    pdl_wait();
    pdl_trigger();
    const int n4 = d / 4;
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (size_t)T * n4) return;
    const int t = (int)(i / n4), c = (int)(i - (size_t)t * n4);
    // all k rows' loads first, then the sum in rank order
    float4 v[kMaxTopK];
    float g[kMaxTopK];
    unsigned kept = 0;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
        v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        g[j] = 0.f;
        if (j < k) {
            const int s = slot[(size_t)t * k + j];
            if (s >= 0) {
                const int r = offset[topk_idx[(size_t)t * k + j]] + s;
                v[j] = reinterpret_cast<const float4*>(y + (size_t)r * d)[c];
                g[j] = topk_gate[(size_t)t * k + j];
                kept |= 1u << j;
            }
        }
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
        if ((kept >> j) & 1u) {
            acc.x = fmaf(g[j], v[j].x, acc.x);
            acc.y = fmaf(g[j], v[j].y, acc.y);
            acc.z = fmaf(g[j], v[j].z, acc.z);
            acc.w = fmaf(g[j], v[j].w, acc.w);
        }
    }
    reinterpret_cast<float4*>(out + (size_t)t * d)[c] = acc;
}

__global__ void zero_kernel(float4* __restrict__ p, size_t n4) {
    pdl_wait();
    pdl_trigger();
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x)
        p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

}  // namespace

cudaError_t launch_combine(const float* y, const int* slot, const int* offset, const int* topk_idx,
                           const float* topk_gate, int T, int k, int d, float* out, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    const size_t n = (size_t)T * (d / 4);
    return launch_pdl(combine_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, y, slot, offset, topk_idx,
                      topk_gate, T, k, d, out);
}

cudaError_t launch_zero(float* p, size_t n, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    const size_t n4 = n / 4;  // n is a multiple of 4 (d is a multiple of 64)
    unsigned blocks = (unsigned)((n4 + 255) / 256);
    if (blocks > 148u * 16u) blocks = 148u * 16u;
    return launch_pdl(zero_kernel, dim3(blocks), dim3(256), 0, s, reinterpret_cast<float4*>(p), n4);
}

}  // namespace moe
