// gate_common.cuh -- device helpers shared by the gate kernels (gate.cu, gate_select.cu).
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace gate {

constexpr int kMaxCand = kMaxCandidates;       // contenders re-scored per token
constexpr float kU = 5.9604644775390625e-08f;  // 2^-24
constexpr int kGateSoftmax = 0, kGateNoisy = 1, kGateCosine = 2;

__device__ __forceinline__ float softplus_f(float z) {
    // log(1 + e^z); the second form is the same function written to avoid overflow of e^z
    return z > 20.0f ? z + log1pf(expf(-z)) : log1pf(expf(z));
}

template <typename T>
__device__ __forceinline__ const T* logit_row(const GateParams& P, int gate, int n) {
    if (gate == kGateCosine) return static_cast<const T*>(P.proj) + (size_t)n * P.d;
    if (gate == kGateNoisy && n >= P.E) return static_cast<const T*>(P.w_noise) + (size_t)(n - P.E) * P.d;
    return static_cast<const T*>(P.w_gate) + (size_t)n * P.d;
}

// monotone map of a float onto uint32 (order of the keys = order of the values; -0 and +0 map alike)
__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t u = __float_as_uint(f + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// (hi, lo) += a * b: for bf16 operands the product is exact in fp32 (8-bit significands), so only the
// addition needs the error-free transformation
template <typename T>
__device__ __forceinline__ void ff_acc(float& hi, float& lo, float a, float b) {
    if constexpr (sizeof(T) == 2) {
        float s, e;
        two_sum(hi, a * b, s, e);
        hi = s;
        lo += e;
    } else {
        ff_fma(hi, lo, a, b);
    }
}

// float-float dot product of two length-d rows by one warp (lanes take 8-element slices); the loads of
// four slices per lane are issued before any arithmetic, and the four slices go to separate (hi, lo)
// accumulators so that their latencies overlap
template <typename T>
__device__ __forceinline__ double warp_dot_ff(const T* a, const T* b, int d, int lane) {
    float hi[4] = {0.f, 0.f, 0.f, 0.f}, lo[4] = {0.f, 0.f, 0.f, 0.f};
    for (int i0 = lane * 8; i0 < d; i0 += 4 * 32 * 8) {
        float va[4][8], vb[4][8];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * 32 * 8;
            if (i < d) {
                load8(a + i, va[u]);
                load8(b + i, vb[u]);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) va[u][j] = vb[u][j] = 0.f;
            }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int u = 0; u < 4; ++u) ff_acc<T>(hi[u], lo[u], va[u][j], vb[u][j]);
    }
    ff_add(hi[0], lo[0], hi[1], lo[1]);
    ff_add(hi[2], lo[2], hi[3], lo[3]);
    ff_add(hi[0], lo[0], hi[2], lo[2]);
    ff_warp_sum(hi[0], lo[0]);
    return (double)hi[0] + (double)lo[0];
}

// float-float dot products of one length-d row a with up to four rows b[0..nb) by one warp: the loads of
// all rows' slices are in flight together (one round of memory latency for all of them, not nb rounds)
template <typename T>
__device__ __forceinline__ void warp_dot_ff4(const T* a, const T* const (&b)[4], int nb, int d, int lane,
                                             double (&out)[4]) {
    float hi[4] = {0.f, 0.f, 0.f, 0.f}, lo[4] = {0.f, 0.f, 0.f, 0.f};
    for (int i = lane * 8; i < d; i += 32 * 8) {
        float va[8], vb[4][8];
        load8(a + i, va);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (u < nb) {
                load8(b[u] + i, vb[u]);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) vb[u][j] = 0.f;
            }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int u = 0; u < 4; ++u) ff_acc<T>(hi[u], lo[u], va[j], vb[u][j]);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        ff_warp_sum(hi[u], lo[u]);
        out[u] = (double)hi[u] + (double)lo[u];
    }
}

}  // namespace gate
}  // namespace moe
