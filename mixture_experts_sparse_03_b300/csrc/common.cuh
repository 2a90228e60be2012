// common.cuh -- device helpers shared by the kernels of libmoe_b300 (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"

namespace moe {

using bf16_t = uint16_t;  // raw bits of a bfloat16; converted with the helpers below

// error word at the start of the workspace: [0] = status code, [1] = which kernel recorded it
enum : int { kErrCheck = 5, kErrTimeout = 6 };
enum : int {
    kWhereGate = 1, kWhereDispatch = 2, kWhereFfnSimt = 3, kWhereGemmProducer = 4, kWhereGemmMma = 5,
    kWhereGemmEpilogue = 6, kWhereCombine = 7, kWhereGateGemm = 8, kWhereRouterStats = 9
};

// ---- programmatic dependent launch ------------------------------------------------------------------
// Every kernel is launched so that the next one in the stream may start (prologue: barriers, TMEM,
// descriptor prefetch) while this one finishes.  A kernel calls pdl_wait() before it touches global
// memory (it returns once the preceding grids have completed and their writes are visible), then
// pdl_trigger() to let its own successor launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

__device__ __forceinline__ void record_error(int* err, int code, int where) {
    if (err != nullptr && atomicCAS(err, 0, code) == 0) atomicExch(err + 1, where);
}

// ---- bf16 <-> fp32 ------------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
__device__ __forceinline__ float bf16_to_f32(bf16_t b) { return __uint_as_float(uint32_t(b) << 16); }

// round to nearest even, two values packed low | high << 16
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// 8 consecutive elements -> fp32 (16-byte aligned source)
__device__ __forceinline__ void load8(const bf16_t* p, float v[8]) {
    uint4 u = *reinterpret_cast<const uint4*>(p);
    v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x); v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
    v[4] = bf16_lo(u.z); v[5] = bf16_hi(u.z); v[6] = bf16_lo(u.w); v[7] = bf16_hi(u.w);
}
__device__ __forceinline__ void load8(const float* p, float v[8]) {
    float4 a = *reinterpret_cast<const float4*>(p);
    float4 b = *reinterpret_cast<const float4*>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ float load1(const bf16_t* p) { return bf16_to_f32(*p); }
__device__ __forceinline__ float load1(const float* p) { return *p; }

__device__ __forceinline__ void store1(bf16_t* p, float v) {
    unsigned short h;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(v));
    *p = h;
}
__device__ __forceinline__ void store1(float* p, float v) { *p = v; }

// ---- float-float (doubled single precision) ------------------------------------------------------
// Knuth's TwoSum and the FMA-based TwoProduct: a + b = s + e and a * b = p + e exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = a + b;
    float bb = s - a;
    e = (a - (s - bb)) + (b - bb);
}
__device__ __forceinline__ void two_prod(float a, float b, float& p, float& e) {
    p = a * b;
    e = fmaf(a, b, -p);
}
// (hi, lo) += a * b, keeping about 48 significant bits
__device__ __forceinline__ void ff_fma(float& hi, float& lo, float a, float b) {
    float p, pe, s, se;
    two_prod(a, b, p, pe);
    two_sum(hi, p, s, se);
    hi = s;
    lo += se + pe;
}
__device__ __forceinline__ void ff_add(float& hi, float& lo, float ohi, float olo) {
    float s, se;
    two_sum(hi, ohi, s, se);
    hi = s;
    lo += se + olo;
}
// Kahan's compensated summation, (hi, lo) += v with lo the running correction of hi: over n addends the
// result hi + lo errs by at most 2u * sum |v| + O(n u^2) (u = 2^-24), at four additions per addend
__device__ __forceinline__ void kahan_add(float& hi, float& lo, float v) {
    const float y = v + lo;
    const float t = hi + y;
    lo = y - (t - hi);
    hi = t;
}
__device__ __forceinline__ void ff_warp_sum(float& hi, float& lo) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        float oh = __shfl_xor_sync(0xffffffffu, hi, off);
        float ol = __shfl_xor_sync(0xffffffffu, lo, off);
        ff_add(hi, lo, oh, ol);
    }
}

// named CTA barrier `id` over `count` threads (whole warps): arrive without waiting, or wait for all
__device__ __forceinline__ void named_bar_arrive(int id, int count) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// GELU with the erf form, z/2 (1 + erf(z / sqrt 2)) (the exact GELU, not the tanh approximation).
// erf comes from Abramowitz & Stegun, Handbook of Mathematical Functions, formula 7.1.26: for x >= 0,
// 1 - erf(x) = t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) e^(-x^2), t = 1 / (1 + p x), |error| <= 1.5e-7.
// With Q = 1 - erf(|z| / sqrt 2), 1 + erf(z / sqrt 2) is 2 - Q for z >= 0 and Q for z < 0, so the
// negative side keeps its small values without cancellation.  The hidden activations are rounded to
// bf16 (relative step 2^-8) right after, far above this error.
__device__ __forceinline__ float gelu_erf(float z) {
    const float x = fabsf(z) * 0.70710678118654752f;
    float t;  // 1 / (1 + p x) with the hardware's approximate reciprocal (relative error ~2^-23)
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(t) : "f"(fmaf(0.3275911f, x, 1.0f)));
    float p = fmaf(t, 1.061405429f, -1.453152027f);
    p = fmaf(t, p, 1.421413741f);
    p = fmaf(t, p, -0.284496736f);
    p = fmaf(t, p, 0.254829592f);
    const float q = p * t * __expf(-x * x);
    return 0.5f * z * (z >= 0.0f ? 2.0f - q : q);
}

// GELU'(z) = Phi(z) + z phi(z) (the derivative of the erf-form GELU), with Phi from the same
// Abramowitz & Stegun 7.1.26 erf as gelu_erf; phi(z) = e^(-z^2/2) / sqrt(2 pi) reuses its exponential.
__device__ __forceinline__ float gelu_grad(float z) {
    const float x = fabsf(z) * 0.70710678118654752f;
    float t;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(t) : "f"(fmaf(0.3275911f, x, 1.0f)));
    float p = fmaf(t, 1.061405429f, -1.453152027f);
    p = fmaf(t, p, 1.421413741f);
    p = fmaf(t, p, -0.284496736f);
    p = fmaf(t, p, 0.254829592f);
    const float ex = __expf(-x * x);  // e^(-z^2 / 2)
    const float q = p * t * ex;
    return 0.5f * (z >= 0.0f ? 2.0f - q : q) + z * ex * 0.3989422804014327f;
}

// expert owning dispatched row r: the e with off[e] <= r < off[e+1] (off ascending, E+1 entries)
__device__ __forceinline__ int expert_of_row(const int* off, int E, int r) {
    int lo = 0, hi = E;  // invariant: off[lo] <= r < off[hi]
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (off[mid] <= r) lo = mid; else hi = mid;
    }
    return lo;
}

}  // namespace moe
