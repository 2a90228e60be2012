// ffn_simt.cu -- grouped expert FFN on CUDA cores (fp32 FMA; the fp32 layer's path and a bf16
// cross-check path).  The expert is Linear -> GELU -> Linear (CANN MOELayer example; Tutel 'ffn').
//
// Dispatched rows are grouped by expert in segments padded to 128 rows, so every 64-row tile belongs
// to one expert (found by binary search in the segment offsets).  Tile 64 x 64, 256 threads, 4 x 4
// outputs per thread, reduction chunks of 32 staged (transposed) in shared memory.  Epilogues:
//   mode 0  hidden = GELU(acc + b1)         stored in the layer dtype (bf16 rounds to nearest even)
//   mode 1  y = acc + b2                    stored fp32
//   mode 2  out[token] += gate * (acc + b2) fp32 atomic add (the fused combine)
// Padding rows (row_token < 0) are computed but never stored.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kTile = 64, kKC = 32, kSS = kTile + 4;

template <typename T>
__global__ void __launch_bounds__(256) ffn_simt_kernel(const FfnParams P) {
    __shared__ __align__(16) float As[kKC * kSS];
    __shared__ __align__(16) float Bs[kKC * kSS];
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x;
    const int r0 = blockIdx.x * kTile;
    const int total = P.offset[P.E];
    if (r0 >= total) return;
    const int e = expert_of_row(P.offset, P.E, r0);
    const int n0 = blockIdx.y * kTile;
    const int K = P.K, N = P.N;
    const T* A = static_cast<const T*>(P.A);
    const T* W = static_cast<const T*>(P.W) + (size_t)e * N * K;
    const int lrow = tid >> 2, lc8 = (tid & 3) * 8;
    const int ty = tid >> 4, tx = tid & 15;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    const T* arow = A + (size_t)(r0 + lrow) * K;
    const T* wrow = (n0 + lrow < N) ? W + (size_t)(n0 + lrow) * K : nullptr;
    for (int k0 = 0; k0 < K; k0 += kKC) {
        float va[8], vb[8];
        load8(arow + k0 + lc8, va);
        if (wrow) load8(wrow + k0 + lc8, vb);
        else {
#pragma unroll
            for (int j = 0; j < 8; ++j) vb[j] = 0.f;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            As[(lc8 + j) * kSS + lrow] = va[j];
            Bs[(lc8 + j) * kSS + lrow] = vb[j];
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < kKC; ++kk) {
            float4 a = *reinterpret_cast<const float4*>(&As[kk * kSS + ty * 4]);
            float4 b = *reinterpret_cast<const float4*>(&Bs[kk * kSS + tx * 4]);
            const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }
    const T* bias = static_cast<const T*>(P.bias);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = r0 + ty * 4 + i;
        const int tok = P.row_token[r];
        if (tok < 0) continue;
        const float g = P.mode == 2 ? P.row_gate[r] : 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n >= N) continue;
            float v = acc[i][j];
            if (bias) v += load1(bias + (size_t)e * N + n);
            if (P.mode == 0) store1(static_cast<T*>(P.C) + (size_t)r * N + n, gelu_erf(v));
            else if (P.mode == 1) static_cast<float*>(P.C)[(size_t)r * N + n] = v;
            else atomicAdd(P.out + (size_t)tok * N + n, g * v);
        }
    }
}

}  // namespace

cudaError_t launch_ffn_simt(const FfnParams& P, cudaStream_t s) {
    if (P.rows_cap <= 0) return cudaSuccess;
    dim3 grid((unsigned)((P.rows_cap + kTile - 1) / kTile), (unsigned)((P.N + kTile - 1) / kTile));
    cudaError_t e = P.bf16 ? launch_pdl(ffn_simt_kernel<bf16_t>, grid, dim3(256), 0, s, P)
                           : launch_pdl(ffn_simt_kernel<float>, grid, dim3(256), 0, s, P);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace moe
