// dispatch.cu -- capacity-limited dispatch: group the (token, expert) pairs by expert, in token order.
//
// Tokens are grouped by the expert they chose before the per-group matmuls ("How sparse activation
// improves efficiency", section 3.1), under a per-expert capacity (capacity_factor in the "Tutel MoE
// guide", where 1.2 admits 20 % more than an even share; the CANN MOELayer of "MoE sparse-compute
// acceleration", section 3.2), with overflow pairs dropped.
// Slot of pair (t, e) = number of pairs of earlier tokens routed to e; kept iff slot < C.
//
// Three steps over blocks of 32 tokens (the gate kernel's blocks, so within moe_forward the gate
// produces step 1 and its last block runs step 2, see scan.cuh):
//   count   per-block expert histogram                          blk_hist[b][e]
//   scan    per expert: exclusive prefix over blocks (in place), total count, kept = min(count, C),
//           padded segment offsets off[e] = sum_{e'<e} roundup(kept[e'], 128), padding rows marked
//   assign  warp 0 walks the block's pairs in token order in chunks of 32; __match_any_sync gives
//           each pair its rank among equal experts in the chunk, a shared running counter per expert
//           carries the order across chunks; then all warps copy the kept rows of x with 16-byte
//           loads and stores (and zero the block's output rows when the combine is fused)
// No step depends on scheduling order, so the result is deterministic.
#include "common.cuh"
#include "kernels.h"
#include "scan.cuh"

namespace moe {

namespace {

constexpr int kBT = kTokensPerBlock;

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__global__ void __launch_bounds__(256) count_kernel(const int* __restrict__ topk_idx, int T, int k, int E,
                                                    int* __restrict__ blk_hist, int* err) {
    __shared__ int hist[kMaxExperts];
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const int t0 = blockIdx.x * kBT;
    const int n = min(kBT, T - t0) * k;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        int e = topk_idx[(size_t)t0 * k + i];
        if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
        else record_error(err, kErrCheck, kWhereDispatch);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) blk_hist[(size_t)blockIdx.x * E + e] = hist[e];
}

// one block of 1024 threads
__global__ void __launch_bounds__(1024) scan_kernel(int* __restrict__ blk_hist, int nblk, int E, int C,
                                                    int* __restrict__ count, int* __restrict__ offset,
                                                    int* __restrict__ row_token, float* __restrict__ row_gate) {
    __shared__ int part[1024];
    __shared__ int padded[kMaxExperts + 1];
    __shared__ int kept[kMaxExperts];
    __shared__ int wsum[33];
    ScanSmem sm{part, padded, kept, wsum};
    scan_experts(blk_hist, nblk, E, C, count, offset, row_token, row_gate, sm);
}

template <typename T>
__global__ void __launch_bounds__(1024) assign_kernel(const T* __restrict__ x, const int* __restrict__ topk_idx,
                                                     const float* __restrict__ topk_gate,
                                                     const int* __restrict__ blk_base, const int* __restrict__ offset,
                                                     int T_, int k, int E, int d, int C, int* __restrict__ slot,
                                                     int* __restrict__ row_token, float* __restrict__ row_gate,
                                                     T* __restrict__ xd, float* __restrict__ out_zero, int* err) {
    __shared__ int running[kMaxExperts];
    __shared__ int prow[kBT * kMaxTopK];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t0 = blockIdx.x * kBT;
    const int ntok = min(kBT, T_ - t0);
    const int npairs = ntok * k;
    for (int e = tid; e < E; e += blockDim.x) running[e] = blk_base[(size_t)blockIdx.x * E + e];
    __syncthreads();
    if (warp == 0) {
        for (int c0 = 0; c0 < npairs; c0 += 32) {
            const int p = c0 + lane;
            const bool valid = p < npairs;
            int e = valid ? topk_idx[(size_t)t0 * k + p] : -1;
            if (valid && (e < 0 || e >= E)) {
                record_error(err, kErrCheck, kWhereDispatch);
                e = -2;  // matches no expert; dropped below
            }
            const unsigned mask = __match_any_sync(0xffffffffu, e);
            const int rank = __popc(mask & lanemask_lt());
            const bool real = valid && e >= 0;
            const int base = real ? running[e] : 0;
            __syncwarp();
            if (real && rank == 0) running[e] = base + __popc(mask);
            __syncwarp();
            if (valid) {
                const int s = base + rank;
                int r = -1;
                if (real && s < C) r = offset[e] + s;
                slot[(size_t)t0 * k + p] = r >= 0 ? s : -1;
                prow[p] = r;
                if (r >= 0) {
                    row_token[r] = t0 + p / k;
                    row_gate[r] = topk_gate[(size_t)t0 * k + p];
                }
            }
        }
    }
    __syncthreads();
    // row gather, 16 bytes per lane per step, four loads in flight per lane
    constexpr int V = 16 / sizeof(T);
    const int nv = d / V;
    for (int p = warp; p < npairs; p += blockDim.x / 32) {
        const int r = prow[p];
        if (r < 0) continue;
        const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)(t0 + p / k) * d);
        uint4* dst = reinterpret_cast<uint4*>(xd + (size_t)r * d);
        for (int i0 = lane; i0 < nv; i0 += 4 * 32) {
            uint4 v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (i0 + j * 32 < nv) v[j] = __ldg(src + i0 + j * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (i0 + j * 32 < nv) dst[i0 + j * 32] = v[j];
        }
    }
    if (out_zero != nullptr) {
        const int n4 = d / 4;
        for (int tt = warp; tt < ntok; tt += blockDim.x / 32) {
            float4* o = reinterpret_cast<float4*>(out_zero + (size_t)(t0 + tt) * d);
            for (int i = lane; i < n4; i += 32) o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
}

}  // namespace

cudaError_t launch_dispatch_count(const int* topk_idx, int T, int k, int E, int* blk_hist, int* err,
                                  cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    count_kernel<<<(T + kBT - 1) / kBT, 256, 0, s>>>(topk_idx, T, k, E, blk_hist, err);
    return cudaGetLastError();
}

cudaError_t launch_dispatch_scan(int* blk_hist, int T, int k, int E, int C, int* count, int* offset,
                                 int* row_token, float* row_gate, cudaStream_t s) {
    (void)k;
    if (T <= 0) return cudaSuccess;
    const int nblk = (T + kBT - 1) / kBT;
    scan_kernel<<<1, 1024, 0, s>>>(blk_hist, nblk, E, C, count, offset, row_token, row_gate);
    return cudaGetLastError();
}

cudaError_t launch_dispatch_assign(const void* x, int bf16, const int* topk_idx, const float* topk_gate,
                                   const int* blk_hist, const int* offset, int T, int k, int E, int d, int C,
                                   int* slot, int* row_token, float* row_gate, void* x_dispatched,
                                   float* out_to_zero, int* err, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    const int blocks = (T + kBT - 1) / kBT;
    if (bf16)
        assign_kernel<bf16_t><<<blocks, 1024, 0, s>>>(static_cast<const bf16_t*>(x), topk_idx, topk_gate, blk_hist,
                                                     offset, T, k, E, d, C, slot, row_token, row_gate,
                                                     static_cast<bf16_t*>(x_dispatched), out_to_zero, err);
    else
        assign_kernel<float><<<blocks, 1024, 0, s>>>(static_cast<const float*>(x), topk_idx, topk_gate, blk_hist,
                                                    offset, T, k, E, d, C, slot, row_token, row_gate,
                                                    static_cast<float*>(x_dispatched), out_to_zero, err);
    return cudaGetLastError();
}

}  // namespace moe
