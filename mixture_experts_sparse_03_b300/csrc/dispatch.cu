// dispatch.cu -- capacity-limited dispatch: group the (token, expert) pairs by expert, in token order.
//
// Tokens are grouped by the expert they chose before the per-group matmuls ("How sparse activation
// improves efficiency", section 3.1), under a per-expert capacity (capacity_factor in the "Tutel MoE
// guide", where 1.2 admits 20 % more than an even share; the CANN MOELayer of "MoE sparse-compute
// acceleration", section 3.2), with overflow pairs dropped.
// Slot of pair (t, e) = number of pairs of earlier tokens routed to e; kept iff slot < C.
//
// Three steps over blocks of 32 tokens (the gate kernels' blocks: the fp32 gate kernel and the fused
// bf16 gate do step 1 on their own tokens and run step 2 in their last block, see scan.cuh; when the
// histogram is small -- the fused gate's usual case -- every gather CTA does step 2's work for its own
// blocks instead, and the gate skips it):
//   rank    a warp per block, 32 blocks per CTA: each pair's rank among the block's pairs of the same
//           expert, in token order (kept in `slot` until the gather), and the block's expert histogram
//           blk_hist[b][e]; the last CTA to finish runs the scan
//   scan    per expert: exclusive prefix over blocks (in place), total count, kept = min(count, C),
//           padded segment offsets off[e] = sum_{e'<e} roundup(kept[e'], 128), padding rows marked
//   gather  one warp per pair: slot = prefix[b][e] + rank, kept iff slot < C, row = off[e] + slot;
//           the row of x is copied with 16-byte loads, eight in flight per lane; the same grid also
//           zeroes the output when the combine is fused into the expert GEMM
// With rank priority (every token's first choice before any second choice) the rank and gather steps
// walk the pairs in (rank, token) order instead: virtual item v = j * T + t stands for pair (t, j), and
// the blocks are 32 consecutive virtual items, so the same rank / scan / gather machinery numbers them.
// No step depends on scheduling order, so the result is deterministic.
#include "common.cuh"
#include "kernels.h"
#include "scan.cuh"

namespace moe {

namespace {

constexpr int kBT = kTokensPerBlock;
constexpr int kGatherWarps = 8;  // warps (pairs) per gather block
constexpr int kRankWarps = 32;   // token blocks per rank CTA, a warp each
static_assert(kGatherWarps <= kBT, "a gather CTA's pairs span at most two token blocks");

__global__ void __launch_bounds__(32 * kRankWarps) rank_kernel(const int* __restrict__ topk_idx, int T, int k,
                                                              int E, int* __restrict__ blk_hist,
                                                              int* __restrict__ rank, int* err, int* ticket, int C,
                                                              int* count, int* offset, int* row_token,
                                                              float* row_gate, int rank_major) {
    extern __shared__ int running_all[];  // [kRankWarps][E]
    __shared__ int part[32 * kRankWarps];
    __shared__ int padded[kMaxExperts + 1];
    __shared__ int kept[kMaxExperts];
    __shared__ int wsum[33];
    __shared__ int last;
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nblk = rank_major ? (int)(((long)T * k + kBT - 1) / kBT) : (T + kBT - 1) / kBT;
    const int b = blockIdx.x * kRankWarps + warp;
    if (b < nblk) {
        int* running = running_all + (size_t)warp * E;
        for (int e = lane; e < E; e += 32) running[e] = 0;
        __syncwarp();
        bool bad = false;
        auto checked = [&](int e) {
            const bool ok = e >= 0 && e < E;
            bad |= !ok;
            return ok ? e : -2;  // an out-of-range id takes no slot
        };
        if (rank_major) {  // 32 virtual items v = j * T + t, item i of the block is pair (t, j)
            const long v0 = (long)b * kBT;
            auto pair_of = [&](int i) { const long v = v0 + i; return (v % T) * k + v / T; };
            rank_pairs_warp_to([&](int i) { return checked(topk_idx[pair_of(i)]); },
                               (int)min((long)kBT, (long)T * k - v0), running,
                               [&](int i, int r) { rank[pair_of(i)] = r; }, lane);
        } else {
            const int t0 = b * kBT;
            const int* ids = topk_idx + (size_t)t0 * k;
            rank_pairs_warp([&](int i) { return checked(ids[i]); }, min(kBT, T - t0) * k, running,
                            rank + (size_t)t0 * k, lane);
        }
        if (bad) record_error(err, kErrCheck, kWhereDispatch);
        __syncwarp();
        for (int e = lane; e < E; e += 32) blk_hist[(size_t)b * E + e] = running[e];
    }
    // the last CTA to finish runs the scan over every block's histogram
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        last = atomicAdd(ticket, 1) == (int)gridDim.x - 1;
        __threadfence();
    }
    __syncthreads();
    if (last) {
        ScanSmem sm{part, padded, kept, wsum};
        scan_experts(blk_hist, nblk, E, C, count, offset, row_token, row_gate, sm);
        if (threadIdx.x == 0) *ticket = 0;  // ready for the next call
    }
}

// Router statistics fused into the gather (moe_forward with MOE_FLAG_ROUTER_STATS): each CTA adds its
// pairs' gates -- every top-k gate, kept or dropped -- to the experts' 64-bit fixed-point sums (a gate is
// a multiple of 2^-32 after rounding, so the sums are exact and independent of the order of the adds)
// and its dropped pairs to a counter; the last CTA to finish (ticket) turns the sums into the importance
// and the two losses, in fp64 in a fixed order, and resets the accumulators for the next call.
__device__ __forceinline__ double block_sum_d256(double v, double* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_sum_d(v);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    double s = 0.0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += red[w];
    return s;
}

__device__ void fused_router_stats(const GatherStats& st, int E, int warp, int lane, int e, float gv, bool counted,
                                   bool dropped) {
    constexpr double kFix = 4294967296.0;  // 2^32
    __shared__ int s_e[kGatherWarps];
    __shared__ unsigned long long s_g[kGatherWarps];
    __shared__ int s_drop[kGatherWarps];
    __shared__ int s_last;
    __shared__ double s_red[kGatherWarps];
    if (lane == 0) {
        s_e[warp] = counted ? e : -1;
        s_g[warp] = counted ? (unsigned long long)llrint((double)gv * kFix) : 0ull;
        s_drop[warp] = dropped ? 1 : 0;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int nd = 0;
        for (int w = 0; w < kGatherWarps; ++w) {
            nd += s_drop[w];
            if (s_e[w] < 0) continue;
            unsigned long long sum = s_g[w];
            for (int v = w + 1; v < kGatherWarps; ++v)  // the CTA's pairs of the same expert, one add
                if (s_e[v] == s_e[w]) { sum += s_g[v]; s_e[v] = -1; }
            atomicAdd(st.acc + s_e[w], sum);
        }
        if (nd) atomicAdd(st.acc + E, (unsigned long long)nd);
        __threadfence();
        s_last = atomicAdd(st.ticket, 1) == (int)gridDim.x - 1;
        __threadfence();
    }
    __syncthreads();
    if (!s_last) return;
    double s = 0.0;
    for (int i = threadIdx.x; i < E; i += blockDim.x) s += (double)__ldcg(st.acc + i) / kFix;
    const double mean = block_sum_d256(s, s_red) / (double)E;
    double ss = 0.0;
    for (int i = threadIdx.x; i < E; i += blockDim.x) {
        const double v = (double)__ldcg(st.acc + i) / kFix;
        st.importance[i] = (float)v;
        ss += (mean - v) * (mean - v);
    }
    ss = block_sum_d256(ss, s_red);
    __syncthreads();
    if (threadIdx.x == 0) {
        st.losses[0] = E > 1 ? (float)(0.1 * sqrt(ss / (double)(E - 1))) : __int_as_float(0x7fc00000);
        st.losses[1] = (float)ss;
        *st.dropped = (long long)__ldcg(st.acc + E);
    }
    __syncthreads();  // every thread has read the sums
    for (int i = threadIdx.x; i <= E; i += blockDim.x) st.acc[i] = 0ull;
    if (threadIdx.x == 0) *st.ticket = 0;
}

// SCAN: blk_hist holds each block's raw expert histogram and every CTA derives what it needs itself
// (E <= kGatherScanMaxE): the prefix of its one or two token blocks, the expert totals and the padded
// segment offsets; CTA 0 writes count and offset, CTA c writes the padding rows of experts c, c + grid,
// ...  Otherwise blk_hist holds the scanned prefixes and offset the segment offsets.
template <typename T, bool SCAN>
__global__ void __launch_bounds__(32 * kGatherWarps) gather_kernel(
    const T* __restrict__ x, const int* __restrict__ topk_idx, const float* __restrict__ topk_gate,
    const int* __restrict__ blk_hist, int* __restrict__ offset, int* __restrict__ count, int T_, int k, int E,
    int d, int C, int* __restrict__ slot, int* __restrict__ row_token, float* __restrict__ row_gate,
    T* __restrict__ xd, float* __restrict__ out_zero, int rank_major, const GatherStats stats) {
    __shared__ int s_pre[2][kGatherScanMaxE];  // prefix of blocks b_lo and b_lo + 1
    __shared__ int s_off[kGatherScanMaxE + 1];
    __shared__ int s_kept[kGatherScanMaxE];
    __shared__ int s_part[3][32 * kGatherWarps];
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31, tid = threadIdx.x;
    const long npairs = (long)T_ * k;
    const long p = (long)blockIdx.x * kGatherWarps + (threadIdx.x >> 5);
    const int t = p < npairs ? (int)(p / k) : 0;
    constexpr int V = 16 / sizeof(T);
    const int nv = d / V;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d);
    // the token's row is known before its routing: its first 8 x 32 16-byte pieces are loaded while the
    // pair's expert, rank and block prefix are still on their way
    uint4 v[8];
    int e = -1, rk = -1;
    float gv = 0.f;
    if (p < npairs) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (lane + j * 32 < nv) v[j] = __ldg(src + lane + j * 32);
        e = topk_idx[p];
        rk = slot[p];  // the block rank, replaced by the slot below
        gv = topk_gate[p];
    }
    const int b_lo = (int)(((long)blockIdx.x * kGatherWarps / k) / kBT);
    if constexpr (SCAN) {
        // thread (g, e) sums rows g, g + G, ... of the histogram: those before b_lo, row b_lo, and all
        const int nblk = (T_ + kBT - 1) / kBT;
        const int G = (32 * kGatherWarps) / E, g = tid / E, e = tid - g * E;
        int lo = 0, mid = 0, tot = 0;
        if (g < G) {
            for (int b = g; b < nblk; b += G) {
                const int c = blk_hist[(size_t)b * E + e];
                tot += c;
                lo += b < b_lo ? c : 0;
                mid += b == b_lo ? c : 0;
            }
        }
        s_part[0][tid] = lo;
        s_part[1][tid] = mid;
        s_part[2][tid] = tot;
        __syncthreads();
        if (tid < E) {
            int a = 0, m = 0, n = 0;
            for (int gg = 0; gg < G; ++gg) {
                a += s_part[0][gg * E + tid];
                m += s_part[1][gg * E + tid];
                n += s_part[2][gg * E + tid];
            }
            s_pre[0][tid] = a;
            s_pre[1][tid] = a + m;
            const int kept = min(n, C);
            s_kept[tid] = kept;
            s_off[tid] = (kept + kRowAlign - 1) / kRowAlign * kRowAlign;  // padded size, scanned below
            if (blockIdx.x == 0 && count != nullptr) count[tid] = n;
        }
        __syncthreads();
        if (tid < 32) {  // exclusive scan of the padded sizes (E <= 64: two per lane)
            const int i0 = 2 * lane, i1 = 2 * lane + 1;
            const int a0 = i0 < E ? s_off[i0] : 0, a1 = i1 < E ? s_off[i1] : 0;
            int inc = a0 + a1;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += u;
            }
            const int ex = inc - a0 - a1;
            __syncwarp();
            if (i0 < E) s_off[i0] = ex;
            if (i1 < E) s_off[i1] = ex + a0;
            if (lane == 31) s_off[E] = inc;
        }
        __syncthreads();
        if (blockIdx.x == 0)
            for (int q = tid; q <= E; q += 32 * kGatherWarps) offset[q] = s_off[q];
        for (int c = blockIdx.x; c < E; c += gridDim.x)  // padding rows of expert c
            for (int i = tid; i < kRowAlign; i += 32 * kGatherWarps) {
                const int r = s_off[c] + s_kept[c] + i;
                if (r < s_off[c + 1]) {
                    row_token[r] = -1;
                    row_gate[r] = 0.f;
                }
            }
    }
    int s_final = -1;  // this pair's slot (the same in every lane of the warp)
    if (p < npairs) {
        int s = -1, r = -1;
        if (rk >= 0 && e >= 0 && e < E) {
            const int b = t / kBT;
            if constexpr (SCAN) {
                s = s_pre[b - b_lo][e] + rk;  // a CTA's 8 pairs span at most two token blocks
                if (s < C) r = s_off[e] + s;
                else s = -1;
            } else {
                // rank priority: the pair's block in (rank, token) order
                const int bb = rank_major ? (int)(((long)(p % k) * T_ + t) / kBT) : b;
                s = blk_hist[(size_t)bb * E + e] + rk;
                if (s < C) r = offset[e] + s;
                else s = -1;
            }
        }
        s_final = s;
        __syncwarp();
        if (lane == 0) {
            slot[p] = s;
            if (r >= 0) {
                row_token[r] = t;
                row_gate[r] = gv;
            }
        }
        if (r >= 0) {
            uint4* dst = reinterpret_cast<uint4*>(xd + (size_t)r * d);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (lane + j * 32 < nv) dst[lane + j * 32] = v[j];
            for (int i0 = lane + 8 * 32; i0 < nv; i0 += 8 * 32) {  // rows longer than 4 KiB
                uint4 w[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (i0 + j * 32 < nv) w[j] = __ldg(src + i0 + j * 32);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (i0 + j * 32 < nv) dst[i0 + j * 32] = w[j];
            }
        }
    }
    if (stats.acc != nullptr) {
        const bool counted = p < npairs && e >= 0 && e < E;
        fused_router_stats(stats, E, threadIdx.x >> 5, lane, e, gv, counted, counted && s_final < 0);
    }
    if (out_zero != nullptr) {
        const size_t n4 = (size_t)T_ * d / 4;
        float4* o = reinterpret_cast<float4*>(out_zero);
        for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x)
            o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

}  // namespace

cudaError_t launch_dispatch_rank(const int* topk_idx, int T, int k, int E, int* blk_hist, int* rank, int* err,
                                 int* ticket, int C, int* count, int* offset, int* row_token, float* row_gate,
                                 int rank_major, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    const int nblk = rank_major ? (int)(((long)T * k + kBT - 1) / kBT) : (T + kBT - 1) / kBT;
    const size_t smem = sizeof(int) * (size_t)kRankWarps * E;
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(rank_kernel, dim3((nblk + kRankWarps - 1) / kRankWarps), dim3(32 * kRankWarps), smem, s,
                      topk_idx, T, k, E, blk_hist, rank, err, ticket, C, count, offset, row_token, row_gate,
                      rank_major);
}

cudaError_t launch_dispatch_gather(const void* x, int bf16, const int* topk_idx, const float* topk_gate,
                                   const int* blk_hist, int* offset, int* count, bool scan, int T, int k, int E,
                                   int d, int C, int* slot, int* row_token, float* row_gate, void* x_dispatched,
                                   float* out_to_zero, int rank_major, const GatherStats& stats, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    if (scan && (E > kGatherScanMaxE || rank_major)) return cudaErrorInvalidValue;
    const long npairs = (long)T * k;
    const unsigned blocks = (unsigned)((npairs + kGatherWarps - 1) / kGatherWarps);
    const dim3 grid(blocks), block(32 * kGatherWarps);
    if (bf16) {
        auto xp = static_cast<const bf16_t*>(x);
        auto xo = static_cast<bf16_t*>(x_dispatched);
        if (scan)
            return launch_pdl(gather_kernel<bf16_t, true>, grid, block, 0, s, xp, topk_idx, topk_gate, blk_hist,
                              offset, count, T, k, E, d, C, slot, row_token, row_gate, xo, out_to_zero, rank_major, stats);
        return launch_pdl(gather_kernel<bf16_t, false>, grid, block, 0, s, xp, topk_idx, topk_gate, blk_hist, offset,
                          count, T, k, E, d, C, slot, row_token, row_gate, xo, out_to_zero, rank_major, stats);
    }
    auto xp = static_cast<const float*>(x);
    auto xo = static_cast<float*>(x_dispatched);
    if (scan)
        return launch_pdl(gather_kernel<float, true>, grid, block, 0, s, xp, topk_idx, topk_gate, blk_hist, offset,
                          count, T, k, E, d, C, slot, row_token, row_gate, xo, out_to_zero, rank_major, stats);
    return launch_pdl(gather_kernel<float, false>, grid, block, 0, s, xp, topk_idx, topk_gate, blk_hist, offset,
                      count, T, k, E, d, C, slot, row_token, row_gate, xo, out_to_zero, rank_major, stats);
}

}  // namespace moe
