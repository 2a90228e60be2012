// scan.cuh -- the block-level steps of the dispatch, shared by the dispatch kernels and the gate
// kernels (which run them on their own block of tokens, and the scan in their last block):
//   rank_pairs_warp  within-block token-order ranks of the (token, expert) pairs + block histogram
//   scan_experts     per-expert prefix over the block histograms, counts, padded segment offsets
//
// Input: blk_hist[b][e] = pairs of token block b routed to expert e.  Output, in place: blk_hist[b][e]
// = pairs of blocks before b routed to e (the first slot block b hands out for e); count[e] = total;
// offset[e] = sum over e' < e of roundup(min(count[e'], C), 128), offset[E] = total rows; padding rows
// [offset[e] + kept[e], offset[e+1]) get row_token -1 and row_gate 0.
#pragma once

#include "common.cuh"

namespace moe {

// One warp numbers the block's pairs in token order (pair i belongs to token i / k, rank i % k): 32 pairs
// at a time, __match_any_sync groups equal experts and each pair's rank among them is the number of
// lower lanes in its group; a shared running count per expert carries the numbering across chunks.
// `running` [E] must be zero on entry and holds the block's expert histogram on exit.  expert_of(i)
// < 0 marks a pair that takes no slot (rank -1, not counted).
// store_rank(i, r) receives pair i's rank (-1 for a pair that takes no slot).
template <typename F, typename S>
__device__ __forceinline__ void rank_pairs_warp_to(F expert_of, int npairs, int* running, S store_rank, int lane) {
    for (int c0 = 0; c0 < npairs; c0 += 32) {
        const int i = c0 + lane;
        const bool valid = i < npairs;
        const int e = valid ? expert_of(i) : -1;
        const unsigned mask = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(mask & lanemask_lt());
        const bool real = valid && e >= 0;
        const int base = real ? running[e] : 0;
        __syncwarp();
        if (real && rank == 0) running[e] = base + __popc(mask);
        __syncwarp();
        if (valid) store_rank(i, real ? base + rank : -1);
    }
}
template <typename F>
__device__ __forceinline__ void rank_pairs_warp(F expert_of, int npairs, int* running, int* rank_out, int lane) {
    rank_pairs_warp_to(expert_of, npairs, running, [&](int i, int r) { rank_out[i] = r; }, lane);
}

struct ScanSmem {
    int* part;     // [blockDim.x]
    int* padded;   // [E + 1]
    int* kept;     // [E]
    int* wsum;     // [33]
};

// The block's global stores all come after its last barrier when E <= blockDim.x (one chunk of experts):
// a barrier that follows stores to global memory costs the block a round trip to L2.
__device__ __forceinline__ void scan_experts(int* blk_hist, int nblk, int E, int C, int* count, int* offset,
                                             int* row_token, float* row_gate, const ScanSmem& sm) {
    constexpr int R = 16;  // block rows a thread keeps in registers between reading and writing them
    const int NT = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool one_chunk = E <= NT;
    int v[R];
    int e = 0, b0 = 0, b1 = 0, run0 = 0;
    bool active = false, last_group = false;
    // thread (g, e) writes the exclusive prefixes of expert e over blocks [b0, b1) (v: the first R counts)
    auto write_back = [&]() {
        int run = run0;
#pragma unroll
        for (int j = 0; j < R; ++j)
            if (b0 + j < b1) {
                blk_hist[(size_t)(b0 + j) * E + e] = run;
                run += v[j];
            }
        for (int i0 = b0 + R; i0 < b1; i0 += 8) {
            int w[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) w[j] = i0 + j < b1 ? __ldcg(blk_hist + (size_t)(i0 + j) * E + e) : 0;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (i0 + j < b1) {
                    blk_hist[(size_t)(i0 + j) * E + e] = run;
                    run += w[j];
                }
        }
        if (last_group) count[e] = run;
    };
    // per chunk of up to NT experts: thread (g, e) owns expert e over the g-th run of `per` blocks, so
    // a warp reads consecutive experts of one block row (coalesced), all of its rows in flight at once
    for (int e0 = 0; e0 < E; e0 += NT) {
        const int ne = min(NT, E - e0);
        const int G = max(1, min(nblk, NT / ne));
        const int per = (nblk + G - 1) / G;
        const int g = tid / ne;
        e = e0 + tid % ne;
        active = g < G;
        last_group = g == G - 1;
        b0 = active ? min(nblk, g * per) : nblk;
        b1 = active ? min(nblk, b0 + per) : nblk;
        int s = 0;
#pragma unroll
        for (int j = 0; j < R; ++j) v[j] = b0 + j < b1 ? __ldcg(blk_hist + (size_t)(b0 + j) * E + e) : 0;
#pragma unroll
        for (int j = 0; j < R; ++j) s += v[j];
        for (int i0 = b0 + R; i0 < b1; i0 += 8) {  // rows beyond the first R: summed now, re-read below
            int w[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) w[j] = i0 + j < b1 ? __ldcg(blk_hist + (size_t)(i0 + j) * E + e) : 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) s += w[j];
        }
        sm.part[tid] = s;
        __syncthreads();
        // inclusive scan over the groups of each expert (Hillis-Steele, stride ne)
        for (int off = 1; off < G; off <<= 1) {
            const int add = (active && g >= off) ? sm.part[tid - off * ne] : 0;
            __syncthreads();
            sm.part[tid] += add;
            __syncthreads();
        }
        if (active) {
            run0 = sm.part[tid] - s;  // blocks of this expert before b0
            if (last_group) {
                const int kept = min(sm.part[tid], C);
                sm.kept[e] = kept;
                sm.padded[e] = (kept + kRowAlign - 1) / kRowAlign * kRowAlign;
            }
            if (!one_chunk) write_back();  // the registers serve the next chunk
        }
        __syncthreads();
    }
    // exclusive scan of the padded sizes by one warp: lane l takes experts [l*per, (l+1)*per)
    if (warp == 0) {
        const int per = (E + 31) / 32;
        const int lo = min(E, lane * per), hi = min(E, lo + per);
        int own = 0;
        for (int i = lo; i < hi; ++i) own += sm.padded[i];
        int inc = own;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, inc, off);
            if (lane >= off) inc += o;
        }
        int run = inc - own;
        for (int i = lo; i < hi; ++i) {
            const int pv = sm.padded[i];
            sm.padded[i] = run;
            run += pv;
        }
        if (lane == 31) sm.padded[E] = inc;
    }
    __syncthreads();
    // global stores only from here on
    if (one_chunk && active) write_back();
    for (int q = tid; q <= E; q += NT) offset[q] = sm.padded[q];
    for (int i = tid; i < E * kRowAlign; i += NT) {
        const int ee = i / kRowAlign;
        const int r = sm.padded[ee] + sm.kept[ee] + i % kRowAlign;
        if (r < sm.padded[ee + 1]) {
            row_token[r] = -1;
            row_gate[r] = 0.f;
        }
    }
}

}  // namespace moe
