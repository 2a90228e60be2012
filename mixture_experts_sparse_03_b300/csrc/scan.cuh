// scan.cuh -- the dispatch scan as a block-level device function, shared by the standalone scan
// kernel and by the last block of the gate kernel (which runs it once every block has written its
// histogram).
//
// Input: blk_hist[b][e] = pairs of token block b routed to expert e.  Output, in place: blk_hist[b][e]
// = pairs of blocks before b routed to e (the first slot block b hands out for e); count[e] = total;
// offset[e] = sum over e' < e of roundup(min(count[e'], C), 128), offset[E] = total rows; padding rows
// [offset[e] + kept[e], offset[e+1]) get row_token -1 and row_gate 0.
#pragma once

#include "common.cuh"

namespace moe {

struct ScanSmem {
    int* part;     // [blockDim.x]
    int* padded;   // [E + 1]
    int* kept;     // [E]
    int* wsum;     // [33]
};

__device__ __forceinline__ void scan_experts(int* blk_hist, int nblk, int E, int C, int* count, int* offset,
                                             int* row_token, float* row_gate, const ScanSmem& sm) {
    const int NT = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int tpe = 1;  // threads per expert, each taking a contiguous range of blocks
    while (tpe * 2 * E <= NT && tpe * 2 <= nblk) tpe *= 2;
    const int groups = NT / tpe;
    for (int e0 = 0; e0 < E; e0 += groups) {
        const int e = e0 + tid / tpe, sub = tid % tpe;
        const bool active = e < E;
        const int per = (nblk + tpe - 1) / tpe;
        const int b0 = min(nblk, sub * per), b1 = min(nblk, b0 + per);
        int s = 0;
        if (active)
            for (int b = b0; b < b1; ++b) s += __ldcg(blk_hist + (size_t)b * E + e);
        sm.part[tid] = s;
        __syncthreads();
        if (active) {
            int run = 0;
            for (int q = 0; q < sub; ++q) run += sm.part[tid - sub + q];
            for (int b = b0; b < b1; ++b) {
                const int c = __ldcg(blk_hist + (size_t)b * E + e);
                blk_hist[(size_t)b * E + e] = run;
                run += c;
            }
            if (sub == tpe - 1) {
                count[e] = run;
                const int kept = min(run, C);
                sm.kept[e] = kept;
                sm.padded[e] = (kept + kRowAlign - 1) / kRowAlign * kRowAlign;
            }
        }
        __syncthreads();
    }
    // exclusive scan of the padded sizes, NT values at a time
    int carry = 0;
    for (int base = 0; base < E; base += NT) {
        const int i = base + tid;
        const int v = i < E ? sm.padded[i] : 0;
        int inc = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, inc, off);
            if (lane >= off) inc += o;
        }
        if (lane == 31) sm.wsum[warp] = inc;
        __syncthreads();
        if (warp == 0) {
            const int nw = NT / 32;
            const int w = lane < nw ? sm.wsum[lane] : 0;
            int winc = w;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, winc, off);
                if (lane >= off) winc += o;
            }
            if (lane < nw) sm.wsum[lane] = winc - w;  // exclusive prefix of the warp totals
            if (lane == 31) sm.wsum[32] = winc;       // total of this chunk
        }
        __syncthreads();
        const int excl = carry + sm.wsum[warp] + inc - v;
        const int total = sm.wsum[32];
        __syncthreads();
        if (i < E) sm.padded[i] = excl;
        carry += total;
        __syncthreads();
    }
    if (tid == 0) sm.padded[E] = carry;
    __syncthreads();
    for (int q = tid; q <= E; q += NT) offset[q] = sm.padded[q];
    for (int i = tid; i < E * kRowAlign; i += NT) {
        const int e = i / kRowAlign;
        const int r = sm.padded[e] + sm.kept[e] + i % kRowAlign;
        if (r < sm.padded[e + 1]) {
            row_token[r] = -1;
            row_gate[r] = 0.f;
        }
    }
}

}  // namespace moe
