// ffn_tc.cu -- grouped expert GEMM on the 5th-generation tensor cores (tcgen05, TMEM accumulators,
// TMA loads), bf16 operands, fp32 accumulation.
//
// Grouping tokens by expert and running one batched matmul per group ("How sparse activation improves
// efficiency", section 3.1), done as one persistent launch over all experts: the dispatched rows are segments of 128-row tiles,
// one expert per tile, and the tiles (m-tile, n-tile) are dealt round-robin to one CTA per SM.
//
// CTA = 6 warps:
//   warp 0     TMA producer: A tile [128 x 64] of the dispatched activations and B tile [256 x 64]
//              of the expert's weight ([E, N, K] tensor map, expert = third coordinate) per stage,
//              128-byte swizzle, into a 4-stage ring guarded by full / empty mbarriers
//   warp 1     allocates 512 TMEM columns (two 128 x 256 fp32 accumulators); one lane issues
//              tcgen05.mma (M = 128, N = 256, K = 16, kind::f16) and tcgen05.commit to release smem
//              stages and to hand finished accumulators to the epilogue
//   warps 2-5  epilogue, one warp per TMEM lane quarter (32 rows): tcgen05.ld of the accumulator, then
//              bias, GELU or gate scaling and the stores, while the MMA warp fills the other accumulator;
//              the bf16 row outputs (H, and Z in the backward's recomputation) go through a per-warp
//              staging tile so that each store instruction writes whole 64-byte row pieces of 8 rows
//              (epilogue_staged), the other modes store from each thread's row (epilogue_cols)
// Every mbarrier wait is bounded: on expiry the kernel records MOE_ERR_DEVICE_TIMEOUT in the error
// word, all roles stop, the producer waits (bounded) for its copies in flight, the MMA warp waits for
// its last MMAs, and the TMEM is freed before the CTA exits.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace moe {

namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64, kStages = 4;
constexpr int kThreads = 192;  // producer warp, MMA warp, 4 epilogue warps (one per TMEM lane quarter)
constexpr uint32_t kABytes = kBM * kBK * 2;           // 16 KiB
constexpr uint32_t kBBytes = kBN * kBK * 2;           // 32 KiB
constexpr uint32_t kStageBytes = kABytes + kBBytes;   // 48 KiB
constexpr uint32_t kTmemCols = 2 * kBN;               // 512

// the epilogue warps' bias buffers follow the ints that start at s_off, 16-byte aligned
__device__ __forceinline__ void* smem_bias_base(int* s_off, int nints) {
    return reinterpret_cast<void*>((reinterpret_cast<uintptr_t>(s_off + nints) + 15) & ~uintptr_t(15));
}
constexpr size_t kBiasSmem = 4 * kBN * sizeof(float) + 16;  // 4 epilogue warps x kBN floats, + alignment
// single-SM kernel: per epilogue warp two 32-row x 64-byte staging tiles for its bf16 outputs (and Z)
constexpr size_t kOutStageSmem = 4 * 2 * 2048 + 16;

struct TcArgs {
    const int* offset;
    const int* row_token;
    const float* row_gate;
    const bf16_t* bias;
    void* C;
    float* out;
    int E, K, N, mode;
    int* err;
    const float* scale;  // block-FP8 weights: fp32 scale per 128 x 128 block, [E, N/128, K/128]
    int stages;          // SM-pair kernel: depth of its TMA ring
    bf16_t* aux;         // modes 3 / 4: the pre-activations Z [rows, N] (read / written)
    int M;               // weight-gradient kernel: rows of each expert's output [M, N]
    int b_mn;            // single-SM kernel: B is [E, K, N] (N contiguous), read MN-major
    float* zero;         // single-SM kernel, forward bf16 row output: cleared by one extra warp, or nullptr
    long long zero_n4;   // its length in float4
};

using namespace tc;

// Epilogue of columns [c_begin, c_end) of one accumulator row (TMEM lane = this thread's row r of the
// tile, token tok, gate g), 32 at a time:
//   mode 0: + b1, GELU(erf), round to bf16, store the hidden row
//   mode 1: + b2, store fp32 y
//   mode 2: + b2, times the row's gate, fp32 atomic add into out[tok] (fused combine)
//   mode 3: (backward) times GELU'(Z[r]) with the saved pre-activations, store bf16 dZ
//   mode 4: + b1, store bf16 Z and bf16 GELU(Z) (the forward that the backward recomputes)
//   mode 5: (backward) fp32 atomic add into out[tok] (gate 1, no bias: the gather-reduce of dx)
// All lanes of the warp call this (tcgen05.ld is warp-wide); rows with tok < 0 store nothing.
// kBwd: the backward's modes (3 - 5) are compiled in; the forward kernels leave them out (registers)
template <bool kBwd = false>
__device__ __forceinline__ void epilogue_cols(const TcArgs& a, uint32_t taddr, int r, int tok, float g,
                                              const float* sbias, int n0, int c_begin, int c_end) {
    for (int c0 = c_begin; c0 < c_end; c0 += 32) {
        uint32_t v[32];
        __syncwarp();
        tmem_ld32(taddr + (uint32_t)c0, v);
        const int n = n0 + c0;
        if (tok < 0 || n >= a.N) continue;
        float f[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[j]);
        if (sbias) {  // the tile's bias slice, staged in shared memory (all lanes read the same words)
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const float4 bb = *reinterpret_cast<const float4*>(sbias + c0 + j);
                f[j] += bb.x;
                f[j + 1] += bb.y;
                f[j + 2] += bb.z;
                f[j + 3] += bb.w;
            }
        }
        if (a.mode == 0) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<bf16_t*>(a.C) + (size_t)r * a.N + n);
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
                uint4 w;
                w.x = pack_bf16x2(gelu_erf(f[j + 0]), gelu_erf(f[j + 1]));
                w.y = pack_bf16x2(gelu_erf(f[j + 2]), gelu_erf(f[j + 3]));
                w.z = pack_bf16x2(gelu_erf(f[j + 4]), gelu_erf(f[j + 5]));
                w.w = pack_bf16x2(gelu_erf(f[j + 6]), gelu_erf(f[j + 7]));
                __stcs(dst + j / 8, w);  // streaming: the hidden rows should not push the weights out of L2
            }
        } else if (a.mode == 1) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.C) + (size_t)r * a.N + n);
#pragma unroll
            for (int j = 0; j < 32; j += 4) __stcs(dst + j / 4, make_float4(f[j], f[j + 1], f[j + 2], f[j + 3]));
        } else if (kBwd && a.mode == 3) {
            const uint4* zs = reinterpret_cast<const uint4*>(a.aux + (size_t)r * a.N + n);
            uint4* dst = reinterpret_cast<uint4*>(static_cast<bf16_t*>(a.C) + (size_t)r * a.N + n);
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
                const uint4 zz = __ldg(zs + j / 8);
                const uint32_t zw[4] = {zz.x, zz.y, zz.z, zz.w};
                uint32_t o[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    o[i] = pack_bf16x2(f[j + 2 * i] * gelu_grad(bf16_lo(zw[i])),
                                       f[j + 2 * i + 1] * gelu_grad(bf16_hi(zw[i])));
                dst[j / 8] = make_uint4(o[0], o[1], o[2], o[3]);
            }
        } else if (kBwd && a.mode == 4) {
            uint4* zd = reinterpret_cast<uint4*>(a.aux + (size_t)r * a.N + n);
            uint4* dst = reinterpret_cast<uint4*>(static_cast<bf16_t*>(a.C) + (size_t)r * a.N + n);
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
                uint32_t zw[4], hw[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    zw[i] = pack_bf16x2(f[j + 2 * i], f[j + 2 * i + 1]);
                    hw[i] = pack_bf16x2(gelu_erf(f[j + 2 * i]), gelu_erf(f[j + 2 * i + 1]));
                }
                zd[j / 8] = make_uint4(zw[0], zw[1], zw[2], zw[3]);
                dst[j / 8] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            }
        } else if (kBwd && a.mode == 5) {
            float4* dst = reinterpret_cast<float4*>(a.out + (size_t)tok * a.N + n);
#pragma unroll
            for (int j = 0; j < 32; j += 4) atomicAdd(dst + j / 4, make_float4(f[j], f[j + 1], f[j + 2], f[j + 3]));
        } else {
            float4* dst = reinterpret_cast<float4*>(a.out + (size_t)tok * a.N + n);
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                atomicAdd(dst + j / 4, make_float4(g * f[j], g * f[j + 1], g * f[j + 2], g * f[j + 3]));
        }
    }
}

// Epilogue of the bf16 modes (0: H = GELU(acc + b1); 4: Z = acc + b1 and H = GELU(Z); 3: dZ = acc * GELU'(Z)),
// 32 columns at a time through this warp's staging tiles (two of 32 rows x 64 bytes; 16-byte chunk c of row t
// at t * 64 + ((c ^ ((t >> 1) & 3)) << 4), so that a quarter warp's 16-byte accesses hit distinct banks both
// along a row and down a column): each thread fills its own row (r0 + lane, token tok), then every store
// instruction writes 8 rows x 64 bytes, four lanes a row; in mode 3 the Z chunk comes in the same way.  Rows
// with tok < 0 are neither loaded nor stored.  All lanes call this (tcgen05.ld and the shuffles are warp-wide).
template <bool kBwd>
__device__ __forceinline__ void epilogue_staged(const TcArgs& a, uint32_t taddr, int r0, int tok, const float* sbias,
                                                int n0, uint8_t* stg, int lane) {
    uint8_t* s0 = stg;         // the output tile (H, or Z in mode 4, or dZ)
    uint8_t* s1 = stg + 2048;  // mode 4: H; mode 3: the Z chunk read
    const int wsw = (lane >> 1) & 3;
    const int rl = lane >> 2, cc = lane & 3;
    for (int c0 = 0; c0 < kBN; c0 += 32) {
        const int n = n0 + c0;
        if (n >= a.N) break;  // N is a multiple of 32: the whole chunk is in or out (the same for the warp)
        __syncwarp();         // the previous chunk's reads of the tiles are done
        if (kBwd && a.mode == 3) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int rr = 8 * i + rl;
                const int rt = __shfl_sync(0xffffffffu, tok, rr);
                uint4 z = make_uint4(0u, 0u, 0u, 0u);
                if (rt >= 0) z = __ldg(reinterpret_cast<const uint4*>(a.aux + (size_t)(r0 + rr) * a.N + n) + cc);
                *reinterpret_cast<uint4*>(s1 + rr * 64 + ((cc ^ ((rr >> 1) & 3)) << 4)) = z;
            }
        }
        uint32_t v[32];
        tmem_ld32(taddr + (uint32_t)c0, v);
        float f[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[j]);
        if (sbias) {
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const float4 bb = *reinterpret_cast<const float4*>(sbias + c0 + j);
                f[j] += bb.x;
                f[j + 1] += bb.y;
                f[j + 2] += bb.z;
                f[j + 3] += bb.w;
            }
        }
        __syncwarp();  // mode 3: the Z chunk is in s1
        uint32_t o0[16], o1[16];
        if (kBwd && a.mode == 3) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint4 zz = *reinterpret_cast<const uint4*>(s1 + lane * 64 + ((c ^ wsw) << 4));
                const uint32_t zw[4] = {zz.x, zz.y, zz.z, zz.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int j = 8 * c + 2 * i;
                    o0[4 * c + i] = pack_bf16x2(f[j] * gelu_grad(bf16_lo(zw[i])), f[j + 1] * gelu_grad(bf16_hi(zw[i])));
                }
            }
        } else if (kBwd && a.mode == 4) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                o0[i] = pack_bf16x2(f[2 * i], f[2 * i + 1]);
                o1[i] = pack_bf16x2(gelu_erf(f[2 * i]), gelu_erf(f[2 * i + 1]));
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) o0[i] = pack_bf16x2(gelu_erf(f[2 * i]), gelu_erf(f[2 * i + 1]));
        }
        const bool two = kBwd && a.mode == 4;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            *reinterpret_cast<uint4*>(s0 + lane * 64 + ((c ^ wsw) << 4)) =
                make_uint4(o0[4 * c], o0[4 * c + 1], o0[4 * c + 2], o0[4 * c + 3]);
            if (two)
                *reinterpret_cast<uint4*>(s1 + lane * 64 + ((c ^ wsw) << 4)) =
                    make_uint4(o1[4 * c], o1[4 * c + 1], o1[4 * c + 2], o1[4 * c + 3]);
        }
        __syncwarp();
        // destinations: mode 0 / 3 -> C; mode 4 -> Z in aux (s0) and H in C (s1)
        bf16_t* d0 = two ? a.aux : static_cast<bf16_t*>(a.C);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int rr = 8 * i + rl;
            const int rt = __shfl_sync(0xffffffffu, tok, rr);
            const int off = rr * 64 + ((cc ^ ((rr >> 1) & 3)) << 4);
            const uint4 w0 = *reinterpret_cast<const uint4*>(s0 + off);
            if (rt >= 0) {
                uint4* g0 = reinterpret_cast<uint4*>(d0 + (size_t)(r0 + rr) * a.N + n) + cc;
                if (a.mode == 0) __stcs(g0, w0);  // streaming: the hidden rows should not push the weights out of L2
                else *g0 = w0;
                if (two)
                    *(reinterpret_cast<uint4*>(static_cast<bf16_t*>(a.C) + (size_t)(r0 + rr) * a.N + n) + cc) =
                        *reinterpret_cast<const uint4*>(s1 + off);
            }
        }
    }
}

// Epilogue of mode 3 (dZ = acc * GELU'(Z), bf16, no bias) for one accumulator row (TMEM lane = this thread's
// row r, token tok): the Z chunk of the next 32 columns is loaded while this chunk is computed, so that the
// latency of the Z loads overlaps the arithmetic instead of stalling every chunk.
__device__ __forceinline__ void epilogue_dz(const TcArgs& a, uint32_t taddr, int r, int tok, int n0) {
    const bf16_t* zrow = a.aux + (size_t)r * a.N;
    bf16_t* drow = static_cast<bf16_t*>(a.C) + (size_t)r * a.N;
    uint4 zc[4], zn[4];
    const bool live = tok >= 0;
    if (live && n0 < a.N) {
#pragma unroll
        for (int i = 0; i < 4; ++i) zc[i] = __ldg(reinterpret_cast<const uint4*>(zrow + n0) + i);
    }
    for (int c0 = 0; c0 < kBN; c0 += 32) {
        const int n = n0 + c0;
        uint32_t v[32];
        __syncwarp();
        tmem_ld32(taddr + (uint32_t)c0, v);
        if (n >= a.N) continue;  // the same for the warp: N is a multiple of 32
        const bool more = live && c0 + 32 < kBN && n + 32 < a.N;
        if (more) {
#pragma unroll
            for (int i = 0; i < 4; ++i) zn[i] = __ldg(reinterpret_cast<const uint4*>(zrow + n + 32) + i);
        }
        if (live) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t zw[4] = {zc[i].x, zc[i].y, zc[i].z, zc[i].w};
                uint32_t o[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int j = 8 * i + 2 * q;
                    o[q] = pack_bf16x2(__uint_as_float(v[j]) * gelu_grad(bf16_lo(zw[q])),
                                       __uint_as_float(v[j + 1]) * gelu_grad(bf16_hi(zw[q])));
                }
                reinterpret_cast<uint4*>(drow + n)[i] = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
        if (more) {
#pragma unroll
            for (int i = 0; i < 4; ++i) zc[i] = zn[i];
        }
    }
}

// One warp stages the bias slice of a tile (kBN columns from n0 of expert e's bias) as fp32 in its own
// shared-memory buffer: eight columns per lane, one 16-byte load each (N is a multiple of 64).
__device__ __forceinline__ const float* stage_bias(const TcArgs& a, float* wbias, int e, int n0, int lane) {
    if (a.bias == nullptr) return nullptr;
    const int n = n0 + lane * 8;
    float bb[8];
    if (n < a.N) {
        load8(a.bias + (size_t)e * a.N + n, bb);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) bb[i] = 0.f;
    }
    __syncwarp();  // the previous tile's reads of the buffer are done
    *reinterpret_cast<float4*>(wbias + lane * 8) = make_float4(bb[0], bb[1], bb[2], bb[3]);
    *reinterpret_cast<float4*>(wbias + lane * 8 + 4) = make_float4(bb[4], bb[5], bb[6], bb[7]);
    __syncwarp();
    return wbias;
}

// kStaged: the bf16 row-output modes (0, 4) with the staged epilogue; the other modes are compiled apart from
// it, so that each keeps its own register allocation.  The forward's up projection (mode 0) has a seventh
// warp that clears a buffer (TcArgs::zero: the fp32 output the fused combine then adds into) while the
// GEMM runs: its 4 bytes per output element are written in the GEMM's shadow, not by the gather.
__host__ __device__ constexpr int tc_threads(bool bwd, bool staged) { return kThreads + (!bwd && staged ? 32 : 0); }
template <bool kBwd, bool kStaged>
__global__ void __launch_bounds__(tc_threads(kBwd, kStaged), 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    // the 128-byte swizzle atoms need 1024-byte aligned tiles in the shared address space
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* sA = base;
    uint8_t* sB = base + kStages * kABytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + kStages * kBBytes);
    // bars: full[kStages], empty[kStages], tfull[2], tempty[2], last
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    int* s_off = reinterpret_cast<int*>(tmem_holder + 4);
    float* s_bias = reinterpret_cast<float*>(smem_bias_base(s_off, a.E + 1));  // [4 warps][kBN]
    uint8_t* s_out = reinterpret_cast<uint8_t*>(smem_bias_base(reinterpret_cast<int*>(s_bias), 4 * kBN));  // [4][4 KiB]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto bar = [&](int i) { return smem_u32(bars + i); };
    const int FULL = 0, EMPTY = kStages, TFULL = 2 * kStages, TEMPTY = 2 * kStages + 2, LAST = 2 * kStages + 4;

    if (threadIdx.x == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        *abort_flag = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(FULL + s), 1);
            mbar_init(bar(EMPTY + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(TFULL + s), 1);
            mbar_init(bar(TEMPTY + s), 4);
        }
        mbar_init(bar(LAST), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    }
    pdl_wait();  // the set-up above overlaps the previous kernel; its outputs are read from here on
    pdl_trigger();
    for (int i = threadIdx.x; i <= a.E; i += blockDim.x) s_off[i] = a.offset[i];
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem_base = *tmem_holder;

    const int total_rows = s_off[a.E];
    const int m_tiles = total_rows / kBM;
    const int n_tiles = (a.N + kBN - 1) / kBN;
    const int num_tiles = m_tiles * n_tiles;
    const int k_iters = a.K / kBK;

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_phase[kStages];
            bool issued[kStages];
            for (int s = 0; s < kStages; ++s) { issued[s] = false; issued_phase[s] = 0; }
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                const int m0 = (tile / n_tiles) * kBM, n0 = (tile % n_tiles) * kBN;
                const int e = expert_of_row(s_off, a.E, m0);
                for (int kb = 0; kb < k_iters; ++kb) {
                    if (!mbar_wait(bar(EMPTY + stage), phase ^ 1u, abort_flag)) { ok = false; break; }
                    mbar_expect_tx(bar(FULL + stage), kStageBytes);
                    tma_load_2d(smem_u32(sA + stage * kABytes), &tmA, bar(FULL + stage), kb * kBK, m0);
                    if (a.b_mn) {  // four boxes of 64 N-columns x 64 K-rows
#pragma unroll
                        for (int j = 0; j < kBN / 64; ++j)
                            tma_load_3d(smem_u32(sB + stage * kBBytes + j * 8192), &tmB, bar(FULL + stage), n0 + 64 * j,
                                        kb * kBK, e);
                    } else {
                        tma_load_3d(smem_u32(sB + stage * kBBytes), &tmB, bar(FULL + stage), kb * kBK, n0, e);
                    }
                    issued[stage] = true;
                    issued_phase[stage] = phase;
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                record_error(a.err, kErrTimeout, kWhereGemmProducer);
                *abort_flag = 1;
                // let every copy this thread started land before the CTA's shared memory goes away
                for (int s = 0; s < kStages; ++s)
                    if (issued[s]) {
                        mbar_wait_bounded(bar(FULL + s), issued_phase[s]);
                    }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(kBM, kBN) | (a.b_mn ? kIdescBMnMajor : 0u);
            int stage = 0;
            uint32_t phase = 0;
            int local = 0;
            bool ok = true, any = false;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x, ++local) {
                const int acc = local & 1;
                const uint32_t acc_phase = (local >> 1) & 1;
                if (!mbar_wait(bar(TEMPTY + acc), acc_phase ^ 1u, abort_flag)) { ok = false; break; }
                fence_after();
                const uint32_t d_tmem = tmem_base + acc * kBN;
                for (int kb = 0; kb < k_iters; ++kb) {
                    if (!mbar_wait(bar(FULL + stage), phase, abort_flag)) { ok = false; break; }
                    fence_after();
                    const uint64_t ad = smem_desc_sw128(smem_u32(sA + stage * kABytes));
                    // K-major B: a K step of 16 is 32 bytes along the row; MN-major: 16 rows of 128 bytes
                    const uint64_t bd = a.b_mn ? smem_desc_sw128_mn(smem_u32(sB + stage * kBBytes))
                                               : smem_desc_sw128(smem_u32(sB + stage * kBBytes));
                    const uint64_t bstep = a.b_mn ? (2048 >> 4) : 2;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        mma_bf16(d_tmem, ad + (uint64_t)(kk * 2), bd + bstep * kk, idesc, (kb | kk) != 0);
                    any = true;
                    commit(bar(EMPTY + stage));
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
                if (ok) commit(bar(TFULL + acc));
            }
            if (!ok) {
                record_error(a.err, kErrTimeout, kWhereGemmMma);
                *abort_flag = 1;
            }
            if (any) {  // all MMAs this thread issued have finished once LAST completes
                commit(bar(LAST));
                mbar_wait_bounded(bar(LAST), 0);
            }
        }
    } else if (warp == kThreads / 32) {
        // the clearing warp (forward up projection only): its CTA's share of the buffer, 16 bytes a lane
        if constexpr (!kBwd && kStaged) {
            if (a.zero != nullptr) {
                const long long per = (a.zero_n4 + gridDim.x - 1) / gridDim.x;
                const long long z0 = (long long)blockIdx.x * per, z1 = min(a.zero_n4, z0 + per);
                float4* z = reinterpret_cast<float4*>(a.zero);
                for (long long i = z0 + lane; i < z1; i += 32) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    } else {
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        int local = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++local) {
            const int acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            // the tile's rows, tokens, gates and bias are fetched while its accumulator is still being filled
            const int m0 = (tile / n_tiles) * kBM, n0 = (tile % n_tiles) * kBN;
            const int e = expert_of_row(s_off, a.E, m0);
            const int r = m0 + row;
            const int tok = a.row_token[r];
            const float g = (a.mode == 2 && tok >= 0) ? a.row_gate[r] : 0.f;
            const float* sb = stage_bias(a, s_bias + q * kBN, e, n0, lane);
            const bool ok = __all_sync(0xffffffffu, mbar_wait(bar(TFULL + acc), acc_phase, abort_flag));
            if (!ok) {
                if (lane == 0) {
                    record_error(a.err, kErrTimeout, kWhereGemmEpilogue);
                    *abort_flag = 1;
                }
                break;
            }
            fence_after();
            if constexpr (kStaged)
                epilogue_staged<kBwd>(a, tmem_base + lane_base + (uint32_t)(acc * kBN), m0 + q * 32, tok, sb, n0,
                                      s_out + q * 4096, lane);
            else if (kBwd && a.mode == 3)
                epilogue_dz(a, tmem_base + lane_base + (uint32_t)(acc * kBN), r, tok, n0);
            else
                epilogue_cols<kBwd>(a, tmem_base + lane_base + (uint32_t)(acc * kBN), r, tok, g, sb, n0, 0, kBN);
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(TEMPTY + acc));
        }
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 1) {
        tmem_free(tmem_base, kTmemCols);
    }
}

// ---- the same GEMM on pairs of SMs (cluster of 2, tcgen05 cta_group::2) -------------------------------
// A pair computes a 256 x 256 tile: each CTA holds 128 rows of A and 128 of the 256 weight rows of B per
// K block (32 KiB a stage, so 6 stages fit), one thread of the even CTA issues M = 256 MMAs that read
// both CTAs' shared memory and write each CTA's 128 accumulator rows into its own TMEM.  Per SM this
// halves the B bytes per FLOP against the single-SM tile, so the ring covers 1.5x the load latency.
// Tiles start on expert segment boundaries: an expert with an odd number of 128-row blocks ends with a
// tile whose upper half is discarded.  Barriers: FULL (even CTA, count 1: its producer expects both
// CTAs' bytes, and both CTAs' copies complete on it), EMPTY and TFULL (both CTAs, by multicast commit),
// TEMPTY (even CTA, count 8: four epilogue warps of each CTA).
constexpr int k2Stages = 6;       // with a bias (its staging buffers take 4 KiB)
constexpr int k2StagesNoBias = 7;  // without one: 224 KiB of ring
constexpr uint32_t k2HalfB = 128 * kBK * 2;            // 16 KiB: 128 of the 256 weight rows
constexpr uint32_t k2StageBytes = kABytes + k2HalfB;   // 32 KiB per CTA

__device__ __forceinline__ void pair_tile(const int* s_tp, const int* s_off, int E, int n_tiles, int tile, int& e,
                                          int& m0, int& n0) {
    const int mt = tile / n_tiles;
    n0 = (tile % n_tiles) * kBN;
    int lo = 0, hi = E;  // s_tp[lo] <= mt < s_tp[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_tp[mid] <= mt) lo = mid; else hi = mid;
    }
    e = lo;
    m0 = s_off[e] + (mt - s_tp[e]) * 256;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_tc_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* sA = base;
    const int NS = a.stages;
    uint8_t* sB = base + NS * kABytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + NS * k2HalfB);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * NS + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    int* s_off = reinterpret_cast<int*>(tmem_holder + 4);
    int* s_tp = s_off + (a.E + 1);  // first 256-row tile of each expert (prefix), E + 1 entries
    float* s_bias = reinterpret_cast<float*>(smem_bias_base(s_off, 2 * (a.E + 1)));  // [4 warps][kBN]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    auto bar = [&](int i) { return smem_u32(bars + i); };
    const int FULL = 0, EMPTY = NS, TFULL = 2 * NS, TEMPTY = 2 * NS + 2, LAST = 2 * NS + 4;

    if (threadIdx.x == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        *abort_flag = 0;
        for (int st = 0; st < NS; ++st) {
            mbar_init(bar(FULL + st), 1);
            mbar_init(bar(EMPTY + st), 1);
        }
        for (int st = 0; st < 2; ++st) {
            mbar_init(bar(TFULL + st), 1);
            mbar_init(bar(TEMPTY + st), 8);
        }
        mbar_init(bar(LAST), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    pdl_wait();  // the set-up above overlaps the previous kernel; its outputs are read from here on
    pdl_trigger();
    for (int i = threadIdx.x; i <= a.E; i += kThreads) s_off[i] = a.offset[i];
    __syncthreads();
    if (threadIdx.x == 0) {  // tiles per expert: its rows (a multiple of 128) in blocks of 256
        int acc = 0;
        for (int e = 0; e < a.E; ++e) {
            s_tp[e] = acc;
            acc += (s_off[e + 1] - s_off[e] + 255) / 256;
        }
        s_tp[a.E] = acc;
    }
    if (warp == 1) tmem_alloc_pair(smem_u32(tmem_holder), kTmemCols);
    fence_before();
    __syncthreads();
    cluster_sync();  // the peer's barriers are initialised before anyone arrives on them
    fence_after();
    const uint32_t tmem_base = *tmem_holder;

    const int n_tiles = (a.N + kBN - 1) / kBN;
    const int num_tiles = s_tp[a.E] * n_tiles;
    const int k_iters = a.K / kBK;
    const int pair_id = blockIdx.x >> 1, num_pairs = gridDim.x >> 1;

    if (warp == 0) {
        if (lane == 0) {
            const uint32_t full0 = mapa_shared(bar(FULL), 0);  // the even CTA's FULL barriers
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true, any = false;
            for (int tile = pair_id; ok && tile < num_tiles; tile += num_pairs) {
                int e, m0, n0;
                pair_tile(s_tp, s_off, a.E, n_tiles, tile, e, m0, n0);
                for (int kb = 0; kb < k_iters; ++kb) {
                    if (!mbar_wait_cluster(bar(EMPTY + stage), phase ^ 1u, abort_flag)) { ok = false; break; }
                    const uint32_t fb = full0 + 8u * (uint32_t)stage;
                    // the even CTA expects both CTAs' bytes (its own arrive is CTA-local and cheap); the odd
                    // CTA's copies may land first, taking the transaction count below zero for a while
                    if (leader) mbar_expect_tx(bar(FULL + stage), 2 * k2StageBytes);
                    tma_load_2d_pair(smem_u32(sA + stage * kABytes), &tmA, fb, kb * kBK, m0 + 128 * (int)rank);
                    tma_load_3d_pair(smem_u32(sB + stage * k2HalfB), &tmB, fb, kb * kBK, n0 + 128 * (int)rank, e);
                    any = true;
                    if (++stage == NS) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                record_error(a.err, kErrTimeout, kWhereGemmProducer);
                *abort_flag = 1;
                // copies in flight signal the even CTA's barriers, which this CTA cannot poll: give them
                // time to land before the shared memory they write is released
                if (any)
                    for (int i = 0; i < 2000; ++i) __nanosleep(1000);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            constexpr uint32_t idesc = idesc_bf16(256, kBN);
            int stage = 0;
            uint32_t phase = 0;
            int local = 0;
            bool ok = true, any = false;
            for (int tile = pair_id; ok && tile < num_tiles; tile += num_pairs, ++local) {
                const int acc = local & 1;
                const uint32_t acc_phase = (local >> 1) & 1;
                if (!mbar_wait_cluster(bar(TEMPTY + acc), acc_phase ^ 1u, abort_flag)) { ok = false; break; }
                fence_after();
                const uint32_t d_tmem = tmem_base + acc * kBN;
                for (int kb = 0; kb < k_iters; ++kb) {
                    if (!mbar_wait_cluster(bar(FULL + stage), phase, abort_flag)) { ok = false; break; }
                    fence_after();
                    const uint64_t ad = smem_desc_sw128(smem_u32(sA + stage * kABytes));
                    const uint64_t bd = smem_desc_sw128(smem_u32(sB + stage * k2HalfB));
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        mma_bf16_pair(d_tmem, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc,
                                      (kb | kk) != 0);
                    any = true;
                    commit_pair_mc(bar(EMPTY + stage), 3);
                    if (++stage == NS) { stage = 0; phase ^= 1u; }
                }
                if (ok) commit_pair_mc(bar(TFULL + acc), 3);
            }
            if (!ok) {
                record_error(a.err, kErrTimeout, kWhereGemmMma);
                *abort_flag = 1;
            }
            if (any) {  // every MMA issued above has finished once LAST completes
                commit_pair_mc(bar(LAST), 1);
                mbar_wait_bounded(bar(LAST), 0);
            }
        }
    } else {
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        const uint32_t tempty0 = mapa_shared(bar(TEMPTY), 0);
        int local = 0;
        for (int tile = pair_id; tile < num_tiles; tile += num_pairs, ++local) {
            const int acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            // the tile's rows, tokens, gates and bias are fetched while its accumulator is still being filled
            int e, m0, n0;
            pair_tile(s_tp, s_off, a.E, n_tiles, tile, e, m0, n0);
            const int r = m0 + 128 * (int)rank + row;
            const int tok = r < s_off[e + 1] ? a.row_token[r] : -1;  // beyond the segment: discarded
            const float g = (a.mode == 2 && tok >= 0) ? a.row_gate[r] : 0.f;
            const float* sb = stage_bias(a, s_bias + q * kBN, e, n0, lane);
            const bool ok = __all_sync(0xffffffffu, mbar_wait_cluster(bar(TFULL + acc), acc_phase, abort_flag));
            if (!ok) {
                if (lane == 0) {
                    record_error(a.err, kErrTimeout, kWhereGemmEpilogue);
                    *abort_flag = 1;
                }
                break;
            }
            fence_after();
            epilogue_cols(a, tmem_base + lane_base + (uint32_t)(acc * kBN), r, tok, g, sb, n0, 0, kBN);
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty0 + 8u * (uint32_t)acc);
        }
    }
    fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs are done with the pair's TMEM and barriers
    fence_after();
    if (warp == 1) tmem_free_pair(tmem_base, kTmemCols);
}

// ---- weight gradients: GEMMs grouped along K ------------------------------------------------------------
// dW[e] [M, N] = sum over the dispatched rows r of expert e of A[r][m] B[r][n], i.e. the contraction runs over
// the expert's own row segment [off[e], off[e+1]).  Both operands are read as stored, A [rows, M] and
// B [rows, N] row-major: MN-major tiles, A as two and B as four TMA boxes of 64 columns x 64 rows per
// K step (the descriptors of gemm_tc_kernel's MN-major B, instruction-descriptor bits 15 and 16); padding
// rows hold zeros in both.  Tiles (e, m-tile, n-tile) are dealt to one CTA per SM; a tile of an expert
// without rows stores zeros.  The epilogue stores fp32 rows m < M of dW[e].
constexpr int kWgStageStride = 36;                                  // floats per staged row
constexpr size_t kWgStageBytes = 4 * 32 * kWgStageStride * sizeof(float);  // 4 epilogue warps
__global__ void __launch_bounds__(kThreads, 1)
    gemm_wgrad_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* sA = base;
    uint8_t* sB = base + kStages * kABytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + kStages * kBBytes);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    int* s_off = reinterpret_cast<int*>(tmem_holder + 4);
    // per epilogue warp a 32 x 32 fp32 staging tile (rows 36 floats apart: conflict-free 16-byte accesses
    // both row-wise and column-wise), so that each output row leaves as whole 128-byte lines
    float* s_stage = reinterpret_cast<float*>(
        (reinterpret_cast<uintptr_t>(s_off + a.E + 1) + 15) & ~static_cast<uintptr_t>(15));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto bar = [&](int i) { return smem_u32(bars + i); };
    const int FULL = 0, EMPTY = kStages, TFULL = 2 * kStages, TEMPTY = 2 * kStages + 2, LAST = 2 * kStages + 4;

    if (threadIdx.x == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        *abort_flag = 0;
        for (int st = 0; st < kStages; ++st) {
            mbar_init(bar(FULL + st), 1);
            mbar_init(bar(EMPTY + st), 1);
        }
        for (int st = 0; st < 2; ++st) {
            mbar_init(bar(TFULL + st), 1);
            mbar_init(bar(TEMPTY + st), 4);
        }
        mbar_init(bar(LAST), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    pdl_wait();
    pdl_trigger();
    for (int i = threadIdx.x; i <= a.E; i += kThreads) s_off[i] = a.offset[i];
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem_base = *tmem_holder;

    const int m_tiles = (a.M + kBM - 1) / kBM;
    const int n_tiles = (a.N + kBN - 1) / kBN;
    const int per_e = m_tiles * n_tiles;
    const int num_tiles = a.E * per_e;
    auto decode = [&](int tile, int& e, int& m0, int& n0, int& k0, int& nk) {
        e = tile / per_e;
        const int rem = tile - e * per_e;
        m0 = (rem / n_tiles) * kBM;
        n0 = (rem % n_tiles) * kBN;
        k0 = s_off[e];
        nk = (s_off[e + 1] - k0) / kBK;
    };

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_phase[kStages];
            bool issued[kStages];
            for (int st = 0; st < kStages; ++st) { issued[st] = false; issued_phase[st] = 0; }
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                int e, m0, n0, k0, nk;
                decode(tile, e, m0, n0, k0, nk);
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(bar(EMPTY + stage), phase ^ 1u, abort_flag)) { ok = false; break; }
                    mbar_expect_tx(bar(FULL + stage), kStageBytes);
                    const int kr = k0 + kb * kBK;
#pragma unroll
                    for (int j = 0; j < kBM / 64; ++j)
                        tma_load_2d(smem_u32(sA + stage * kABytes + j * 8192), &tmA, bar(FULL + stage), m0 + 64 * j, kr);
#pragma unroll
                    for (int j = 0; j < kBN / 64; ++j)
                        tma_load_2d(smem_u32(sB + stage * kBBytes + j * 8192), &tmB, bar(FULL + stage), n0 + 64 * j, kr);
                    issued[stage] = true;
                    issued_phase[stage] = phase;
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                record_error(a.err, kErrTimeout, kWhereGemmProducer);
                *abort_flag = 1;
                for (int st = 0; st < kStages; ++st)
                    if (issued[st]) mbar_wait_bounded(bar(FULL + st), issued_phase[st]);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(kBM, kBN) | kIdescAMnMajor | kIdescBMnMajor;
            int stage = 0;
            uint32_t phase = 0;
            int local = 0;
            bool ok = true, any = false;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x, ++local) {
                int e, m0, n0, k0, nk;
                decode(tile, e, m0, n0, k0, nk);
                const int acc = local & 1;
                const uint32_t acc_phase = (local >> 1) & 1;
                if (!mbar_wait(bar(TEMPTY + acc), acc_phase ^ 1u, abort_flag)) { ok = false; break; }
                fence_after();
                const uint32_t d_tmem = tmem_base + acc * kBN;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(bar(FULL + stage), phase, abort_flag)) { ok = false; break; }
                    fence_after();
                    // MN-major operands: a K step of 16 is 16 rows of 128 bytes
                    const uint64_t ad = smem_desc_sw128_mn(smem_u32(sA + stage * kABytes));
                    const uint64_t bd = smem_desc_sw128_mn(smem_u32(sB + stage * kBBytes));
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        mma_bf16(d_tmem, ad + (uint64_t)(kk * 128), bd + (uint64_t)(kk * 128), idesc, (kb | kk) != 0);
                    any = true;
                    commit(bar(EMPTY + stage));
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                if (nk > 0) commit(bar(TFULL + acc));
                else mbar_arrive(bar(TFULL + acc));  // nothing to wait for: the epilogue stores zeros
            }
            if (!ok) {
                record_error(a.err, kErrTimeout, kWhereGemmMma);
                *abort_flag = 1;
            }
            if (any) {
                commit(bar(LAST));
                mbar_wait_bounded(bar(LAST), 0);
            }
        }
    } else {
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        int local = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++local) {
            int e, m0, n0, k0, nk;
            decode(tile, e, m0, n0, k0, nk);
            const int acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            const int m = m0 + row;
            const bool ok = __all_sync(0xffffffffu, mbar_wait(bar(TFULL + acc), acc_phase, abort_flag));
            if (!ok) {
                if (lane == 0) {
                    record_error(a.err, kErrTimeout, kWhereGemmEpilogue);
                    *abort_flag = 1;
                }
                break;
            }
            fence_after();
            if (nk > 0) {
                // each 32-column chunk: this thread's row into the staging tile, then 4 rows x 128 bytes per
                // store instruction (8 lanes a row)
                float* stg = s_stage + q * (32 * kWgStageStride);
                const int mr = (lane & 7) * 4;
#pragma unroll 1
                for (int c0 = 0; c0 < kBN; c0 += 32) {
                    uint32_t v[32];
                    __syncwarp();
                    tmem_ld32(tmem_base + lane_base + (uint32_t)(acc * kBN + c0), v);
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4*>(stg + lane * kWgStageStride + j) =
                            make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]), __uint_as_float(v[j + 2]),
                                        __uint_as_float(v[j + 3]));
                    __syncwarp();
                    const int n = n0 + c0 + mr;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int rr = 4 * i + (lane >> 3);
                        const int mrow = m0 + q * 32 + rr;
                        const float4 val = *reinterpret_cast<const float4*>(stg + rr * kWgStageStride + mr);
                        if (mrow < a.M && n < a.N)
                            __stcs(reinterpret_cast<float4*>(static_cast<float*>(a.C) + ((size_t)e * a.M + mrow) * a.N + n),
                                   val);
                    }
                }
            } else if (m < a.M) {  // an expert without rows: its gradient is zero
                float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.C) + ((size_t)e * a.M + m) * a.N + n0);
                for (int c = 0; c < kBN && n0 + c < a.N; c += 4) dst[c / 4] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(TEMPTY + acc));
        }
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 1) tmem_free(tmem_base, kTmemCols);
}

// ---- the single-SM GEMM with block-FP8 weights ----------------------------------------------------
// The expert weight arrives as FP8 E4M3 codes ([E, N, K], one byte each) with one fp32 scale per 128 x 128
// block ([E, N/128, K/128]).  HBM carries one byte per weight, and the codes come from DRAM while the
// activations (A) mostly come from L2, so they travel in separate rings: a deep ring of code tiles
// (256 x 64 bytes, no swizzle) that keeps enough bytes in flight to cover the DRAM latency, and a short
// ring of bf16 A tiles, each fed by its own producer thread.  Eight converter warps turn each code tile
// into bf16 (code value x scale, exact for power-of-two scales) in the 128-byte-swizzled K-major layout
// the MMA reads, into one of a few bf16 B buffers, then release the code tile; the MMAs (kind::f16) and
// the epilogue are those of gemm_tc_kernel.  In the swapped kernel (at most 64 rows per expert) the
// converters form two groups that take alternate K blocks, so that one group's chain of waits, loads,
// conversion, proxy fence and arrival overlaps the other's.  Barriers: FULLA / EMPTYA (A ring), FULLB /
// EMPTYB (code ring, released by the converter warps), BREADY / BEMPTY (bf16 buffers, freed by the MMA's
// commit), TFULL / TEMPTY (accumulators), LAST.
constexpr int kF8ARing = 4;     // A tiles come from L2: a few stages cover its latency
constexpr int kF8BRingMax = 12;  // code tiles come from DRAM: as many as fit
#ifndef MOE_F8_SWAP_GROUPS
#define MOE_F8_SWAP_GROUPS 2
#endif
#ifndef MOE_F8_SWAP_BUFS
#define MOE_F8_SWAP_BUFS 4
#endif
// widened-weight buffers (bf16 tiles in shared memory; in the swapped kernel, A operands in tensor memory)
// and converter groups: each group widens every kGroups-th K block, so that the groups' chains of waits,
// loads, conversion, fence and arrival overlap; a group needs a buffer of its own
__host__ __device__ constexpr int f8_bufs(bool swap) { return swap ? MOE_F8_SWAP_BUFS : 2; }
__host__ __device__ constexpr int f8_groups(bool swap) { return swap ? MOE_F8_SWAP_GROUPS : 1; }
constexpr uint32_t kB8Bytes = kBN * kBK;  // 16 KiB of codes per K block
// converter warps: 8 in the 128-row kernel (its registers allow no more); 8 per group in the swapped one
// (a warp per lane quarter and half of the 256-row tile)
__host__ __device__ constexpr int f8_conv_warps(bool swap) { return swap ? 8 * f8_groups(true) : 8; }
// + the converters + the A producer: 480 threads (swapped kernel, two groups: 736)
__host__ __device__ constexpr int f8_threads(bool swap) { return kThreads + 32 * f8_conv_warps(swap) + 32; }
constexpr int kF8Block = 128;                                  // scale block edge
constexpr int kSwapRows = 64;                                  // swapped kernel: rows per tile (MMA N)
constexpr uint32_t kSwapABytes = kSwapRows * kBK * 2;          // its A tiles: 8 KiB
constexpr int kSwapTmemA = 256;  // swapped kernel: first tensor-memory column of the widened weights

// 16 E4M3 codes (one row's K block of 16) times `scale` -> 16 bf16 in two 16-byte chunks
__device__ __forceinline__ void e4m3x16_to_bf16(const uint4 v, float scale, uint4& lo, uint4& hi) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const __half2_raw hr =
                __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[i] >> (16 * hf)), __NV_E4M3);
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
            o[2 * i + hf] = pack_bf16x2(f.x * scale, f.y * scale);
        }
    }
    lo = make_uint4(o[0], o[1], o[2], o[3]);
    hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// kSwap (few rows per expert, e.g. decode): the roles of the operands swap.  The weights become the MMA's
// M side (two M = 128 halves of the 256-row code tile) and the expert's rows the N side, 64 rows a tile
// (a 64-row chunk of the expert's segment; chunks past its last real row are skipped by every role), so
// the tensor work per weight byte follows the real rows instead of 128-row padded tiles; the epilogue
// reads the accumulator transposed (a lane per output feature, a column per row).
template <bool kSwap>
__global__ void __launch_bounds__(f8_threads(kSwap), 1)
    gemm_fp8w_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB8,
                     const TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    constexpr int kConvWarps = f8_conv_warps(kSwap), kNThreads = f8_threads(kSwap);
    constexpr int kBufs = f8_bufs(kSwap), kGroups = f8_groups(kSwap), kGroupWarps = kConvWarps / kGroups;
    static_assert(kGroups >= 1 && kBufs >= kGroups && kBufs >= 2 && kConvWarps % kGroups == 0 &&
                      (1024 % (32 * kGroupWarps)) == 0 && kGroupWarps <= 16,
                  "converter groups");
    static_assert(!kSwap || (kGroupWarps == 8 && kSwapTmemA + kBufs * 64 <= 512), "swapped kernel's tensor memory");
    const int NB = a.stages;  // depth of the code ring (host: as deep as shared memory allows, <= 8)
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    constexpr uint32_t kASlot = kSwap ? kSwapABytes : kABytes;
    uint8_t* sA = base;                              // [kF8ARing] bf16 A tiles, 128-byte swizzle
    uint8_t* sBb = sA + kF8ARing * kASlot;           // [kBufs] bf16 B tiles, 128-byte swizzle (not swapped)
    uint8_t* sB8 = sBb + (kSwap ? 0 : kBufs * kBBytes);  // [NB] code tiles (swapped: 64-byte swizzle)
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB8 + NB * kB8Bytes);
    const int FULLA = 0, EMPTYA = kF8ARing, BREADY = 2 * kF8ARing, BEMPTY = BREADY + kBufs,
              TFULL = BEMPTY + kBufs, TEMPTY = TFULL + 2, LAST = TEMPTY + 2, FULLB = LAST + 1, EMPTYB = FULLB + NB,
              NBARS = EMPTYB + NB;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + NBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    int* s_off = reinterpret_cast<int*>(tmem_holder + 4);
    float* s_bias = reinterpret_cast<float*>(smem_bias_base(s_off, a.E + 1));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto bar = [&](int i) { return smem_u32(bars + i); };

    if (threadIdx.x == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB8);
        *abort_flag = 0;
        for (int i = 0; i < kF8ARing; ++i) {
            mbar_init(bar(FULLA + i), 1);
            mbar_init(bar(EMPTYA + i), 1);
        }
        for (int i = 0; i < kBufs; ++i) {
            mbar_init(bar(BREADY + i), kGroupWarps);
            mbar_init(bar(BEMPTY + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(TFULL + i), 1);
            mbar_init(bar(TEMPTY + i), 4);
        }
        mbar_init(bar(LAST), 1);
        for (int i = 0; i < NB; ++i) {
            mbar_init(bar(FULLB + i), 1);
            mbar_init(bar(EMPTYB + i), kGroupWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // swapped: 2 accumulators x 2 halves x 64 rows, then kBufs widened A operands (2 halves x 32 columns)
    constexpr uint32_t kCols = kTmemCols;
    if (warp == 1) tmem_alloc(smem_u32(tmem_holder), kCols);
    pdl_wait();
    pdl_trigger();
    for (int i = threadIdx.x; i <= a.E; i += kNThreads) s_off[i] = a.offset[i];
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem_base = *tmem_holder;

    const int total_rows = s_off[a.E];
    constexpr int kRowsPerTile = kSwap ? kSwapRows : kBM;
    const int m_tiles = total_rows / kRowsPerTile;
    const int n_tiles = (a.N + kBN - 1) / kBN;
    const int num_tiles = m_tiles * n_tiles;
    const int k_iters = a.K / kBK;
    // tile -> first row, first weight row, expert; a swapped tile whose first row is padding holds no real
    // row (real rows are a prefix of each segment) and is skipped by every role alike
    auto tile_at = [&](int tile, int& m0, int& n0, int& e) {
        m0 = (tile / n_tiles) * kRowsPerTile;
        n0 = (tile % n_tiles) * kBN;
        e = expert_of_row(s_off, a.E, m0);
        return !kSwap || a.row_token[m0] >= 0;
    };
    const int a_warp = kNThreads / 32 - 1;  // the last warp issues the A loads

    if (warp == 0 || warp == a_warp) {
        // warp 0: the code tiles, NB deep; the last warp: the A tiles, kF8ARing deep
        if (lane == 0) {
            const bool is_b = warp == 0;
            const int depth = is_b ? NB : kF8ARing;
            const int FULL = is_b ? FULLB : FULLA, EMPTY = is_b ? EMPTYB : EMPTYA;
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_phase[kF8BRingMax];
            bool issued[kF8BRingMax];
            for (int i = 0; i < kF8BRingMax; ++i) { issued[i] = false; issued_phase[i] = 0; }
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                int m0, n0, e;
                if (!tile_at(tile, m0, n0, e)) continue;
                for (int kb = 0; kb < k_iters; ++kb) {
                    if (!mbar_wait(bar(EMPTY + stage), phase ^ 1u, abort_flag)) { ok = false; break; }
                    if (is_b) {
                        mbar_expect_tx(bar(FULL + stage), kB8Bytes);
                        tma_load_3d(smem_u32(sB8 + stage * kB8Bytes), &tmB8, bar(FULL + stage), kb * kBK, n0, e);
                    } else {
                        mbar_expect_tx(bar(FULL + stage), kASlot);
                        tma_load_2d(smem_u32(sA + stage * kASlot), &tmA, bar(FULL + stage), kb * kBK, m0);
                    }
                    issued[stage] = true;
                    issued_phase[stage] = phase;
                    if (++stage == depth) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                record_error(a.err, kErrTimeout, kWhereGemmProducer);
                *abort_flag = 1;
                for (int i = 0; i < depth; ++i)
                    if (issued[i]) mbar_wait_bounded(bar(FULL + i), issued_phase[i]);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = kSwap ? idesc_bf16(128, kSwapRows) : idesc_bf16(kBM, kBN);
            int stage = 0, buf = 0;
            uint32_t phase = 0, bphase = 0;
            int local = 0;
            bool ok = true, any = false;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                int m0, n0, e;
                if (!tile_at(tile, m0, n0, e)) continue;
                const int acc = local & 1;
                const uint32_t acc_phase = (local >> 1) & 1;
                ++local;
                if (!mbar_wait(bar(TEMPTY + acc), acc_phase ^ 1u, abort_flag)) { ok = false; break; }
                fence_after();
                const uint32_t d_tmem = tmem_base + acc * (kSwap ? 2 * kSwapRows : kBN);
                for (int kb = 0; kb < k_iters; ++kb) {
                    if (!mbar_wait(bar(FULLA + stage), phase, abort_flag) ||
                        !mbar_wait(bar(BREADY + buf), bphase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    const uint64_t ad = smem_desc_sw128(smem_u32(sA + stage * kASlot));
                    const uint64_t bd = smem_desc_sw128(smem_u32(sBb + buf * kBBytes));
                    if constexpr (kSwap) {
                        // D[half] (128 weight rows x 64 rows) += W[half] (A operand, tensor memory: 32 columns
                        // of bf16 pairs per half, 8 per K step of 16) x X^T (B operand, shared memory)
                        const uint32_t wa = tmem_base + (uint32_t)(kSwapTmemA + buf * 64);
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk) {
                            mma_bf16_tmem_a(d_tmem, wa + kk * 8, ad + (uint64_t)(kk * 2), idesc, (kb | kk) != 0);
                            mma_bf16_tmem_a(d_tmem + kSwapRows, wa + 32 + kk * 8, ad + (uint64_t)(kk * 2), idesc,
                                            (kb | kk) != 0);
                        }
                    } else {
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk)
                            mma_bf16(d_tmem, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc, (kb | kk) != 0);
                    }
                    any = true;
                    commit(bar(EMPTYA + stage));
                    commit(bar(BEMPTY + buf));
                    if (++stage == kF8ARing) { stage = 0; phase ^= 1u; }
                    if (++buf == kBufs) { buf = 0; bphase ^= 1u; }
                }
                if (ok) commit(bar(TFULL + acc));
            }
            if (!ok) {
                record_error(a.err, kErrTimeout, kWhereGemmMma);
                *abort_flag = 1;
            }
            if (any) {
                commit(bar(LAST));
                mbar_wait_bounded(bar(LAST), 0);
            }
        }
    } else if (kSwap && warp < kThreads / 32) {
        // a lane per output feature n (TMEM lane), a column per row of the 64-row chunk
        const int q = warp & 3;
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        int local = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            int m0, n0, e;
            if (!tile_at(tile, m0, n0, e)) continue;
            const int acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            ++local;
            const int tok_lo = a.row_token[m0 + lane], tok_hi = a.row_token[m0 + 32 + lane];
            const float g_lo = (a.mode == 2 && tok_lo >= 0) ? a.row_gate[m0 + lane] : 0.f;
            const float g_hi = (a.mode == 2 && tok_hi >= 0) ? a.row_gate[m0 + 32 + lane] : 0.f;
            const bool ok = __all_sync(0xffffffffu, mbar_wait(bar(TFULL + acc), acc_phase, abort_flag));
            if (!ok) {
                if (lane == 0) {
                    record_error(a.err, kErrTimeout, kWhereGemmEpilogue);
                    *abort_flag = 1;
                }
                break;
            }
            fence_after();
#pragma unroll 1
            for (int hf = 0; hf < 2; ++hf) {
                const int n = n0 + hf * 128 + q * 32 + lane;
                const float bn = (a.bias != nullptr && n < a.N) ? bf16_to_f32(a.bias[(size_t)e * a.N + n]) : 0.f;
#pragma unroll 1
                for (int jh = 0; jh < 2; ++jh) {
                    uint32_t v[32];
                    __syncwarp();
                    tmem_ld32(tmem_base + lane_base + (uint32_t)(acc * 2 * kSwapRows + hf * kSwapRows + jh * 32), v);
                    for (int j = 0; j < 32; ++j) {
                        const int tok = __shfl_sync(0xffffffffu, jh ? tok_hi : tok_lo, j);
                        if (tok < 0) continue;  // padding row (the same for the whole warp)
                        const float gj = __shfl_sync(0xffffffffu, jh ? g_hi : g_lo, j);
                        if (n >= a.N) continue;
                        const int r = m0 + jh * 32 + j;
                        const float f = __uint_as_float(v[j]) + bn;
                        if (a.mode == 0) {
                            static_cast<bf16_t*>(a.C)[(size_t)r * a.N + n] =
                                (bf16_t)(pack_bf16x2(gelu_erf(f), 0.f) & 0xffffu);
                        } else if (a.mode == 1) {
                            static_cast<float*>(a.C)[(size_t)r * a.N + n] = f;
                        } else {
                            atomicAdd(a.out + (size_t)tok * a.N + n, gj * f);
                        }
                    }
                }
            }
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(TEMPTY + acc));
        }
    } else if (warp < kThreads / 32) {
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        int local = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++local) {
            const int acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            const int m0 = (tile / n_tiles) * kBM, n0 = (tile % n_tiles) * kBN;
            const int e = expert_of_row(s_off, a.E, m0);
            const int r = m0 + row;
            const int tok = a.row_token[r];
            const float g = (a.mode == 2 && tok >= 0) ? a.row_gate[r] : 0.f;
            const float* sb = stage_bias(a, s_bias + q * kBN, e, n0, lane);
            const bool ok = __all_sync(0xffffffffu, mbar_wait(bar(TFULL + acc), acc_phase, abort_flag));
            if (!ok) {
                if (lane == 0) {
                    record_error(a.err, kErrTimeout, kWhereGemmEpilogue);
                    *abort_flag = 1;
                }
                break;
            }
            fence_after();
            epilogue_cols(a, tmem_base + lane_base + (uint32_t)(acc * kBN), r, tok, g, sb, n0, 0, kBN);
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(TEMPTY + acc));
        }
    } else if constexpr (kSwap) {
        // converter warps (swapped kernel), kGroups groups of 8: group g widens the K blocks whose running count
        // over the CTA's tiles is g mod kGroups.  Warp (half hf, lane quarter q) widens weight rows
        // hf * 128 + q * 32 + lane: each thread one row of 64 codes (four 16-byte chunks; the 64-byte swizzle of
        // the code tiles puts chunk c of row r at c ^ ((r >> 1) & 3), so a quarter warp's loads hit all banks),
        // and stores its 32 bf16 pairs into its lane of the tensor-memory A operand.
        const int cw = warp - kThreads / 32;
        const int grp = cw / 8, hf = (cw % 8) >> 2, q = warp & 3;
        const int row = hf * 128 + q * 32 + lane;
        const int swz = (row >> 1) & 3;
        const uint32_t tl = (uint32_t)(q * 32) << 16;
        const int nbn = a.N / kF8Block, nbk = a.K / kF8Block;
        int stage = grp, buf = grp;
        uint32_t phase = 0, bphase = 0;
        int count = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
            int m0, n0, e;
            if (!tile_at(tile, m0, n0, e)) continue;
            // this row's 128-row scale block (rows past N are zero codes); its scale for the group's next K
            // block is loaded one iteration ahead
            const int nb = n0 / kF8Block + hf;
            const float* sp = a.scale + ((size_t)e * nbn + nb) * nbk;
            const bool has = nb < nbn;
            const int kb_first = (grp - count % kGroups + kGroups) % kGroups;
            count += k_iters;
            float nsc = 0.f;
            if (has && kb_first < k_iters) nsc = __ldg(sp + (kb_first * kBK) / kF8Block);
            for (int kb = kb_first; kb < k_iters; kb += kGroups) {
                const float sc = nsc;
                if (has && kb + kGroups < k_iters) nsc = __ldg(sp + ((kb + kGroups) * kBK) / kF8Block);
                const bool got = mbar_wait(bar(FULLB + stage), phase, abort_flag) &&
                                 mbar_wait(bar(BEMPTY + buf), bphase ^ 1u, abort_flag);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                fence_after();  // the MMAs that read this buffer before have finished (their commit)
                const uint8_t* src = sB8 + stage * kB8Bytes + row * kBK;
                uint4 v[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) v[c] = *reinterpret_cast<const uint4*>(src + ((c ^ swz) << 4));
                uint32_t o[32];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint4 lo, hi;
                    e4m3x16_to_bf16(v[c], sc, lo, hi);
                    o[8 * c + 0] = lo.x; o[8 * c + 1] = lo.y; o[8 * c + 2] = lo.z; o[8 * c + 3] = lo.w;
                    o[8 * c + 4] = hi.x; o[8 * c + 5] = hi.y; o[8 * c + 6] = hi.z; o[8 * c + 7] = hi.w;
                }
                tmem_st32(tmem_base + tl + (uint32_t)(kSwapTmemA + buf * 64 + hf * 32), o);
                tmem_wait_st();
                fence_before();  // the MMA thread reads these columns after the barrier below
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar(BREADY + buf));
                    mbar_arrive(bar(EMPTYB + stage));
                }
                stage += kGroups;
                if (stage >= NB) { stage -= NB; phase ^= 1u; }
                buf += kGroups;
                if (buf >= kBufs) { buf -= kBufs; bphase ^= 1u; }
            }
        }
        if (!ok && lane == 0) {
            record_error(a.err, kErrTimeout, kWhereGemmProducer);
            *abort_flag = 1;
        }
    } else {
        // converter warps, kGroups groups of kGroupWarps: group g widens the K blocks whose running count over
        // the CTA's tiles is g mod kGroups; its thread gt handles the 16-byte pieces gt + i * 32 * kGroupWarps
        // of the 256 x 64 codes (row = piece / 4, K bytes 16 * (piece % 4) ..), rows 8 * kGroupWarps apart
        constexpr int kPieces = 1024 / (32 * kGroupWarps), kRowStep = 8 * kGroupWarps;
        const int ct = threadIdx.x - kThreads;
        const int grp = ct / (32 * kGroupWarps), gt = ct % (32 * kGroupWarps);
        const int r0 = gt >> 2, j = gt & 3;
        const int nbn = a.N / kF8Block, nbk = a.K / kF8Block;
        int stage = grp, buf = grp;  // ring positions of K block number grp (the host keeps NB >= kGroups)
        uint32_t phase = 0, bphase = 0;
        int count = 0;  // K blocks of the tiles before this one
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
            int m0, n0, e;
            if (!tile_at(tile, m0, n0, e)) continue;
            // the two 128-row scale blocks of this tile's 256 weight rows (rows past N are zero codes); the
            // scales of the group's next K block are loaded one of its iterations ahead
            const int nb0 = n0 / kF8Block;
            const float* sp = a.scale + ((size_t)e * nbn) * nbk;
            auto load_scales = [&](int kb_, float& s0, float& s1) {
                const int kbs = (kb_ * kBK) / kF8Block;
                s0 = nb0 < nbn ? __ldg(sp + (size_t)nb0 * nbk + kbs) : 0.f;
                s1 = nb0 + 1 < nbn ? __ldg(sp + (size_t)(nb0 + 1) * nbk + kbs) : 0.f;
            };
            const int kb_first = (grp - count % kGroups + kGroups) % kGroups;
            count += k_iters;
            float nsc0 = 0.f, nsc1 = 0.f;
            if (kb_first < k_iters) load_scales(kb_first, nsc0, nsc1);
            for (int kb = kb_first; kb < k_iters; kb += kGroups) {
                const float sc0 = nsc0, sc1 = nsc1;
                if (kb + kGroups < k_iters) load_scales(kb + kGroups, nsc0, nsc1);
                const bool got = mbar_wait(bar(FULLB + stage), phase, abort_flag) &&
                                 mbar_wait(bar(BEMPTY + buf), bphase ^ 1u, abort_flag);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                const uint8_t* src = sB8 + stage * kB8Bytes;
                uint8_t* dst = sBb + buf * kBBytes;
#pragma unroll
                for (int i = 0; i < kPieces; ++i) {
                    const int r = r0 + kRowStep * i;
                    const uint4 v = *reinterpret_cast<const uint4*>(src + r * kBK + j * 16);
                    uint4 lo, hi;
                    e4m3x16_to_bf16(v, r < kF8Block ? sc0 : sc1, lo, hi);
                    uint8_t* drow = dst + (r >> 3) * 1024 + (r & 7) * 128;
                    *reinterpret_cast<uint4*>(drow + (((2 * j) ^ (r & 7)) << 4)) = lo;
                    *reinterpret_cast<uint4*>(drow + (((2 * j + 1) ^ (r & 7)) << 4)) = hi;
                }
                fence_proxy_async_smem();  // the MMA reads these bytes through the async proxy
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar(BREADY + buf));
                    mbar_arrive(bar(EMPTYB + stage));  // the code tile is read: its stage may refill
                }
                stage += kGroups;
                if (stage >= NB) { stage -= NB; phase ^= 1u; }
                buf += kGroups;
                if (buf >= kBufs) { buf -= kBufs; bphase ^= 1u; }
            }
        }
        if (!ok && lane == 0) {
            record_error(a.err, kErrTimeout, kWhereGemmProducer);
            *abort_flag = 1;
        }
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 1) tmem_free(tmem_base, kCols);
}

// ---- host side ----------------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

struct MapKey {
    const void* ptr;
    uint64_t d0, d1, d2;
    uint32_t b1;
    uint32_t kind;  // 0: bf16, 128-byte swizzle; 1: bytes, no swizzle; 2: bytes, 64-byte swizzle
    bool operator==(const MapKey& o) const {
        return ptr == o.ptr && d0 == o.d0 && d1 == o.d1 && d2 == o.d2 && b1 == o.b1 && kind == o.kind;
    }
};
struct MapEntry {
    MapKey key;
    CUtensorMap map;
};
std::mutex g_map_mutex;
MapEntry g_maps[64];
int g_maps_used = 0, g_maps_next = 0;

}  // namespace

namespace {
bool tma_map_kind(const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b1, uint32_t kind,
                  CUtensorMap* out) {
    const MapKey key{ptr, d0, d1, d2, b1, kind};
    std::lock_guard<std::mutex> lock(g_map_mutex);
    for (int i = 0; i < g_maps_used; ++i)
        if (g_maps[i].key == key) { *out = g_maps[i].map; return true; }
    auto fn = encode_fn();
    if (!fn) return false;
    CUtensorMap m;
    const cuuint32_t rank = d2 > 0 ? 3 : 2;
    const uint64_t es_bytes = kind == 0 ? 2 : 1;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {d0 * es_bytes, d0 * d1 * es_bytes};
    cuuint32_t box[3] = {(cuuint32_t)kBK, b1, 1};  // 64 elements of K: 128 bytes (bf16) or 64 (codes)
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(&m, kind == 0 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, rank,
                    const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    kind == 0 ? CU_TENSOR_MAP_SWIZZLE_128B
                              : (kind == 2 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE),
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    MapEntry& slot = g_maps[g_maps_next];
    slot.key = key;
    slot.map = m;
    g_maps_next = (g_maps_next + 1) % 64;
    if (g_maps_used < 64) ++g_maps_used;
    *out = m;
    return true;
}
}  // namespace

bool tma_map_bf16(const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b1, CUtensorMap* out) {
    return tma_map_kind(ptr, d0, d1, d2, b1, 0, out);
}

// clusters of two of the pair kernel that can be resident at once (cached per shared-memory size)
int pair_clusters(size_t smem) {
    static size_t cached_smem = 0;
    static int cached = 0;
    if (cached_smem == smem && cached > 0) return cached;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 74, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_pair_kernel, &cfg) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        n = device_sm_count() / 2;
    }
    cached_smem = smem;
    cached = n;
    return n;
}

int device_sm_count() {
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
    }
    return n;
}

size_t ffn_tc_smem_bytes(int E) {
    return 1024 + (size_t)kStages * kStageBytes + (2 * kStages + 5) * 8 + 16 + 4 * (size_t)(E + 1) + kBiasSmem +
           kOutStageSmem;
}

size_t ffn_tc_pair_smem_bytes(int E, bool bias, int ns) {
    return 1024 + (size_t)ns * k2StageBytes + (2 * ns + 5) * 8 + 16 + 8 * (size_t)(E + 1) + (bias ? kBiasSmem : 0);
}

// the SM-pair kernel's ring depth: one stage more when there is no bias to stage and it fits
int pair_stages(int E, bool bias) {
    return !bias && ffn_tc_pair_smem_bytes(E, false, k2StagesNoBias) <= 227 * 1024 ? k2StagesNoBias : k2Stages;
}

cudaError_t launch_wgrad_tc(const WgradParams& P, cudaStream_t s) {
    if (P.M <= 0 || P.N <= 0 || P.E <= 0) return cudaSuccess;
    const int a_ld = P.a_ld > 0 ? P.a_ld : P.M;
    if (a_ld < P.M || a_ld % 8 || P.N % 8 || P.rows <= 0 || P.rows_b <= 0) return cudaErrorInvalidValue;
    CUtensorMap ma, mb;  // boxes of 64 columns x 64 rows
    if (!tma_map_bf16(P.A, (uint64_t)a_ld, (uint64_t)P.rows, 0, 64, &ma)) return cudaErrorInvalidValue;
    if (!tma_map_bf16(P.B, (uint64_t)P.N, (uint64_t)P.rows_b, 0, 64, &mb)) return cudaErrorInvalidValue;
    TcArgs a{};
    a.offset = P.offset;
    a.C = P.dW;
    a.E = P.E;
    a.K = 0;
    a.N = P.N;
    a.M = P.M;
    a.mode = 1;
    a.err = P.err;
    const size_t smem = 1024 + (size_t)kStages * kStageBytes + (2 * kStages + 5) * 8 + 16 + 4 * (size_t)(P.E + 1) + 16 +
                        kWgStageBytes;
    if (smem > 227 * 1024) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(gemm_wgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t tiles = (int64_t)P.E * ((P.M + kBM - 1) / kBM) * ((P.N + kBN - 1) / kBN);
    int grid = device_sm_count();
    if (tiles < grid) grid = (int)tiles;
    return launch_pdl(gemm_wgrad_kernel, dim3(grid), dim3(kThreads), smem, s, ma, mb, a);
}

size_t ffn_fp8_smem_bytes(int E, bool bias, int nb, bool swap) {
    return 1024 + (size_t)kF8ARing * (swap ? kSwapABytes : kABytes) + (swap ? 0 : (size_t)f8_bufs(swap) * kBBytes) +
           (size_t)nb * kB8Bytes + (2 * kF8ARing + 2 * f8_bufs(swap) + 5 + 2 * nb) * 8 + 16 +
           4 * (size_t)(E + 1) + (bias && !swap ? kBiasSmem : 0);
}

// the code ring as deep as shared memory allows (at most kF8BRingMax, at least 2 and the converter groups)
int fp8_ring_depth(int E, bool bias, bool swap) {
    const int lo = f8_groups(swap) > 2 ? f8_groups(swap) : 2;
    int nb = kF8BRingMax;
    while (nb > lo && ffn_fp8_smem_bytes(E, bias, nb, swap) > 227 * 1024) --nb;
    return nb;
}

cudaError_t launch_ffn_tc(const FfnParams& P, cudaStream_t s) {
    if (!P.bf16) return cudaErrorInvalidValue;
    if (P.w_scale != nullptr && P.zero != nullptr) return cudaErrorInvalidValue;
    if (P.rows_cap <= 0) return P.zero != nullptr ? cudaMemsetAsync(P.zero, 0, (size_t)P.zero_n * 4, s) : cudaSuccess;
    CUtensorMap ma, mb;
    if (P.w_scale != nullptr) {  // block-FP8 weights: byte codes, single-SM tiles
        if (P.K % kF8Block || P.N % kF8Block) return cudaErrorInvalidValue;
        // no expert holds more than 64 rows (decode): the swapped kernel, 64-row chunks of each segment
        const bool swap = P.max_rows > 0 && P.max_rows <= kSwapRows;
        const int rows_box = swap ? kSwapRows : kBM;
        if (!tma_map_bf16(P.A, (uint64_t)P.K, (uint64_t)P.rows_cap, 0, rows_box, &ma)) return cudaErrorInvalidValue;
        if (!tma_map_kind(P.W, (uint64_t)P.K, (uint64_t)P.N, (uint64_t)P.E, kBN, swap ? 2 : 1, &mb))
            return cudaErrorInvalidValue;
        const bool bias = P.bias != nullptr;
        const int nb = fp8_ring_depth(P.E, bias, swap);
        TcArgs a8{P.offset, P.row_token, P.row_gate, static_cast<const bf16_t*>(P.bias), P.C, P.out,
                  P.E, P.K, P.N, P.mode, P.err, P.w_scale, nb, static_cast<bf16_t*>(P.aux), 0};
        const size_t smem8 = ffn_fp8_smem_bytes(P.E, bias, nb, swap);
        if (smem8 > 227 * 1024) return cudaErrorInvalidValue;
        auto kern8 = swap ? gemm_fp8w_kernel<true> : gemm_fp8w_kernel<false>;
        cudaError_t e8 = cudaFuncSetAttribute(kern8, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem8);
        if (e8 != cudaSuccess) return e8;
        const int64_t tiles8 = (P.rows_cap / rows_box) * (int64_t)((P.N + kBN - 1) / kBN);
        int grid8 = device_sm_count();
        if (tiles8 < grid8) grid8 = (int)(tiles8 > 0 ? tiles8 : 1);
        return launch_pdl(kern8, dim3(grid8), dim3(f8_threads(swap)), smem8, s, ma, mb, a8);
    }
    if (!tma_map_bf16(P.A, (uint64_t)P.K, (uint64_t)P.rows_cap, 0, kBM, &ma)) return cudaErrorInvalidValue;
    if (P.w_kn) {  // W [E, K, N]: boxes of 64 N-columns x 64 K-rows, single-SM kernel only
        if (P.pair || P.N % 64) return cudaErrorInvalidValue;
        if (!tma_map_bf16(P.W, (uint64_t)P.N, (uint64_t)P.K, (uint64_t)P.E, 64, &mb)) return cudaErrorInvalidValue;
    } else if (!tma_map_bf16(P.W, (uint64_t)P.K, (uint64_t)P.N, (uint64_t)P.E, kBN, &mb)) {
        return cudaErrorInvalidValue;
    }
    TcArgs a;
    a.offset = P.offset;
    a.row_token = P.row_token;
    a.row_gate = P.row_gate;
    a.bias = static_cast<const bf16_t*>(P.bias);
    a.C = P.C;
    a.out = P.out;
    a.E = P.E;
    a.K = P.K;
    a.N = P.N;
    a.mode = P.mode;
    a.err = P.err;
    a.scale = nullptr;
    a.stages = kStages;
    a.aux = static_cast<bf16_t*>(P.aux);
    a.M = 0;
    a.b_mn = P.w_kn;
    a.zero = nullptr;
    a.zero_n4 = 0;
    if (P.zero != nullptr && (P.pair || P.mode != 0 || P.zero_n % 4 != 0 ||
                              (reinterpret_cast<uintptr_t>(P.zero) & 15)))
        return cudaErrorInvalidValue;  // only the single-SM up projection clears a buffer
    if (P.pair) {
        // pairs of SMs: B boxes of 128 weight rows (half of a 256-wide tile), grid = 2 x the clusters that fit
        CUtensorMap mb2;
        if (!tma_map_bf16(P.W, (uint64_t)P.K, (uint64_t)P.N, (uint64_t)P.E, 128, &mb2)) return cudaErrorInvalidValue;
        a.stages = pair_stages(P.E, P.bias != nullptr);
        const size_t smem2 = ffn_tc_pair_smem_bytes(P.E, P.bias != nullptr, a.stages);
        cudaError_t e2 =
            cudaFuncSetAttribute(gemm_tc_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2);
        if (e2 != cudaSuccess) return e2;
        const int64_t max_tiles = (P.rows_cap / kBM + P.E) / 2 * (int64_t)((P.N + kBN - 1) / kBN) + 1;
        int pairs = pair_clusters(smem2);
        if (max_tiles < pairs) pairs = (int)max_tiles;
            return launch_pdl(gemm_tc_pair_kernel, dim3(2 * pairs), dim3(kThreads), smem2, s, ma, mb2, a);
    }
    const size_t smem = ffn_tc_smem_bytes(P.E);
    const bool bwd = P.mode >= 3, staged = P.mode == 0 || P.mode == 4;
    auto kern = bwd ? (staged ? gemm_tc_kernel<true, true> : gemm_tc_kernel<true, false>)
                    : (staged ? gemm_tc_kernel<false, true> : gemm_tc_kernel<false, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t max_tiles = (P.rows_cap / kBM) * (int64_t)((P.N + kBN - 1) / kBN);
    int grid = device_sm_count();
    if (max_tiles < grid) grid = (int)(max_tiles > 0 ? max_tiles : 1);
    if (P.zero != nullptr) {
        if (2 * grid < device_sm_count()) {  // few tiles: the CTAs' clearing warps would be too few
            cudaError_t ez = cudaMemsetAsync(P.zero, 0, (size_t)P.zero_n * 4, s);
            if (ez != cudaSuccess) return ez;
        } else {
            a.zero = P.zero;
            a.zero_n4 = P.zero_n / 4;
        }
    }
    return launch_pdl(kern, dim3(grid), dim3(tc_threads(bwd, staged)), smem, s, ma, mb, a);
}

}  // namespace moe
