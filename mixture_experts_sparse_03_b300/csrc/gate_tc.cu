// gate_tc.cu -- the gate's logits GEMM on the tensor cores: L = x W^T in fp32 for bf16 layers.
//
// The logits of every gate type are one GEMM with the activations: the softmax gate's x W_g^T (a single
// linear layer before the softmax, "How sparse activation improves efficiency", section 2.1), the
// noisy gate's clean and noise linear maps x W_g^T and x W_n^T ("MoE sparse-compute acceleration",
// section 2.1, NoisyTopKGating), and the cosine gate's projection x P^T (Tutel's cosine_top in the
// "Tutel MoE guide").  This kernel computes it with tcgen05.mma (kind::f16: bf16 operands, products
// exact, fp32 accumulation in TMEM) fed by TMA, and writes fp32 partial logits; the selection kernel
// (gate.cu) sums the partials, scores, picks the top-k, and re-scores near ties exactly.
//
// Grid (m-tile, n-tile, split): 128 tokens x BN logits x a range of 64-wide K blocks per CTA.  The
// weight rows are one or two tensors (w_gate, then w_noise for the noisy gate); an n-tile never
// straddles them.  Small token counts split K across CTAs so that about one CTA per SM streams the
// weights; the splits' partials are summed in a fixed order by the selection kernel (deterministic).
//
// CTA = 6 warps: warp 0 issues the TMA loads into a ring of stages; warp 1 allocates TMEM and one lane
// issues the MMAs, each 64-wide K block into a fresh accumulator (two, alternating); warps 2-5 add
// every block's accumulator into float-float sums (so the tensor cores' fp32 rounding only ever spans
// 64 products and the error bound does not grow with d), compute the squared norms of the x rows
// (n-tile 0) and weight rows (m-tile 0) from the shared-memory tiles -- the selection kernel bounds
// each logit's error by them -- and store the logits.
// Every mbarrier wait is bounded; on expiry the kernel records MOE_ERR_DEVICE_TIMEOUT, waits (bounded)
// for its own copies and MMAs, frees its TMEM and returns.
#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace moe {

namespace {

using namespace tc;

constexpr int kGM = 128, kGK = 64, kGStages = 4, kGThreads = 192;
constexpr int kGMaxBN = 64;  // logits per n-tile: the epilogue holds 64 float-float sums per row
constexpr uint32_t kGABytes = kGM * kGK * 2;  // 16 KiB

struct GemmArgs {
    float* part;       // [S][T][Np]
    float* xn2_part;   // [S][T]
    float* wn2_part;   // [S][Np]
    const bf16_t* x;   // [T, d]
    const bf16_t* w0;  // [N0, d]
    const bf16_t* w1;  // [N1, d] or nullptr
    int T, d, N0, N1, Np, BN, nt0, per, kb;
    int* err;
};

// sum of squares of the 64 bf16 of one 128-byte row of a swizzled tile (the swizzle only permutes the
// row's 16-byte chunks, so the sum is over the same elements)
__device__ __forceinline__ float sumsq_tile_row(const uint8_t* row) {
    float s[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 u = *reinterpret_cast<const uint4*>(row + c * 16);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
        s[c] = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float lo = bf16_lo(w[j]), hi = bf16_hi(w[j]);
            s[c] = fmaf(lo, lo, s[c]);
            s[c] = fmaf(hi, hi, s[c]);
        }
    }
    return ((s[0] + s[1]) + (s[2] + s[3])) + ((s[4] + s[5]) + (s[6] + s[7]));
}

__global__ void __launch_bounds__(kGThreads, 1)
    gate_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                     const __grid_constant__ CUtensorMap tmB1, const GemmArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t b_bytes = (uint32_t)a.BN * kGK * 2;
    const uint32_t stage_bytes = kGABytes + b_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + kGStages * stage_bytes);
    // bars: full[kGStages], empty[kGStages], chunk_full[2], chunk_empty[2], last
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * kGStages + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    const int FULL = 0, EMPTY = kGStages, CFULL = 2 * kGStages, CEMPTY = 2 * kGStages + 2, LAST = 2 * kGStages + 4;
    auto bar = [&](int i) { return smem_u32(bars + i); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mt = blockIdx.x, nt = blockIdx.y, split = blockIdx.z;
    const bool second = nt >= a.nt0;                        // tile of w_noise (noisy gate)
    const int n_local = (second ? nt - a.nt0 : nt) * a.BN;  // first weight row of the tile
    const int n_map = second ? a.N1 : a.N0;                 // rows of that weight tensor
    const int col0 = (second ? a.N0 : 0) + n_local;         // first output column
    const int m0 = mt * kGM;
    const int kb0 = split * a.per, kb1 = min(a.kb, kb0 + a.per);
    const int nkb = kb1 - kb0;
    const bool x_norms = a.xn2_part != nullptr && nt == 0;
    const bool w_norms = a.wn2_part != nullptr && mt == 0;
    const bool readers = x_norms || w_norms;  // epilogue warps read the smem tiles too
    uint32_t tcols = 32;
    while (tcols < 2u * (uint32_t)a.BN) tcols <<= 1;

    if (threadIdx.x == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(second ? &tmB1 : &tmB0);
        *abort_flag = 0;
        for (int s = 0; s < kGStages; ++s) {
            mbar_init(bar(FULL + s), 1);
            mbar_init(bar(EMPTY + s), readers ? 5 : 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(CFULL + s), 1);
            mbar_init(bar(CEMPTY + s), 4);
        }
        mbar_init(bar(LAST), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_holder), tcols);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            const CUtensorMap* mb = second ? &tmB1 : &tmB0;
            uint32_t issued_phase[kGStages];
            bool issued[kGStages];
            for (int s = 0; s < kGStages; ++s) { issued[s] = false; issued_phase[s] = 0; }
            bool ok = true;
            int stage = 0;
            uint32_t phase = 0;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait(bar(EMPTY + stage), phase ^ 1u, abort_flag)) { ok = false; break; }
                uint8_t* st = base + stage * stage_bytes;
                mbar_expect_tx(bar(FULL + stage), stage_bytes);
                tma_load_2d(smem_u32(st), &tmA, bar(FULL + stage), kb * kGK, m0);
                tma_load_2d(smem_u32(st + kGABytes), mb, bar(FULL + stage), kb * kGK, n_local);
                issued[stage] = true;
                issued_phase[stage] = phase;
                if (++stage == kGStages) { stage = 0; phase ^= 1u; }
            }
            if (!ok) {
                record_error(a.err, kErrTimeout, kWhereGateGemm);
                *abort_flag = 1;
                for (int s = 0; s < kGStages; ++s)
                    if (issued[s]) mbar_wait_bounded(bar(FULL + s), issued_phase[s]);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // each 64-wide K block goes to a fresh accumulator (two, alternating), which the epilogue
            // adds into float-float sums: the tensor cores' rounding only ever spans 64 products
            const uint32_t idesc = idesc_bf16(kGM, a.BN);
            bool ok = true, any = false;
            int stage = 0;
            uint32_t phase = 0;
            for (int i = 0; i < nkb; ++i) {
                const int buf = i & 1;
                if (!mbar_wait(bar(CEMPTY + buf), ((i >> 1) & 1) ^ 1u, abort_flag)) { ok = false; break; }
                if (!mbar_wait(bar(FULL + stage), phase, abort_flag)) { ok = false; break; }
                fence_after();
                uint8_t* st = base + stage * stage_bytes;
                const uint64_t ad = smem_desc_sw128(smem_u32(st));
                const uint64_t bd = smem_desc_sw128(smem_u32(st + kGABytes));
                const uint32_t d_tmem = tmem_base + (uint32_t)(buf * a.BN);
#pragma unroll
                for (int kk = 0; kk < kGK / 16; ++kk)
                    mma_bf16(d_tmem, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc, kk != 0);
                any = true;
                commit(bar(EMPTY + stage));
                commit(bar(CFULL + buf));
                if (++stage == kGStages) { stage = 0; phase ^= 1u; }
            }
            if (!ok) {
                record_error(a.err, kErrTimeout, kWhereGateGemm);
                *abort_flag = 1;
            }
            if (any) {  // every MMA issued above has finished once LAST completes
                commit(bar(LAST));
                mbar_wait_bounded(bar(LAST), 0);
            }
        }
    } else {
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int r = q * 32 + lane;
        const int et = threadIdx.x - 64;  // 0..127
        const int ncols = min(a.BN, n_map - n_local);
        float hi[64], lo[64];
#pragma unroll
        for (int j = 0; j < 64; ++j) hi[j] = lo[j] = 0.f;
        float xs = 0.f, wsq = 0.f;
        bool ok = true;
        int stage = 0;
        uint32_t phase = 0;
        for (int i = 0; i < nkb && ok; ++i) {
            if (readers) {  // squared norms of this row of x and of this weight row, from the smem tiles
                ok = __all_sync(0xffffffffu, mbar_wait(bar(FULL + stage), phase, abort_flag));
                if (!ok) break;
                const uint8_t* st = base + stage * stage_bytes;
                if (x_norms) xs += sumsq_tile_row(st + r * 128);
                if (w_norms && et < a.BN) wsq += sumsq_tile_row(st + kGABytes + et * 128);
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(EMPTY + stage));
                if (++stage == kGStages) { stage = 0; phase ^= 1u; }
            }
            const int buf = i & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(bar(CFULL + buf), (i >> 1) & 1, abort_flag));
            if (!ok) break;
            fence_after();
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 16) {
                if (c0 < a.BN) {
                    uint32_t v[16];
                    tmem_ld16(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * a.BN + c0), v);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        float s_, e_;
                        two_sum(hi[c0 + j], __uint_as_float(v[j]), s_, e_);
                        hi[c0 + j] = s_;
                        lo[c0 + j] += e_;
                    }
                }
            }
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(CEMPTY + buf));
        }
        if (!ok) {
            if (lane == 0) {
                record_error(a.err, kErrTimeout, kWhereGateGemm);
                *abort_flag = 1;
            }
        } else {
            const int row = m0 + r;
            if (row < a.T) {
                float* dst = a.part + ((size_t)split * a.T + row) * a.Np + col0;
#pragma unroll
                for (int j = 0; j < 64; ++j)
                    if (j < ncols) dst[j] = hi[j] + lo[j];
                if (x_norms) a.xn2_part[(size_t)split * a.T + row] = xs;
            }
            if (w_norms && et < ncols) a.wn2_part[(size_t)split * a.Np + col0 + et] = wsq;
        }
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 1) tmem_free(tmem_base, tcols);
}

}  // namespace

GateGemmPlan gate_gemm_plan(int T, int d, int N0, int N1, int sms) {
    GateGemmPlan g{};
    const int nmax = N0 > N1 ? N0 : N1;
    g.BN = nmax >= kGMaxBN ? kGMaxBN : (nmax + 15) / 16 * 16;
    if (g.BN < 16) g.BN = 16;
    g.nt0 = (N0 + g.BN - 1) / g.BN;
    g.nt1 = N1 > 0 ? (N1 + g.BN - 1) / g.BN : 0;
    g.mt = (T + kGM - 1) / kGM;
    g.kb = d / kGK;
    g.Np = N0 + N1;
    const long tiles = (long)g.mt * (g.nt0 + g.nt1);
    int S = (tiles <= 0 || tiles >= sms) ? 1 : (int)(sms / tiles);
    if (S > kGateMaxSplits) S = kGateMaxSplits;
    if (S > g.kb) S = g.kb;
    if (S < 1) S = 1;
    g.per = (g.kb + S - 1) / S;
    g.S = (g.kb + g.per - 1) / g.per;
    g.smem = 1024 + (size_t)kGStages * (kGABytes + (size_t)g.BN * kGK * 2) + (2 * kGStages + 5) * 8 + 16;
    return g;
}

cudaError_t launch_gate_gemm(const GateGemmPlan& g, const void* x, const void* w0, const void* w1, int T, int d,
                             int N0, int N1, float* part, float* xn2_part, float* wn2_part, int* err,
                             cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    CUtensorMap ma, mb0, mb1;
    if (!tma_map_bf16(x, (uint64_t)d, (uint64_t)T, 0, kGM, &ma)) return cudaErrorInvalidValue;
    if (!tma_map_bf16(w0, (uint64_t)d, (uint64_t)N0, 0, (uint32_t)g.BN, &mb0)) return cudaErrorInvalidValue;
    if (N1 > 0) {
        if (!tma_map_bf16(w1, (uint64_t)d, (uint64_t)N1, 0, (uint32_t)g.BN, &mb1)) return cudaErrorInvalidValue;
    } else {
        mb1 = mb0;
    }
    GemmArgs a;
    a.part = part;
    a.xn2_part = xn2_part;
    a.wn2_part = wn2_part;
    a.x = static_cast<const bf16_t*>(x);
    a.w0 = static_cast<const bf16_t*>(w0);
    a.w1 = static_cast<const bf16_t*>(w1);
    a.T = T;
    a.d = d;
    a.N0 = N0;
    a.N1 = N1;
    a.Np = g.Np;
    a.BN = g.BN;
    a.nt0 = g.nt0;
    a.per = g.per;
    a.kb = g.kb;
    a.err = err;
    cudaError_t e = cudaFuncSetAttribute(gate_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)g.smem);
    if (e != cudaSuccess) return e;
    dim3 grid(g.mt, g.nt0 + g.nt1, g.S);
    gate_gemm_kernel<<<grid, kGThreads, g.smem, s>>>(ma, mb0, mb1, a);
    return cudaGetLastError();
}

}  // namespace moe
