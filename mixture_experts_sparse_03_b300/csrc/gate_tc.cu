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
// weight rows are one or two tensors (w_gate, then w_noise for the noisy gate); an n-tile holds both
// halves only when each has the same <= 64 rows (a multiple of 8): two TMA boxes fill the tile, w_gate's
// rows then w_noise's, so that x is read once per token tile.  Tiles are up to 128 logits wide when
// 64-wide ones would need more than one wave of CTAs.  Small token counts split K across CTAs so that
// about one CTA per SM streams the weights; the splits' partials are summed in a fixed order by the
// selection kernel (deterministic).
//
// CTA = 12 warps: warp 0 issues the TMA loads into a ring of stages; warp 1 allocates TMEM and one lane
// issues the MMAs, each 128-wide chunk of K (two blocks) into a fresh accumulator (up to 8 in rotation,
// 512 TMEM columns); warps 2-9 (a TMEM lane quarter each, and one of two 64-column halves of the tile) add
// every chunk's accumulator into compensated (Kahan) sums, so the tensor cores' fp32 rounding only ever
// spans 128 products and the error bound does not grow with d; warps 10-11 compute the squared norms of the x
// rows (n-tile 0) and weight rows (m-tile 0) from the shared-memory tiles -- the selection kernel bounds
// each logit's error by them.  The logits leave through a shared-memory staging tile, a row at a time.
// When one CTA can hold every logit of its tokens (softmax gate, E <= 64) the selection runs in the same
// launch: a cluster of up to four CTAs per 128-token tile splits K, the CTAs add their compensated
// partials through distributed shared memory, and each selects its share of the rows, a warp per token
// (select_row): top-k, near-tie re-scoring, gates; then the dispatch's pair ranks and block histograms,
// and the dispatch scan in the last CTA -- the whole gate in one launch.
// Every mbarrier wait is bounded; on expiry the kernel records MOE_ERR_DEVICE_TIMEOUT, waits (bounded)
// for its own copies and MMAs, frees its TMEM and returns.
#include "common.cuh"
#include "gate_common.cuh"
#include "kernels.h"
#include "scan.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

using namespace tc;
using gate::kMaxCand;
using gate::kU;
using gate::order_key;

constexpr int kGM = 128, kGK = 64;
constexpr int kGMaxStages = 12;  // TMA ring depth: as many stages as fit (the CTAs are few and latency-bound)
constexpr int kGThreads = 384;  // producer, MMA, 8 accumulation warps, 2 norm warps
constexpr int kGAccWarps = 8, kGNormWarp0 = 10;
constexpr int kGChunks = 8;     // TMEM accumulators the MMAs rotate through (at most; 512 columns in all)
constexpr int kGKChunk = 2;     // 64-wide K blocks an accumulator sums (8 MMA steps) before it is added
constexpr int kGMaxBN = 128;    // logits per n-tile: two accumulation warps per row, 64 compensated sums each
constexpr int kGFusedMaxBN = 64;  // fused selection: every logit of a token in one accumulation warp
constexpr int kGStageStride = 64 + 4;  // epilogue staging: floats per row (16-byte stores conflict-free)
constexpr uint32_t kGABytes = kGM * kGK * 2;  // 16 KiB
constexpr int kGMaxCluster = 4;  // fused gate: CTAs splitting K per token tile (at most one per row quarter)

// fused gate: each CTA's compensated partial logits (hi [BN][128], lo [BN][128], column-major so that a
// warp reads 32 consecutive rows), x-row norms [128] and weight-row norms [kGFusedMaxBN] over its K range
__host__ __device__ constexpr size_t red_bytes(int BN) { return (size_t)(2 * BN * kGM + kGM + kGFusedMaxBN) * 4; }

struct GemmArgs {
    float* part;       // [S][T][Np]
    float* xn2_part;   // [S][T]
    float* wn2_part;   // [S][Np]
    const bf16_t* x;   // [T, d]
    const bf16_t* w0;  // [N0, d]
    const bf16_t* w1;  // [N1, d] or nullptr
    int T, d, N0, N1, Np, BN, nt0, per, kb, stages;
    int both;          // 1: one n-tile holds w_gate's N0 rows, then w_noise's N1 = N0 rows
    int nch;           // TMEM accumulators in rotation
    int* err;
};

// sum of squares of the 64 bf16 of one 128-byte row of a swizzled tile (the swizzle only permutes the
// row's 16-byte chunks, so the sum is over the same elements).  Row r reads its chunks starting at chunk
// r mod 8: rows are 128 bytes apart, so in the same chunk order eight consecutive rows would hit the same
// four banks; rotated, each group of eight lanes covers all 32 banks.
__device__ __forceinline__ float sumsq_tile_row(const uint8_t* row, int r) {
    float s[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 u = *reinterpret_cast<const uint4*>(row + ((c + r) & 7) * 16);
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

constexpr int kGWarps = kGThreads / 32;
constexpr int kLgStride = kGFusedMaxBN + 1;  // row stride of the logits staged for the selection

// Fused selection smem (softmax gate, all logits of a token in one CTA): per row the top-(k+1) values
// and ids and the chosen ids, the rows' x norms and the weight-row norms, per warp the contenders of a
// re-scored row, per row quarter the dispatch rank counters, and the dispatch scan's scratch.
struct FusedSmem {
    float selv[kGM][kMaxTopK + 1];
    int seli[kGM][kMaxTopK + 1];
    int fidx[kGM][kMaxTopK];
    float xn2[kGM];
    float wn2[kGFusedMaxBN];
    int cand[kGWarps][kMaxCand];
    double ex[kGWarps][kMaxCand];
    int running[4][kGFusedMaxBN];
    int part[kGThreads];
    int padded[kGFusedMaxBN + 1];
    int kept[kGFusedMaxBN];
    int wsum[33];
    int last;
};

// Selection of one token by one warp from its fp32 logits lrow[0..E) (E <= 64; lane l holds experts l
// and l + 32): the error bound of each logit from the tensor-core accumulation bound cb |x| |w_e|, the
// top-(k+1) by warp reductions over order keys (ties -> lower expert id), then the ids and gates, or --
// when two of the top-(k+1) lie within twice the bound -- float-float re-scoring of every expert within
// twice the bound of the k-th best, a warp dot product per contender, and the k best of those.
__device__ __forceinline__ void select_row(const GateParams& P, FusedSmem& fs, const float* lrow, int rr, int t,
                                           int w, int lane) {
    const int E = P.E, k = P.k, ksel = min(k + 1, E);
    const bool h0 = lane < E, h1 = lane + 32 < E;
    const float v0 = h0 ? lrow[lane] : 0.f, v1 = h1 ? lrow[lane + 32] : 0.f;
    const float xn = sqrtf(fs.xn2[rr]);
    float dm = 0.f;
    if (h0) dm = P.cb * xn * sqrtf(fs.wn2[lane]) + 4.f * kU * fabsf(v0);
    if (h1) dm = fmaxf(dm, P.cb * xn * sqrtf(fs.wn2[lane + 32]) + 4.f * kU * fabsf(v1));
    const float two_d = 2.f * (warp_max(dm) * 1.0625f);
    const uint32_t key0 = order_key(v0), key1 = order_key(v1);
    bool t0 = !h0, t1 = !h1;  // taken (or absent)
    for (int s2 = 0; s2 < ksel; ++s2) {
        // the lane's best untaken expert (its lower id wins a tie), then the warp's
        const bool use1 = !t1 && (t0 || key1 > key0);
        const bool has = !t0 || !t1;
        const uint32_t bk = use1 ? key1 : key0;
        const uint32_t wk = __reduce_max_sync(0xffffffffu, has ? bk : 0u);
        const int wi = (int)__reduce_min_sync(0xffffffffu, has && bk == wk ? (uint32_t)(use1 ? lane + 32 : lane) : 0xffffffffu);
        if (wi == lane) t0 = true;
        if (wi == lane + 32) t1 = true;
        const float wv = __shfl_sync(0xffffffffu, wi < 32 ? v0 : v1, wi & 31);
        if (lane == 0) {
            fs.selv[rr][s2] = wv;
            fs.seli[rr][s2] = wi;
        }
    }
    __syncwarp();
    bool refine = false;
    for (int s2 = 1; s2 < k; ++s2) refine |= !(fs.selv[rr][s2 - 1] - fs.selv[rr][s2] > two_d);
    if (k < E) refine |= !(fs.selv[rr][k - 1] - fs.selv[rr][k] > two_d);
    const float m = fs.selv[rr][0];
    float den_all = 0.f;
    if (P.norm == 0) den_all = warp_sum((h0 ? expf(v0 - m) : 0.f) + (h1 ? expf(v1 - m) : 0.f));
    if (!refine) {
        float den = den_all;
        if (P.norm != 0) {
            den = 0.f;
            for (int s2 = 0; s2 < k; ++s2) den += expf(fs.selv[rr][s2] - m);
        }
        if (lane < k) {
            P.topk_idx[(size_t)t * k + lane] = fs.seli[rr][lane];
            P.topk_gate[(size_t)t * k + lane] = expf(fs.selv[rr][lane] - m) / den;
            fs.fidx[rr][lane] = fs.seli[rr][lane];
        }
        return;
    }
    // contenders, in expert order
    const float thr = fs.selv[rr][k - 1] - two_d;
    const bool c0 = h0 && !(v0 < thr), c1 = h1 && !(v1 < thr);
    const unsigned m0b = __ballot_sync(0xffffffffu, c0), m1b = __ballot_sync(0xffffffffu, c1);
    const int n0 = __popc(m0b), cnt = n0 + __popc(m1b);  // at most 64 = kMaxCand
    if (c0) fs.cand[w][__popc(m0b & lanemask_lt())] = lane;
    if (c1) fs.cand[w][n0 + __popc(m1b & lanemask_lt())] = lane + 32;
    __syncwarp();
    const bf16_t* xr = static_cast<const bf16_t*>(P.x) + (size_t)t * P.d;
    for (int c0 = 0; c0 < cnt; c0 += 4) {  // four contenders per pass, their loads in flight together
        const int nb = min(4, cnt - c0);
        const bf16_t* rows[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            rows[u] = static_cast<const bf16_t*>(P.w_gate) + (size_t)fs.cand[w][c0 + min(u, nb - 1)] * P.d;
        double v[4];
        gate::warp_dot_ff4<bf16_t>(xr, rows, nb, P.d, lane, v);
        if (lane == 0)
            for (int u = 0; u < nb; ++u) fs.ex[w][c0 + u] = v[u];
    }
    __syncwarp();
    // k rounds of a warp argmax over the contenders' exact scores (equal scores -> lower expert id)
    bool u0 = lane >= cnt, u1 = lane + 32 >= cnt;
    for (int s2 = 0; s2 < k; ++s2) {
        double bv = -INFINITY;
        int bid = INT_MAX, bc = -1;
        if (!u0) { bv = fs.ex[w][lane]; bid = fs.cand[w][lane]; bc = lane; }
        if (!u1 && (bc < 0 || fs.ex[w][lane + 32] > bv)) {
            bv = fs.ex[w][lane + 32];
            bid = fs.cand[w][lane + 32];
            bc = lane + 32;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const double ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oid = __shfl_xor_sync(0xffffffffu, bid, off);
            const int oc = __shfl_xor_sync(0xffffffffu, bc, off);
            if (oc >= 0 && (bc < 0 || ov > bv || (ov == bv && oid < bid))) {
                bv = ov;
                bid = oid;
                bc = oc;
            }
        }
        if (bc < 0) {  // fewer than k contenders: only a NaN logit leaves the top k out
            if (lane == 0) record_error(P.err, kErrCheck, kWhereGateGemm);
            bc = 0;
            bid = fs.cand[w][0];
        }
        if (bc == lane) u0 = true;
        if (bc == lane + 32) u1 = true;
        if (lane == 0) fs.fidx[rr][s2] = bid;
    }
    __syncwarp();
    // gates from the fp32 logits of the chosen experts
    float den = den_all;
    if (P.norm != 0) {
        den = 0.f;
        for (int s2 = 0; s2 < k; ++s2) den += expf(lrow[fs.fidx[rr][s2]] - m);
    }
    if (lane < k) {
        const int e = fs.fidx[rr][lane];
        P.topk_idx[(size_t)t * k + lane] = e;
        P.topk_gate[(size_t)t * k + lane] = expf(lrow[e] - m) / den;
    }
}

template <bool FUSED, int BNC>
__global__ void __launch_bounds__(kGThreads, 1)
    gate_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                     const __grid_constant__ CUtensorMap tmB1, const GemmArgs a, const GateParams P) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t b_bytes = (uint32_t)a.BN * kGK * 2;
    const uint32_t stage_bytes = kGABytes + b_bytes;
    const int NS = a.stages;
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + NS * stage_bytes);
    // bars: full[NS], empty[NS], chunk_full[kGChunks], chunk_empty[kGChunks], last
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * NS + 2 * kGChunks + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    FusedSmem& fs = *reinterpret_cast<FusedSmem*>(tmem_holder + 4);
    float* red = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(&fs) + sizeof(FusedSmem));  // fused only
    const int FULL = 0, EMPTY = NS, CFULL = 2 * NS, CEMPTY = 2 * NS + kGChunks, LAST = 2 * NS + 2 * kGChunks;
    auto bar = [&](int i) { return smem_u32(bars + i); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // fused: grid (cs, m-tiles) in clusters of cs CTAs, CTA `split` of a cluster taking the split-th range
    // of K blocks of the cluster's token tile; otherwise grid (m-tiles, n-tiles, splits)
    const int mt = FUSED ? blockIdx.y : blockIdx.x, nt = FUSED ? 0 : blockIdx.y;
    const int split = FUSED ? blockIdx.x : blockIdx.z;
    const int cs = FUSED ? (int)gridDim.x : 1;
    const bool second = !a.both && nt >= a.nt0;             // tile of w_noise (noisy gate)
    const int n_local = (second ? nt - a.nt0 : nt) * a.BN;  // first weight row of the tile
    const int n_map = a.both ? a.BN : second ? a.N1 : a.N0;  // rows of that weight tensor (both: of the two)
    const int col0 = (second ? a.N0 : 0) + n_local;         // first output column
    const int m0 = mt * kGM;
    const int kb0 = split * a.per, kb1 = min(a.kb, kb0 + a.per);
    const int nkb = kb1 - kb0;
    const int ncols = min(a.BN, n_map - n_local);
    const bool x_norms = FUSED || (a.xn2_part != nullptr && nt == 0);
    const bool w_norms = FUSED || (a.wn2_part != nullptr && mt == 0);
    const bool readers = x_norms || w_norms;  // the norm warps read the smem tiles too
    const int nch = a.nch;
    uint32_t tcols = 32;
    while (tcols < (uint32_t)(nch * a.BN)) tcols <<= 1;

    if (threadIdx.x == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(second ? &tmB1 : &tmB0);
        *abort_flag = 0;
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar(FULL + s), 1);
            mbar_init(bar(EMPTY + s), readers ? 3 : 1);  // the MMAs' commit and the two norm warps
        }
        for (int s = 0; s < kGChunks; ++s) {
            mbar_init(bar(CFULL + s), 1);
            mbar_init(bar(CEMPTY + s), a.BN > 64 ? 8 : 4);  // the accumulation warps with columns
        }
        mbar_init(bar(LAST), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_holder), tcols);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem_base = *tmem_holder;
    pdl_wait();  // the set-up above overlaps the previous kernel; its outputs are read below
    pdl_trigger();

    float hi[BNC], lo[BNC];  // accumulation warps: the compensated sums (value hi + lo) of row r
#pragma unroll
    for (int j = 0; j < BNC; ++j) hi[j] = lo[j] = 0.f;
    if (warp == 0) {
        if (lane == 0) {
            const CUtensorMap* mb = second ? &tmB1 : &tmB0;
            uint32_t issued_phase[kGMaxStages];
            bool issued[kGMaxStages];
            for (int s = 0; s < kGMaxStages; ++s) { issued[s] = false; issued_phase[s] = 0; }
            bool ok = true;
            int stage = 0;
            uint32_t phase = 0;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait(bar(EMPTY + stage), phase ^ 1u, abort_flag)) { ok = false; break; }
                uint8_t* st = base + stage * stage_bytes;
                mbar_expect_tx(bar(FULL + stage), stage_bytes);
                tma_load_2d(smem_u32(st), &tmA, bar(FULL + stage), kb * kGK, m0);
                tma_load_2d(smem_u32(st + kGABytes), mb, bar(FULL + stage), kb * kGK, n_local);
                if (a.both)  // w_noise's rows below w_gate's (N0 a multiple of 8: whole swizzle atoms)
                    tma_load_2d(smem_u32(st + kGABytes + (uint32_t)a.N0 * 128u), &tmB1, bar(FULL + stage),
                                kb * kGK, 0);
                issued[stage] = true;
                issued_phase[stage] = phase;
                if (++stage == NS) { stage = 0; phase ^= 1u; }
            }
            if (!ok) {
                record_error(a.err, kErrTimeout, kWhereGateGemm);
                *abort_flag = 1;
                for (int s = 0; s < NS; ++s)
                    if (issued[s]) mbar_wait_bounded(bar(FULL + s), issued_phase[s]);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // each chunk of kGKChunk K blocks (128 products) goes to a fresh accumulator (nch of them, in
            // turn), which the accumulation warps add into compensated sums: the tensor cores' rounding only
            // ever spans 128 products, and the MMAs run up to nch chunks ahead of the additions
            const uint32_t idesc = idesc_bf16(kGM, a.BN);
            bool ok = true, any = false;
            int stage = 0;
            uint32_t phase = 0;
            for (int i = 0; i < nkb; ++i) {
                const int ci = i / kGKChunk, buf = ci % nch;
                const bool first = i % kGKChunk == 0, last = i % kGKChunk == kGKChunk - 1 || i == nkb - 1;
                if (first && !mbar_wait(bar(CEMPTY + buf), ((ci / nch) & 1) ^ 1u, abort_flag)) { ok = false; break; }
                if (!mbar_wait(bar(FULL + stage), phase, abort_flag)) { ok = false; break; }
                fence_after();
                uint8_t* st = base + stage * stage_bytes;
                const uint64_t ad = smem_desc_sw128(smem_u32(st));
                const uint64_t bd = smem_desc_sw128(smem_u32(st + kGABytes));
                const uint32_t d_tmem = tmem_base + (uint32_t)(buf * a.BN);
#pragma unroll
                for (int kk = 0; kk < kGK / 16; ++kk)
                    mma_bf16(d_tmem, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc, !first || kk != 0);
                any = true;
                commit(bar(EMPTY + stage));
                if (last) commit(bar(CFULL + buf));
                if (++stage == NS) { stage = 0; phase ^= 1u; }
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
    } else if (warp >= kGNormWarp0) {
        // norm warps: squared norms of the x rows and weight rows over this CTA's K range, from the tiles;
        // thread nr takes rows nr and nr + 64
        const int nr = threadIdx.x - 32 * kGNormWarp0;  // 0..63
        float xs0 = 0.f, xs1 = 0.f, ws0 = 0.f, ws1 = 0.f;
        bool ok = true;
        int stage = 0;
        uint32_t phase = 0;
        for (int i = 0; i < nkb && readers; ++i) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(FULL + stage), phase, abort_flag));
            if (!ok) break;
            const uint8_t* st = base + stage * stage_bytes;
            if (x_norms) {
                xs0 += sumsq_tile_row(st + nr * 128, nr);
                xs1 += sumsq_tile_row(st + (nr + 64) * 128, nr + 64);
            }
            if (w_norms && nr < a.BN) ws0 += sumsq_tile_row(st + kGABytes + nr * 128, nr);
            if (w_norms && nr + 64 < a.BN) ws1 += sumsq_tile_row(st + kGABytes + (nr + 64) * 128, nr + 64);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(EMPTY + stage));
            if (++stage == NS) { stage = 0; phase ^= 1u; }
        }
        if (!ok) {
            if (lane == 0) {
                record_error(a.err, kErrTimeout, kWhereGateGemm);
                *abort_flag = 1;
            }
        } else if constexpr (!FUSED) {
            if (x_norms && m0 + nr < a.T) a.xn2_part[(size_t)split * a.T + m0 + nr] = xs0;
            if (x_norms && m0 + nr + 64 < a.T) a.xn2_part[(size_t)split * a.T + m0 + nr + 64] = xs1;
            if (w_norms && nr < ncols) a.wn2_part[(size_t)split * a.Np + col0 + nr] = ws0;
            if (w_norms && nr + 64 < ncols) a.wn2_part[(size_t)split * a.Np + col0 + nr + 64] = ws1;
        } else {
            red[2 * a.BN * kGM + nr] = xs0;
            red[2 * a.BN * kGM + nr + 64] = xs1;
            red[2 * a.BN * kGM + kGM + nr] = nr < ncols ? ws0 : 0.f;  // fused: BN <= 64
        }
        // the stage ring is read no more: the accumulation warps may stage the logits in it
        if constexpr (!FUSED) named_bar_arrive(1, 32 * (kGAccWarps + 2));
    } else {
        // accumulation warps: a TMEM lane quarter (32 rows) and a 64-column half of the tile each
        const int q = warp & 3;
        const int r = q * 32 + lane;
        const int cb = ((warp - 2) >> 2) * 64;  // the warp's first column
        const bool active = cb < a.BN;          // tiles of <= 64 logits leave warps 6-9 idle
        // G = 64 / BNC accumulators per round: their TMEM loads are in flight together, then added.
        // Compensated summation (Kahan: value = hi + lo, lo the running correction): the sum of n blocks
        // errs by at most 2u * sum |block| + O(n u^2) (Higham, Accuracy and Stability of Numerical
        // Algorithms, section 4.3) at four additions per block.
        constexpr int G = 64 / BNC;
        const int nck = (nkb + kGKChunk - 1) / kGKChunk;  // accumulator chunks
        bool ok = true;
        for (int i0 = 0; i0 < nck && ok && active; i0 += G) {
            const int ng = min(G, nck - i0);
            for (int j = 0; j < ng && ok; ++j)
                ok = __all_sync(0xffffffffu, mbar_wait(bar(CFULL + (i0 + j) % nch), ((i0 + j) / nch) & 1,
                                                       abort_flag));
            if (!ok) break;
            fence_after();
            if constexpr (BNC == 64) {  // one accumulator per round, loaded 16 columns at a time
                const uint32_t tb =
                    tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)((i0 % nch) * a.BN + cb);
#pragma unroll
                for (int c0 = 0; c0 < 64; c0 += 16) {
                    if (cb + c0 < a.BN) {
                        uint32_t v[16];
                        tmem_ld16(tb + (uint32_t)c0, v);
#pragma unroll
                        for (int c = 0; c < 16; ++c) kahan_add(hi[c0 + c], lo[c0 + c], __uint_as_float(v[c]));
                    }
                }
            } else {
            uint32_t v[G][BNC];
#pragma unroll
            for (int j = 0; j < G; ++j)
#pragma unroll
                for (int c0 = 0; c0 < BNC; c0 += 16)
                    if (j < ng && c0 < a.BN)
                        tmem_ld16_async(tmem_base + ((uint32_t)(q * 32) << 16) +
                                            (uint32_t)(((i0 + j) % nch) * a.BN + c0),
                                        *reinterpret_cast<uint32_t(*)[16]>(&v[j][c0]));
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < G; ++j)
#pragma unroll
                for (int c = 0; c < BNC; ++c)
                    if (j < ng && c < a.BN) kahan_add(hi[c], lo[c], __uint_as_float(v[j][c]));  // K order
            }
            fence_before();
            __syncwarp();
            if (lane == 0)
                for (int j = 0; j < ng; ++j) mbar_arrive(bar(CEMPTY + (i0 + j) % nch));
        }
        if (!ok) {
            if (lane == 0) {
                record_error(a.err, kErrTimeout, kWhereGateGemm);
                *abort_flag = 1;
            }
        }
        if constexpr (!FUSED) {
            // through a staging tile in the (finished) stage ring: each thread writes its row, then the
            // warp stores row after row, 128 contiguous bytes per instruction
            named_bar_sync(1, 32 * (kGAccWarps + 2));  // every norm warp is done with the ring
            float* stg = reinterpret_cast<float*>(base) + (size_t)(warp - 2) * 32 * kGStageStride;
            const int wcols = min(min(BNC, a.BN - cb), ncols - cb);
            if (ok && active && wcols > 0) {
#pragma unroll
                for (int j = 0; j < BNC; j += 4)
                    *reinterpret_cast<float4*>(stg + lane * kGStageStride + j) =
                        make_float4(hi[j] + lo[j], hi[j + 1] + lo[j + 1], hi[j + 2] + lo[j + 2], hi[j + 3] + lo[j + 3]);
                __syncwarp();
                const int rows = min(32, a.T - (m0 + q * 32));
                float* dst = a.part + ((size_t)split * a.T + m0 + q * 32) * a.Np + col0 + cb;
#pragma unroll
                for (int rr = 0; rr < 32; ++rr)
#pragma unroll
                    for (int c0 = 0; c0 < BNC; c0 += 32)
                        if (rr < rows && c0 + lane < wcols)
                            dst[(size_t)rr * a.Np + c0 + lane] = stg[rr * kGStageStride + c0 + lane];
            }
        } else if (active) {
#pragma unroll
            for (int j = 0; j < BNC; ++j)
                if (j < a.BN) {
                    red[j * kGM + r] = hi[j];
                    red[(a.BN + j) * kGM + r] = lo[j];
                }
        }
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 1) tmem_free(tmem_base, tcols);
    if constexpr (FUSED) {
        if (cs > 1) cluster_sync();  // every CTA's partials (written before the barrier above) are visible
        // the CTA that selects row quarter q (q = split, split + cs, ...) adds the cluster's partials into
        // the quarter's accumulation warp: its own first, then the others in rank order (a fixed order), and
        // stages the logits in the stage ring, which the finished K loop no longer uses
        float* lg = reinterpret_cast<float*>(base);  // [kGM][kLgStride]
        const int q = warp & 3;
        if (warp >= 2 && warp < 6 && q % cs == split) {
            const int r = q * 32 + lane;
            float xs = red[2 * a.BN * kGM + r];
            // generic pointers into the other CTAs' shared memory (rank order): plain loads the compiler can
            // issue together
            const int np = cs - 1;  // peer u is CTA u, or u + 1 from this CTA's rank on
            const float* rp[kGMaxCluster - 1];
#pragma unroll
            for (int u = 0; u < kGMaxCluster - 1; ++u)
                rp[u] = static_cast<const float*>(
                    __cluster_map_shared_rank(red, (unsigned)min(u < split ? u : u + 1, cs - 1)));
#pragma unroll
            for (int j = 0; j < BNC; ++j)
                if (j < a.BN) {
                    float ph[kGMaxCluster - 1], pl[kGMaxCluster - 1];
#pragma unroll
                    for (int u = 0; u < kGMaxCluster - 1; ++u)
                        if (u < np) {
                            ph[u] = rp[u][j * kGM + r];
                            pl[u] = rp[u][(a.BN + j) * kGM + r];
                        }
#pragma unroll
                    for (int u = 0; u < kGMaxCluster - 1; ++u)
                        if (u < np) ff_add(hi[j], lo[j], ph[u], pl[u]);
                }
#pragma unroll
            for (int u = 0; u < kGMaxCluster - 1; ++u)
                if (u < np) xs += rp[u][2 * a.BN * kGM + r];
#pragma unroll
            for (int j = 0; j < BNC; ++j)
                if (j < a.BN) lg[r * kLgStride + j] = hi[j] + lo[j];
            fs.xn2[r] = xs;
            if (q == split) {  // the first quarter's warp also sums the weight-row norms
                for (int j = lane; j < kGFusedMaxBN; j += 32) {
                    float w = 0.f;
                    for (int c = 0; c < cs; ++c)
                        w += static_cast<const float*>(__cluster_map_shared_rank(red, (unsigned)c))[2 * a.BN * kGM + kGM + j];
                    fs.wn2[j] = w;
                }
            }
        }
        if (cs > 1) cluster_arrive();  // done reading the other CTAs' shared memory
        __syncthreads();
        // selection: a warp per row of the CTA's quarters
        const int nown = (4 - split + cs - 1) / cs;  // quarters this CTA selects
        for (int i = warp; i < 32 * nown; i += kGWarps) {
            const int rr = (split + cs * (i >> 5)) * 32 + (i & 31);
            if (m0 + rr < P.T) select_row(P, fs, lg + rr * kLgStride, rr, m0 + rr, warp, lane);
        }
        __syncthreads();
        // the dispatch's first step, a warp per 32-token block: pair ranks in token order, block histogram
        if (P.blk_hist != nullptr && warp < nown) {
            const int qq = split + cs * warp;
            const int t0 = m0 + qq * 32, ntok = min(32, P.T - t0), E = P.E, k = P.k;
            if (ntok > 0) {
                for (int e = lane; e < E; e += 32) fs.running[warp][e] = 0;
                __syncwarp();
                rank_pairs_warp([&](int i) { return fs.fidx[qq * 32 + i / k][i % k]; }, ntok * k, fs.running[warp],
                                P.slot + (size_t)t0 * k, lane);
                __syncwarp();
                for (int e = lane; e < E; e += 32) P.blk_hist[(size_t)(t0 / 32) * E + e] = fs.running[warp][e];
            }
        }
        __syncthreads();
        // the dispatch scan runs in the last CTA to finish its blocks' histograms
        if (P.blk_hist != nullptr && P.ticket != nullptr) {
            if (threadIdx.x == 0) {
                __threadfence();
                fs.last = atomicAdd(P.ticket, 1) == (int)(gridDim.x * gridDim.y) - 1;
                __threadfence();
            }
            __syncthreads();
            if (fs.last) {
                ScanSmem sm{fs.part, fs.padded, fs.kept, fs.wsum};
                const int nblk = (P.T + kTokensPerBlock - 1) / kTokensPerBlock;
                scan_experts(P.blk_hist, nblk, P.E, P.C, P.count, P.offset, P.row_token, P.row_gate, sm);
                if (threadIdx.x == 0) *P.ticket = 0;  // ready for the next call
            }
        }
        if (cs > 1) cluster_wait();  // no CTA leaves while another may still read its shared memory
    }
}

}  // namespace

GateGemmPlan gate_gemm_plan(int T, int d, int N0, int N1, int sms, bool fuse_select) {
    GateGemmPlan g{};
    g.fused = fuse_select && N1 == 0 && N0 <= kGFusedMaxBN;
    g.cs = 1;
    if (g.fused) {
        // a cluster of cs CTAs per token tile splits K; their compensated partials meet in shared memory,
        // so the selecting CTA still sees every logit of its tokens.  As many as keep one wave.
        const long mtiles = (T + kGM - 1) / kGM;
        for (int c = kGMaxCluster; c > 1; c >>= 1)
            if (c <= d / kGK && mtiles * c <= sms) { g.cs = c; break; }
        sms = 1;  // no split-K partials in global memory
    }
    g.mt = (T + kGM - 1) / kGM;
    const int nmax = N0 > N1 ? N0 : N1;
    // 64-wide tiles, or up to 128 wide when 64-wide ones would take more than one wave
    const long tiles64 = (long)g.mt * ((N0 + 63) / 64 + (N1 + 63) / 64);
    const int bn_max = !g.fused && tiles64 > sms ? kGMaxBN : kGFusedMaxBN;
    g.both = !g.fused && N1 == N0 && 2 * N0 <= bn_max && N0 % 8 == 0;
    if (g.both) {
        g.BN = 2 * N0;  // one tile: w_gate's rows, then w_noise's
        g.nt0 = 1;
        g.nt1 = 0;
    } else {
        g.BN = nmax >= bn_max ? bn_max : (nmax + 15) / 16 * 16;
        if (g.BN < 16) g.BN = 16;
        g.nt0 = (N0 + g.BN - 1) / g.BN;
        g.nt1 = N1 > 0 ? (N1 + g.BN - 1) / g.BN : 0;
    }
    g.nch = 512 / g.BN < kGChunks ? 512 / g.BN : kGChunks;
    g.kb = d / kGK;
    g.Np = N0 + N1;
    const long tiles = (long)g.mt * (g.nt0 + g.nt1);
    int S = (tiles <= 0 || tiles >= sms) ? 1 : (int)(sms / tiles);
    if (S > kGateMaxSplits) S = kGateMaxSplits;
    if (S > g.kb) S = g.kb;
    if (S < 1) S = 1;
    g.per = (g.kb + S * g.cs - 1) / (S * g.cs);
    g.S = g.fused ? 1 : (g.kb + g.per - 1) / g.per;
    const size_t stage_bytes = kGABytes + (size_t)g.BN * kGK * 2;
    const size_t fixed = 1024 + 16 + (g.fused ? sizeof(FusedSmem) + red_bytes(g.BN) : 0) + (2 * kGChunks + 1) * 8;
    g.stages = (int)((200 * 1024 - fixed) / (stage_bytes + 16));
    if (g.stages > kGMaxStages) g.stages = kGMaxStages;
    if (g.stages > g.per) g.stages = g.per < 2 ? 2 : g.per;
    // after the K loop the stage ring holds the fused selection's logits, or the epilogue's staging tiles
    const size_t after = g.fused ? (size_t)kGM * kLgStride * 4
                                 : (size_t)(g.BN > 64 ? kGAccWarps : 4) * 32 * kGStageStride * 4;
    while ((size_t)g.stages * stage_bytes < after) ++g.stages;
    g.smem = fixed + (size_t)g.stages * (stage_bytes + 16);
    return g;
}

cudaError_t launch_gate_gemm(const GateGemmPlan& g, const void* x, const void* w0, const void* w1, int T, int d,
                             int N0, int N1, float* part, float* xn2_part, float* wn2_part, int* err,
                             const GateParams* sel, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    CUtensorMap ma, mb0, mb1;
    if (!tma_map_bf16(x, (uint64_t)d, (uint64_t)T, 0, kGM, &ma)) return cudaErrorInvalidValue;
    const uint32_t box_rows = (uint32_t)(g.both ? N0 : g.BN);
    if (!tma_map_bf16(w0, (uint64_t)d, (uint64_t)N0, 0, box_rows, &mb0)) return cudaErrorInvalidValue;
    if (N1 > 0) {
        if (!tma_map_bf16(w1, (uint64_t)d, (uint64_t)N1, 0, box_rows, &mb1)) return cudaErrorInvalidValue;
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
    a.stages = g.stages;
    a.both = g.both ? 1 : 0;
    a.nch = g.nch;
    a.err = err;
    const dim3 grid = g.fused ? dim3(g.cs, g.mt, 1) : dim3(g.mt, g.nt0 + g.nt1, g.S);
    if (g.fused && sel == nullptr) return cudaErrorInvalidValue;
    const GateParams none{};
    auto go = [&](auto kern, const GateParams& p) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)g.smem);
        if (e != cudaSuccess) return e;
        if (!g.fused || g.cs == 1) return launch_pdl(kern, grid, dim3(kGThreads), g.smem, s, ma, mb0, mb1, a, p);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = dim3(kGThreads);
        cfg.dynamicSmemBytes = g.smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)g.cs;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        return cudaLaunchKernelEx(&cfg, kern, ma, mb0, mb1, a, p);
    };
    cudaError_t e;
    if (g.fused)
        e = g.BN <= 16 ? go(gate_gemm_kernel<true, 16>, *sel)
            : g.BN <= 32 ? go(gate_gemm_kernel<true, 32>, *sel) : go(gate_gemm_kernel<true, 64>, *sel);
    else
        e = g.BN <= 16 ? go(gate_gemm_kernel<false, 16>, none)
            : g.BN <= 32 ? go(gate_gemm_kernel<false, 32>, none) : go(gate_gemm_kernel<false, 64>, none);  // per warp
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace moe
