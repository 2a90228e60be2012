// gate.cu -- fused gate: logits GEMM, softmax / noisy / cosine scoring, per-token top-k, gate weights.
//
// The gate follows NoisyTopKGating ("MoE sparse-compute acceleration", section 2.1: clean and noise
// linear maps without bias, noise scaled by softplus, topk of the noisy logits, softmax over the k
// chosen), the single linear + softmax gate ("How sparse activation improves efficiency", section 2.1;
// Tutel top.py), the full-softmax top-1 gate of the MOELayer on "PyTorch-CUDA-v2.6 and MoE", and
// Tutel's cosine_top ("Tutel MoE guide"; scored as cos(x P, e_j) / temperature).  "MoE on a single
// card" (section 3.3) recommends fusing the gate with the expert selection in one CUDA kernel; this is
// that kernel.
//
// One block = 32 tokens, three phases:
//  1. logits [32, N] into shared memory (N = E, 2E for the noisy gate, cos_dim for the cosine gate).
//     Small gates (N <= 16, N * d <= 16384: the weight fits in shared memory) use 512 threads, one warp
//     per token (two per warp in turn), the weight staged once per block; larger gates use 256 threads
//     and a tiled SIMT GEMM over 32-wide reduction chunks.  Either way products are summed in fp32
//     over chunks of at most 32, and the chunk sums are added with TwoSum compensation, so each
//     logit's error is at most 31 u sum|x_i w_i| + u |logit| <= 33 u |x| |w| (u = 2^-24;
//     Cauchy-Schwarz), a bound the kernel evaluates per token from the row norms.
//  2. one warp per token: scores, top-(k+1) by warp-shuffle argmax (ties -> lower expert id), and a
//     bound on the fp32 score error.  If two of the top-k scores, or the k-th and (k+1)-th, lie within
//     twice that bound, the token is queued for re-scoring; otherwise its choice is provably the
//     exact one and the gates are written.
//  3. the whole block re-scores each queued token's contenders (every expert whose fp32 score is
//     within twice the bound of the k-th best) with float-float dot products (TwoProduct/TwoSum,
//     about 48 bits) and picks the top-k of those by the exact scores.
// The gate weights use the fp32 scores (they are continuous in the scores; only the choice is
// discrete).  Optionally the block also writes the expert histogram of its 32 tokens (the first step
// of the dispatch), and the last block to finish runs the dispatch scan over all histograms.
#include <float.h>
#include <math.h>

#include "common.cuh"
#include "gate_common.cuh"
#include "kernels.h"
#include "scan.cuh"

namespace moe {

namespace {

using namespace gate;

constexpr int kBT = kTokensPerBlock;   // 32 tokens per block
constexpr int kSmallElems = 16384;     // N * d at or below which the weight is staged whole
constexpr int kKC = 32;                // reduction chunk
constexpr int kXSS = kBT + 1;          // shared stride of the transposed x tile

struct Layout {
    int N;       // logits per token
    int BN;      // logits per pass
    int stage;   // cosine: expert embeddings staged (transposed) in shared memory
    size_t logits, xs, ws, wst, wn2, xn2, sc, embs, embn, selv, seli, rl_tok, rl_n, rl_m, rl_den, rl_cand,
        rl_sc, fidx, hist, ex, uex, nref, scan_part, scan_padded, scan_kept, scan_wsum, total;
};

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

__host__ __device__ inline Layout make_layout(int gate, int E, int p, int d, int BN, int stage, bool small,
                                              int nthreads, bool pre = false) {
    const int nwarps = nthreads / 32;
    Layout L;
    L.N = gate == kGateSoftmax ? E : gate == kGateNoisy ? 2 * E : p;
    L.BN = BN;
    L.stage = stage;
    size_t o = 0;
    auto take = [&](size_t bytes, size_t al) { o = align_up(o, al); size_t r = o; o += bytes; return r; };
    L.logits = take(sizeof(float) * kBT * L.N, 16);
    L.xs = take(small ? 0 : sizeof(float) * kKC * kXSS, 16);
    L.ws = take(small ? 0 : sizeof(float) * kKC * (BN + 1), 16);
    L.wst = take(small ? sizeof(float) * (size_t)L.N * d : 0, 16);
    L.wn2 = take(sizeof(float) * L.N, 16);
    L.xn2 = take(sizeof(float) * kBT, 16);
    L.sc = take(sizeof(float) * nwarps * E, 16);
    L.embs = take(stage ? sizeof(float) * E * p : 0, 16);
    L.embn = take(gate == kGateCosine ? sizeof(float) * E : 0, 16);
    L.selv = take(sizeof(float) * nwarps * (kMaxTopK + 1), 16);
    L.seli = take(sizeof(int) * nwarps * (kMaxTopK + 1), 16);
    L.rl_tok = take(sizeof(int) * kBT, 16);
    L.rl_n = take(sizeof(int) * kBT, 16);
    L.rl_m = take(sizeof(float) * kBT, 16);
    L.rl_den = take(sizeof(float) * kBT, 16);
    L.rl_cand = take(sizeof(int) * kBT * kMaxCand, 16);
    L.rl_sc = take(sizeof(float) * kBT * kMaxCand, 16);
    L.fidx = take(sizeof(int) * kBT * kMaxTopK, 16);
    L.hist = take(sizeof(int) * E, 16);
    L.ex = take(sizeof(double) * kMaxCand, 16);
    L.uex = take(gate == kGateCosine ? sizeof(double) * p : 0, 16);
    L.nref = take(sizeof(int) * 4, 16);
    L.scan_part = take(sizeof(int) * nthreads, 16);
    L.scan_padded = take(sizeof(int) * (E + 1), 16);
    L.scan_kept = take(sizeof(int) * E, 16);
    L.scan_wsum = take(sizeof(int) * 33, 16);
    L.total = align_up(o, 16);
    return L;
}

// phase-1 variants: logits by the tiled SIMT GEMM or by the small-gate SIMT path
constexpr int kPh1Tiled = 0, kPh1Small = 1;

template <typename T, int GATE, int TM, int TN, int TX, int PH1>
__global__ void __launch_bounds__(PH1 == kPh1Small ? 512 : 256) gate_kernel(const GateParams P, const int stage) {
    pdl_wait();
    pdl_trigger();
    constexpr bool SMALL = PH1 == kPh1Small;
    constexpr int NT = SMALL ? 512 : 256;
    constexpr int NW = NT / 32;
    constexpr int TY = 256 / TX;
    constexpr int BN = TN * TX;
    static_assert(PH1 != kPh1Tiled || TM * TY == kBT, "a block covers 32 tokens");
    extern __shared__ __align__(16) unsigned char smem[];
    const Layout L = make_layout(GATE, P.E, P.p, P.d, BN, stage, SMALL, NT);
    float* logits = reinterpret_cast<float*>(smem + L.logits);
    float* xs = reinterpret_cast<float*>(smem + L.xs);
    float* ws = reinterpret_cast<float*>(smem + L.ws);
    float* wst = reinterpret_cast<float*>(smem + L.wst);
    float* wn2 = reinterpret_cast<float*>(smem + L.wn2);
    float* xn2 = reinterpret_cast<float*>(smem + L.xn2);
    float* scw = reinterpret_cast<float*>(smem + L.sc);
    float* embs = reinterpret_cast<float*>(smem + L.embs);
    float* embn = reinterpret_cast<float*>(smem + L.embn);
    float* selv_all = reinterpret_cast<float*>(smem + L.selv);
    int* seli_all = reinterpret_cast<int*>(smem + L.seli);
    int* rl_tok = reinterpret_cast<int*>(smem + L.rl_tok);
    int* rl_n = reinterpret_cast<int*>(smem + L.rl_n);
    float* rl_m = reinterpret_cast<float*>(smem + L.rl_m);
    float* rl_den = reinterpret_cast<float*>(smem + L.rl_den);
    int* rl_cand = reinterpret_cast<int*>(smem + L.rl_cand);
    float* rl_sc = reinterpret_cast<float*>(smem + L.rl_sc);
    int* fidx = reinterpret_cast<int*>(smem + L.fidx);
    int* hist = reinterpret_cast<int*>(smem + L.hist);
    double* ex = reinterpret_cast<double*>(smem + L.ex);
    double* uex = reinterpret_cast<double*>(smem + L.uex);
    int* nref = reinterpret_cast<int*>(smem + L.nref);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tok0 = blockIdx.x * kBT;
    const int ntok = min(kBT, P.T - tok0);
    const int N = L.N, d = P.d, E = P.E, k = P.k;
    const T* x = static_cast<const T*>(P.x);
    constexpr int WSS = BN + 1;

    if (tid == 0) nref[0] = 0;

    // ---------------------------------------------------------------- phase 1: logits [32, N]
    if constexpr (SMALL) {
        // stage the N weight rows (fp32) and their squared norms
        for (int i = tid * 8; i < N * d; i += NT * 8) {
            const int n = i / d, c = i % d;
            float v[8];
            load8(logit_row<T>(P, GATE, n) + c, v);
#pragma unroll
            for (int j = 0; j < 8; ++j) wst[i + j] = v[j];
        }
        __syncthreads();
        for (int n = warp; n < N; n += NW) {
            float q = 0.f;
            for (int c = lane; c < d; c += 32) q = fmaf(wst[n * d + c], wst[n * d + c], q);
            q = warp_sum(q);
            if (lane == 0) wn2[n] = q;
        }
        // one warp per token: lane owns the 8-element slices lane*8 + 256*j of the row
        for (int tt = warp; tt < kBT; tt += NW) {
            float hi[16], lo[16];
#pragma unroll
            for (int n = 0; n < 16; ++n) hi[n] = lo[n] = 0.f;
            float sq = 0.f;
            if (tt < ntok) {
                const T* xr = x + (size_t)(tok0 + tt) * d;
                for (int c0 = lane * 8; c0 < d; c0 += 4 * 256) {  // up to 4 slices = 32 products per chunk
                    float xv[4][8];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int c = c0 + j * 256;
                        if (c < d) load8(xr + c, xv[j]);
                        else {
#pragma unroll
                            for (int q = 0; q < 8; ++q) xv[j][q] = 0.f;
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int q = 0; q < 8; ++q) sq = fmaf(xv[j][q], xv[j][q], sq);
#pragma unroll
                    for (int n = 0; n < 16; ++n) {
                        if (n >= N) break;
                        float c = 0.f;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int col = c0 + j * 256;
                            if (col < d) {
                                const float4 w0 = *reinterpret_cast<const float4*>(wst + n * d + col);
                                const float4 w1 = *reinterpret_cast<const float4*>(wst + n * d + col + 4);
                                c = fmaf(xv[j][0], w0.x, c); c = fmaf(xv[j][1], w0.y, c);
                                c = fmaf(xv[j][2], w0.z, c); c = fmaf(xv[j][3], w0.w, c);
                                c = fmaf(xv[j][4], w1.x, c); c = fmaf(xv[j][5], w1.y, c);
                                c = fmaf(xv[j][6], w1.z, c); c = fmaf(xv[j][7], w1.w, c);
                            }
                        }
                        float s_, e_;
                        two_sum(hi[n], c, s_, e_);
                        hi[n] = s_;
                        lo[n] += e_;
                    }
                }
            }
            // compensated butterfly: every lane ends with the full sums
#pragma unroll
            for (int n = 0; n < 16; ++n) {
                if (n >= N) break;
                ff_warp_sum(hi[n], lo[n]);
                if (lane == n) logits[tt * N + n] = hi[n] + lo[n];
            }
            sq = warp_sum(sq);
            if (lane == 0) xn2[tt] = sq;
        }
    } else {
    const int ty = tid / TX, tx = tid % TX;
    const int lrow = tid >> 2, lc8 = (tid & 3) * 8;  // loaders: 4 threads per row, 8 elements each
    const T* xrow = (tid < 4 * kBT && lrow < ntok) ? x + (size_t)(tok0 + lrow) * d : nullptr;
    float sqx = 0.f;
    for (int n0 = 0; n0 < N; n0 += BN) {
        float hi[TM][TN], lo[TM][TN];
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) hi[i][j] = lo[i][j] = 0.f;
        float sqw = 0.f;
        const T* wrow = (tid < 4 * BN && n0 + lrow < N) ? logit_row<T>(P, GATE, n0 + lrow) : nullptr;
        for (int k0 = 0; k0 < d; k0 += kKC) {
            if (tid < 4 * kBT) {
                float v[8];
                if (xrow) load8(xrow + k0 + lc8, v);
                else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) v[j] = 0.f;
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    xs[(lc8 + j) * kXSS + lrow] = v[j];
                    if (n0 == 0) sqx = fmaf(v[j], v[j], sqx);
                }
            }
            if (tid < 4 * BN) {
                float v[8];
                if (wrow) load8(wrow + k0 + lc8, v);
                else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) v[j] = 0.f;
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    ws[(lc8 + j) * WSS + lrow] = v[j];
                    sqw = fmaf(v[j], v[j], sqw);
                }
            }
            __syncthreads();
            float c[TM][TN];
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) c[i][j] = 0.f;
#pragma unroll 8
            for (int kk = 0; kk < kKC; ++kk) {
                float a[TM], b[TN];
#pragma unroll
                for (int i = 0; i < TM; ++i) a[i] = xs[kk * kXSS + ty * TM + i];
#pragma unroll
                for (int j = 0; j < TN; ++j) b[j] = ws[kk * WSS + tx * TN + j];
#pragma unroll
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int j = 0; j < TN; ++j) c[i][j] = fmaf(a[i], b[j], c[i][j]);
            }
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) {
                    float s, e;
                    two_sum(hi[i][j], c[i][j], s, e);
                    hi[i][j] = s;
                    lo[i][j] += e;
                }
            __syncthreads();
        }
        sqw += __shfl_xor_sync(0xffffffffu, sqw, 1);
        sqw += __shfl_xor_sync(0xffffffffu, sqw, 2);
        if (tid < 4 * BN && (tid & 3) == 0 && n0 + lrow < N) wn2[n0 + lrow] = sqw;
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) {
                int n = n0 + tx * TN + j;
                if (n < N) logits[(ty * TM + i) * N + n] = hi[i][j] + lo[i][j];
            }
    }
    sqx += __shfl_xor_sync(0xffffffffu, sqx, 1);
    sqx += __shfl_xor_sync(0xffffffffu, sqx, 2);
    if (tid < 4 * kBT && (tid & 3) == 0) xn2[lrow] = sqx;
    }  // tiled phase 1

    if (GATE == kGateCosine) {  // expert embedding norms (and a transposed copy if it fits)
        const T* emb = static_cast<const T*>(P.emb);
        for (int e = warp; e < E; e += NW) {
            float s = 0.f;
            for (int j = lane * 8; j < P.p; j += 32 * 8) {
                float v[8];
                load8(emb + (size_t)e * P.p + j, v);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    s = fmaf(v[q], v[q], s);
                    if (stage) embs[(j + q) * E + e] = v[q];
                }
            }
            s = warp_sum(s);
            if (lane == 0) embn[e] = sqrtf(s);
        }
    }
    __syncthreads();

    // ---------------------------------------------------------------- phase 2: one warp per token
    float* sc = scw + warp * E;
    float* selv = selv_all + warp * (kMaxTopK + 1);
    int* seli = seli_all + warp * (kMaxTopK + 1);
    const int ksel = min(k + 1, E);
    for (int tt = warp; tt < ntok; tt += NW) {
        const int t = tok0 + tt;
        const float* Lr = logits + tt * N;
        const float xn = sqrtf(xn2[tt]);
        float dmax = 0.f;
        if (GATE == kGateSoftmax) {
            for (int e = lane; e < E; e += 32) {
                float s = Lr[e];
                sc[e] = s;
                dmax = fmaxf(dmax, P.cb * xn * sqrtf(wn2[e]) + 4.f * kU * fabsf(s));
            }
        } else if (GATE == kGateNoisy) {
            for (int e = lane; e < E; e += 32) {
                float c = Lr[e], z = Lr[E + e];
                float ep = P.eps[(size_t)t * E + e];
                float sp = softplus_f(z);
                float s = fmaf(ep, sp, c);
                sc[e] = s;
                float bc = P.cb * xn * sqrtf(wn2[e]) + 4.f * kU * fabsf(c);
                float bz = P.cb * xn * sqrtf(wn2[E + e]) + 4.f * kU * fabsf(z);
                dmax = fmaxf(dmax, bc + fabsf(ep) * (bz + 8.f * kU * (sp + 1.f)) + 4.f * kU * fabsf(s));
            }
        } else {
            const int p = P.p;
            float nu2 = 0.f, D2 = 0.f;
            for (int j = lane; j < p; j += 32) {
                float u = Lr[j];
                nu2 = fmaf(u, u, nu2);
                float du = P.cb * xn * sqrtf(wn2[j]) + 4.f * kU * fabsf(u);
                D2 = fmaf(du, du, D2);
            }
            nu2 = warp_sum(nu2);
            D2 = warp_sum(D2);
            const float nu = sqrtf(nu2), Dl = sqrtf(D2);
            // |cos(u~, e) - cos(u, e)| <= 2 |u~ - u| / |u|; fp32 dot, norms and divisions add (2p + 8) u
            const float rel = nu > 2.f * Dl ? (2.f * p + 8.f) * kU + 2.f * Dl / (nu - Dl) : INFINITY;
            const float nuc = fmaxf(nu, 1e-12f);
            const T* emb = static_cast<const T*>(P.emb);
            for (int e = lane; e < E; e += 32) {
                float dot = 0.f;
                if (stage) {
                    for (int j = 0; j < p; ++j) dot = fmaf(Lr[j], embs[j * E + e], dot);
                } else {
                    for (int j = 0; j < p; ++j) dot = fmaf(Lr[j], load1(emb + (size_t)e * p + j), dot);
                }
                float s = dot / (nuc * fmaxf(embn[e], 1e-12f)) * P.inv_temp;
                sc[e] = s;
                dmax = fmaxf(dmax, rel * P.inv_temp + 4.f * kU * fabsf(s));
            }
        }
        dmax = warp_max(dmax) * 1.0625f;
        __syncwarp();

        // top-(k+1) by repeated warp argmax; a lane owns experts lane, lane+32, ...
        uint32_t taken = 0;
        for (int r = 0; r < ksel; ++r) {
            float bv = -INFINITY;
            int bi = INT_MAX;
            for (int i = 0, e = lane; e < E; ++i, e += 32) {
                if ((taken >> i) & 1u) continue;
                float v = sc[e];
                if (bi == INT_MAX || v > bv) { bv = v; bi = e; }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                if (oi != INT_MAX && (bi == INT_MAX || ov > bv || (ov == bv && oi < bi))) { bv = ov; bi = oi; }
            }
            if (bi != INT_MAX && lane == (bi & 31)) taken |= 1u << (bi >> 5);
            if (lane == 0) { selv[r] = bv; seli[r] = bi; }
            __syncwarp();
        }
        bool refine = false;
        const float two_d = 2.f * dmax;
        for (int r = 1; r < k; ++r) refine |= !(selv[r - 1] - selv[r] > two_d);
        if (k < E) refine |= !(selv[k - 1] - selv[k] > two_d);
        const float m = selv[0];
        float den_all = 0.f;
        if (P.norm == 0) {
            float s = 0.f;
            for (int e = lane; e < E; e += 32) s += expf(sc[e] - m);
            den_all = warp_sum(s);
        }
        if (!refine) {
            float den = den_all;
            if (P.norm != 0) {
                den = 0.f;
                for (int r = 0; r < k; ++r) den += expf(selv[r] - m);
            }
            if (lane < k) {
                P.topk_idx[(size_t)t * k + lane] = seli[lane];
                P.topk_gate[(size_t)t * k + lane] = expf(selv[lane] - m) / den;
                fidx[tt * kMaxTopK + lane] = seli[lane];
            }
        } else {
            int q = 0;
            if (lane == 0) q = atomicAdd(nref, 1);
            q = __shfl_sync(0xffffffffu, q, 0);
            const float thr = selv[k - 1] - two_d;
            int cnt = 0;
            for (int base = 0; base < E; base += 32) {
                int e = base + lane;
                bool pred = e < E && !(sc[e] < thr);
                unsigned mask = __ballot_sync(0xffffffffu, pred);
                int pos = cnt + __popc(mask & lanemask_lt());
                if (pred && pos < kMaxCand) {
                    rl_cand[q * kMaxCand + pos] = e;
                    rl_sc[q * kMaxCand + pos] = sc[e];
                }
                cnt += __popc(mask);
            }
            if (cnt > kMaxCand) {
                if (lane == 0) record_error(P.err, kErrCheck, kWhereGate);
                cnt = kMaxCand;
            }
            if (lane == 0) {
                rl_tok[q] = tt;
                rl_n[q] = cnt;
                rl_m[q] = m;
                rl_den[q] = den_all;
            }
        }
        __syncwarp();
    }
    __syncthreads();

    // ---------------------------------------------------------------- phase 3: exact re-scoring
    const int nq = nref[0];
    for (int q = 0; q < nq; ++q) {
        const int tt = rl_tok[q], t = tok0 + tt, nc = rl_n[q];
        const T* xr = x + (size_t)t * d;
        const int* cand = rl_cand + q * kMaxCand;
        if (GATE == kGateCosine) {
            const T* proj = static_cast<const T*>(P.proj);
            for (int j = warp; j < P.p; j += NW) {
                double u = warp_dot_ff<T>(xr, proj + (size_t)j * d, d, lane);
                if (lane == 0) uex[j] = u;
            }
            __syncthreads();
            const T* emb = static_cast<const T*>(P.emb);
            for (int c = warp; c < nc; c += NW) {
                const int e = cand[c];
                double dot = 0.0, ne2 = 0.0, nu2 = 0.0;
                for (int j = lane; j < P.p; j += 32) {
                    double uj = uex[j];
                    double ej = (double)load1(emb + (size_t)e * P.p + j);
                    dot = fma(uj, ej, dot);
                    ne2 = fma(ej, ej, ne2);
                    nu2 = fma(uj, uj, nu2);
                }
                dot = warp_sum_d(dot);
                ne2 = warp_sum_d(ne2);
                nu2 = warp_sum_d(nu2);
                if (lane == 0) ex[c] = dot / (fmax(sqrt(nu2), 1e-12) * fmax(sqrt(ne2), 1e-12)) / P.temp;
            }
        } else {
            for (int c = warp; c < nc; c += NW) {
                const int e = cand[c];
                double s = warp_dot_ff<T>(xr, logit_row<T>(P, GATE, e), d, lane);
                if (GATE == kGateNoisy) {
                    double z = warp_dot_ff<T>(xr, logit_row<T>(P, GATE, E + e), d, lane);
                    s += (double)P.eps[(size_t)t * E + e] * log1p(exp(z));
                }
                if (lane == 0) ex[c] = s;
            }
        }
        __syncthreads();
        if (tid == 0) {
            uint64_t used = 0;
            int chosen[kMaxTopK];
            for (int r = 0; r < k; ++r) {
                int best = -1;
                for (int c = 0; c < nc; ++c) {
                    if ((used >> c) & 1ull) continue;
                    if (best < 0 || ex[c] > ex[best] || (ex[c] == ex[best] && cand[c] < cand[best])) best = c;
                }
                used |= 1ull << best;
                chosen[r] = best;
            }
            const float m = rl_m[q];
            float den = rl_den[q];
            if (P.norm != 0) {
                den = 0.f;
                for (int r = 0; r < k; ++r) den += expf(rl_sc[q * kMaxCand + chosen[r]] - m);
            }
            for (int r = 0; r < k; ++r) {
                const int c = chosen[r];
                P.topk_idx[(size_t)t * k + r] = cand[c];
                P.topk_gate[(size_t)t * k + r] = expf(rl_sc[q * kMaxCand + c] - m) / den;
                fidx[tt * kMaxTopK + r] = cand[c];
            }
        }
        __syncthreads();
    }

    // ---------------------------------------------------------------- block ranks and expert histogram
    if (P.blk_hist != nullptr) {
        for (int e = tid; e < E; e += NT) hist[e] = 0;
        __syncthreads();
        if (warp == 0)
            rank_pairs_warp([&](int i) { return fidx[(i / k) * kMaxTopK + i % k]; }, ntok * k, hist,
                            P.slot + (size_t)tok0 * k, lane);
        __syncthreads();
        for (int e = tid; e < E; e += NT) P.blk_hist[(size_t)blockIdx.x * E + e] = hist[e];
        if (P.ticket != nullptr) {  // the last block to finish runs the dispatch scan
            __syncthreads();  // the block's histogram is written; thread 0 publishes it with the ticket
            if (tid == 0) {
                __threadfence();
                nref[1] = atomicAdd(P.ticket, 1);
                __threadfence();
            }
            __syncthreads();
            if (nref[1] == (int)gridDim.x - 1) {
                ScanSmem sm;
                sm.part = reinterpret_cast<int*>(smem + L.scan_part);
                sm.padded = reinterpret_cast<int*>(smem + L.scan_padded);
                sm.kept = reinterpret_cast<int*>(smem + L.scan_kept);
                sm.wsum = reinterpret_cast<int*>(smem + L.scan_wsum);
                scan_experts(P.blk_hist, gridDim.x, E, P.C, P.count, P.offset, P.row_token, P.row_gate, sm);
                if (tid == 0) *P.ticket = 0;  // ready for the next call
            }
        }
    }
}

bool use_small(int gate, int E, int p, int d) {
    const int N = gate == kGateSoftmax ? E : gate == kGateNoisy ? 2 * E : p;
    return N <= 16 && N * d <= kSmallElems;
}

template <typename T, int GATE, int TM, int TN, int TX, int PH1>
cudaError_t launch_cfg(const GateParams& P, cudaStream_t s) {
    constexpr int BN = TN * TX;
    constexpr bool SMALL = PH1 == kPh1Small;
    constexpr int NT = SMALL ? 512 : 256;
    Layout L0 = make_layout(GATE, P.E, P.p, P.d, BN, 0, SMALL, NT);
    int stage = 0;
    if (GATE == kGateCosine) {
        Layout L1 = make_layout(GATE, P.E, P.p, P.d, BN, 1, SMALL, NT);
        if (L1.total <= 200 * 1024) { stage = 1; L0 = L1; }
    }
    auto kern = gate_kernel<T, GATE, TM, TN, TX, PH1>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L0.total);
    if (e != cudaSuccess) return e;
    const int blocks = (P.T + kBT - 1) / kBT;
    return launch_pdl(kern, dim3(blocks), dim3(NT), L0.total, s, P, stage);
}

template <typename T, int GATE>
cudaError_t launch_gate_t(const GateParams& P, cudaStream_t s) {
    const int N = GATE == kGateSoftmax ? P.E : GATE == kGateNoisy ? 2 * P.E : P.p;
    if (use_small(GATE, P.E, P.p, P.d)) return launch_cfg<T, GATE, 1, 1, 8, kPh1Small>(P, s);
    if (N <= 8) return launch_cfg<T, GATE, 1, 1, 8, kPh1Tiled>(P, s);
    if (N <= 16) return launch_cfg<T, GATE, 1, 2, 8, kPh1Tiled>(P, s);
    if (N <= 32) return launch_cfg<T, GATE, 2, 2, 16, kPh1Tiled>(P, s);
    return launch_cfg<T, GATE, 2, 4, 16, kPh1Tiled>(P, s);
}

template <typename T>
cudaError_t launch_gate_d(const GateParams& P, cudaStream_t s) {
    switch (P.gate) {
        case kGateSoftmax: return launch_gate_t<T, kGateSoftmax>(P, s);
        case kGateNoisy: return launch_gate_t<T, kGateNoisy>(P, s);
        default: return launch_gate_t<T, kGateCosine>(P, s);
    }
}

}  // namespace

size_t gate_smem_bytes(int gate, int E, int p, int d) {
    const int N = gate == kGateSoftmax ? E : gate == kGateNoisy ? 2 * E : p;
    const bool small = use_small(gate, E, p, d);
    const int BN = small ? 8 : N <= 8 ? 8 : N <= 16 ? 16 : N <= 32 ? 32 : 64;
    return make_layout(gate, E, p, d, BN, 0, small, small ? 512 : 256).total;
}

cudaError_t launch_gate(const GateParams& P, cudaStream_t s) {
    if (P.T <= 0) return cudaSuccess;
    if (P.part != nullptr) return launch_gate_select(P, s);  // logits precomputed on the tensor cores
    return P.bf16 ? launch_gate_d<bf16_t>(P, s) : launch_gate_d<float>(P, s);
}

}  // namespace moe
