// gate_select.cu -- scores, per-token top-k and gate weights from the tensor-core logits (bf16 layers).
//
// The logits come from gate_tc.cu as fp32 partial sums over splits of d, with the squared norms of the
// x rows and weight rows.  Three kernels:
//   select   one warp per token, 32 tokens per CTA: sums the token's partials in split order and forms
//            the scores -- softmax gate: the logit; noisy gate: clean + eps * softplus(noise)
//            (NoisyTopKGating, "MoE sparse-compute acceleration", section 2.1); cosine gate:
//            cos(u, e_j) / temperature with u = x P^T (Tutel's cosine_top), the dot products u . e_j of
//            the CTA's 32 tokens computed together from shared memory, 4 tokens x 4 experts a lane
//            in registers (the warp per token keeps the norms and the selection) -- with a bound on each
//            score's error from the tensor-core accumulation bound cb |x| |w|, and picks the top-(k+1)
//            by warp-shuffle argmax (ties -> lower expert id).  If two of them lie within twice the
//            bound, the token goes to a global queue with its contenders (every expert within twice the
//            bound of the k-th best); otherwise it gets its ids and gate weights here.
//   fold     cosine gate only: v_e = P^T e_e in float-float for every expert that contends somewhere.
//            u . e_e = x . v_e, and |u| and the temperature are common to all experts, so x . v_e / |e_e|
//            orders the experts exactly as cos(u, e_e) / temperature does.
//   rescore  every SM works through the queue, a token per CTA and a warp per contender: float-float
//            dot products (about 48 bits) give the contenders' scores, and the k best of those win.
// The gate weights always come from the fp32 scores (softmax over the k chosen, or over all E for top-1
// layers); the re-scoring only decides which experts are chosen.
#include <float.h>
#include <math.h>

#include "common.cuh"
#include "gate_common.cuh"
#include "kernels.h"
#include "scan.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

using namespace gate;

constexpr int kBT = kTokensPerBlock;  // tokens per CTA, one warp each
constexpr int kSelThreads = 32 * kBT;
constexpr int kSel = kMaxTopK + 1;

struct SelLayout {
    size_t logits, sc, wn2, embs, embn, tokn, cpart, selv, seli, cand, total;
};

// cosine scores from staged embeddings: the dot products u . e of the CTA's 32 tokens are split over
// kCosSlices ranges of the p components, a warp per (range, group of kCosGroup experts), lane = token
constexpr int kCosSlices = 8;
constexpr int kCosGroup = 16;
// row stride of the staged logits: the cosine gate's u rows are padded to an odd length so that the
// score loop's 32 lanes (32 token rows, one component each) fall in distinct banks
__host__ __device__ inline int sel_ld(int gate, int N) { return gate == kGateCosine ? N + 1 : N; }
__host__ __device__ inline int e32(int E) { return (E + kCosGroup - 1) / kCosGroup * kCosGroup; }

__host__ __device__ inline size_t al16(size_t v) { return (v + 15) / 16 * 16; }

__host__ __device__ inline SelLayout sel_layout(int gate, int E, int p, int stage) {
    const int N = gate == kGateSoftmax ? E : gate == kGateNoisy ? 2 * E : p;
    const bool cos = gate == kGateCosine;
    SelLayout L;
    size_t o = 0;
    auto take = [&](size_t bytes, size_t al) { o = (o + al - 1) / al * al; size_t r = o; o += bytes; return r; };
    L.logits = take(4 * (size_t)kBT * sel_ld(gate, N), 16);
    L.sc = take(cos ? 4 * (size_t)kBT * E : 0, 16);
    L.wn2 = take(4 * (size_t)N, 16);
    L.embs = take(stage ? 4 * (size_t)p * e32(E) : 0, 16);  // transposed [p][E rounded up to 16], zero-filled
    L.embn = take(cos ? 4 * (size_t)E : 0, 16);
    L.tokn = take(cos ? 4 * 2 * (size_t)kBT : 0, 16);
    L.cpart = take(stage ? 4 * (size_t)kCosSlices * kBT * e32(E) : 0, 16);
    L.selv = take(4 * kBT * kSel, 16);
    L.seli = take(4 * kBT * kSel, 16);
    L.cand = take(4 * kBT * kMaxCand, 16);
    L.total = al16(o);
    return L;
}

template <typename T, int GATE>
__global__ void __launch_bounds__(kSelThreads) gate_select_kernel(const GateParams P, const int stage) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ __align__(16) unsigned char smem[];
    const SelLayout L = sel_layout(GATE, P.E, P.p, stage);
    float* logits = reinterpret_cast<float*>(smem + L.logits);
    float* scs = reinterpret_cast<float*>(smem + L.sc);
    float* wn2 = reinterpret_cast<float*>(smem + L.wn2);
    float* embs = reinterpret_cast<float*>(smem + L.embs);
    float* embn = reinterpret_cast<float*>(smem + L.embn);
    float* tok_nuc = reinterpret_cast<float*>(smem + L.tokn);  // cosine: per token max(|u|, tiny)
    float* tok_rel = tok_nuc + kBT;                              // and the relative error bound of its cosines
    float* cpart = reinterpret_cast<float*>(smem + L.cpart);     // cosine: [slice][token][expert] partial dots
    float* selv_all = reinterpret_cast<float*>(smem + L.selv);
    int* seli_all = reinterpret_cast<int*>(smem + L.seli);
    int* cand_all = reinterpret_cast<int*>(smem + L.cand);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tok0 = blockIdx.x * kBT;
    const int ntok = min(kBT, P.T - tok0);
    const int E = P.E, k = P.k;
    const int N = GATE == kGateSoftmax ? E : GATE == kGateNoisy ? 2 * E : P.p;
    const int ldL = sel_ld(GATE, N);

    // ---- CTA: weight-row squared norms (sum of the split partials); cosine: embedding norms
    for (int n = tid; n < N; n += kSelThreads) {
        float q = 0.f;
        for (int s0 = 0; s0 < P.S; s0 += 8) {
            float a[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) a[j] = s0 + j < P.S ? P.wn2p[(size_t)(s0 + j) * P.Np + n] : 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) q += a[j];
        }
        wn2[n] = q;
    }
    if (GATE == kGateCosine) {
        const T* emb = static_cast<const T*>(P.emb);
        for (int e = warp; e < E; e += kBT) {
            float s = 0.f;
            for (int j = lane * 8; j < P.p; j += 32 * 8) {
                float v[8];
                load8(emb + (size_t)e * P.p + j, v);
#pragma unroll
                for (int q = 0; q < 8; ++q) s = fmaf(v[q], v[q], s);
            }
            s = warp_sum(s);
            if (lane == 0) embn[e] = sqrtf(s);
        }
        // the embeddings transposed into shared memory as fp32 [p][E32] (E32: E rounded up to 16, the
        // extra columns zero), so that the score loop reads 4 experts of a component with one broadcast
        // 16-byte load; consecutive threads take consecutive experts (p is a multiple of 8)
        if (stage) {
            const int E32 = e32(E), pc = P.p / 8;
            for (int i = tid; i < E32 * pc; i += kSelThreads) {
                const int e = i % E32, j = (i / E32) * 8;
                float v[8];
                if (e < E) {
                    load8(emb + (size_t)e * P.p + j, v);
                } else {
#pragma unroll
                    for (int q = 0; q < 8; ++q) v[q] = 0.f;
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) embs[(size_t)(j + q) * E32 + e] = v[q];
            }
        }
    }
    __syncthreads();

    // ---- one warp per token: the partial logits summed, and the scores (cosine with staged embeddings:
    // the norms of u here, the scores by the whole CTA below)
    const int tt = warp, t = tok0 + tt;
    float* selv = selv_all + tt * kSel;
    int* seli = seli_all + tt * kSel;
    int* cand = cand_all + tt * kMaxCand;
    float* Lr = logits + (size_t)tt * ldL;
    float* sc = GATE == kGateCosine ? scs + (size_t)tt * E : Lr;  // scores (in place unless cosine)
    const bool blocked = GATE == kGateCosine && stage;  // CTA-wide score step between two barriers
    float dmax = 0.f;
    if (tt < ntok) {
        float xq = 0.f;
        for (int sp = lane; sp < P.S; sp += 32) xq += P.xn2p[(size_t)sp * P.T + t];
        // the noisy gate's eps entries of experts lane and lane + 32 are loaded now, with the partials,
        // instead of after them (further ones when they are needed)
        float ep0 = 0.f, ep1 = 0.f;
        if (GATE == kGateNoisy) {
            if (lane < E) ep0 = P.eps[(size_t)t * E + lane];
            if (lane + 32 < E) ep1 = P.eps[(size_t)t * E + lane + 32];
        }
        // the splits' partials, summed in split order: a lane takes columns lane + 32 c, eight columns
        // of two splits (sixteen loads) in flight at a time
        {
            const float* src = P.part + (size_t)t * P.Np + lane;
            const size_t stride = (size_t)P.T * P.Np;
            const int ncl = (N + 31) / 32;
            for (int c0 = 0; c0 < ncl; c0 += 8) {
                float v[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) v[j] = 0.f;
                for (int s0 = 0; s0 < P.S; s0 += 2) {
                    float a[2][8];
#pragma unroll
                    for (int u = 0; u < 2; ++u)
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const bool ok = s0 + u < P.S && lane + 32 * (c0 + j) < N;
                            a[u][j] = ok ? src[(size_t)(s0 + u) * stride + 32 * (c0 + j)] : 0.f;
                        }
#pragma unroll
                    for (int u = 0; u < 2; ++u)
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            if (s0 + u < P.S) v[j] += a[u][j];
                }
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (lane + 32 * (c0 + j) < N) Lr[lane + 32 * (c0 + j)] = v[j];
            }
        }
        const float xn = sqrtf(warp_sum(xq));
        __syncwarp();
        if (GATE == kGateSoftmax) {
            for (int e = lane; e < E; e += 32) dmax = fmaxf(dmax, P.cb * xn * sqrtf(wn2[e]) + 4.f * kU * fabsf(Lr[e]));
        } else if (GATE == kGateNoisy) {
            for (int e = lane; e < E; e += 32) {
                const float c = Lr[e], z = Lr[E + e];
                const float ep = e == lane ? ep0 : e == lane + 32 ? ep1 : P.eps[(size_t)t * E + e];
                const float sp = softplus_f(z);
                const float s = fmaf(ep, sp, c);
                sc[e] = s;
                const float bc = P.cb * xn * sqrtf(wn2[e]) + 4.f * kU * fabsf(c);
                const float bz = P.cb * xn * sqrtf(wn2[E + e]) + 4.f * kU * fabsf(z);
                // softplus' slope is below 1, so an error in z moves softplus(z) by at most that much
                dmax = fmaxf(dmax, bc + fabsf(ep) * (bz + 8.f * kU * (sp + 1.f)) + 4.f * kU * fabsf(s));
            }
        } else {
            const int p = P.p;
            float nu2 = 0.f, D2 = 0.f;
            for (int j = lane; j < p; j += 32) {
                const float u = Lr[j];
                nu2 = fmaf(u, u, nu2);
                const float du = P.cb * xn * sqrtf(wn2[j]) + 4.f * kU * fabsf(u);
                D2 = fmaf(du, du, D2);
            }
            nu2 = warp_sum(nu2);
            D2 = warp_sum(D2);
            const float nu = sqrtf(nu2), Dl = sqrtf(D2);
            // |cos(u~, e) - cos(u, e)| <= 2 |u~ - u| / |u|; the fp32 dot, norms and division add (2p + 8) u
            const float rel = nu > 2.f * Dl ? (2.f * p + 8.f) * kU + 2.f * Dl / (nu - Dl) : INFINITY;
            const float nuc = fmaxf(nu, 1e-12f);
            if (blocked) {
                if (lane == 0) {
                    tok_nuc[tt] = nuc;
                    tok_rel[tt] = rel;
                }
            } else {
                const T* emb = static_cast<const T*>(P.emb);
                for (int e = lane; e < E; e += 32) {
                    // four interleaved partial sums (p is a multiple of 8); the error stays within the
                    // (2p + 8) u bound of a p-term dot product
                    float d4[4] = {0.f, 0.f, 0.f, 0.f};
                    for (int j = 0; j < p; j += 8) {
                        float ev[8];
                        load8(emb + (size_t)e * p + j, ev);
#pragma unroll
                        for (int q = 0; q < 8; ++q) d4[q & 3] = fmaf(Lr[j + q], ev[q], d4[q & 3]);
                    }
                    const float dot = (d4[0] + d4[1]) + (d4[2] + d4[3]);
                    const float s = dot / (nuc * fmaxf(embn[e], 1e-12f)) * P.inv_temp;
                    sc[e] = s;
                    dmax = fmaxf(dmax, rel * P.inv_temp + 4.f * kU * fabsf(s));
                }
            }
        }
    }
    if (blocked) {
        // cosine scores of the CTA's tokens: warp task (expert group g of kCosGroup, component range r)
        // covers the 32 tokens, lane (a, b) four tokens a + 8 i and four experts 4 b + q of the group, their
        // 16 partial dots in registers: per component four loads of u (eight distinct rows, odd stride:
        // conflict-free) and four of the experts' values (four distinct addresses) for 16 FMAs.  The ranges'
        // partial sums are then added in range order; a p-term dot product summed in this order stays within
        // the (2p + 8) u bound.
        __syncthreads();
        const int p = P.p, E32 = e32(E), ngr = E32 / kCosGroup, jl = p / kCosSlices;  // p: a multiple of 8
        const int la = lane & 7, lb = lane >> 3;
        for (int task = warp; task < ngr * kCosSlices; task += kBT) {
            const int g = task / kCosSlices, r = task % kCosSlices;
            float acc[4][4];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[a][q] = 0.f;
            const float* ur = logits + (size_t)la * ldL;
            const float* er = embs + g * kCosGroup + 4 * lb;
#pragma unroll 2
            for (int j = r * jl; j < (r + 1) * jl; ++j) {
                float u[4], ev[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) u[a] = ur[(size_t)(8 * a) * ldL + j];
#pragma unroll
                for (int q = 0; q < 4; ++q) ev[q] = er[(size_t)j * E32 + q];
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[a][q] = fmaf(u[a], ev[q], acc[a][q]);
            }
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    cpart[((size_t)r * kBT + la + 8 * a) * E32 + g * kCosGroup + 4 * lb + q] = acc[a][q];
        }
        __syncthreads();
        for (int i = tid; i < ntok * E; i += kSelThreads) {
            const int tq = i / E, e = i - tq * E;
            float dot = 0.f;
#pragma unroll
            for (int r = 0; r < kCosSlices; ++r) dot += cpart[((size_t)r * kBT + tq) * E32 + e];
            scs[(size_t)tq * E + e] = dot / (tok_nuc[tq] * fmaxf(embn[e], 1e-12f)) * P.inv_temp;
        }
        __syncthreads();
        if (tt < ntok) {
            float smax = 0.f;
            for (int e = lane; e < E; e += 32) smax = fmaxf(smax, fabsf(sc[e]));
            dmax = tok_rel[tt] * P.inv_temp + 4.f * kU * smax;
        }
    }
    if (tt < ntok) {
        dmax = warp_max(dmax) * 1.0625f;
        __syncwarp();

        // top-(k+1) by repeated warp argmax (ties -> lower expert id); a lane owns experts lane, lane + 32,
        // ...; each round takes the lane's best untaken key, then the warp's maximum key and the lowest
        // expert id holding it with two redux instructions
        const int ksel = min(k + 1, E);
        uint32_t taken = 0;
        for (int r = 0; r < ksel; ++r) {
            uint32_t bk = 0;
            int bi = INT_MAX;
            for (int i = 0, e = lane; e < E; ++i, e += 32) {
                if ((taken >> i) & 1u) continue;
                const uint32_t key = order_key(sc[e]);
                if (bi == INT_MAX || key > bk) { bk = key; bi = e; }
            }
            const uint32_t wk = __reduce_max_sync(0xffffffffu, bi != INT_MAX ? bk : 0u);
            const int wi = (int)__reduce_min_sync(0xffffffffu, (bi != INT_MAX && bk == wk) ? (uint32_t)bi : 0xffffffffu);
            if (lane == (wi & 31)) taken |= 1u << (wi >> 5);
            if (lane == 0) { selv[r] = sc[wi]; seli[r] = wi; }
        }
        __syncwarp();
        const float two_d = 2.f * dmax;
        bool refine = false;
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
            }
        } else {
            // contenders: every expert whose score is within twice the bound of the k-th best
            const float thr = selv[k - 1] - two_d;
            int cnt = 0;
            for (int base = 0; base < E; base += 32) {
                const int e = base + lane;
                const bool pred = e < E && !(sc[e] < thr);
                const unsigned mask = __ballot_sync(0xffffffffu, pred);
                const int pos = cnt + __popc(mask & lanemask_lt());
                if (pred && pos < kMaxCand) cand[pos] = e;
                cnt += __popc(mask);
            }
            if (cnt > kMaxCand) {
                if (lane == 0) record_error(P.err, kErrCheck, kWhereGate);
                cnt = kMaxCand;
            }
            __syncwarp();
            // the queue entry: token, contenders, the fp32 maximum score and softmax denominator, the
            // contenders' ids and fp32 scores
            int q = 0;
            if (lane == 0) q = atomicAdd(P.rq_count, 1);
            q = __shfl_sync(0xffffffffu, q, 0);
            int* ent = P.rq + (size_t)q * kRescoreInts;
            if (lane == 0) {
                ent[0] = t;
                ent[1] = cnt;
                ent[2] = __float_as_int(m);
                ent[3] = __float_as_int(den_all);
            }
            for (int c = lane; c < cnt; c += 32) {
                ent[4 + c] = cand[c];
                ent[4 + kMaxCand + c] = __float_as_int(sc[cand[c]]);
                if (GATE == kGateCosine) P.need[cand[c]] = 1;
            }
        }
    }
}

// ---- fold: v_e[i] = sum_j P[j][i] e_e[j] for the flagged experts, float-float (hi, lo) per entry.
// A CTA covers kFoldCols columns of P for a group of 32 experts: it stages the column strip of P and
// the group's embeddings (transposed, fp32) in shared memory a chunk of kFoldChunk rows at a time, and
// thread (column c, expert lane) accumulates over j in two interleaved float-float chains.
constexpr int kFoldCols = 8;
constexpr int kFoldChunk = 256;
constexpr int kFoldThreads = 32 * kFoldCols;

template <typename T>
__global__ void __launch_bounds__(kFoldThreads) gate_cos_fold_kernel(const GateParams P) {
    __shared__ float ps[kFoldChunk][kFoldCols];
    __shared__ float es[kFoldChunk][33];
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, lane = tid & 31, c = tid >> 5;
    const int E = P.E, d = P.d, p = P.p;
    const int i0 = blockIdx.x * kFoldCols, e0 = blockIdx.y * 32;
    const int e = e0 + lane;
    const bool mine = e < E && P.need[e] != 0;
    if (__syncthreads_or(mine) == 0) return;  // no expert of the group contends anywhere
    const T* proj = static_cast<const T*>(P.proj);
    const T* emb = static_cast<const T*>(P.emb);
    float hi[2] = {0.f, 0.f}, lo[2] = {0.f, 0.f};
    for (int j0 = 0; j0 < p; j0 += kFoldChunk) {
        const int nj = min(kFoldChunk, p - j0);
        __syncthreads();
        // a row of the strip is one 16-byte load (d and i0 are multiples of 8), and so are eight
        // consecutive entries of an embedding (p and j0 are multiples of 8)
#pragma unroll 2
        for (int j = tid; j < nj; j += kFoldThreads) {
            float v[8];
            load8(proj + (size_t)(j0 + j) * d + i0, v);
#pragma unroll
            for (int cc = 0; cc < kFoldCols; ++cc) ps[j][cc] = v[cc];
        }
        const int nv = nj / 8;
#pragma unroll 4
        for (int q = tid; q < 32 * nv; q += kFoldThreads) {
            const int ee = q / nv, j = (q % nv) * 8;
            float v[8];
            if (e0 + ee < E) {
                load8(emb + (size_t)(e0 + ee) * p + j0 + j, v);
            } else {
#pragma unroll
                for (int u = 0; u < 8; ++u) v[u] = 0.f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) es[j + u][ee] = v[u];
        }
        __syncthreads();
#pragma unroll 4
        for (int j = 0; j < nj; j += 2) {  // p is a multiple of 8
            ff_fma(hi[0], lo[0], ps[j][c], es[j][lane]);
            ff_fma(hi[1], lo[1], ps[j + 1][c], es[j + 1][lane]);
        }
    }
    ff_add(hi[0], lo[0], hi[1], lo[1]);
    if (mine) P.cosv[(size_t)e * d + i0 + c] = make_float2(hi[0], lo[0]);
}

// x . v_e by one warp, float-float: x_i * hi_i exactly (TwoProduct), x_i * lo_i in fp32 (its error is
// below 2^-48 |x_i v_i|); lanes take 8-element slices
template <typename T>
__device__ __forceinline__ double warp_dot_folded(const T* x, const float2* v, int d, int lane) {
    float hi[2] = {0.f, 0.f}, lo[2] = {0.f, 0.f};
    for (int i0 = lane * 8; i0 < d; i0 += 2 * 32 * 8) {
        float xa[2][8];
        float4 va[2][4];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int i = i0 + u * 32 * 8;
            if (i < d) {
                load8(x + i, xa[u]);
                const float4* vp = reinterpret_cast<const float4*>(v + i);
#pragma unroll
                for (int q = 0; q < 4; ++q) va[u][q] = vp[q];
            } else {
#pragma unroll
                for (int q = 0; q < 8; ++q) xa[u][q] = 0.f;
#pragma unroll
                for (int q = 0; q < 4; ++q) va[u][q] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                ff_fma(hi[u], lo[u], xa[u][2 * q], va[u][q].x);
                lo[u] = fmaf(xa[u][2 * q], va[u][q].y, lo[u]);
                ff_fma(hi[u], lo[u], xa[u][2 * q + 1], va[u][q].z);
                lo[u] = fmaf(xa[u][2 * q + 1], va[u][q].w, lo[u]);
            }
    }
    ff_add(hi[0], lo[0], hi[1], lo[1]);
    ff_warp_sum(hi[0], lo[0]);
    return (double)hi[0] + (double)lo[0];
}

// ---- rescore: CTA q takes queue entries q, q + gridDim.x, ...; warps take the entry's contenders
template <typename T, int GATE, int NW>
__global__ void __launch_bounds__(32 * NW) gate_rescore_kernel(const GateParams P) {
    __shared__ int cnd[kMaxCand];
    __shared__ float csc[kMaxCand];
    __shared__ double ex[kMaxCand];
    __shared__ int hdr[4];
    __shared__ int chosen[kMaxTopK];
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int E = P.E, k = P.k, d = P.d;
    const int nq = *P.rq_count;
    for (int q = blockIdx.x; q < nq; q += gridDim.x) {
        const int* ent = P.rq + (size_t)q * kRescoreInts;
        if (tid < 4) hdr[tid] = ent[tid];
        __syncthreads();
        const int nc = hdr[1];
        for (int c = tid; c < nc; c += 32 * NW) {
            cnd[c] = ent[4 + c];
            csc[c] = __int_as_float(ent[4 + kMaxCand + c]);
        }
        __syncthreads();
        const int t = hdr[0];
        const T* xr = static_cast<const T*>(P.x) + (size_t)t * d;
        for (int c = warp; c < nc; c += NW) {
            const int e = cnd[c];
            double sv;
            if (GATE == kGateCosine) {
                const T* er = static_cast<const T*>(P.emb) + (size_t)e * P.p;
                double ne2 = 0.0;
                for (int j = lane; j < P.p; j += 32) {
                    const double v = (double)load1(er + j);
                    ne2 = fma(v, v, ne2);
                }
                ne2 = warp_sum_d(ne2);
                sv = warp_dot_folded<T>(xr, P.cosv + (size_t)e * d, d, lane) / fmax(sqrt(ne2), 1e-12);
            } else {
                sv = warp_dot_ff<T>(xr, logit_row<T>(P, GATE, e), d, lane);
                if (GATE == kGateNoisy) {
                    const double z = warp_dot_ff<T>(xr, logit_row<T>(P, GATE, E + e), d, lane);
                    sv += (double)P.eps[(size_t)t * E + e] * log1p(exp(z));
                }
            }
            if (lane == 0) ex[c] = sv;
        }
        __syncthreads();
        if (warp == 0) {
            // k rounds of a warp argmax over the contenders (a lane holds contenders lane and lane + 32);
            // equal scores go to the lower expert id
            bool used0 = lane >= nc, used1 = lane + 32 >= nc;
            for (int r = 0; r < k; ++r) {
                double bv = -INFINITY;
                int bid = INT_MAX, bc = -1;
                if (!used0) { bv = ex[lane]; bid = cnd[lane]; bc = lane; }
                if (!used1 && (bc < 0 || ex[lane + 32] > bv || (ex[lane + 32] == bv && cnd[lane + 32] < bid))) {
                    bv = ex[lane + 32];
                    bid = cnd[lane + 32];
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
                if (bc < 0) {  // fewer than k contenders: only a NaN score leaves the top k out
                    if (lane == 0) record_error(P.err, kErrCheck, kWhereGate);
                    bc = 0;
                }
                if (bc == lane) used0 = true;
                if (bc == lane + 32) used1 = true;
                if (lane == 0) chosen[r] = bc;
            }
            __syncwarp();
            const float m = __int_as_float(hdr[2]);
            float den = __int_as_float(hdr[3]);
            if (P.norm != 0) {
                den = 0.f;
                for (int r = 0; r < k; ++r) den += expf(csc[chosen[r]] - m);
            }
            if (lane < k) {
                P.topk_idx[(size_t)t * k + lane] = cnd[chosen[lane]];
                P.topk_gate[(size_t)t * k + lane] = expf(csc[chosen[lane]] - m) / den;
            }
        }
        __syncthreads();
    }
}

template <typename T, int GATE>
cudaError_t launch_sel(const GateParams& P, cudaStream_t s) {
    int stage = 0;
    SelLayout L = sel_layout(GATE, P.E, P.p, 0);
    if (GATE == kGateCosine) {
        const SelLayout L1 = sel_layout(GATE, P.E, P.p, 1);
        if (L1.total <= 200 * 1024) { stage = 1; L = L1; }
    }
    auto kern = gate_select_kernel<T, GATE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3((P.T + kBT - 1) / kBT), dim3(kSelThreads), L.total, s, P, stage);
}

}  // namespace

size_t gate_select_smem_bytes(int gate, int E, int p) { return sel_layout(gate, E, p, 0).total; }

cudaError_t launch_gate_rescore(const GateParams& P, cudaStream_t s) {
    if (P.T <= 0) return cudaSuccess;
    if (!P.bf16 || P.rq_count == nullptr) return cudaErrorInvalidValue;
    // eight warps per CTA and four CTAs per SM: queued tokens mostly have k + 1 contenders.  Many experts
    // make long contender lists more likely: there sixteen warps and two CTAs per SM.
    const int sms = device_sm_count();
    if (P.E >= 128) {
        const dim3 grid((unsigned)(2 * sms));
        switch (P.gate) {
            case kGateSoftmax: return launch_pdl(gate_rescore_kernel<bf16_t, kGateSoftmax, 16>, grid, dim3(512), 0, s, P);
            case kGateNoisy: return launch_pdl(gate_rescore_kernel<bf16_t, kGateNoisy, 16>, grid, dim3(512), 0, s, P);
            default: return launch_pdl(gate_rescore_kernel<bf16_t, kGateCosine, 16>, grid, dim3(512), 0, s, P);
        }
    }
    const dim3 grid((unsigned)(4 * sms));
    switch (P.gate) {
        case kGateSoftmax: return launch_pdl(gate_rescore_kernel<bf16_t, kGateSoftmax, 8>, grid, dim3(256), 0, s, P);
        case kGateNoisy: return launch_pdl(gate_rescore_kernel<bf16_t, kGateNoisy, 8>, grid, dim3(256), 0, s, P);
        default: return launch_pdl(gate_rescore_kernel<bf16_t, kGateCosine, 8>, grid, dim3(256), 0, s, P);
    }
}

cudaError_t launch_gate_cos_fold(const GateParams& P, cudaStream_t s) {
    if (P.T <= 0) return cudaSuccess;
    if (!P.bf16 || P.gate != kGateCosine || P.need == nullptr || P.cosv == nullptr) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)(P.d / kFoldCols), (unsigned)((P.E + 31) / 32));  // d is a multiple of 8
    return launch_pdl(gate_cos_fold_kernel<bf16_t>, grid, dim3(kFoldThreads), 0, s, P);
}

cudaError_t launch_gate_select(const GateParams& P, cudaStream_t s) {
    if (P.T <= 0) return cudaSuccess;
    if (!P.bf16) return cudaErrorInvalidValue;
    switch (P.gate) {
        case kGateSoftmax: return launch_sel<bf16_t, kGateSoftmax>(P, s);
        case kGateNoisy: return launch_sel<bf16_t, kGateNoisy>(P, s);
        default: return launch_sel<bf16_t, kGateCosine>(P, s);
    }
}

}  // namespace moe
