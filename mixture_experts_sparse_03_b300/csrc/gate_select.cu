// gate_select.cu -- scores, per-token top-k and gate weights from the tensor-core logits (bf16 layers).
//
// The logits come from gate_tc.cu as fp32 partial sums over splits of d, with the squared norms of the
// x rows and weight rows.  One warp per token, 32 tokens (one dispatch block) per CTA:
//   1. the warp sums its token's partials in split order, forms the scores -- softmax gate: the logit;
//      noisy gate: clean + eps * softplus(noise) (NoisyTopKGating, "MoE sparse-compute acceleration",
//      section 2.1); cosine gate: cos(u, e_j) / temperature with u = x P^T (Tutel's cosine_top) -- and
//      a bound on each score's error from the tensor-core accumulation bound cb |x| |w|;
//   2. picks the top-(k+1) by warp-shuffle argmax (ties -> lower expert id);
//   3. if two of them lie within twice the bound, queues the token; the CTA then re-scores each queued
//      token's contenders with float-float dot products (about 48 bits), a warp per contender (the
//      cosine gate first recomputes all of u, a warp per component), and picks by those scores;
//   4. writes ids and gate weights (softmax over the k chosen scores, or the full softmax for top-1
//      layers), the CTA's expert histogram, and the last CTA to finish runs the dispatch scan.
#include <float.h>
#include <math.h>

#include "common.cuh"
#include "gate_common.cuh"
#include "kernels.h"
#include "scan.cuh"

namespace moe {

namespace {

using namespace gate;

constexpr int kBT = kTokensPerBlock;  // tokens per CTA, one warp each
constexpr int kSelThreads = 32 * kBT;
constexpr int kSel = kMaxTopK + 1;

struct SelLayout {
    size_t logits, sc, wn2, embs, embn, selv, seli, cand, candn, exs, fidx, hist, queue, nq, uex, cm, cden,
        scan_part, scan_padded, scan_kept, scan_wsum, total;
};

__host__ __device__ inline size_t al16(size_t v) { return (v + 15) / 16 * 16; }

__host__ __device__ inline SelLayout sel_layout(int gate, int E, int p, int stage) {
    const int N = gate == kGateSoftmax ? E : gate == kGateNoisy ? 2 * E : p;
    const bool cos = gate == kGateCosine;
    SelLayout L;
    size_t o = 0;
    auto take = [&](size_t bytes, size_t al) { o = (o + al - 1) / al * al; size_t r = o; o += bytes; return r; };
    L.logits = take(4 * (size_t)kBT * N, 16);
    L.sc = take(cos ? 4 * (size_t)kBT * E : 0, 16);
    L.wn2 = take(4 * (size_t)N, 16);
    L.embs = take(stage ? 4 * (size_t)p * E : 0, 16);
    L.embn = take(cos ? 4 * (size_t)E : 0, 16);
    L.selv = take(4 * kBT * kSel, 16);
    L.seli = take(4 * kBT * kSel, 16);
    L.cand = take(4 * kBT * kMaxCand, 16);
    L.candn = take(4 * kBT, 16);
    L.exs = take(8 * kBT * kMaxCand, 16);
    L.fidx = take(4 * kBT * kMaxTopK, 16);
    L.hist = take(4 * (size_t)E, 16);
    L.queue = take(4 * kBT, 16);
    L.nq = take(16, 16);
    L.uex = take(cos ? 8 * (size_t)p : 0, 16);
    L.cm = take(4 * kBT, 16);
    L.cden = take(4 * kBT, 16);
    L.scan_part = take(4 * kSelThreads, 16);
    L.scan_padded = take(4 * (size_t)(E + 1), 16);
    L.scan_kept = take(4 * (size_t)E, 16);
    L.scan_wsum = take(4 * 33, 16);
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
    float* selv_all = reinterpret_cast<float*>(smem + L.selv);
    int* seli_all = reinterpret_cast<int*>(smem + L.seli);
    int* cand_all = reinterpret_cast<int*>(smem + L.cand);
    int* candn = reinterpret_cast<int*>(smem + L.candn);
    double* exs_all = reinterpret_cast<double*>(smem + L.exs);
    int* fidx = reinterpret_cast<int*>(smem + L.fidx);
    int* hist = reinterpret_cast<int*>(smem + L.hist);
    int* queue = reinterpret_cast<int*>(smem + L.queue);
    int* nq = reinterpret_cast<int*>(smem + L.nq);
    double* uex = reinterpret_cast<double*>(smem + L.uex);
    float* cm = reinterpret_cast<float*>(smem + L.cm);
    float* cden = reinterpret_cast<float*>(smem + L.cden);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tok0 = blockIdx.x * kBT;
    const int ntok = min(kBT, P.T - tok0);
    const int E = P.E, k = P.k, d = P.d;
    const int N = GATE == kGateSoftmax ? E : GATE == kGateNoisy ? 2 * E : P.p;
    const T* x = static_cast<const T*>(P.x);

    if (tid == 0) nq[0] = 0;
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

    // ---- one warp per token
    const int tt = warp, t = tok0 + tt;
    float* selv = selv_all + tt * kSel;
    int* seli = seli_all + tt * kSel;
    int* cand = cand_all + tt * kMaxCand;
    if (tt < ntok) {
        float* Lr = logits + (size_t)tt * N;
        float xq = 0.f;
        for (int sp = lane; sp < P.S; sp += 32) xq += P.xn2p[(size_t)sp * P.T + t];
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
        float* sc = GATE == kGateCosine ? scs + (size_t)tt * E : Lr;  // scores (in place unless cosine)
        float dmax = 0.f;
        if (GATE == kGateSoftmax) {
            for (int e = lane; e < E; e += 32) dmax = fmaxf(dmax, P.cb * xn * sqrtf(wn2[e]) + 4.f * kU * fabsf(Lr[e]));
        } else if (GATE == kGateNoisy) {
            for (int e = lane; e < E; e += 32) {
                const float c = Lr[e], z = Lr[E + e];
                const float ep = P.eps[(size_t)t * E + e];
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
            const T* emb = static_cast<const T*>(P.emb);
            for (int e = lane; e < E; e += 32) {
                float dot = 0.f;
                if (stage) {
                    for (int j = 0; j < p; ++j) dot = fmaf(Lr[j], embs[j * E + e], dot);
                } else {
                    for (int j = 0; j < p; ++j) dot = fmaf(Lr[j], load1(emb + (size_t)e * p + j), dot);
                }
                const float s = dot / (nuc * fmaxf(embn[e], 1e-12f)) * P.inv_temp;
                sc[e] = s;
                dmax = fmaxf(dmax, rel * P.inv_temp + 4.f * kU * fabsf(s));
            }
        }
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
                fidx[tt * kMaxTopK + lane] = seli[lane];
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
            if (lane == 0) {  // the CTA re-scores its queued tokens together below
                const int q = atomicAdd(nq, 1);
                queue[q] = tt;
                candn[tt] = cnt;
                cm[tt] = m;
                cden[tt] = den_all;
            }
        }
    }
    __syncthreads();

    // ---- exact re-scoring of the queued tokens, one at a time by the whole CTA: a warp per contender
    // (softmax / noisy), or first a warp per component of u = x P^T and then per contender (cosine)
    {
        const int nqueued = nq[0];
        for (int qi = 0; qi < nqueued; ++qi) {
            const int tq = queue[qi], tg = tok0 + tq, nc = candn[tq];
            const int* cnd = cand_all + tq * kMaxCand;
            double* ex = exs_all + tq * kMaxCand;
            const T* xr = x + (size_t)tg * d;
            if (GATE == kGateCosine) {
                const T* proj = static_cast<const T*>(P.proj);
                for (int j = warp; j < P.p; j += kBT) {
                    const double u = warp_dot_ff<T>(xr, proj + (size_t)j * d, d, lane);
                    if (lane == 0) uex[j] = u;
                }
                __syncthreads();
                const T* emb = static_cast<const T*>(P.emb);
                for (int c = warp; c < nc; c += kBT) {
                    const int e = cnd[c];
                    double dot = 0.0, ne2 = 0.0, nu2 = 0.0;
                    for (int j = lane; j < P.p; j += 32) {
                        const double uj = uex[j];
                        const double ej = (double)load1(emb + (size_t)e * P.p + j);
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
                for (int c = warp; c < nc; c += kBT) {
                    const int e = cnd[c];
                    double sv = warp_dot_ff<T>(xr, logit_row<T>(P, GATE, e), d, lane);
                    if (GATE == kGateNoisy) {
                        const double z = warp_dot_ff<T>(xr, logit_row<T>(P, GATE, E + e), d, lane);
                        sv += (double)P.eps[(size_t)tg * E + e] * log1p(exp(z));
                    }
                    if (lane == 0) ex[c] = sv;
                }
            }
            __syncthreads();
            if (tid == 0) {
                const float* sc = GATE == kGateCosine ? scs + (size_t)tq * E : logits + (size_t)tq * N;
                uint64_t used = 0;
                int chosen[kMaxTopK];
                for (int r = 0; r < k; ++r) {
                    int best = -1;
                    for (int c = 0; c < nc; ++c) {
                        if ((used >> c) & 1ull) continue;
                        if (best < 0 || ex[c] > ex[best] || (ex[c] == ex[best] && cnd[c] < cnd[best])) best = c;
                    }
                    used |= 1ull << best;
                    chosen[r] = cnd[best];
                }
                const float m = cm[tq];
                float den = cden[tq];
                if (P.norm != 0) {
                    den = 0.f;
                    for (int r = 0; r < k; ++r) den += expf(sc[chosen[r]] - m);
                }
                for (int r = 0; r < k; ++r) {
                    P.topk_idx[(size_t)tg * k + r] = chosen[r];
                    P.topk_gate[(size_t)tg * k + r] = expf(sc[chosen[r]] - m) / den;
                    fidx[tq * kMaxTopK + r] = chosen[r];
                }
            }
            __syncthreads();
        }
    }

    // ---- the dispatch's first step on the CTA's tokens (pair ranks in token order, expert histogram);
    // the last CTA to finish runs the dispatch scan
    if (P.blk_hist != nullptr) {
        for (int e = tid; e < E; e += kSelThreads) hist[e] = 0;
        __syncthreads();
        if (warp == 0)
            rank_pairs_warp([&](int i) { return fidx[(i / k) * kMaxTopK + i % k]; }, ntok * k, hist,
                            P.slot + (size_t)tok0 * k, lane);
        __syncthreads();
        for (int e = tid; e < E; e += kSelThreads) P.blk_hist[(size_t)blockIdx.x * E + e] = hist[e];
        if (P.ticket != nullptr) {
            __syncthreads();  // the block's histogram is written; thread 0 publishes it with the ticket
            if (tid == 0) {
                __threadfence();
                nq[1] = atomicAdd(P.ticket, 1);
                __threadfence();
            }
            __syncthreads();
            if (nq[1] == (int)gridDim.x - 1) {
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
