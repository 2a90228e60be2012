// bwd.cu -- the data-movement kernels of the layer's backward pass (the GEMMs are in ffn_tc.cu).
//
// Only the top-k paths carry gradients ("MoE sparse-compute acceleration", section 2.1: the sparse gate
// matrix is zero elsewhere).  With the forward recomputed (routing, dispatch, Z = X_d W1^T + b1,
// H = GELU(Z), y = H W2^T + b2 per dispatched row), the backward needs:
//   dy_kernel         dY[r] = gate_r dout[token_r] (bf16), zero for padding rows
//   gate_grad_kernel  per token: dg_j = dout_t . y_r for its kept pairs, the scores' gradient through the
//                     softmax (over the k chosen scores, or over all E), and for the noisy gate the noise
//                     logits' gradient ds eps sigmoid(x W_n^T); a bf16 row [ds | dn | 0] per token
//   zero_pad_rows     zeros in the padding rows of X_d, H and dZ, which the weight-gradient GEMMs contract
//                     over together with the real rows
//   segment_colsum    bias gradients: column sums of dY / dZ over each expert's row segment (fp32; their
//                     padding rows are zero)
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

// Padding rows (row_token < 0) below *row_limit of up to three bf16 buffers [rows, w_i] (w_i a multiple of 8,
// or a null buffer) become zero: a warp per row, 16-byte stores; real rows are not touched.
__global__ void __launch_bounds__(256) zero_pad_rows_kernel(bf16_t* __restrict__ p0, int w0, bf16_t* __restrict__ p1,
                                                           int w1, bf16_t* __restrict__ p2, int w2, int rows,
                                                           const int* __restrict__ row_token,
                                                           const int* __restrict__ row_limit) {
    pdl_wait();
    pdl_trigger();
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (r >= rows || r >= *row_limit || row_token[r] >= 0) return;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    bf16_t* const ps[3] = {p0, p1, p2};
    const int ws[3] = {w0, w1, w2};
#pragma unroll
    for (int b = 0; b < 3; ++b)
        if (ps[b] != nullptr)
            for (int c = lane * 8; c < ws[b]; c += 256) *reinterpret_cast<uint4*>(ps[b] + (size_t)r * ws[b] + c) = z;
}

// dY[r][:] = gate_r * dout[token_r][:] in bf16 (a warp per row, 8 columns per lane per step); rows of
// padding and rows from *row_limit on (past the last expert's segment: row_token never written) get 0
__global__ void __launch_bounds__(256) dy_kernel(const float* __restrict__ dout, const int* __restrict__ row_token,
                                                const float* __restrict__ row_gate, int rows, int d,
                                                const int* __restrict__ row_limit, bf16_t* __restrict__ dY) {
    pdl_wait();
    pdl_trigger();
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (r >= rows) return;
    const int t = r < *row_limit ? row_token[r] : -1;
    const float g = t >= 0 ? row_gate[r] : 0.f;
    uint4* dst = reinterpret_cast<uint4*>(dY + (size_t)r * d);
    for (int c = lane * 8; c < d; c += 256) {
        float v[8];
        if (t >= 0) {
            load8(dout + (size_t)t * d + c, v);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = 0.f;
        }
        dst[c / 8] = make_uint4(pack_bf16x2(g * v[0], g * v[1]), pack_bf16x2(g * v[2], g * v[3]),
                                pack_bf16x2(g * v[4], g * v[5]), pack_bf16x2(g * v[6], g * v[7]));
    }
}

// One warp per token.  dg_j = dout_t . y_r for each kept pair (slot >= 0, row r = offset[e] + slot), 0 for a
// dropped pair; then ds over the experts:
//   norm topk: ds_{e_j} = g_j (dg_j - sum_j' g_j' dg_j');  norm all: ds_e = sum_j dg_j g_j ([e = e_j] - p_e)
// with p the softmax of the token's scores over all E (scores from the logits: clean, or clean +
// eps softplus(noise) for the noisy gate); the noisy gate adds dn_e = ds_e eps_e sigmoid(noise_e).  The
// token's row of dS [Tp, Np] bf16 gets [ds (E) | dn (E, noisy) | 0].
__global__ void __launch_bounds__(256) gate_grad_kernel(const float* __restrict__ dout, const float* __restrict__ y,
                                                       const int* __restrict__ topk_idx,
                                                       const float* __restrict__ topk_gate,
                                                       const int* __restrict__ slot, const int* __restrict__ offset,
                                                       const float* __restrict__ logits, const float* __restrict__ eps,
                                                       int T, int Tp, int d, int E, int k, int noisy, int norm_all,
                                                       int Np, bf16_t* __restrict__ dS) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (t >= Tp) return;
    bf16_t* row = dS + (size_t)t * Np;
    if (t >= T) {
        for (int c = lane; c < Np; c += 32) row[c] = 0;
        return;
    }
    float dg[kMaxTopK], g[kMaxTopK];
    int ids[kMaxTopK];
    float sum = 0.f;
    for (int j = 0; j < k; ++j) {
        const int e = topk_idx[(size_t)t * k + j];
        const int sl = slot[(size_t)t * k + j];
        ids[j] = e;
        g[j] = topk_gate[(size_t)t * k + j];
        float acc = 0.f;
        if (sl >= 0) {
            const float* yr = y + (size_t)(offset[e] + sl) * d;
            const float* go = dout + (size_t)t * d;
            for (int c = lane * 4; c < d; c += 128) {
                const float4 a = *reinterpret_cast<const float4*>(go + c);
                const float4 b = *reinterpret_cast<const float4*>(yr + c);
                acc = fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, fmaf(a.w, b.w, acc))));
            }
            acc = warp_sum(acc);
        }
        dg[j] = acc;
        sum += g[j] * acc;
    }
    const float* lg = logits + (size_t)t * (noisy ? 2 * E : E);
    auto score = [&](int e) {
        float s = lg[e];
        if (noisy) {
            const float n = lg[E + e];
            s += eps[(size_t)t * E + e] * (n > 20.f ? n : log1pf(__expf(n)));
        }
        return s;
    };
    float m = -INFINITY, den = 0.f;
    if (norm_all) {
        for (int e = lane; e < E; e += 32) m = fmaxf(m, score(e));
        m = warp_max(m);
        for (int e = lane; e < E; e += 32) den += __expf(score(e) - m);
        den = warp_sum(den);
    }
    for (int e = lane; e < E; e += 32) {
        float ds = 0.f;
        if (norm_all) {
            const float p = __expf(score(e) - m) / den;
            for (int j = 0; j < k; ++j) ds += dg[j] * g[j] * ((ids[j] == e ? 1.f : 0.f) - p);
        } else {
            for (int j = 0; j < k; ++j)
                if (ids[j] == e) ds = g[j] * (dg[j] - sum);
        }
        row[e] = (bf16_t)(pack_bf16x2(ds, 0.f) & 0xffffu);
        if (noisy) {
            const float n = lg[E + e];
            const float sig = 1.f / (1.f + __expf(-n));
            const float dn = ds * eps[(size_t)t * E + e] * sig;
            row[E + e] = (bf16_t)(pack_bf16x2(dn, 0.f) & 0xffffu);
        }
    }
    for (int c = (noisy ? 2 * E : E) + lane; c < Np; c += 32) row[c] = 0;
}

// db[e][c] = sum over the rows r in [offset[e], offset[e+1]) of src[r][c] (fp32; the padding rows of src hold
// zeros).  A CTA per (256 columns, expert): warp w sums the rows w, w + 8, ... of the segment, eight columns a
// lane (16-byte loads, two rows in flight), then the eight warps' partials are added in warp order
// (deterministic).
__global__ void __launch_bounds__(256) segment_colsum_kernel(const bf16_t* __restrict__ src, const int* __restrict__ offset,
                                                            int C, float* __restrict__ db) {
    __shared__ float part[8][256];
    pdl_wait();
    pdl_trigger();
    const int e = blockIdx.y, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c0 = blockIdx.x * 256 + lane * 8;
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
    if (c0 < C) {
        const int r1 = offset[e + 1];
        int r = offset[e] + w;
        for (; r + 8 < r1; r += 16) {
            float a[8], b[8];
            load8(src + (size_t)r * C + c0, a);
            load8(src + (size_t)(r + 8) * C + c0, b);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] += a[j] + b[j];
        }
        if (r < r1) {
            float a[8];
            load8(src + (size_t)r * C + c0, a);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] += a[j];
        }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) part[w][lane * 8 + j] = acc[j];
    __syncthreads();
    const int c = blockIdx.x * 256 + threadIdx.x;
    if (c < C) {
        float t = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) t += part[q][threadIdx.x];
        db[(size_t)e * C + c] = t;
    }
}

// WcatT [d][Np] = [W_g ; W_n ; 0]^T (a thread per element; the gate weights are small)
__global__ void gate_weights_t_kernel(const bf16_t* __restrict__ wg, const bf16_t* __restrict__ wn, int E, int d,
                                      int Np, bf16_t* __restrict__ out) {
    pdl_wait();
    pdl_trigger();
    const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long)d * Np) return;
    const int m = (int)(i / Np), n = (int)(i % Np);
    bf16_t v = 0;
    if (n < E) v = wg[(size_t)n * d + m];
    else if (wn != nullptr && n < 2 * E) v = wn[(size_t)(n - E) * d + m];
    out[i] = v;
}

// row_token of the gate-path GEMM: identity for t < T, -1 for the padding up to Tp; offset {0, Tp}
__global__ void iota_rows_kernel(int* __restrict__ rows, int T, int Tp, int* __restrict__ off2) {
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < Tp) rows[i] = i < T ? i : -1;
    if (i == 0) { off2[0] = 0; off2[1] = Tp; }
}

}  // namespace

cudaError_t launch_zero_pad_rows(void* p0, int w0, void* p1, int w1, void* p2, int w2, int rows,
                                 const int* row_token, const int* row_limit, cudaStream_t s) {
    if (rows <= 0) return cudaSuccess;
    return launch_pdl(zero_pad_rows_kernel, dim3((rows + 7) / 8), dim3(256), 0, s, static_cast<bf16_t*>(p0), w0,
                      static_cast<bf16_t*>(p1), w1, static_cast<bf16_t*>(p2), w2, rows, row_token, row_limit);
}

cudaError_t launch_bwd_dy(const float* dout, const int* row_token, const float* row_gate, int rows, int d,
                          const int* row_limit, void* dY, cudaStream_t s) {
    if (rows <= 0) return cudaSuccess;
    return launch_pdl(dy_kernel, dim3((rows + 7) / 8), dim3(256), 0, s, dout, row_token, row_gate, rows, d, row_limit,
                      static_cast<bf16_t*>(dY));
}

cudaError_t launch_bwd_gate(const float* dout, const float* y, const int* topk_idx, const float* topk_gate,
                            const int* slot, const int* offset, const float* logits, const float* eps, int T, int Tp,
                            int d, int E, int k, int noisy, int norm_all, int Np, void* dS, cudaStream_t s) {
    if (Tp <= 0) return cudaSuccess;
    return launch_pdl(gate_grad_kernel, dim3((Tp + 7) / 8), dim3(256), 0, s, dout, y, topk_idx, topk_gate, slot, offset,
                      logits, eps, T, Tp, d, E, k, noisy, norm_all, Np, static_cast<bf16_t*>(dS));
}

cudaError_t launch_segment_colsum(const void* src, const int* offset, int E, int C, float* db, cudaStream_t s) {
    if (E <= 0 || C <= 0) return cudaSuccess;
    if (C % 8) return cudaErrorInvalidValue;
    return launch_pdl(segment_colsum_kernel, dim3((C + 255) / 256, E), dim3(256), 0, s, static_cast<const bf16_t*>(src),
                      offset, C, db);
}

cudaError_t launch_gate_weights_t(const void* wg, const void* wn, int E, int d, int Np, void* out, cudaStream_t s) {
    const long n = (long)d * Np;
    return launch_pdl(gate_weights_t_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s,
                      static_cast<const bf16_t*>(wg), static_cast<const bf16_t*>(wn), E, d, Np, static_cast<bf16_t*>(out));
}

cudaError_t launch_iota_rows(int* rows, int T, int Tp, int* off2, cudaStream_t s) {
    return launch_pdl(iota_rows_kernel, dim3((Tp + 255) / 256), dim3(256), 0, s, rows, T, Tp, off2);
}

}  // namespace moe
