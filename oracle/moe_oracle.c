/*
 * moe_oracle.c -- plain, slow, single-threaded fp64 reference of the sparse MoE layer forward pass.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU-baseline leg use it.
 * It shares no code, header, table or constant with the CUDA library and includes nothing from it.
 *
 * Every value is read from the caller's fp32 or bf16 buffers and widened exactly to double; all
 * arithmetic is double precision, in loops, with no BLAS, threads, SIMD intrinsics or reordering
 * beyond what each function's definition states.
 *
 * The steps follow the pages in order:
 *   1. gate scores   -- "MoE sparse-compute acceleration" section 2.1 (NoisyTopKGating: clean and noise
 *                       linear maps without bias, noise scaled by softplus); "How sparse activation
 *                       improves efficiency" section 2.1 (one linear layer and a softmax); "Tutel MoE
 *                       guide", gate types top / cosine_top.  The cosine form cos(x P, e_j) / temperature is the reading
 *                       the workload definition fixes, since the pages give no formula for it.
 *   2. top-k + gates -- NoisyTopKGating: topk of the logits, softmax over the k selected; the top-1
 *                       MOELayer of "PyTorch-CUDA-v2.6 and MoE": softmax over all
 *                       experts, the max weight multiplies the output.
 *   3. dispatch      -- "How sparse activation improves efficiency" section 3.1 (group tokens by
 *                       chosen expert); "Tutel MoE guide" capacity_factor (1.2 admits 20 % above an
 *                       even share); overflow dropped.
 *   4. expert FFN    -- CANN MOELayer example: Linear(d, 4d) -> GELU -> Linear(4d, d).
 *   5. combine       -- "MoE on a single card" section 1.2: Output = sum_i g_i(x) E_i(x).
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared moe_oracle.c -lm  (oracle/__init__.py does this).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_F32 0
#define OR_BF16 1
#define OR_F64 2

#define GATE_SOFTMAX 0
#define GATE_NOISY 1
#define GATE_COSINE 2

#define NORM_ALL 0
#define NORM_TOPK 1

/* Exact widening of element i of a fp32, bf16 or fp64 buffer.  A bf16 value is the upper half of the
 * fp32 with the same sign, exponent and leading 7 mantissa bits. */
static double elem(const void *base, size_t i, int dtype)
{
    if (dtype == OR_F64) return ((const double *)base)[i];
    if (dtype == OR_BF16) {
        uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float *)base)[i];
}

/* sum_i a[i] * b[i], i = 0..n-1, accumulated left to right in double (a and b of element types adt, bdt). */
static double dot_rows(const void *a, size_t a_off, int adt, const void *b, size_t b_off, int bdt, int n)
{
    double s = 0.0;
    for (int i = 0; i < n; ++i)
        s += elem(a, a_off + (size_t)i, adt) * elem(b, b_off + (size_t)i, bdt);
    return s;
}

static double softplus(double z) { return log1p(exp(z)); }

static double gelu_erf(double z) { return 0.5 * z * (1.0 + erf(z / sqrt(2.0))); }

/* ---- step 1: selection scores s[t][e] ------------------------------------------------------------
 * SOFTMAX: s = x . W_g[e]
 * NOISY:   s = x . W_g[e] + eps[t][e] * softplus(x . W_n[e])
 * COSINE:  u = P x (u_j = x . P[j], j < p);  s = (u . emb[e]) / (max(|u|,1e-12) max(|emb[e]|,1e-12)) / temp
 */
void oracle_gate_scores(int gate_type, int T, int d, int E, int p, double temperature, int dtype,
                        const void *x, const void *w_gate, const void *w_noise, const float *eps,
                        const void *proj, const void *emb, double *scores)
{
    double *u = NULL;
    if (gate_type == GATE_COSINE)
        u = (double *)malloc(sizeof(double) * (size_t)(p > 0 ? p : 1));
    for (int t = 0; t < T; ++t) {
        size_t xo = (size_t)t * (size_t)d;
        if (gate_type == GATE_COSINE) {
            double nu2 = 0.0;
            for (int j = 0; j < p; ++j) {
                u[j] = dot_rows(x, xo, dtype, proj, (size_t)j * (size_t)d, dtype, d);
                nu2 += u[j] * u[j];
            }
            double nu = sqrt(nu2);
            if (nu < 1e-12) nu = 1e-12;
            for (int e = 0; e < E; ++e) {
                double num = 0.0, ne2 = 0.0;
                for (int j = 0; j < p; ++j) {
                    double ej = elem(emb, (size_t)e * (size_t)p + (size_t)j, dtype);
                    num += u[j] * ej;
                    ne2 += ej * ej;
                }
                double ne = sqrt(ne2);
                if (ne < 1e-12) ne = 1e-12;
                scores[(size_t)t * E + e] = num / (nu * ne) / temperature;
            }
        } else {
            for (int e = 0; e < E; ++e) {
                double s = dot_rows(x, xo, dtype, w_gate, (size_t)e * (size_t)d, dtype, d);
                if (gate_type == GATE_NOISY) {
                    double noise = dot_rows(x, xo, dtype, w_noise, (size_t)e * (size_t)d, dtype, d);
                    s += (double)eps[(size_t)t * E + e] * softplus(noise);
                }
                scores[(size_t)t * E + e] = s;
            }
        }
    }
    free(u);
}

/* ---- step 2: top-k by score, ties to the lower expert id, and the gate weights -------------------
 * k rounds of argmax over the experts not yet chosen; a later expert replaces the running best only
 * if its score is strictly greater, so equal scores keep the lower id.  With m the best score:
 *   NORM_ALL:  g_j = exp(s_j - m) / sum_{all e} exp(s_e - m)
 *   NORM_TOPK: g_j = exp(s_j - m) / sum_{chosen e} exp(s_e - m)
 */
void oracle_topk(int T, int E, int k, int norm, const double *scores, int32_t *idx, double *gate)
{
    char *taken = (char *)malloc((size_t)(E > 0 ? E : 1));
    for (int t = 0; t < T; ++t) {
        const double *s = scores + (size_t)t * E;
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || s[e] > s[best]) best = e;
            }
            taken[best] = 1;
            idx[(size_t)t * k + j] = best;
        }
        double m = s[idx[(size_t)t * k]];
        double den = 0.0;
        if (norm == NORM_ALL) {
            for (int e = 0; e < E; ++e) den += exp(s[e] - m);
        } else {
            for (int j = 0; j < k; ++j) den += exp(s[idx[(size_t)t * k + j]] - m);
        }
        for (int j = 0; j < k; ++j)
            gate[(size_t)t * k + j] = exp(s[idx[(size_t)t * k + j]] - m) / den;
    }
    free(taken);
}

/* ---- step 3: capacity ----------------------------------------------------------------------------
 * C = ceil(capacity_factor * T * k / E), the product and quotient evaluated in double, left to right;
 * an explicit capacity >= 0 overrides it. */
int oracle_capacity(int T, int E, int k, double capacity_factor, int capacity)
{
    if (capacity >= 0) return capacity;
    return (int)ceil(capacity_factor * (double)T * (double)k / (double)E);
}

/* Walk the pairs in priority order.  Each pair takes the next free position of its expert's queue; the
 * pair is kept if that position is < C, else dropped (slot -1).  count[e] is the number of pairs routed
 * to e before the limit.
 *   PRIORITY_TOKEN: token order (t = 0..T-1, then rank j = 0..k-1) -- the workloads' "capacity slots in
 *                   token order";
 *   PRIORITY_RANK:  rank order (every token's first choice, in token order, then every second choice,
 *                   ...) -- the other reading of the "Tutel MoE guide"'s capacity_factor rule, where a
 *                   token's lower-ranked choices never push out another token's first choice. */
#define PRIORITY_TOKEN 0
#define PRIORITY_RANK 1
void oracle_dispatch(int T, int E, int k, int C, int priority, const int32_t *idx, int32_t *slot,
                     int32_t *count)
{
    for (int e = 0; e < E; ++e) count[e] = 0;
    if (priority == PRIORITY_RANK) {
        for (int r = 0; r < k; ++r)
            for (int tok = 0; tok < T; ++tok) {
                const size_t i = (size_t)tok * k + r;
                const int q = count[idx[i]]++;
                slot[i] = q < C ? q : -1;
            }
        return;
    }
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            int e = idx[(size_t)t * k + j];
            int pos = count[e]++;
            slot[(size_t)t * k + j] = pos < C ? pos : -1;
        }
    }
}

/* ---- step 4: one expert on one token ------------------------------------------------------------
 * y = W2 GELU(W1 x + b1) + b2, W1 [h, d], W2 [d, h] (rows = output features).  b1 / b2 may be NULL.
 * x and the biases have element type `dtype`, the weights `wdtype` (fp64 for dequantised weights). */
void oracle_expert(int d, int h, int dtype, int wdtype, const void *x, size_t x_off, const void *w1,
                   size_t w1_off, const void *b1, size_t b1_off, const void *w2, size_t w2_off,
                   const void *b2, size_t b2_off, double *y)
{
    double *a = (double *)malloc(sizeof(double) * (size_t)h);
    for (int n = 0; n < h; ++n) {
        double z = dot_rows(x, x_off, dtype, w1, w1_off + (size_t)n * (size_t)d, wdtype, d);
        if (b1) z += elem(b1, b1_off + (size_t)n, dtype);
        a[n] = gelu_erf(z);
    }
    for (int n = 0; n < d; ++n) {
        double z = 0.0;
        for (int i = 0; i < h; ++i)
            z += a[i] * elem(w2, w2_off + (size_t)n * (size_t)h + (size_t)i, wdtype);
        if (b2) z += elem(b2, b2_off + (size_t)n, dtype);
        y[n] = z;
    }
    free(a);
}

/* ---- block-FP8 expert weights -----------------------------------------------------------------------
 * "MoE architecture: breaking the single-card compute bottleneck", section 1.3 (FP8 weights shrink the
 * model) and the Block FP8 rows of the "Tutel MoE guide" throughput table.  The pages fix no format;
 * the reading taken: each weight matrix [rows, cols] is stored as FP8 E4M3 codes plus one fp32 scale
 * per block x block tile, and the layer computes with the dequantised weight  code value * scale.
 * An E4M3 code is sign (bit 7), exponent field E (bits 6..3, bias 7) and mantissa field M (bits 2..0):
 * E > 0: (1 + M/8) * 2^(E-7);  E = 0: (M/8) * 2^-6 (subnormal);  E = 15 and M = 7 is NaN. */
static double e4m3_value(uint8_t code)
{
    const int sign = code >> 7, ex = (code >> 3) & 15, man = code & 7;
    double mag;
    if (ex == 15 && man == 7) return NAN;
    if (ex == 0)
        mag = ldexp((double)man / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)man / 8.0, ex - 7);
    return sign ? -mag : mag;
}

/* out[r][c] = e4m3(q[r][c]) * scale[r / block][c / block]; scale is [ceil(rows/block), ceil(cols/block)]. */
void oracle_dequant_block_fp8(int rows, int cols, int block, const uint8_t *q, const float *scale, double *out)
{
    const int sc = (cols + block - 1) / block;
    for (int r = 0; r < rows; ++r)
        for (int c = 0; c < cols; ++c)
            out[(size_t)r * cols + c] =
                e4m3_value(q[(size_t)r * cols + c]) * (double)scale[(size_t)(r / block) * sc + (c / block)];
}

/* ---- step 5: combine, for a list of tokens -------------------------------------------------------
 * out[i] = sum over ranks j of token tokens[i] with slot >= 0 of gate[t][j] * expert_{idx[t][j]}(x_t);
 * a token whose pairs were all dropped gets 0.  out is [ntok, d]. */
void oracle_combine_tokens(int d, int h, int k, int dtype, int wdtype, const int32_t *tokens, int ntok,
                           const void *x, const int32_t *idx, const double *gate,
                           const int32_t *slot, const void *w1, const void *b1, const void *w2,
                           const void *b2, double *out)
{
    double *y = (double *)malloc(sizeof(double) * (size_t)d);
    for (int i = 0; i < ntok; ++i) {
        int t = tokens[i];
        double *o = out + (size_t)i * (size_t)d;
        for (int n = 0; n < d; ++n) o[n] = 0.0;
        for (int j = 0; j < k; ++j) {
            if (slot[(size_t)t * k + j] < 0) continue;
            size_t e = (size_t)idx[(size_t)t * k + j];
            oracle_expert(d, h, dtype, wdtype, x, (size_t)t * (size_t)d, w1, e * (size_t)h * (size_t)d, b1,
                          e * (size_t)h, w2, e * (size_t)d * (size_t)h, b2, e * (size_t)d, y);
            double g = gate[(size_t)t * k + j];
            for (int n = 0; n < d; ++n) o[n] += g * y[n];
        }
    }
    free(y);
}

/* ---- router statistics -----------------------------------------------------------------------------
 * "MoE sparse-compute acceleration" section 4.1: the importance of expert e is the column sum of the
 * dense gate matrix, sum over tokens of the gate the token gives e (0 where e is not among its top k);
 * expert_importance_loss = 0.1 * std(importance) with torch.std's default (n - 1 in the denominator,
 * NaN for a single expert).  "MoE architecture: breaking the single-card compute bottleneck", load
 * balancing: load_balance_loss = sum_e (mean_load - load_e)^2 with load_e the same column sums.  The
 * dropped pairs are those the capacity limit refused (slot -1).  Sums in token order, then rank. */
void oracle_router_stats(int T, int E, int k, const int32_t *idx, const double *gate, const int32_t *slot,
                         double *importance, double *importance_loss, double *load_balance_loss,
                         int64_t *dropped)
{
    for (int e = 0; e < E; ++e) importance[e] = 0.0;
    int64_t drops = 0;
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            size_t i = (size_t)t * (size_t)k + (size_t)j;
            importance[idx[i]] += gate[i];
            if (slot && slot[i] < 0) ++drops;
        }
    double mean = 0.0;
    for (int e = 0; e < E; ++e) mean += importance[e];
    mean /= (double)E;
    double ss = 0.0;
    for (int e = 0; e < E; ++e) ss += (mean - importance[e]) * (mean - importance[e]);
    *load_balance_loss = ss;
    *importance_loss = E > 1 ? 0.1 * sqrt(ss / (double)(E - 1)) : NAN;
    *dropped = drops;
}

/* ---- backward of the layer ------------------------------------------------------------------------
 * "MoE sparse-compute acceleration", section 2.1: only the top-k paths carry gradients (the sparse gate
 * matrix is zero elsewhere, so nothing flows to the other experts or through the choice itself).  Given
 * dout = dL/dout [T, d] (fp64), the layer is recomputed (scores, top-k, gates, capacity dispatch) and for
 * every kept pair (t, e, gate g), with z = W1[e] x_t + b1[e], a = GELU(z), y = W2[e] a + b2[e]:
 *   dg = dout_t . y          dy = g dout_t         dW2[e] += dy a^T     db2[e] += dy
 *   da = W2[e]^T dy          dz = da * GELU'(z)    dW1[e] += dz x_t^T   db1[e] += dz     dx_t += W1[e]^T dz
 * with GELU'(z) = Phi(z) + z phi(z); a dropped pair has dg = 0.  The gates' gradient reaches the scores:
 *   NORM_TOPK (softmax over the k chosen scores): ds_{e_j} = g_j (dg_j - sum_j' g_j' dg_j'), 0 elsewhere;
 *   NORM_ALL (the chosen entries of the softmax over all E): ds_e = sum_j dg_j g_j ([e = e_j] - p_e).
 * and the scores' reaches the gate weights and x:
 *   SOFTMAX: s = x W_g^T                       dW_g[e] += ds_e x_t,  dx_t += sum_e ds_e W_g[e]
 *   NOISY:   s = x W_g^T + eps softplus(x W_n^T)  additionally dn_e = ds_e eps_e sigmoid(x . W_n[e]):
 *            dW_n[e] += dn_e x_t,  dx_t += sum_e dn_e W_n[e]
 * (softplus' = sigmoid).  The cosine gate's backward is not part of this oracle.  Outputs are written
 * (not accumulated); dw_noise may be NULL for the softmax gate, db1 / db2 are written even without biases. */
static double gelu_grad(double z)
{
    const double pi = 3.14159265358979323846;
    return 0.5 * (1.0 + erf(z * sqrt(0.5))) + z * exp(-0.5 * z * z) / sqrt(2.0 * pi);
}

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

void oracle_backward(int gate_type, int norm, int T, int d, int h, int E, int k, int C, int priority, int dtype,
                     const void *x, const void *w_gate, const void *w_noise, const float *eps, const void *w1,
                     const void *b1, const void *w2, const void *b2, const double *dout, double *dx,
                     double *dw_gate, double *dw_noise, double *dw1, double *db1, double *dw2, double *db2)
{
    double *scores = (double *)malloc(sizeof(double) * (size_t)T * E);
    int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * (size_t)T * k);
    double *gate = (double *)malloc(sizeof(double) * (size_t)T * k);
    int32_t *slot = (int32_t *)malloc(sizeof(int32_t) * (size_t)T * k);
    int32_t *count = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    double *z = (double *)malloc(sizeof(double) * (size_t)h);
    double *a = (double *)malloc(sizeof(double) * (size_t)h);
    double *da = (double *)malloc(sizeof(double) * (size_t)h);
    double *dg = (double *)malloc(sizeof(double) * (size_t)k);
    double *ds = (double *)malloc(sizeof(double) * (size_t)E);
    double *p = (double *)malloc(sizeof(double) * (size_t)E);
    oracle_gate_scores(gate_type, T, d, E, 0, 1.0, dtype, x, w_gate, w_noise, eps, NULL, NULL, scores);
    oracle_topk(T, E, k, norm, scores, idx, gate);
    oracle_dispatch(T, E, k, C, priority, idx, slot, count);
    memset(dx, 0, sizeof(double) * (size_t)T * d);
    memset(dw_gate, 0, sizeof(double) * (size_t)E * d);
    if (dw_noise) memset(dw_noise, 0, sizeof(double) * (size_t)E * d);
    memset(dw1, 0, sizeof(double) * (size_t)E * h * d);
    memset(db1, 0, sizeof(double) * (size_t)E * h);
    memset(dw2, 0, sizeof(double) * (size_t)E * d * h);
    memset(db2, 0, sizeof(double) * (size_t)E * d);
    for (int t = 0; t < T; ++t) {
        const size_t xo = (size_t)t * d;
        const double *go = dout + xo;
        double *gx = dx + xo;
        /* the experts */
        for (int j = 0; j < k; ++j) {
            const size_t i = (size_t)t * k + j;
            dg[j] = 0.0;
            if (slot[i] < 0) continue;
            const size_t e = (size_t)idx[i];
            const double g = gate[i];
            for (int n = 0; n < h; ++n) {
                z[n] = dot_rows(x, xo, dtype, w1, (e * h + n) * (size_t)d, dtype, d);
                if (b1) z[n] += elem(b1, e * h + n, dtype);
                a[n] = gelu_erf(z[n]);
                da[n] = 0.0;
            }
            for (int m = 0; m < d; ++m) {
                double y = 0.0;
                for (int n = 0; n < h; ++n) y += a[n] * elem(w2, (e * d + m) * (size_t)h + n, dtype);
                if (b2) y += elem(b2, e * d + m, dtype);
                dg[j] += go[m] * y;
                const double dy = g * go[m];
                db2[e * d + m] += dy;
                for (int n = 0; n < h; ++n) {
                    dw2[(e * d + m) * (size_t)h + n] += dy * a[n];
                    da[n] += elem(w2, (e * d + m) * (size_t)h + n, dtype) * dy;
                }
            }
            for (int n = 0; n < h; ++n) {
                const double dz = da[n] * gelu_grad(z[n]);
                db1[e * h + n] += dz;
                for (int m = 0; m < d; ++m) {
                    dw1[(e * h + n) * (size_t)d + m] += dz * elem(x, xo + m, dtype);
                    gx[m] += elem(w1, (e * h + n) * (size_t)d + m, dtype) * dz;
                }
            }
        }
        /* the gates -> the scores */
        for (int e = 0; e < E; ++e) ds[e] = 0.0;
        if (norm == NORM_TOPK) {
            double sum = 0.0;
            for (int j = 0; j < k; ++j) sum += gate[(size_t)t * k + j] * dg[j];
            for (int j = 0; j < k; ++j) ds[idx[(size_t)t * k + j]] = gate[(size_t)t * k + j] * (dg[j] - sum);
        } else {
            const double *s = scores + (size_t)t * E;
            double m = s[0], den = 0.0;
            for (int e = 1; e < E; ++e) if (s[e] > m) m = s[e];
            for (int e = 0; e < E; ++e) p[e] = exp(s[e] - m);
            for (int e = 0; e < E; ++e) den += p[e];
            for (int e = 0; e < E; ++e) p[e] /= den;
            for (int j = 0; j < k; ++j) {
                const double gj = gate[(size_t)t * k + j];
                for (int e = 0; e < E; ++e) ds[e] += dg[j] * gj * ((e == idx[(size_t)t * k + j] ? 1.0 : 0.0) - p[e]);
            }
        }
        /* the scores -> the gate weights and x */
        for (int e = 0; e < E; ++e) {
            if (ds[e] == 0.0) continue;
            for (int m = 0; m < d; ++m) {
                dw_gate[(size_t)e * d + m] += ds[e] * elem(x, xo + m, dtype);
                gx[m] += ds[e] * elem(w_gate, (size_t)e * d + m, dtype);
            }
            if (gate_type == GATE_NOISY) {
                const double nl = dot_rows(x, xo, dtype, w_noise, (size_t)e * d, dtype, d);
                const double dn = ds[e] * (double)eps[(size_t)t * E + e] * sigmoid(nl);
                for (int m = 0; m < d; ++m) {
                    dw_noise[(size_t)e * d + m] += dn * elem(x, xo + m, dtype);
                    gx[m] += dn * elem(w_noise, (size_t)e * d + m, dtype);
                }
            }
        }
    }
    free(scores); free(idx); free(gate); free(slot); free(count);
    free(z); free(a); free(da); free(dg); free(ds); free(p);
}

/* Single entries of the backward above, for layers too large for the whole of it (test support): the same
 * definitions, evaluated one output at a time from the routing of the whole layer (scores, idx, gate,
 * slot, as oracle_gate_scores / oracle_topk / oracle_dispatch give them).
 *   dx_rows[i][:]  = dx of token tok[i]: for each of its kept pairs, W1[e]^T dz with
 *                    dz = (W2[e]^T g dout_t) * GELU'(z), plus the scores' gradient through W_g (and W_n)
 *   dw1_v[i], db1_v[i] = dW1[e][n][m] and db1[e][n] for (e, n, m) = s1[3i .. 3i+2]: sums over the kept pairs
 *                    (t, e) of dz_t[n] x_t[m] and dz_t[n]
 *   dw2_v[i], db2_v[i] = dW2[e][m][n] and db2[e][m] for (e, m, n) = s2[3i .. 3i+2]: sums over the kept pairs
 *                    of g dout_t[m] GELU(z_t[n]) and g dout_t[m]
 * Pairs are visited in token order, ranks in order, as in oracle_backward. */
static void pair_hidden(int d, int h, int dtype, const void *x, size_t xo, const void *w1, const void *b1, size_t e,
                        int n, double *z_out)
{
    double z = dot_rows(x, xo, dtype, w1, (e * h + n) * (size_t)d, dtype, d);
    if (b1 != NULL) z = z + elem(b1, e * (size_t)h + n, dtype);
    *z_out = z;
}

void oracle_backward_sampled(int gate_type, int norm, int T, int d, int h, int E, int k, int dtype,
                             const void *x, const void *w_gate, const void *w_noise, const float *eps,
                             const void *w1, const void *b1, const void *w2, const void *b2, const double *dout,
                             const double *scores, const int32_t *idx, const double *gate, const int32_t *slot,
                             int nt, const int32_t *tok, double *dx_rows, int n1, const int32_t *s1, double *dw1_v,
                             double *db1_v, int n2, const int32_t *s2, double *dw2_v, double *db2_v)
{
    double *z = (double *)malloc(sizeof(double) * (size_t)h);
    double *a = (double *)malloc(sizeof(double) * (size_t)h);
    double *da = (double *)malloc(sizeof(double) * (size_t)h);
    double *dg = (double *)malloc(sizeof(double) * (size_t)k);
    double *ds = (double *)malloc(sizeof(double) * (size_t)E);
    double *p = (double *)malloc(sizeof(double) * (size_t)E);
    for (int i = 0; i < nt; ++i) {
        const int t = tok[i];
        const size_t xo = (size_t)t * d;
        const double *go = dout + xo;
        double *gx = dx_rows + (size_t)i * d;
        for (int m = 0; m < d; ++m) gx[m] = 0.0;
        for (int j = 0; j < k; ++j) {
            const size_t q = (size_t)t * k + j;
            dg[j] = 0.0;
            if (slot[q] < 0) continue;
            const size_t e = (size_t)idx[q];
            const double g = gate[q];
            for (int n = 0; n < h; ++n) {
                pair_hidden(d, h, dtype, x, xo, w1, b1, e, n, &z[n]);
                a[n] = gelu_erf(z[n]);
                da[n] = 0.0;
            }
            for (int m = 0; m < d; ++m) {
                double y = 0.0;
                for (int n = 0; n < h; ++n) y += a[n] * elem(w2, (e * d + m) * (size_t)h + n, dtype);
                if (b2) y += elem(b2, e * d + m, dtype);
                dg[j] += go[m] * y;
                const double dy = g * go[m];
                for (int n = 0; n < h; ++n) da[n] += elem(w2, (e * d + m) * (size_t)h + n, dtype) * dy;
            }
            for (int n = 0; n < h; ++n) {
                const double dzn = da[n] * gelu_grad(z[n]);
                for (int m = 0; m < d; ++m) gx[m] += elem(w1, (e * h + n) * (size_t)d + m, dtype) * dzn;
            }
        }
        for (int e = 0; e < E; ++e) ds[e] = 0.0;
        if (norm == NORM_TOPK) {
            double sum = 0.0;
            for (int j = 0; j < k; ++j) sum += gate[(size_t)t * k + j] * dg[j];
            for (int j = 0; j < k; ++j) {
                const size_t q = (size_t)t * k + j;
                ds[idx[q]] = gate[q] * (dg[j] - sum);
            }
        } else {
            const double *s = scores + (size_t)t * E;
            double mx = s[0], den = 0.0;
            for (int e = 1; e < E; ++e) if (s[e] > mx) mx = s[e];
            for (int e = 0; e < E; ++e) p[e] = exp(s[e] - mx);
            for (int e = 0; e < E; ++e) den += p[e];
            for (int e = 0; e < E; ++e) p[e] /= den;
            for (int j = 0; j < k; ++j) {
                const double gj = gate[(size_t)t * k + j];
                const int ej = idx[(size_t)t * k + j];
                for (int e = 0; e < E; ++e) ds[e] += dg[j] * gj * ((e == ej ? 1.0 : 0.0) - p[e]);
            }
        }
        for (int e = 0; e < E; ++e) {
            if (ds[e] == 0.0) continue;
            for (int m = 0; m < d; ++m) gx[m] = gx[m] + ds[e] * elem(w_gate, (size_t)e * d + m, dtype);
            if (gate_type == GATE_NOISY) {
                const double nl = dot_rows(x, xo, dtype, w_noise, (size_t)e * d, dtype, d);
                const double ept = (double)eps[(size_t)t * E + e];
                const double dn = ds[e] * ept * sigmoid(nl);
                for (int m = 0; m < d; ++m) gx[m] += dn * elem(w_noise, (size_t)e * d + m, dtype);
            }
        }
    }
    for (int i = 0; i < n1; ++i) {
        const size_t e = (size_t)s1[3 * i];
        const int n = s1[3 * i + 1], m = s1[3 * i + 2];
        double w = 0.0, b = 0.0;
        for (int t = 0; t < T; ++t)
            for (int j = 0; j < k; ++j) {
                const size_t q = (size_t)t * k + j;
                if (slot[q] < 0 || (size_t)idx[q] != e) continue;
                const size_t xo = (size_t)t * d;
                double zn;
                pair_hidden(d, h, dtype, x, xo, w1, b1, e, n, &zn);
                double dan = 0.0;
                for (int mm = 0; mm < d; ++mm)
                    dan += elem(w2, (e * d + mm) * (size_t)h + n, dtype) * (gate[q] * dout[xo + mm]);
                const double dzn = dan * gelu_grad(zn);
                w += dzn * elem(x, xo + m, dtype);
                b += dzn;
            }
        dw1_v[i] = w;
        db1_v[i] = b;
    }
    for (int i = 0; i < n2; ++i) {
        const size_t e = (size_t)s2[3 * i];
        const int m = s2[3 * i + 1], n = s2[3 * i + 2];
        double w = 0.0, b = 0.0;
        for (int t = 0; t < T; ++t)
            for (int j = 0; j < k; ++j) {
                const size_t q = (size_t)t * k + j;
                if (slot[q] < 0 || (size_t)idx[q] != e) continue;
                const size_t xo = (size_t)t * d;
                double zn;
                pair_hidden(d, h, dtype, x, xo, w1, b1, e, n, &zn);
                const double dy = gate[q] * dout[xo + m];
                w += dy * gelu_erf(zn);
                b += dy;
            }
        dw2_v[i] = w;
        db2_v[i] = b;
    }
    free(z); free(a); free(da); free(dg); free(ds); free(p);
}
