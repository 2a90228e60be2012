/*
 * moe_b300.h -- C ABI of a sparsely activated Mixture-of-Experts (MoE) layer, forward pass, on one
 * NVIDIA B300 (sm_103a).
 *
 * The layer computes  Output(x) = sum_i g_i(x) * E_i(x)  over the top-k experts chosen for each token
 * ("MoE on a single card", section 1.2, the formula for Output; "MoE sparse-compute acceleration",
 * section 2.1, NoisyTopKGating; "Tutel MoE guide", gate types top / cosine_top and capacity_factor).
 * It runs as five steps, each of which is also an entry point:
 *
 *   moe_route       gate GEMM + softmax / noisy / cosine scoring + per-token top-k and gate weights
 *   moe_dispatch    per-expert counts, capacity slots in token order, drop-on-overflow, row gather
 *   moe_expert_ffn  grouped per-expert Linear -> GELU -> Linear over the dispatched rows only
 *   moe_combine     gate-weighted sum of the expert outputs back into token order
 *   moe_forward     all of the above in one call
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Ownership.  The caller allocates and owns every buffer.  The library never allocates or frees
 *    device memory.  It keeps no state between calls except a small host-side cache of TMA tensor
 *    descriptors (keyed by pointer and shape) and the optional trace hook (moe_trace_events).
 *  - Pointers.  Tensor arguments are DEVICE pointers (cudaMalloc / torch CUDA tensors), contiguous,
 *    row-major, 16-byte aligned.  `stream` is a cudaStream_t passed as void*; NULL means the legacy
 *    default stream.
 *  - Asynchrony.  Calls enqueue work on `stream` and return; they never synchronise.  Outputs are
 *    valid once the stream has reached that point.  No call performs a host<->device copy.
 *  - Validation.  Every argument is checked on the host before anything is launched.  A failed check
 *    returns a status other than MOE_OK and launches nothing.  Nothing is thrown across the ABI.
 *  - Device-side errors.  Kernels that wait on barriers give up after a bounded number of polls and
 *    record an error word at the start of the workspace; moe_device_status() reads it.
 *  - Empty input.  T = 0 is valid: every call returns MOE_OK and launches nothing.
 *  - dtype.  x and every weight tensor share one element type (moe_config.dtype): MOE_BF16 (the tensor
 *    core path: bf16 operands, fp32 accumulation) or MOE_F32 (fp32 FMA on CUDA cores, no TF32).  The
 *    gate logits, scores and gate weights are always fp32; the layer output is always fp32.
 *  - Layouts.  Linear weights use the [out_features, in_features] layout, so both GEMM operands are
 *    contiguous along the reduction dimension:
 *        w_gate, w_noise [E, d]      proj [cos_dim, d]      expert_emb [E, cos_dim]
 *        w1 [E, h, d]   b1 [E, h]    w2 [E, d, h]   b2 [E, d]
 *    with T = tokens, d = model_dim, h = hidden_size_per_expert, E = num_experts, k = top_k.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes -------------------------------------------------------------------------- */
typedef int32_t moe_status;
#define MOE_OK                  0
#define MOE_ERR_INVALID_ARG     1 /* a pointer, size or enum is out of its documented range          */
#define MOE_ERR_UNSUPPORTED     2 /* valid in principle, outside what the library implements         */
#define MOE_ERR_WORKSPACE       3 /* workspace NULL, misaligned or smaller than moe_workspace_size() */
#define MOE_ERR_CUDA            4 /* a CUDA runtime call failed (launch, memset, descriptor encode)  */
#define MOE_ERR_DEVICE_CHECK    5 /* a kernel's own bounds check failed (see moe_device_status)      */
#define MOE_ERR_DEVICE_TIMEOUT  6 /* a kernel's bounded barrier wait ran out (see moe_device_status)  */

/* ---- enums ----------------------------------------------------------------------------------- */
/* Gate types.  SOFTMAX: s = x W_g^T (one linear layer and a softmax, "How sparse activation improves
 * efficiency", section 2.1; Tutel top.py).  NOISY: s = x W_g^T + eps * softplus(x W_n^T) ("MoE sparse-compute acceleration",
 * section 2.1, NoisyTopKGating; eps is supplied by the caller as an fp32 [T, E] tensor).  COSINE:
 * s_e = cos(x P^T, emb_e) / cos_temperature (Tutel cosine_top; the projection P and the expert
 * embeddings emb are inputs). */
#define MOE_GATE_SOFTMAX 0
#define MOE_GATE_NOISY   1
#define MOE_GATE_COSINE  2

/* Gate normalisation.  ALL: g = full softmax over all E scores, not renormalised (the top-1 layer of
 * "PyTorch-CUDA-v2.6 and MoE", which multiplies by the max softmax weight).
 * TOPK: softmax over the k selected scores (NoisyTopKGating's F.softmax(top_k_logits)). */
#define MOE_GATE_NORM_ALL  0
#define MOE_GATE_NORM_TOPK 1

#define MOE_F32  0
#define MOE_BF16 1

/* ---- configuration -------------------------------------------------------------------------- */
typedef struct moe_config {
    int32_t tokens;                 /* T >= 0                                                        */
    int32_t model_dim;              /* d, multiple of 64                                             */
    int32_t hidden_size_per_expert; /* h, multiple of 64                                             */
    int32_t num_experts;            /* E, 1..1024 (1..512 for the noisy gate)                        */
    int32_t top_k;                  /* k, 1..min(E, 16)                                              */
    int32_t capacity;               /* < 0: ceil(capacity_factor * T * k / E) evaluated in double,
                                       left to right; >= 0: that capacity (T makes the layer dropless) */
    double  capacity_factor;        /* > 0, used when capacity < 0                                   */
    int32_t gate_type;              /* MOE_GATE_*                                                    */
    int32_t gate_norm;              /* MOE_GATE_NORM_*                                               */
    int32_t cos_dim;                /* cosine gate: projection width p, multiple of 8, 8..1024       */
    int32_t dtype;                  /* MOE_F32 or MOE_BF16                                           */
    double  cos_temperature;        /* cosine gate: scores are divided by this (> 0)                 */
    int32_t flags;                  /* MOE_FLAG_* bits, 0 for the default path                       */
    int32_t reserved;               /* must be 0                                                     */
} moe_config;

/* flags: MOE_FLAG_SIMT_FFN runs the expert FFN of a bf16 layer on CUDA cores instead of the tcgen05
 * tensor-core kernel (a slow cross-check path); MOE_FLAG_UNFUSED_COMBINE makes moe_forward write
 * per-row expert outputs and combine them in a separate gather pass even when k <= 2. */
#define MOE_FLAG_SIMT_FFN         1
#define MOE_FLAG_UNFUSED_COMBINE  2
/* The bf16 expert GEMMs run either on single SMs (128 x 256 tiles) or on pairs of SMs (256 x 256 tiles,
 * tcgen05 cta_group::2); by default pairs are used when T * k / E >= 2048 or when d <= 1024 and
 * T * k / E >= 1024, and for the second (down) projection alone when 512 <= d <= 1024 and
 * T * k / E >= 512.  These flags force one. */
#define MOE_FLAG_FFN_ONE_SM       4
#define MOE_FLAG_FFN_SM_PAIR      8
/* Capacity priority.  By default slots are handed out in token order (token t's pairs before token
 * t + 1's; the workloads' "capacity slots in token order").  MOE_FLAG_RANK_MAJOR hands them out in rank
 * order instead: every token's first choice, in token order, then every token's second choice, ... --
 * the other reading of the "Tutel MoE guide"'s capacity_factor rule, under which a token's lower-ranked
 * choices never take a slot from another token's first choice.  It changes which pairs overflow, not
 * how a kept pair is computed.  Applies to moe_forward, moe_dispatch and moe_dispatch_static_scratch. */
#define MOE_FLAG_RANK_MAJOR      16
/* Router statistics fused into the forward: with MOE_FLAG_ROUTER_STATS, moe_forward / moe_forward_fp8
 * also compute what moe_router_stats computes (expert importance, the importance and load-balance losses,
 * the dropped pairs) inside their dispatch kernel -- no extra kernel launch -- and keep them in the
 * workspace until the next call; moe_router_stats_result() copies them out. */
#define MOE_FLAG_ROUTER_STATS    32

/* ---- sizes ------------------------------------------------------------------------------------ */
/* Per-expert capacity C the dispatch step enforces, or -1 if the config is invalid. */
MOE_API int32_t moe_capacity(const moe_config* cfg);

/* Upper bound on the number of dispatched rows: each expert's kept rows are padded to a multiple of
 * 128, so rows <= min(T*k + 127*E, E*roundup(C,128)).  x_dispatched / row_token / row_gate /
 * y_dispatched passed to moe_dispatch / moe_expert_ffn / moe_combine need this many rows.
 * Returns -1 if the config is invalid. */
MOE_API int64_t moe_dispatch_rows(const moe_config* cfg);

/* Bytes of device workspace that every entry point below accepts (one size for all of them).
 * Returns 0 if the config is invalid.  The workspace must be 256-byte aligned (cudaMalloc memory is);
 * it needs no initialisation and may be reused by consecutive calls on one stream; calls running
 * concurrently need separate workspaces. */
MOE_API size_t moe_workspace_size(const moe_config* cfg);

/* ---- step 1+2: routing ------------------------------------------------------------------------ */
/* Gate logits, scores, per-token top-k and gate weights.
 *   x          [T, d] dtype          w_gate [E, d] dtype (all gate types except COSINE)
 *   w_noise    [E, d] dtype          NOISY only, else NULL
 *   noise_eps  [T, E] fp32           NOISY only, else NULL (the standard-normal draws)
 *   proj       [cos_dim, d] dtype    COSINE only, else NULL
 *   expert_emb [E, cos_dim] dtype    COSINE only, else NULL
 * Outputs:
 *   topk_idx   [T, k] int32          expert ids in rank order, best first; ties go to the lower id
 *   topk_gate  [T, k] fp32           gate weight of each chosen expert (see MOE_GATE_NORM_*)
 * Selection is made on the scores (before the softmax).  Scores are first computed in fp32 (for
 * MOE_BF16 the logits come from the tensor cores, see moe_gate_logits; for MOE_F32 from CUDA-core FMA
 * with compensated sums), each with an error bound; when two scores of a token are closer than twice
 * that bound, the contenders are recomputed with a doubled-precision (float-float) dot product, so the
 * chosen set and its order equal those of exact arithmetic except for differences below about 1e-12 of
 * the score scale.  `workspace` (moe_workspace_size bytes) holds the partial logits. */
MOE_API moe_status moe_route(const moe_config* cfg, const void* x, const void* w_gate, const void* w_noise,
                     const float* noise_eps, const void* proj, const void* expert_emb,
                     int32_t* topk_idx, float* topk_gate, void* workspace, size_t workspace_bytes,
                     void* stream);

/* ---- step 1 alone: gate logits ---------------------------------------------------------------- */
/* The gate GEMM of a MOE_BF16 layer on the tensor cores (tcgen05: exact bf16 products, fp32
 * accumulation within each 128-wide chunk of d, chunks added with compensated sums on the CUDA cores):
 *   SOFTMAX  logits [T, E]      = x W_g^T     (the single linear layer before the softmax, "How sparse
 *                                              activation improves efficiency", section 2.1)
 *   NOISY    logits [T, 2E]     = [x W_g^T, x W_n^T]  (clean and noise logits of NoisyTopKGating,
 *                                              "MoE sparse-compute acceleration", section 2.1)
 *   COSINE   logits [T, cos_dim] = x P^T      (the projection of Tutel's cosine_top)
 * fp32, row-major, overwritten.  Error: |logit - exact| <= 64 * 2^-23 * sum_i |x_i w_i|, the bound
 * moe_route assumes for this GEMM (44.5 * 2^-23 from the measured rounding of the tensor cores and the
 * compensated sums, with a margin).  noise_eps and expert_emb are not used.  MOE_F32 layers return MOE_ERR_UNSUPPORTED (their logits are computed inside
 * moe_route's CUDA-core kernel). */
MOE_API moe_status moe_gate_logits(const moe_config* cfg, const void* x, const void* w_gate, const void* w_noise,
                           const void* proj, float* logits, void* workspace, size_t workspace_bytes,
                           void* stream);

/* ---- step 3: capacity-limited dispatch -------------------------------------------------------- */
/* Groups the (token, expert) pairs by expert, ahead of one batched matmul per group ("How sparse
 * activation improves efficiency", section 3.1), under a per-expert capacity C (capacity_factor of the
 * "Tutel MoE guide" and of CANN's MOELayer in "MoE sparse-compute acceleration", section 3.2).  Slots
 * are handed out in token order (for one expert, token t precedes token t+1; a token never picks an
 * expert twice), or in rank order with MOE_FLAG_RANK_MAJOR; a pair whose slot is >= C is dropped.
 * Outputs:
 *   slot          [T, k] int32   slot of each pair in its expert's queue, -1 if dropped
 *   expert_count  [E]    int32   pairs routed to each expert before the capacity limit
 *   expert_offset [E+1]  int32   first dispatched row of each expert; expert e owns rows
 *                                [off[e], off[e+1]), of which the first min(count[e], C) are real and
 *                                the rest (up to a multiple of 128) are padding
 *   row_token     [rows] int32   token of each dispatched row, -1 for padding rows
 *   row_gate      [rows] fp32    gate weight of each dispatched row, 0 for padding rows
 *   x_dispatched  [rows, d]      copy of x[row_token[r]] for every real row (padding rows untouched)
 * rows = moe_dispatch_rows(cfg).  Deterministic: no result depends on thread scheduling. */
MOE_API moe_status moe_dispatch(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                        const float* topk_gate, int32_t* slot, int32_t* expert_count,
                        int32_t* expert_offset, int32_t* row_token, float* row_gate,
                        void* x_dispatched, void* workspace, size_t workspace_bytes, void* stream);

/* ---- step 3 without a caller workspace ----------------------------------------------------------- */
/* The pages have no counterpart to this entry point; it exists for callers that cannot allocate device
 * memory: code running inside another framework's memory pool or a plugin host that hands out only the
 * tensors it owns, and programs that must not allocate after start-up.  They still pass every input and
 * output, but have no way to provide moe_dispatch's workspace.
 *
 * Same arguments, results and ordering guarantees as moe_dispatch, without `workspace` and
 * `workspace_bytes`.  The scratch moe_dispatch keeps in the workspace (an error word and the per-block
 * expert histogram of ceil(T/32) x E ints) lives instead in one fixed device array inside the library,
 * 256 + 4 * MOE_DISPATCH_STATIC_MAX_HIST bytes (1 MiB), which every GPU that loads the library holds
 * until the process exits.  The call allocates nothing (no cudaMalloc, no allocator of any library).
 *  - Limit.  Configs with ceil(T/32) * E > MOE_DISPATCH_STATIC_MAX_HIST return MOE_ERR_UNSUPPORTED and
 *    launch nothing (e.g. T = 16384 allows E <= 511; T = 65536 allows E <= 127).  With
 *    MOE_FLAG_RANK_MAJOR the histogram has ceil(T*k/32) rows instead of ceil(T/32).
 *  - Set-up.  The first call on each device looks up the array's device address (cudaGetSymbolAddress)
 *    with that device current; make that first call before any stream capture.  The address is kept
 *    per device and context: after a device reset (cudaDeviceReset) the next call looks it up again,
 *    and should likewise come before any stream capture.
 *  - Config errors.  A config moe_dispatch rejects is rejected with the same status.
 *  - Sharing.  Every call on a device uses the same array, which keeps the last call's contents (the
 *    call clears what must start at zero).  Calls whose kernels overlap on the GPU (other streams, other
 *    host threads) race on it and give wrong results: serialise them, e.g. on one stream.
 *  - Errors.  Host-side checks return a status as moe_dispatch does.  Expert ids outside [0, E) in
 *    topk_idx are treated as dropped (slot -1, not counted); the device error word of this variant is not
 *    readable by the caller (moe_device_status needs a workspace). */
#define MOE_DISPATCH_STATIC_MAX_HIST 262080
MOE_API moe_status moe_dispatch_static_scratch(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                                       const float* topk_gate, int32_t* slot, int32_t* expert_count,
                                       int32_t* expert_offset, int32_t* row_token, float* row_gate,
                                       void* x_dispatched, void* stream);

/* ---- steps 4+5: grouped expert FFN ------------------------------------------------------------ */
/* For every real dispatched row r of expert e:  y_r = W2[e] GELU(W1[e] x_r + b1[e]) + b2[e], with
 * GELU(z) = z/2 (1 + erf(z / sqrt 2)) (the expert of CANN's MOELayer example: Linear(d, 4d), GELU,
 * Linear(4d, d); Tutel's 'ffn' expert type).  b1 / b2 may be NULL (no bias).
 *   y_dispatched != NULL: y_dispatched [rows, d] fp32 receives y_r for each real row (padding rows
 *                         are left untouched); `out` is ignored and may be NULL.
 *   y_dispatched == NULL: the combine is fused into the second GEMM: out [T, d] fp32 is overwritten
 *                         with sum_r row_gate[r] * y_r over the real rows of each token (0 for a
 *                         token with none).  With top_k <= 2 the result is bitwise deterministic;
 *                         with top_k > 2 the order of the fp32 additions may vary between runs.
 * The hidden activations (bf16 for MOE_BF16, fp32 for MOE_F32) live in the workspace. */
MOE_API moe_status moe_expert_ffn(const moe_config* cfg, const void* x_dispatched,
                          const int32_t* expert_offset, const int32_t* row_token,
                          const float* row_gate, const void* w1, const void* b1, const void* w2,
                          const void* b2, float* y_dispatched, float* out, void* workspace,
                          size_t workspace_bytes, void* stream);

/* ---- step 5 (unfused): combine ----------------------------------------------------------------- */
/* out[t] = sum over j < k with slot[t,j] >= 0 of topk_gate[t,j] * y_dispatched[off[e] + slot[t,j]],
 * e = topk_idx[t,j], summed in rank order j = 0..k-1 (deterministic); 0 for a token whose pairs were
 * all dropped (Output = sum_i g_i(x) E_i(x), "MoE on a single card", section 1.2).  out [T, d] fp32 is
 * overwritten. */
MOE_API moe_status moe_combine(const moe_config* cfg, const float* y_dispatched, const int32_t* slot,
                       const int32_t* expert_offset, const int32_t* topk_idx,
                       const float* topk_gate, float* out, void* stream);

/* ---- router statistics ------------------------------------------------------------------------- */
/* Statistics of one routing, for monitoring expert load and for the auxiliary losses the pages add:
 *   importance[e]   = sum over tokens of the gate the token gives expert e (0 where e is not among
 *                     its top k): the column sums of the dense gate matrix ("MoE sparse-compute
 *                     acceleration", section 4.1); utilisation = importance / T
 *   losses[0]       = expert_importance_loss = 0.1 * std(importance), std with E - 1 in the
 *                     denominator (section 4.1; NaN when E = 1)
 *   losses[1]       = load_balance_loss = sum_e (mean_e importance - importance[e])^2 ("MoE
 *                     architecture: breaking the single-card compute bottleneck", load balancing)
 *   *dropped        = pairs the capacity limit refused (slot < 0), if slot and dropped are not NULL
 * topk_idx [T, k] int32 and topk_gate [T, k] fp32 as moe_route writes them (gates in [0, 1]); slot
 * [T, k] as moe_dispatch / moe_forward write it, or NULL.  importance [E] fp32 and losses [2] fp32 are
 * device buffers, dropped a device int64 or NULL.  Each gate is added as a multiple of 2^-32 (rounded
 * to nearest) in 64-bit integers, so the sums are exact and independent of the order the GPU adds them
 * in: importance[e] is within (pairs of e) * 2^-33 of the exact sum before its rounding to fp32, and
 * the losses are computed in fp64 from those sums.  An expert id outside [0, E) or a gate outside
 * [0, 1] records MOE_ERR_DEVICE_CHECK and is skipped.  Uses the workspace (moe_workspace_size). */
MOE_API moe_status moe_router_stats(const moe_config* cfg, const int32_t* topk_idx, const float* topk_gate,
                            const int32_t* slot, float* importance, float* losses, int64_t* dropped,
                            void* workspace, size_t workspace_bytes, void* stream);

/* The statistics of the last moe_forward / moe_forward_fp8 made with MOE_FLAG_ROUTER_STATS on this
 * workspace (same definitions and exact fixed-point sums as moe_router_stats): enqueues device-to-device
 * copies on `stream` into importance [E] fp32, losses [2] fp32 (importance loss, load-balance loss) and
 * dropped (int64); any of the three may be NULL.  MOE_ERR_INVALID_ARG if cfg lacks the flag. */
MOE_API moe_status moe_router_stats_result(const moe_config* cfg, const void* workspace, size_t workspace_bytes,
                                   float* importance, float* losses, int64_t* dropped, void* stream);

/* ---- whole layer ------------------------------------------------------------------------------ */
/* moe_route -> moe_dispatch -> moe_expert_ffn (+ fused or separate combine) on `stream`, with every
 * intermediate in the workspace.  out [T, d] fp32 is overwritten.  expert_count (may be NULL)
 * receives the per-expert pre-capacity counts.  The fused combine is used when top_k <= 2 and the
 * gather combine otherwise, so the output is bitwise deterministic for every k. */
MOE_API moe_status moe_forward(const moe_config* cfg, const void* x, const void* w_gate,
                       const void* w_noise, const float* noise_eps, const void* proj,
                       const void* expert_emb, const void* w1, const void* b1, const void* w2,
                       const void* b2, float* out, int32_t* expert_count, void* workspace,
                       size_t workspace_bytes, void* stream);

/* ---- backward --------------------------------------------------------------------------------- */
/* Gradients of the layer for a loss L with dL/dout = dout [T, d] fp32 ("MoE sparse-compute acceleration",
 * section 2.1: only the top-k paths carry gradients -- the sparse gate matrix is zero elsewhere, so nothing
 * flows to unchosen experts, through the choice itself, or through dropped pairs):
 *   dx [T, d], dw_gate [E, d], dw_noise [E, d] (noisy gate; may be NULL for softmax), dw1 [E, h, d],
 *   dw2 [E, d, h], db1 [E, h] and db2 [E, d] (each may be NULL), all fp32 and overwritten.
 * For every kept pair (t, e, gate g) with z = W1[e] x_t + b1[e], y = W2[e] GELU(z) + b2[e]:
 *   dg = dout_t . y;  dW2[e] += g dout_t GELU(z)^T;  dz = (W2[e]^T g dout_t) * GELU'(z);  dW1[e] += dz x_t^T;
 *   dx_t += W1[e]^T dz;  and through the gates (softmax over the k chosen scores, or over all E for
 *   MOE_GATE_NORM_ALL) to the scores, W_g (and for the noisy gate, through eps softplus(x W_n^T), to W_n)
 *   and x.  The call recomputes the forward (routing, dispatch, the expert FFN keeping Z = W1 x + b1 in
 *   bf16) and runs the backward GEMMs on the tensor cores: the data gradients grouped by expert over the
 *   dispatched rows (reading W1 and W2 as stored, MN-major), the weight gradients contracting over each
 *   expert's rows.  Intermediate gradients (dY = g dout per row, dZ, the scores' gradient) are rounded to
 *   bf16 for the GEMMs; dx is accumulated with fp32 atomics (not bitwise reproducible).
 * Supported: bf16 layers with the softmax or noisy gate (else MOE_ERR_UNSUPPORTED, also for
 * MOE_FLAG_SIMT_FFN).  workspace: moe_backward_workspace_size(cfg) bytes (it includes the forward's). */
MOE_API size_t moe_backward_workspace_size(const moe_config* cfg);
MOE_API moe_status moe_backward(const moe_config* cfg, const void* x, const void* w_gate, const void* w_noise,
                        const float* noise_eps, const void* w1, const void* b1, const void* w2, const void* b2,
                        const float* dout, float* dx, float* dw_gate, float* dw_noise, float* dw1, float* db1,
                        float* dw2, float* db2, void* workspace, size_t workspace_bytes, void* stream);

/* ---- block-FP8 expert weights --------------------------------------------------------------------- */
/* The same FFN step and whole layer with the expert weights stored as block FP8 ("MoE architecture:
 * breaking the single-card compute bottleneck", section 1.3: FP8 weights shrink the model; the Block FP8
 * rows of the "Tutel MoE guide" throughput table).  Reading taken (the pages fix no format):
 *   w1_q [E, h, d], w2_q [E, d, h]   uint8 FP8 E4M3 codes (sign, 4 exponent bits with bias 7, 3 mantissa
 *                                     bits; exponent field 0 is subnormal; 0x7F / 0xFF are NaN)
 *   w1_scale [E, h/128, d/128], w2_scale [E, d/128, h/128]  fp32, one scale per 128 x 128 block
 * and the layer computes with the dequantised weights  code value * scale  (everything else as in
 * moe_expert_ffn / moe_forward: bf16 activations, fp32 accumulation).  The kernel widens the codes to bf16
 * in shared memory (exact when the scales are powers of two, else the product is rounded to bf16) and
 * streams one byte per weight from HBM.  Requires dtype MOE_BF16, d and h multiples of 128 and no
 * MOE_FLAG_SIMT_FFN (else MOE_ERR_UNSUPPORTED); scales must be 4-byte aligned; the expert GEMMs run on
 * single SMs whatever MOE_FLAG_FFN_SM_PAIR says.  Workspace, outputs and errors as the bf16 calls. */
MOE_API moe_status moe_expert_ffn_fp8(const moe_config* cfg, const void* x_dispatched,
                              const int32_t* expert_offset, const int32_t* row_token, const float* row_gate,
                              const uint8_t* w1_q, const float* w1_scale, const void* b1,
                              const uint8_t* w2_q, const float* w2_scale, const void* b2,
                              float* y_dispatched, float* out, void* workspace, size_t workspace_bytes,
                              void* stream);
MOE_API moe_status moe_forward_fp8(const moe_config* cfg, const void* x, const void* w_gate,
                           const void* w_noise, const float* noise_eps, const void* proj,
                           const void* expert_emb, const uint8_t* w1_q, const float* w1_scale,
                           const void* b1, const uint8_t* w2_q, const float* w2_scale, const void* b2,
                           float* out, int32_t* expert_count, void* workspace, size_t workspace_bytes,
                           void* stream);

/* ---- diagnostics ------------------------------------------------------------------------------ */
/* Synchronises `stream`, reads and clears the error word at the start of `workspace` and returns
 * MOE_OK, MOE_ERR_DEVICE_CHECK or MOE_ERR_DEVICE_TIMEOUT.  If `info` is not NULL it receives a code
 * saying which kernel recorded the error (0 if none). */
MOE_API moe_status moe_device_status(void* workspace, size_t workspace_bytes, int32_t* info, void* stream);

/* Profiling hook.  With events != NULL (an array of `capacity` cudaEvent_t, each passed as void*),
 * the library records events[0] on the launch stream before the first kernel it launches after this
 * call, and events[i] right after the i-th such kernel, until `capacity` events are used; n kernels
 * thus use n + 1 events and kernel i ran between events[i] and events[i+1].  moe_trace_count()
 * returns how many events the current (or, once turned off, the last) trace recorded.  events == NULL
 * turns the hook off.  While `stream` is being captured the events are recorded with
 * cudaEventRecordExternal, so the graph gets event-record nodes and every replay of it times its
 * kernels with no host gaps between them.  Not thread-safe; meant for benchmarks.
 * Every compute entry point also opens an NVTX range named after itself for the length of the call
 * (a no-op unless a profiler is attached). */
MOE_API void    moe_trace_events(void** events, int32_t capacity);
MOE_API int32_t moe_trace_count(void);

/* Number of kernels moe_forward launches for this config (for launch accounting), -1 if invalid. */
MOE_API int32_t moe_forward_launches(const moe_config* cfg);

/* Human-readable name of a status code (static storage). */
MOE_API const char* moe_status_string(moe_status status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
