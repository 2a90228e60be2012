// dispatch_noalloc.cu -- moe_dispatch for callers that cannot allocate device memory.
//
// moe_dispatch needs a little device scratch besides its outputs: an error word and the per-block
// expert histogram ([ceil(T/32), E] ints) that carries the token-order slot numbering across blocks.
// It normally lives in the caller's workspace.  Some callers have no way to provide one: code running
// inside another framework's memory pool or a plugin host that hands out only the tensors it owns,
// and callers that must not allocate after start-up (no cudaMalloc, no allocator call on the hot
// path).  moe_dispatch_static_scratch keeps that scratch in a fixed array compiled into the library
// instead, and otherwise runs exactly the kernels moe_dispatch runs.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "kernels.h"
#include "moe_b300.h"

namespace {

using namespace moe;

constexpr int kHeaderInts = 64;  // error word, its info and padding: 256 bytes before the histogram
constexpr int kScratchInts = kHeaderInts + MOE_DISPATCH_STATIC_MAX_HIST;
static_assert(MOE_DISPATCH_STATIC_MAX_HIST % 64 == 0, "histogram section keeps 256-byte alignment");

// The scratch itself: one copy per device that loads the library, held until the process exits.
static __device__ __align__(256) int32_t g_dispatch_scratch[kScratchInts];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
int32_t* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_dispatch_scratch on the current device.  On the host the symbol names a host
// stand-in, so its address must be looked up once per device, with that device current.
moe_status scratch_for_current_device(int32_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return MOE_ERR_CUDA;
        }
        g_scratch_ptr[dev] = static_cast<int32_t*>(p);
    }
    *out = g_scratch_ptr[dev];
    return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

moe_status moe_dispatch_static_scratch(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                                       const float* topk_gate, int32_t* slot, int32_t* expert_count,
                                       int32_t* expert_offset, int32_t* row_token, float* row_gate,
                                       void* x_dispatched, void* stream) {
    // sizes and capacity exactly as moe_dispatch derives them (moe_capacity validates the config)
    const int32_t C = moe_capacity(cfg);
    if (C < 0) return MOE_ERR_INVALID_ARG;
    const int T = cfg->tokens, k = cfg->top_k, E = cfg->num_experts, d = cfg->model_dim;
    if (T == 0) return MOE_OK;
    const int64_t nblk = ((int64_t)T + kTokensPerBlock - 1) / kTokensPerBlock;
    if (nblk * E > (int64_t)MOE_DISPATCH_STATIC_MAX_HIST) return MOE_ERR_UNSUPPORTED;
    const void* ptrs[] = {x, topk_idx, topk_gate, slot, expert_count, expert_offset, row_token, row_gate, x_dispatched};
    for (const void* q : ptrs)
        if (!q || !aligned16(q)) return MOE_ERR_INVALID_ARG;
    int32_t* scratch = nullptr;
    moe_status st = scratch_for_current_device(&scratch);
    if (st != MOE_OK) return st;
    int* err = scratch;
    int* hist = scratch + kHeaderInts;
    const int Ceff = C < T ? C : T;
    const int bf16 = cfg->dtype == MOE_BF16;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the error word and the rank step's CTA ticket must start at zero; the histogram is written in full
    // before it is read
    if (cudaMemsetAsync(err, 0, 16, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (launch_dispatch_rank(topk_idx, T, k, E, hist, slot, err, err + 2, Ceff, expert_count, expert_offset,
                             row_token, row_gate, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (launch_dispatch_gather(x, bf16, topk_idx, topk_gate, hist, expert_offset, nullptr, false, T, k, E, d, Ceff,
                               slot, row_token,
                               row_gate, x_dispatched, nullptr, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

}  // extern "C"
