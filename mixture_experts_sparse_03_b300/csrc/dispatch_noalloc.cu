// dispatch_noalloc.cu -- moe_dispatch for callers that cannot allocate device memory.
//
// moe_dispatch needs a little device scratch besides its outputs: an error word and the per-block
// expert histogram ([ceil(T/32), E] ints) that carries the token-order slot numbering across blocks.
// It normally lives in the caller's workspace.  Some callers have no way to provide one: code running
// inside another framework's memory pool or a plugin host that hands out only the tensors it owns,
// and callers that must not allocate after start-up (no cudaMalloc, no allocator call on the hot
// path).  moe_dispatch_static_scratch keeps that scratch in a fixed array compiled into the library
// instead, and otherwise runs exactly the kernels moe_dispatch runs.
#include <cuda.h>
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
struct ScratchAddr {
    unsigned long long ctx_id;  // the context the address belongs to (0: none looked up yet)
    int32_t* ptr;
};
ScratchAddr g_scratch[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (0 if there is none or the driver cannot say).
// Context ids are never reused within a process, so a device reset, which destroys the primary
// context and the module holding the array, changes the id and forces a fresh look-up.
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static bool resolved = false;
    if (!resolved) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
        cudaGetLastError();
        resolved = true;
    }
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of g_dispatch_scratch on the current device.  On the host the symbol names a host
// stand-in, so its device address is looked up with cudaGetSymbolAddress, with the device current:
// once per device and context (the first call on a device, and the first after a device reset).
moe_status scratch_for_current_device(int32_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    unsigned long long id = current_context_id();
    if (id == 0 || g_scratch[dev].ctx_id != id) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return MOE_ERR_CUDA;
        }
        // the look-up makes the device's primary context current if nothing was; key the address by it
        if (id == 0) id = current_context_id();
        g_scratch[dev] = ScratchAddr{id, static_cast<int32_t*>(p)};  // id 0: look up again next call
    }
    *out = g_scratch[dev].ptr;
    return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

moe_status moe_dispatch_static_scratch(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                                       const float* topk_gate, int32_t* slot, int32_t* expert_count,
                                       int32_t* expert_offset, int32_t* row_token, float* row_gate,
                                       void* x_dispatched, void* stream) {
    // the config is validated by the same planner as moe_dispatch's, with the same status; sizes and
    // capacity exactly as moe_dispatch derives them
    const moe_status plan = config_status(cfg);
    if (plan != MOE_OK) return plan;
    const int32_t C = moe_capacity(cfg);
    const int T = cfg->tokens, k = cfg->top_k, E = cfg->num_experts, d = cfg->model_dim;
    if (T == 0) return MOE_OK;
    const int rank_major = (cfg->flags & MOE_FLAG_RANK_MAJOR) != 0;
    const int64_t nblk = dispatch_hist_blocks(T, k, rank_major);
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
                             row_token, row_gate, rank_major, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (launch_dispatch_gather(x, bf16, topk_idx, topk_gate, hist, expert_offset, nullptr, false, T, k, E, d, Ceff,
                               slot, row_token,
                               row_gate, x_dispatched, nullptr, rank_major, GatherStats{}, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

}  // extern "C"
