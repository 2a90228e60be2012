// router_stats.cu -- statistics of one routing: expert importance, the importance and load-balance
// losses, and the pairs the capacity limit dropped.
//
// importance[e] is the column sum of the dense gate matrix (the gate each token gives e, 0 where e is
// not among its top k), expert_importance_loss = 0.1 * std(importance) with E - 1 in the denominator
// ("MoE sparse-compute acceleration", section 4.1), load_balance_loss = sum_e (mean - importance[e])^2
// ("MoE architecture: breaking the single-card compute bottleneck", load balancing).
//
// One grid-stride pass over the (token, rank) pairs: each gate, rounded to a multiple of 2^-32, is
// added to its expert's 64-bit integer accumulator in shared memory, and each block adds its nonzero
// accumulators to the global ones once, so the sums are exact and do not depend on the order of the
// atomic adds (the result is the same on every run); each warp counts its dropped pairs with a ballot.  The last block to finish (ticket) converts the sums and computes the two losses in
// fp64, a thread per expert and a block reduction in a fixed order.
#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"  // device_sm_count

namespace moe {

namespace {

constexpr int kStatsThreads = 256;
constexpr double kFix = 4294967296.0;  // 2^32: fixed-point scale of the gate sums

__device__ __forceinline__ double block_sum_d(double v, double* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_sum_d(v);
    __syncthreads();  // red may still be read from a previous call
    if (lane == 0) red[warp] = v;
    __syncthreads();
    double s = 0.0;
    for (int w = 0; w < kStatsThreads / 32; ++w) s += red[w];  // every thread, in warp order
    return s;
}

__global__ void __launch_bounds__(kStatsThreads) router_stats_kernel(
    const int* __restrict__ topk_idx, const float* __restrict__ topk_gate, const int* __restrict__ slot,
    long long npairs, int E, unsigned long long* acc, unsigned long long* drops, int* ticket, int* err,
    float* importance, float* losses, long long* dropped) {
    __shared__ double red[kStatsThreads / 32];
    __shared__ int last;
    extern __shared__ unsigned long long s_acc[];  // [E]
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    for (int e = threadIdx.x; e < E; e += kStatsThreads) s_acc[e] = 0ull;
    __syncthreads();
    unsigned long long nd = 0;
    for (long long p = (long long)blockIdx.x * kStatsThreads + threadIdx.x; p - lane < npairs;
         p += (long long)gridDim.x * kStatsThreads) {
        const bool in = p < npairs;
        if (in) {
            const int e = topk_idx[p];
            const float g = topk_gate[p];
            if (e < 0 || e >= E || !(g >= 0.f && g <= 1.f)) {
                record_error(err, kErrCheck, kWhereRouterStats);
            } else {
                atomicAdd(s_acc + e, (unsigned long long)llrint((double)g * kFix));
            }
        }
        if (slot != nullptr) nd += __popc(__ballot_sync(0xffffffffu, in && slot[p] < 0));
    }
    if (slot != nullptr && lane == 0 && nd != 0) atomicAdd(drops, nd);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kStatsThreads)
        if (s_acc[e] != 0ull) atomicAdd(acc + e, s_acc[e]);
    // the last block to finish turns the sums into the statistics
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        last = atomicAdd(ticket, 1) == (int)gridDim.x - 1;
        __threadfence();
    }
    __syncthreads();
    if (!last) return;
    double s = 0.0;
    for (int e = threadIdx.x; e < E; e += kStatsThreads) s += (double)__ldcg(acc + e) / kFix;
    const double mean = block_sum_d(s, red) / (double)E;
    double ss = 0.0;
    for (int e = threadIdx.x; e < E; e += kStatsThreads) {
        const double v = (double)__ldcg(acc + e) / kFix;
        importance[e] = (float)v;
        ss += (mean - v) * (mean - v);
    }
    ss = block_sum_d(ss, red);
    if (threadIdx.x == 0) {
        losses[0] = E > 1 ? (float)(0.1 * sqrt(ss / (double)(E - 1))) : __int_as_float(0x7fc00000);
        losses[1] = (float)ss;
        if (dropped != nullptr) *dropped = slot != nullptr ? (long long)__ldcg(drops) : 0;
        *ticket = 0;
    }
}

}  // namespace

cudaError_t launch_router_stats(const int* topk_idx, const float* topk_gate, const int* slot, int T, int k, int E,
                                void* scratch, int* err, float* importance, float* losses, long long* dropped,
                                cudaStream_t s) {
    // scratch: E + 1 uint64 (the expert sums, the drop count) then the ticket, all zero on entry
    unsigned long long* acc = static_cast<unsigned long long*>(scratch);
    int* ticket = reinterpret_cast<int*>(acc + E + 1);
    const long long npairs = (long long)T * k;
    long long blocks = (npairs + kStatsThreads - 1) / kStatsThreads;
    const long long cap = 4LL * device_sm_count();
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_pdl(router_stats_kernel, dim3((unsigned)blocks), dim3(kStatsThreads), sizeof(unsigned long long) * E, s,
                      topk_idx, topk_gate,
                      slot, npairs, E, acc, acc + E, ticket, err, importance, losses, dropped);
}

}  // namespace moe
