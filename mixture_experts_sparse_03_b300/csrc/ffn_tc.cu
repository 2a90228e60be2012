// ffn_tc.cu -- grouped expert GEMM on the 5th-generation tensor cores (tcgen05, TMEM accumulators,
// TMA loads), bf16 operands, fp32 accumulation.
//
// Grouping tokens by expert and running one batched matmul per group ("How sparse activation improves
// efficiency", section 3.1), done as one persistent launch over all experts: the dispatched rows are segments of 128-row tiles,
// one expert per tile, and the tiles (m-tile, n-tile) are dealt round-robin to one CTA per SM.
//
// CTA = 6 warps:
//   warp 0     TMA producer: A tile [128 x 64] of the dispatched activations and B tile [256 x 64]
//              of the expert's weight ([E, N, K] tensor map, expert = third coordinate) per stage,
//              128-byte swizzle, into a 4-stage ring guarded by full / empty mbarriers
//   warp 1     allocates 512 TMEM columns (two 128 x 256 fp32 accumulators); one lane issues
//              tcgen05.mma (M = 128, N = 256, K = 16, kind::f16) and tcgen05.commit to release smem
//              stages and to hand finished accumulators to the epilogue
//   warps 2-5  epilogue: tcgen05.ld of the accumulator (each warp its 32 TMEM lanes = 32 rows), then
//              mode 0: + b1, GELU(erf), round to bf16, store the hidden row
//              mode 1: + b2, store fp32 y
//              mode 2: + b2, times the row's gate, fp32 atomic add into out[token] (fused combine)
//              while the MMA warp fills the other accumulator
// Every mbarrier wait is bounded: on expiry the kernel records MOE_ERR_DEVICE_TIMEOUT in the error
// word, all roles stop, the producer waits (bounded) for its copies in flight, the MMA warp waits for
// its last MMAs, and the TMEM is freed before the CTA exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kBM = 128, kBN = 256, kBK = 64, kStages = 4;
constexpr int kThreads = 192;
constexpr uint32_t kABytes = kBM * kBK * 2;           // 16 KiB
constexpr uint32_t kBBytes = kBN * kBK * 2;           // 32 KiB
constexpr uint32_t kStageBytes = kABytes + kBBytes;   // 48 KiB
constexpr uint32_t kTmemCols = 2 * kBN;               // 512
constexpr uint32_t kSpinLimit = 1u << 22;             // polls before a wait gives up (about a second)

struct TcArgs {
    const int* offset;
    const int* row_token;
    const float* row_gate;
    const bf16_t* bias;
    void* C;
    float* out;
    int E, K, N, mode;
    int* err;
};

// ---- PTX wrappers ------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// bounded wait; false if it gave up or another role already gave up
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    for (uint32_t i = 0; i < kSpinLimit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 255u && *abort_flag) return false;
        if (i > 1024u) __nanosleep(64);
    }
    return false;
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(map), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(map), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}
// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane (base lane + i), columns c..c+31
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
          "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
          "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
          "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row groups 1024 bytes apart
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);         // start address
    d |= (uint64_t)(16u >> 4) << 16;                 // leading byte offset (unused with this swizzle)
    d |= (uint64_t)(1024u >> 4) << 32;               // stride byte offset: next 8-row group
    d |= (uint64_t)1 << 46;                          // descriptor version
    d |= (uint64_t)2 << 61;                          // 128-byte swizzle
    return d;
}
// instruction descriptor, kind::f16: D fp32, A and B bf16, both K-major, M x N
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    // the 128-byte swizzle atoms need 1024-byte aligned tiles in the shared address space
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* sA = base;
    uint8_t* sB = base + kStages * kABytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + kStages * kBBytes);
    // bars: full[kStages], empty[kStages], tfull[2], tempty[2], last
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    int* s_off = reinterpret_cast<int*>(tmem_holder + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto bar = [&](int i) { return smem_u32(bars + i); };
    const int FULL = 0, EMPTY = kStages, TFULL = 2 * kStages, TEMPTY = 2 * kStages + 2, LAST = 2 * kStages + 4;

    for (int i = threadIdx.x; i <= a.E; i += kThreads) s_off[i] = a.offset[i];
    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(FULL + s), 1);
            mbar_init(bar(EMPTY + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(TFULL + s), 1);
            mbar_init(bar(TEMPTY + s), 4);
        }
        mbar_init(bar(LAST), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    const int total_rows = s_off[a.E];
    const int m_tiles = total_rows / kBM;
    const int n_tiles = (a.N + kBN - 1) / kBN;
    const int num_tiles = m_tiles * n_tiles;
    const int k_iters = a.K / kBK;

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_phase[kStages];
            bool issued[kStages];
            for (int s = 0; s < kStages; ++s) { issued[s] = false; issued_phase[s] = 0; }
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                const int m0 = (tile / n_tiles) * kBM, n0 = (tile % n_tiles) * kBN;
                const int e = expert_of_row(s_off, a.E, m0);
                for (int kb = 0; kb < k_iters; ++kb) {
                    if (!mbar_wait(bar(EMPTY + stage), phase ^ 1u, abort_flag)) { ok = false; break; }
                    mbar_expect_tx(bar(FULL + stage), kStageBytes);
                    tma_load_2d(smem_u32(sA + stage * kABytes), &tmA, bar(FULL + stage), kb * kBK, m0);
                    tma_load_3d(smem_u32(sB + stage * kBBytes), &tmB, bar(FULL + stage), kb * kBK, n0, e);
                    issued[stage] = true;
                    issued_phase[stage] = phase;
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                record_error(a.err, kErrTimeout, kWhereGemmProducer);
                *abort_flag = 1;
                // let every copy this thread started land before the CTA's shared memory goes away
                for (int s = 0; s < kStages; ++s)
                    if (issued[s]) {
                        for (uint32_t i = 0; i < kSpinLimit && !mbar_try_wait(bar(FULL + s), issued_phase[s]); ++i)
                            __nanosleep(64);
                    }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(kBM, kBN);
            int stage = 0;
            uint32_t phase = 0;
            int local = 0;
            bool ok = true, any = false;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x, ++local) {
                const int acc = local & 1;
                const uint32_t acc_phase = (local >> 1) & 1;
                if (!mbar_wait(bar(TEMPTY + acc), acc_phase ^ 1u, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * kBN;
                for (int kb = 0; kb < k_iters; ++kb) {
                    if (!mbar_wait(bar(FULL + stage), phase, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t ad = smem_desc_sw128(smem_u32(sA + stage * kABytes));
                    const uint64_t bd = smem_desc_sw128(smem_u32(sB + stage * kBBytes));
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        tc_mma(d_tmem, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc, (kb | kk) != 0);
                    any = true;
                    tc_commit(bar(EMPTY + stage));
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
                if (ok) tc_commit(bar(TFULL + acc));
            }
            if (!ok) {
                record_error(a.err, kErrTimeout, kWhereGemmMma);
                *abort_flag = 1;
            }
            if (any) {  // all MMAs this thread issued have finished once LAST completes
                tc_commit(bar(LAST));
                for (uint32_t i = 0; i < kSpinLimit && !mbar_try_wait(bar(LAST), 0); ++i) __nanosleep(64);
            }
        }
    } else {
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        int local = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++local) {
            const int acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            const bool ok = __all_sync(0xffffffffu, mbar_wait(bar(TFULL + acc), acc_phase, abort_flag));
            if (!ok) {
                if (lane == 0) {
                    record_error(a.err, kErrTimeout, kWhereGemmEpilogue);
                    *abort_flag = 1;
                }
                break;
            }
            tc_fence_after();
            const int m0 = (tile / n_tiles) * kBM, n0 = (tile % n_tiles) * kBN;
            const int e = expert_of_row(s_off, a.E, m0);
            const int r = m0 + row;
            const int tok = a.row_token[r];
            const float g = (a.mode == 2 && tok >= 0) ? a.row_gate[r] : 0.f;
            const bf16_t* bias = a.bias ? a.bias + (size_t)e * a.N : nullptr;
            for (int c0 = 0; c0 < kBN; c0 += 32) {
                uint32_t v[32];
                __syncwarp();
                tmem_ld32(tmem_base + lane_base + (uint32_t)(acc * kBN + c0), v);
                const int n = n0 + c0;
                if (tok >= 0 && n < a.N) {
                float f[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[j]);
                if (bias) {
#pragma unroll
                    for (int j = 0; j < 32; j += 8) {
                        float b[8];
                        load8(bias + n + j, b);
#pragma unroll
                        for (int i = 0; i < 8; ++i) f[j + i] += b[i];
                    }
                }
                if (a.mode == 0) {
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<bf16_t*>(a.C) + (size_t)r * a.N + n);
#pragma unroll
                    for (int j = 0; j < 32; j += 8) {
                        uint4 w;
                        w.x = pack_bf16x2(gelu_erf(f[j + 0]), gelu_erf(f[j + 1]));
                        w.y = pack_bf16x2(gelu_erf(f[j + 2]), gelu_erf(f[j + 3]));
                        w.z = pack_bf16x2(gelu_erf(f[j + 4]), gelu_erf(f[j + 5]));
                        w.w = pack_bf16x2(gelu_erf(f[j + 6]), gelu_erf(f[j + 7]));
                        dst[j / 8] = w;
                    }
                } else if (a.mode == 1) {
                    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.C) + (size_t)r * a.N + n);
#pragma unroll
                    for (int j = 0; j < 32; j += 4) dst[j / 4] = make_float4(f[j], f[j + 1], f[j + 2], f[j + 3]);
                } else {
                    float4* dst = reinterpret_cast<float4*>(a.out + (size_t)tok * a.N + n);
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        atomicAdd(dst + j / 4, make_float4(g * f[j], g * f[j + 1], g * f[j + 2], g * f[j + 3]));
                }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(TEMPTY + acc));
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                     : "memory");
    }
}

// ---- host side ----------------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

struct MapKey {
    const void* ptr;
    uint64_t d0, d1, d2;
    uint32_t b1;
    bool operator==(const MapKey& o) const {
        return ptr == o.ptr && d0 == o.d0 && d1 == o.d1 && d2 == o.d2 && b1 == o.b1;
    }
};
struct MapEntry {
    MapKey key;
    CUtensorMap map;
};
std::mutex g_map_mutex;
MapEntry g_maps[64];
int g_maps_used = 0, g_maps_next = 0;

// bf16 tensor [d2][d1][d0] (d0 contiguous) tiled in boxes of 64 x b1 (x 1), 128-byte swizzle
bool get_map(const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b1, CUtensorMap* out) {
    const MapKey key{ptr, d0, d1, d2, b1};
    std::lock_guard<std::mutex> lock(g_map_mutex);
    for (int i = 0; i < g_maps_used; ++i)
        if (g_maps[i].key == key) { *out = g_maps[i].map; return true; }
    auto fn = encode_fn();
    if (!fn) return false;
    CUtensorMap m;
    const cuuint32_t rank = d2 > 0 ? 3 : 2;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
    cuuint32_t box[3] = {(cuuint32_t)kBK, b1, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(ptr), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    MapEntry& slot = g_maps[g_maps_next];
    slot.key = key;
    slot.map = m;
    g_maps_next = (g_maps_next + 1) % 64;
    if (g_maps_used < 64) ++g_maps_used;
    *out = m;
    return true;
}

int num_sms() {
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
    }
    return n;
}

}  // namespace

size_t ffn_tc_smem_bytes(int E) {
    return 1024 + (size_t)kStages * kStageBytes + (2 * kStages + 5) * 8 + 16 + 4 * (size_t)(E + 1);
}

cudaError_t launch_ffn_tc(const FfnParams& P, cudaStream_t s) {
    if (!P.bf16) return cudaErrorInvalidValue;
    if (P.rows_cap <= 0) return cudaSuccess;
    CUtensorMap ma, mb;
    if (!get_map(P.A, (uint64_t)P.K, (uint64_t)P.rows_cap, 0, kBM, &ma)) return cudaErrorInvalidValue;
    if (!get_map(P.W, (uint64_t)P.K, (uint64_t)P.N, (uint64_t)P.E, kBN, &mb)) return cudaErrorInvalidValue;
    TcArgs a;
    a.offset = P.offset;
    a.row_token = P.row_token;
    a.row_gate = P.row_gate;
    a.bias = static_cast<const bf16_t*>(P.bias);
    a.C = P.C;
    a.out = P.out;
    a.E = P.E;
    a.K = P.K;
    a.N = P.N;
    a.mode = P.mode;
    a.err = P.err;
    const size_t smem = ffn_tc_smem_bytes(P.E);
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t max_tiles = (P.rows_cap / kBM) * (int64_t)((P.N + kBN - 1) / kBN);
    int grid = num_sms();
    if (max_tiles < grid) grid = (int)(max_tiles > 0 ? max_tiles : 1);
    gemm_tc_kernel<<<grid, kThreads, smem, s>>>(ma, mb, a);
    return cudaGetLastError();
}

}  // namespace moe
