// Dense BF16 split-K GEMM C = A . W^T on tcgen05 (sm_103a) -- the kernel the
// split-K wave model of gpu-kernels-explained "Split-K, streams and overlap"
// describes: 128 x 128 output tiles, k cut into `split` slices, each slice's
// partial sum written as an FP32 plane and added by a second pass.
//
// One CTA = one 128 x 128 tile over one k slice.  Warp 0 (one thread) loads
// 128 x 64 tiles of A and W by TMA (128-byte swizzle, K-major) into a
// STAGES-deep ring; warp 1 allocates tensor memory; one thread each of warps
// 1 and 2 issues tcgen05.mma (A and B from shared memory) for alternate k
// stages into its own 128 x 128 FP32 accumulator in tensor memory -- a single
// issuing thread spends tens of ns per MMA, as much as the MMA's tensor time;
// warps 3-6 read both accumulators back with tcgen05.ld (lane = row of C),
// add them in a fixed order and store the sum.  All waits are bounded
// (qmm_sm100.cuh).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "qmm_device.cuh"
#include "qmm_internal.h"
#include "qmm_sm100.cuh"

namespace qmm {

namespace {

constexpr int kTile = 128, kKStep = 64, kMaxStagesG = 8;
constexpr int kIssuers = 2;                       // MMA issuers, one accumulator each
constexpr int kThreadsG = 32 * (1 + kIssuers + 4);  // producer, issuers, epilogue
constexpr int kOpBytes = kTile * kKStep * 2;  // one operand tile per stage: 16 KB
constexpr uint32_t kIdescG = idesc_bf16_f32(kTile, kTile);

// K-major 128-byte-swizzle descriptor for an operand held in shared memory
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) { return sdesc_kmajor_sw128(saddr); }

__device__ __forceinline__ void umma_bf16_ss(uint32_t d, uint64_t adesc, uint64_t bdesc,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

struct GemmTcParams {
    void* out;
    int* status;
    int M, N, K, split, out_mode, stages;
};

__global__ void __launch_bounds__(kThreadsG, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap amap,
                   const __grid_constant__ CUtensorMap bmap, const GemmTcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int stages = p.stages;
    uint8_t* ring = base;  // per stage: A tile then W tile
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + stages * 2 * kOpBytes);
    uint64_t* empty = full + kMaxStagesG;
    uint64_t* acc_full = empty + kMaxStagesG;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
    __shared__ int abort_flag;
    volatile int* abort = &abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n0 = blockIdx.x * kTile, m0 = blockIdx.y * kTile, part = blockIdx.z;
    const int T = p.K / kKStep;
    const int nt = T / p.split + (part < T % p.split ? 1 : 0);
    const int t0 = part * (T / p.split) + (part < T % p.split ? part : T % p.split);

    pdl_trigger();
    if (tid == 0) {
        abort_flag = 0;
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, kIssuers);
        mbar_fence_init();
        tma_prefetch_map(&amap);
        tma_prefetch_map(&bmap);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kIssuers * kTile);
        tmem_relinquish();
    }
    pdl_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        int issued = 0;
        for (int i = 0; i < nt; ++i) {
            const int s = i % stages;
            if (!mbar_wait(&empty[s], ((i / stages) & 1) ^ 1, abort, p.status)) break;
            mbar_arrive_expect_tx(&full[s], 2 * kOpBytes);
            const int k = (t0 + i) * kKStep;
            tma_load_2d(ring + s * 2 * kOpBytes, &amap, &full[s], k, m0);
            tma_load_2d(ring + s * 2 * kOpBytes + kOpBytes, &bmap, &full[s], k, n0);
            issued = i + 1;
        }
        if (*abort) {
            const int first = issued > stages ? issued - stages : 0;
            for (int i = first; i < issued; ++i)
                mbar_wait(&full[i % stages], (i / stages) & 1, nullptr, p.status);
        }
    } else if (warp >= 1 && warp <= kIssuers) {
      if (lane == 0) {
        const int c = warp - 1;
        const uint32_t dacc = tmem + c * kTile;
        for (int i = c; i < nt; i += kIssuers) {
            const int s = i % stages;
            if (!mbar_wait(&full[s], (i / stages) & 1, abort, p.status)) break;
            tc_fence_after();
            const uint32_t a_sm = smem_addr(ring + s * 2 * kOpBytes);
            const uint32_t b_sm = a_sm + kOpBytes;
#pragma unroll
            for (int kk = 0; kk < kKStep / 16; ++kk)
                umma_bf16_ss(dacc, sdesc(a_sm + kk * 32), sdesc(b_sm + kk * 32), kIdescG,
                             (i != c) || kk != 0);
            umma_commit(&empty[s]);
        }
        umma_commit(acc_full);
      }
    } else if (warp > kIssuers) {
        // epilogue (warps kIssuers+1 .. kIssuers+4, whole warps only: the
        // warp-wide waits and tcgen05.ld need all 32 lanes): warp w reads
        // tensor-memory lanes 32*(w%4).. = rows of C
        const int quarter = warp & 3;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const int m = m0 + quarter * 32 + lane;
        if (mbar_wait_warp(acc_full, 0, abort, p.status)) {
            tc_fence_after();
            const size_t plane = static_cast<size_t>(part) * p.M * p.N;
#pragma unroll 1
            for (int c = 0; c < kTile / 16; ++c) {
                uint32_t d[16];
                tmem_ld16(tmem + lane_base + c * 16, d);
                tmem_ld_wait();
                static_assert(kIssuers == 2, "the epilogue adds two accumulators");
                if (nt > 1) {  // the second accumulator received stages
                    uint32_t e[16];
                    tmem_ld16(tmem + lane_base + kTile + c * 16, e);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        d[j] = __float_as_uint(__uint_as_float(d[j]) + __uint_as_float(e[j]));
                }
                const int n = n0 + c * 16;
                if (m >= p.M) continue;
                const size_t o = plane + static_cast<size_t>(m) * p.N + n;
                if (p.out_mode == kOutBf16) {
                    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + o;
                    if (n + 16 <= p.N && (p.N & 7) == 0) {
                        uint4 v0, v1;
                        v0.x = pack_bf16x2(__uint_as_float(d[0]), __uint_as_float(d[1]));
                        v0.y = pack_bf16x2(__uint_as_float(d[2]), __uint_as_float(d[3]));
                        v0.z = pack_bf16x2(__uint_as_float(d[4]), __uint_as_float(d[5]));
                        v0.w = pack_bf16x2(__uint_as_float(d[6]), __uint_as_float(d[7]));
                        v1.x = pack_bf16x2(__uint_as_float(d[8]), __uint_as_float(d[9]));
                        v1.y = pack_bf16x2(__uint_as_float(d[10]), __uint_as_float(d[11]));
                        v1.z = pack_bf16x2(__uint_as_float(d[12]), __uint_as_float(d[13]));
                        v1.w = pack_bf16x2(__uint_as_float(d[14]), __uint_as_float(d[15]));
                        reinterpret_cast<uint4*>(dst)[0] = v0;
                        reinterpret_cast<uint4*>(dst)[1] = v1;
                    } else {
                        for (int j = 0; j < 16 && n + j < p.N; ++j)
                            dst[j] = __float2bfloat16_rn(__uint_as_float(d[j]));
                    }
                } else {
                    float* dst = static_cast<float*>(p.out) + o;
                    if (n + 16 <= p.N && (p.N & 3) == 0) {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            reinterpret_cast<float4*>(dst)[j] =
                                make_float4(__uint_as_float(d[4 * j]), __uint_as_float(d[4 * j + 1]),
                                            __uint_as_float(d[4 * j + 2]),
                                            __uint_as_float(d[4 * j + 3]));
                    } else {
                        for (int j = 0; j < 16 && n + j < p.N; ++j) dst[j] = __uint_as_float(d[j]);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        if (lane == 0 && *abort) mbar_wait(acc_full, 0, nullptr, p.status);
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kIssuers * kTile);
    }
}

}  // namespace

bool encode_2d(CUtensorMap* map, CUtensorMapDataType type, const void* ptr, uint64_t rows,
               uint64_t cols, int elem, uint32_t box_rows, uint32_t box_cols,
               CUtensorMapSwizzle swizzle);
int* tc_status_ptr();

int launch_gemm_tc(const void* A, const void* W, void* out, int out_mode, int M, int N, int K,
                   int split, void* stream) {
    static int limit = -1;
    static std::once_flag once;
    std::call_once(once, [] {
        limit = set_max_dynamic_smem(reinterpret_cast<const void*>(gemm_tc_kernel));
    });
    if (limit < 0) return cudaErrorInvalidValue;
    GemmTcParams p;
    p.out = out;
    p.status = tc_status_ptr();
    if (!p.status) return cudaErrorInvalidSymbol;
    p.M = M;
    p.N = N;
    p.K = K;
    p.split = split;
    p.out_mode = out_mode;
    const size_t fixed = 1024 + (2 * kMaxStagesG + 1) * 8 + 16 + 128;
    // stage s of the ring goes to issuer s % kIssuers; a multiple of kIssuers
    // stages keeps each slot's laps with one issuer, so its parity waits are
    // sound (a waiter that skipped a lap could take a two-laps-old completion)
    int stages = kMaxStagesG;
    while (stages > kIssuers &&
           (fixed + stages * 2 * kOpBytes > static_cast<size_t>(limit) || stages % kIssuers))
        --stages;
    p.stages = stages;
    CUtensorMap amap, bmap;
    if (!encode_2d(&amap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, M, K, 2, kTile, kKStep,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&bmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W, N, K, 2, kTile, kKStep,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    LaunchAttrs la;
    apply_pdl(cfg, la);
    cfg.gridDim = dim3((N + kTile - 1) / kTile, (M + kTile - 1) / kTile, split);
    cfg.blockDim = dim3(kThreadsG, 1, 1);
    cfg.dynamicSmemBytes = fixed + stages * 2 * kOpBytes;
    cfg.stream = static_cast<cudaStream_t>(stream);
    return cudaLaunchKernelEx(&cfg, gemm_tc_kernel, amap, bmap, p);
}

}  // namespace qmm
