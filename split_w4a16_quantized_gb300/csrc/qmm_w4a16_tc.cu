// W4A16-g128 partition / unsplit matmul on the 5th-generation tensor cores
// (tcgen05, sm_103a).
//
// A CTA owns 128 weight rows (output columns n0..n0+127) x BNA activation
// rows (m0..m0+BNA-1) over one partition of the reduction axis (tiny-llm
// book, "Week 2 Day 7: Split-K Prefill", Task 2: grid z = partition, equal
// partitions on 128-group boundaries, each writes its own partial plane, no
// atomics).  The product is computed transposed, C^T tile = W . A^T:
//   - MMA A operand = dequantized weights, 128 rows x 16 k, held in TENSOR
//     MEMORY (lane = weight row).  The weights go packed HBM -> shared memory
//     (TMA) -> registers (unpack + dequant) -> tensor memory (tcgen05.st);
//     BF16 weights never travel through shared memory, whose bandwidth a
//     dequantized operand would otherwise exhaust at HBM rate.
//   - MMA B operand = activations, BNA rows x 16 k, loaded by TMA into
//     128-byte-swizzled shared memory (K-major).
//   - D = FP32 accumulator in tensor memory, 128 lanes x BNA columns.
// Warp roles (12 warps):
//   warp 0      TMA producer (one thread): per 128-group one 8 KB weight box
//               and two activation boxes into a STAGES-deep ring;
//   warp 1      tensor-memory allocator; one thread issues tcgen05.mma;
//   warps 4-11  dequantizers, then the epilogue: warp w serves lanes
//               32*(w%4).. of tensor memory and the groups of parity
//               (w-4)/4, writing into one of two tensor-memory A buffers.
// Every mbarrier wait is bounded (qmm_sm100.cuh): a wait that runs out sets
// the status word, the CTA stops issuing work, waits (bounded) for what is in
// flight, frees its tensor memory and exits.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "qmm_device.cuh"
#include "qmm_internal.h"
#include "qmm_sm100.cuh"

namespace qmm {

__device__ int g_tc_status = 0;

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// 2-D row-major tensor [rows, cols] of `elem` bytes, box [box_rows, box_cols]
bool encode_2d(CUtensorMap* map, CUtensorMapDataType type, const void* ptr, uint64_t rows,
               uint64_t cols, int elem, uint32_t box_rows, uint32_t box_cols,
               CUtensorMapSwizzle swizzle) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * elem};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, type, 2, const_cast<void*>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int* tc_status_ptr() {
    static int* ptr = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_tc_status) == cudaSuccess) ptr = static_cast<int*>(p);
    });
    return ptr;
}


namespace {

constexpr int kWRows = 128;              // weight rows per CTA (MMA M)
constexpr int kWStage = kWRows * 64;     // packed weight bytes per group
constexpr int kMaxStages = 8;
constexpr int kThreads = 384;

struct TcParams {
    const uint16_t* scales;
    const uint16_t* biases;
    void* out;
    int* status;
    int M, Kred, Nout, G, gpp, out_mode, stages;
};

template <int BNA>
struct TcCfg {
    static_assert(BNA % 16 == 0 && BNA >= 16 && BNA <= 256, "MMA N");
    static constexpr int ACT_BOX = BNA * 128;       // one 64-k activation box
    static constexpr int ACT_STAGE = 2 * ACT_BOX;   // one 128-group
    static constexpr int ACOL = BNA < 64 ? 64 : BNA;  // first A-buffer column
    static constexpr int NEED = ACOL + 2 * 64;
    static constexpr int TMEM_COLS = NEED <= 128 ? 128 : NEED <= 256 ? 256 : 512;
    static constexpr uint32_t IDESC = idesc_bf16_f32(kWRows, BNA);
};

// pair (q[2c], q[2c+1]) of a packed word as BF16 (128 + q): byte c of x holds
// both nibbles; byte c of x >> 4 has the odd one in its low nibble.
__device__ __forceinline__ uint32_t natural_pair(uint32_t x, uint32_t x4, uint32_t sel) {
    return nibbles_to_bf16x2_biased(__byte_perm(x, x4, sel));
}

// 64 BF16 pairs of one weight row and group, in k order (pair c = k 2c, 2c+1)
__device__ __forceinline__ void dequant_row_group(const uint4 wv[4], uint32_t ss, uint32_t bb,
                                                  uint32_t out[64]) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const uint32_t x = j % 4 == 0 ? wv[j / 4].x : j % 4 == 1 ? wv[j / 4].y
                         : j % 4 == 2 ? wv[j / 4].z : wv[j / 4].w;
        const uint32_t x4 = x >> 4;
        const uint32_t sel[4] = {0x4400u, 0x5511u, 0x6622u, 0x7733u};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t q = fma_bf16x2(natural_pair(x, x4, sel[c]), kBf16x2One, kBf16x2Neg128);
            out[4 * j + c] = fma_bf16x2(q, ss, bb);
        }
    }
}

template <int BNA>
__global__ void __launch_bounds__(kThreads, 1)
    w4a16_tc_kernel(const __grid_constant__ CUtensorMap wmap,
                    const __grid_constant__ CUtensorMap amap, const TcParams p) {
    using C = TcCfg<BNA>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int stages = p.stages;
    uint8_t* aring = base;                                  // stages x ACT_STAGE
    uint8_t* wring = aring + stages * C::ACT_STAGE;         // stages x kWStage
    // per-group scales and biases of this CTA's rows: sc[gi * 128 + r], bi[...]
    uint16_t* sc = reinterpret_cast<uint16_t*>(wring + stages * kWStage);
    uint16_t* bi = sc + p.gpp * kWRows;
    uint32_t* sb = reinterpret_cast<uint32_t*>(bi + p.gpp * kWRows);  // end of the tables
    uint64_t* bars = reinterpret_cast<uint64_t*>(sb);
    uint64_t* full = bars;
    uint64_t* empty = bars + kMaxStages;
    uint64_t* a_full = bars + 2 * kMaxStages;
    uint64_t* a_empty = a_full + 2;
    uint64_t* acc_full = a_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
    __shared__ int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n0 = blockIdx.x * kWRows, m0 = blockIdx.y * BNA, part = blockIdx.z;
    const int ngrp = p.gpp, gbeg = part * p.gpp;
    volatile int* abort = &abort_flag;

    pdl_trigger();
    if (tid == 0) {
        abort_flag = 0;
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1 + 4);  // MMA commit + the four dequant warps
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&a_full[b], 4);
            mbar_init(&a_empty[b], 1);
        }
        mbar_init(acc_full, 1);
        mbar_fence_init();
        tma_prefetch_map(&wmap);
        tma_prefetch_map(&amap);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    pdl_wait();  // global memory is read only after the previous kernel is done
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ---- TMA producer ----
        int issued = 0;
        for (int i = 0; i < ngrp; ++i) {
            const int s = i % stages;
            if (!mbar_wait(&empty[s], ((i / stages) & 1) ^ 1, abort, p.status)) break;
            mbar_arrive_expect_tx(&full[s], kWStage + C::ACT_STAGE);
            const int g = gbeg + i;
            tma_load_2d(wring + s * kWStage, &wmap, &full[s], g * 16, n0);
            tma_load_2d(aring + s * C::ACT_STAGE, &amap, &full[s], g * kGroup, m0);
            tma_load_2d(aring + s * C::ACT_STAGE + C::ACT_BOX, &amap, &full[s], g * kGroup + 64,
                        m0);
            issued = i + 1;
        }
        if (*abort) {  // let copies in flight land before the CTA exits
            const int first = issued > stages ? issued - stages : 0;
            for (int i = first; i < issued; ++i)
                mbar_wait(&full[i % stages], (i / stages) & 1, nullptr, p.status);
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer ----
        for (int i = 0; i < ngrp; ++i) {
            const int s = i % stages, ab = i & 1;
            if (!mbar_wait(&full[s], (i / stages) & 1, abort, p.status)) break;
            if (!mbar_wait(&a_full[ab], (i >> 1) & 1, abort, p.status)) break;
            tc_fence_after();
            const uint32_t a_tm = tmem + C::ACOL + ab * 64;
            const uint32_t b_sm = smem_addr(aring + s * C::ACT_STAGE);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t bdesc = sdesc_kmajor_sw128(b_sm + (kk >> 2) * C::ACT_BOX + (kk & 3) * 32);
                umma_bf16_tmem_a(tmem, a_tm + kk * 8, bdesc, C::IDESC, (i | kk) != 0);
            }
            umma_commit(&empty[s]);
            umma_commit(&a_empty[ab]);
        }
        umma_commit(acc_full);
    } else if (warp >= 4) {
        // ---- dequantizers ----
        // scales (threads 128..255) and biases (256..383) of this CTA's rows for
        // every group, loaded while the first TMA copies are in flight
        {
            const int t = tid - 128, r = t & (kWRows - 1);
            load_group_row(t < kWRows ? p.scales : p.biases, p.Nout, p.G, n0 + r, gbeg, ngrp,
                           (t < kWRows ? sc : bi) + r, kWRows);
        }
        asm volatile("bar.sync 1, %0;\n" ::"n"(kThreads - 128) : "memory");
        const int quarter = warp & 3, par = (warp - 4) >> 2;
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        for (int i = par; i < ngrp; i += 2) {
            const int s = i % stages, ab = i & 1;
            if (!mbar_wait_warp(&full[s], (i / stages) & 1, abort, p.status)) break;
            const uint8_t* wr = wring + s * kWStage + row * 64;
            uint4 wv[4];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                wv[c] = *reinterpret_cast<const uint4*>(wr + ((c ^ ((row >> 1) & 3)) << 4));
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            uint32_t w[64];
            dequant_row_group(wv, bf16_pair(sc[i * kWRows + row]), bf16_pair(bi[i * kWRows + row]),
                              w);
            if (!mbar_wait_warp(&a_empty[ab], ((i >> 1) & 1) ^ 1, abort, p.status)) break;
            const uint32_t ta = tmem + lane_base + C::ACOL + ab * 64;
            tmem_st16(ta + 0, w);
            tmem_st16(ta + 16, w + 16);
            tmem_st16(ta + 32, w + 32);
            tmem_st16(ta + 48, w + 48);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_full[ab]);
        }
        // ---- epilogue: D lane = weight row, column = activation row ----
        if (mbar_wait_warp(acc_full, 0, abort, p.status)) {
            tc_fence_after();
            const int n = n0 + row;
            const size_t plane = static_cast<size_t>(part) * p.M * p.Nout;
            for (int c = par; c < BNA / 16; c += 2) {
                uint32_t d[16];
                tmem_ld16(tmem + lane_base + c * 16, d);
                tmem_ld_wait();
                if (n < p.Nout) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int m = m0 + c * 16 + j;
                        if (m < p.M) {
                            const size_t o = plane + static_cast<size_t>(m) * p.Nout + n;
                            const float f = __uint_as_float(d[j]);
                            if (p.out_mode == kOutBf16)
                                static_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(f);
                            else
                                static_cast<float*>(p.out)[o] = f;
                        }
                    }
                }
            }
        }
    }

    // ---- teardown: every MMA has finished before tensor memory is freed ----
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        if (lane == 0 && *abort) mbar_wait(acc_full, 0, nullptr, p.status);
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int BNA>
int launch_tc(const void* A, const uint32_t* Wq, const void* scales, const void* biases,
              void* out, int out_mode, int M, int Kred, int Nout, int split, cudaStream_t st) {
    using C = TcCfg<BNA>;
    auto kern = w4a16_tc_kernel<BNA>;
    static int limit = -1;
    static std::once_flag once;
    std::call_once(once, [&] { limit = set_max_dynamic_smem(reinterpret_cast<const void*>(kern)); });
    if (limit < 0) return cudaErrorInvalidValue;
    int* status = tc_status_ptr();
    if (!status) return cudaErrorInvalidSymbol;

    TcParams p;
    p.scales = static_cast<const uint16_t*>(scales);
    p.biases = static_cast<const uint16_t*>(biases);
    p.out = out;
    p.status = status;
    p.M = M;
    p.Kred = Kred;
    p.Nout = Nout;
    p.G = Kred / kGroup;
    p.gpp = p.G / split;
    p.out_mode = out_mode;
    // alignment slack + scale/bias table + barriers and tensor-memory slot,
    // with room for the kernel's few bytes of static shared memory
    const size_t fixed = 1024 + static_cast<size_t>(p.gpp) * kWRows * 4 +
                         (2 * kMaxStages + 5) * 8 + 16 + 128;
    const size_t per_stage = C::ACT_STAGE + kWStage;
    int stages = kMaxStages;
    while (stages > 2 && fixed + stages * per_stage > static_cast<size_t>(limit)) --stages;
    if (fixed + stages * per_stage > static_cast<size_t>(limit)) return cudaErrorInvalidValue;
    p.stages = stages;

    CUtensorMap wmap, amap;
    if (!encode_2d(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, Wq, Nout, Kred / 8, 4, kWRows, 16,
                   CU_TENSOR_MAP_SWIZZLE_64B) ||
        !encode_2d(&amap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, M, Kred, 2, BNA, 64,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;

    cudaLaunchConfig_t cfg = {};
    LaunchAttrs la;
    apply_pdl(cfg, la);
    cfg.gridDim = dim3((Nout + kWRows - 1) / kWRows, (M + BNA - 1) / BNA, split);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = fixed + stages * per_stage;
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, kern, wmap, amap, p);
}

}  // namespace

int launch_w4a16_tc(int bm, const void* A, const uint32_t* Wq, const void* scales,
                    const void* biases, void* out, int out_mode, int M, int Kred, int Nout,
                    int split, void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (bm) {
        case 16: return launch_tc<16>(A, Wq, scales, biases, out, out_mode, M, Kred, Nout, split, st);
        case 32: return launch_tc<32>(A, Wq, scales, biases, out, out_mode, M, Kred, Nout, split, st);
        case 64: return launch_tc<64>(A, Wq, scales, biases, out, out_mode, M, Kred, Nout, split, st);
        case 128: return launch_tc<128>(A, Wq, scales, biases, out, out_mode, M, Kred, Nout, split, st);
        case 256: return launch_tc<256>(A, Wq, scales, biases, out, out_mode, M, Kred, Nout, split, st);
        default: return cudaErrorInvalidValue;
    }
}

int read_tc_status(int* out, bool clear) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_tc_status, sizeof(int));
    if (e != cudaSuccess) return e;
    if (clear && v != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_tc_status, &zero, sizeof(int));
        if (e != cudaSuccess) return e;
    }
    *out = v;
    return cudaSuccess;
}

}  // namespace qmm
