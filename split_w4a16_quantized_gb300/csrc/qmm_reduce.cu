// Split-K reduce (tiny-llm book, "Week 2 Day 7: Split-K Prefill", Task 4):
// C[m, n] = BF16(sum_p partial[p, m, n]), summed in FP32 in ascending p and
// rounded once.  The planes are contiguous [split, M, Nout]; the kernel
// treats them as flat vectors of M*Nout elements.  Each thread owns eight
// consecutive outputs (16-byte loads of every plane, one 16-byte store);
// a scalar path serves plane lengths that are not a multiple of eight.
// The grid is sized in multiples of the SM count and strides over the rest.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "qmm.h"
#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qmm {
namespace {

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float v[8]) {
    const uint4 u = __ldcs(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ void load8(const float* p, float v[8]) {
    const float4 a = __ldcs(reinterpret_cast<const float4*>(p));
    const float4 b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ float load1(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ float load1(const float* p) { return *p; }

template <typename T>
__global__ void __launch_bounds__(256) reduce_vec8(const T* __restrict__ partials, int split,
                                                   int64_t plane, __nv_bfloat16* __restrict__ C) {
    const int64_t nvec = plane / 8;
    pdl_trigger();
    pdl_wait();
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < nvec;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.f;
        // up to eight planes' loads in flight at once, then added in
        // ascending plane order (the sum's order does not change)
        for (int p0 = 0; p0 < split; p0 += 8) {
            float v[8][8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (p0 + q < split) load8(partials + (p0 + q) * plane + i * 8, v[q]);
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (p0 + q < split) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[j] += v[q][j];
                }
        }
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        *reinterpret_cast<uint4*>(C + i * 8) = o;
    }
}

template <typename T>
__global__ void __launch_bounds__(256) reduce_scalar(const T* __restrict__ partials, int split,
                                                     int64_t plane, __nv_bfloat16* __restrict__ C) {
    pdl_trigger();
    pdl_wait();
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < plane;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float acc = 0.f;
        for (int p = 0; p < split; ++p) acc += load1(partials + p * plane + i);
        C[i] = __float2bfloat16_rn(acc);
    }
}

int num_sms() {
    static int sms = 0;
    static std::once_flag once;
    std::call_once(once, [] {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            sms = 148;
    });
    return sms;
}

template <typename T>
int launch_typed(const T* partials, int split, int64_t plane, __nv_bfloat16* C,
                 cudaStream_t stream) {
    const bool vec = plane % 8 == 0;
    const int64_t work = vec ? plane / 8 : plane;
    int64_t blocks = (work + 255) / 256;
    const int64_t max_blocks = static_cast<int64_t>(num_sms()) * 8;
    if (blocks > max_blocks) blocks = max_blocks;
    cudaLaunchConfig_t cfg = {};
    LaunchAttrs la;
    apply_pdl(cfg, la);
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    if (vec) return cudaLaunchKernelEx(&cfg, reduce_vec8<T>, partials, split, plane, C);
    return cudaLaunchKernelEx(&cfg, reduce_scalar<T>, partials, split, plane, C);
}

}  // namespace

int launch_reduce(const void* partials, int partial_dtype, int split, int M, int Nout, void* C,
                  void* stream) {
    const int64_t plane = static_cast<int64_t>(M) * Nout;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    __nv_bfloat16* c = static_cast<__nv_bfloat16*>(C);
    if (partial_dtype == QMM_PARTIAL_F32)
        return launch_typed(static_cast<const float*>(partials), split, plane, c, st);
    return launch_typed(static_cast<const __nv_bfloat16*>(partials), split, plane, c, st);
}

}  // namespace qmm
