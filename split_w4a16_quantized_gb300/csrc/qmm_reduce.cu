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

// Eight consecutive partial values of one plane: a 16-byte load (BF16) or two
// (FP32), kept raw until the ordered sum.
template <typename T>
struct Raw8;
template <>
struct Raw8<__nv_bfloat16> {
    uint4 u;
    __device__ __forceinline__ void load(const __nv_bfloat16* p) {
        u = __ldcs(reinterpret_cast<const uint4*>(p));
    }
    __device__ __forceinline__ void add_to(float acc[8]) const {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc[2 * i] += __uint_as_float(w[i] << 16);
            acc[2 * i + 1] += __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
};
template <>
struct Raw8<float> {
    float4 a, b;
    __device__ __forceinline__ void load(const float* p) {
        a = __ldcs(reinterpret_cast<const float4*>(p));
        b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
    }
    __device__ __forceinline__ void add_to(float acc[8]) const {
        acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
        acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
    }
};

__device__ __forceinline__ float load1(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ float load1(const float* p) { return *p; }

// KC planes' loads are in flight at once (KC >= split where possible, so the
// register footprint -- and the CTAs an SM holds -- follows the split).
template <typename T, int KC>
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
        // a chunk of KC planes' loads in flight at once, then the adds in
        // ascending plane order
        for (int p0 = 0; p0 < split; p0 += KC) {
            Raw8<T> r[KC];
#pragma unroll
            for (int q = 0; q < KC; ++q)
                if (p0 + q < split) r[q].load(partials + (p0 + q) * plane + i * 8);
#pragma unroll
            for (int q = 0; q < KC; ++q)
                if (p0 + q < split) r[q].add_to(acc);
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

// Several calls' reduces in one launch.  Work item w of the launch belongs to
// the call whose [begin, next begin) range holds it; a call with planes a
// multiple of eight long takes items of eight outputs, the others one.  Each
// output is the same ascending FP32 sum as in the kernels above.
struct RedItem {
    const void* partials;
    __nv_bfloat16* C;
    int64_t plane;  // M * Nout
    int64_t begin;  // first work item of the call
    int split;
    int vec;        // 1: items of eight outputs
};
struct RedGroup {
    int n;
    int64_t total;
    RedItem item[kMaxGroupCalls];
};

template <typename T>
__global__ void __launch_bounds__(256) reduce_group(const __grid_constant__ RedGroup g) {
    constexpr int KC = 8;
    pdl_trigger();
    pdl_wait();
    for (int64_t w = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; w < g.total;
         w += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        int c = 0;
        while (c + 1 < g.n && w >= g.item[c + 1].begin) ++c;
        const RedItem& it = g.item[c];
        const T* P = static_cast<const T*>(it.partials);
        const int64_t i = w - it.begin;
        if (it.vec) {
            float acc[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = 0.f;
            for (int p0 = 0; p0 < it.split; p0 += KC) {
                Raw8<T> r[KC];
#pragma unroll
                for (int q = 0; q < KC; ++q)
                    if (p0 + q < it.split) r[q].load(P + (p0 + q) * it.plane + i * 8);
#pragma unroll
                for (int q = 0; q < KC; ++q)
                    if (p0 + q < it.split) r[q].add_to(acc);
            }
            uint4 o;
            o.x = pack_bf16x2(acc[0], acc[1]);
            o.y = pack_bf16x2(acc[2], acc[3]);
            o.z = pack_bf16x2(acc[4], acc[5]);
            o.w = pack_bf16x2(acc[6], acc[7]);
            *reinterpret_cast<uint4*>(it.C + i * 8) = o;
        } else {
            float acc = 0.f;
            for (int p = 0; p < it.split; ++p) acc += load1(P + p * it.plane + i);
            it.C[i] = __float2bfloat16_rn(acc);
        }
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
    // one thread per eight outputs (grid-stride beyond 16 CTAs per SM)
    int64_t blocks = (work + 255) / 256;
    const int64_t max_blocks = static_cast<int64_t>(num_sms()) * 16;
    if (blocks > max_blocks) blocks = max_blocks;
    cudaLaunchConfig_t cfg = {};
    LaunchAttrs la;
    apply_pdl(cfg, la);
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    if (vec) {
        constexpr int kMax = sizeof(T) == 2 ? 16 : 8;
        if (split <= 2) return cudaLaunchKernelEx(&cfg, reduce_vec8<T, 2>, partials, split, plane, C);
        if (split <= 4) return cudaLaunchKernelEx(&cfg, reduce_vec8<T, 4>, partials, split, plane, C);
        if (split <= 8 || kMax == 8)
            return cudaLaunchKernelEx(&cfg, reduce_vec8<T, 8>, partials, split, plane, C);
        return cudaLaunchKernelEx(&cfg, reduce_vec8<T, kMax>, partials, split, plane, C);
    }
    return cudaLaunchKernelEx(&cfg, reduce_scalar<T>, partials, split, plane, C);
}

}  // namespace

int launch_reduce_group(const ReduceCall* calls, int n, int partial_dtype, void* stream) {
    if (n < 1 || n > kMaxGroupCalls) return cudaErrorInvalidValue;
    RedGroup g;
    g.n = n;
    int64_t total = 0;
    for (int i = 0; i < n; ++i) {
        RedItem& it = g.item[i];
        it.partials = calls[i].partials;
        it.C = static_cast<__nv_bfloat16*>(calls[i].C);
        it.plane = static_cast<int64_t>(calls[i].M) * calls[i].Nout;
        it.split = calls[i].split;
        it.vec = it.plane % 8 == 0 ? 1 : 0;
        it.begin = total;
        total += it.vec ? it.plane / 8 : it.plane;
    }
    g.total = total;
    int64_t blocks = (total + 255) / 256;
    const int64_t max_blocks = static_cast<int64_t>(num_sms()) * 16;
    if (blocks > max_blocks) blocks = max_blocks;
    cudaLaunchConfig_t cfg = {};
    LaunchAttrs la;
    apply_pdl(cfg, la);
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = static_cast<cudaStream_t>(stream);
    if (partial_dtype == QMM_PARTIAL_F32) return cudaLaunchKernelEx(&cfg, reduce_group<float>, g);
    return cudaLaunchKernelEx(&cfg, reduce_group<__nv_bfloat16>, g);
}

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
