// Dense BF16 split-K GEMM C = A . W^T (gpu-kernels-explained, "Split-K,
// streams and overlap": 128 x 128 output tiles, k cut into `split` slices,
// FP32 partial planes added by a second pass).
//
// CTA tile 128 x 128 x 32, eight warps (2 x 4, warp tile 64 x 32), a 4-deep
// cp.async ring, ldmatrix fragment loads from XOR-swizzled 64-byte rows and
// mma.sync m16n8k16 with FP32 accumulation.  Slice p of the K/64 k-tiles
// is [t0, t0 + nt) with nt = T/split + (p < T mod split).
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qmm {
namespace {

constexpr int GB_M = 128, GB_N = 128, GB_K = 32, GB_STAGES = 4, GB_THREADS = 256;
constexpr int GB_TILE = GB_M * GB_K * 2;  // bytes of one operand tile (A and W alike)
constexpr int GB_SMEM = GB_STAGES * 2 * GB_TILE;

struct GemmParams {
    const uint16_t* A;  // [M, K]
    const uint16_t* W;  // [N, K]
    void* out;          // BF16 C or FP32 planes [split, M, N]
    int M, N, K, split, out_mode;
};

// byte offset of 16-byte chunk c (0..3) of tile row r
__device__ __forceinline__ int gb_off(int r, int c) { return r * 64 + ((c ^ ((r >> 1) & 3)) << 4); }

__global__ void __launch_bounds__(GB_THREADS) gemm_kernel(const GemmParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wm = warp >> 2, wn = warp & 3, g8 = lane >> 2, t4 = lane & 3;
    const int m0 = blockIdx.y * GB_M, n0 = blockIdx.x * GB_N, part = blockIdx.z;
    const int T = p.K / 64;
    const int nt = T / p.split + (part < T % p.split ? 1 : 0);
    const int t0 = part * (T / p.split) + (part < T % p.split ? part : T % p.split);
    const int kbeg = t0 * 64, nk = nt * 2;
    pdl_trigger();
    pdl_wait();

    auto load = [&](int i, int slot) {
        uint8_t* as = smem + slot * 2 * GB_TILE;
        uint8_t* bs = as + GB_TILE;
        const int k = kbeg + i * GB_K;
        for (int c = tid; c < GB_M * 4; c += GB_THREADS) {
            const int r = c >> 2, ch = c & 3;
            const int m = m0 + r, n = n0 + r;
            const bool okm = m < p.M, okn = n < p.N;
            cp_async16(smem_addr(as + gb_off(r, ch)),
                       p.A + static_cast<size_t>(okm ? m : 0) * p.K + k + ch * 8, okm);
            cp_async16(smem_addr(bs + gb_off(r, ch)),
                       p.W + static_cast<size_t>(okn ? n : 0) * p.K + k + ch * 8, okn);
        }
    };

    float acc[4][4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[a][b][c] = 0.f;

#pragma unroll
    for (int s = 0; s < GB_STAGES - 1; ++s) {
        if (s < nk) load(s, s);
        cp_async_commit();
    }
    for (int i = 0; i < nk; ++i) {
        cp_async_wait<GB_STAGES - 2>();
        __syncthreads();
        if (i + GB_STAGES - 1 < nk) load(i + GB_STAGES - 1, (i + GB_STAGES - 1) % GB_STAGES);
        cp_async_commit();
        const uint8_t* as = smem + (i % GB_STAGES) * 2 * GB_TILE;
        const uint8_t* bs = as + GB_TILE;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            uint32_t af[4][4], bf[2][4];
#pragma unroll
            for (int mi = 0; mi < 4; ++mi) {
                const int r = wm * 64 + mi * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
                ldmatrix_x4(af[mi], smem_addr(as + gb_off(r, 2 * ks + (lane >> 4))));
            }
#pragma unroll
            for (int nj = 0; nj < 2; ++nj) {
                const int r = wn * 32 + nj * 16 + (lane & 7) + 8 * (lane >> 4);
                ldmatrix_x4(bf[nj], smem_addr(bs + gb_off(r, 2 * ks + ((lane >> 3) & 1))));
            }
#pragma unroll
            for (int mi = 0; mi < 4; ++mi)
#pragma unroll
                for (int ni = 0; ni < 4; ++ni)
                    mma_bf16_16816(acc[mi][ni], af[mi], bf[ni >> 1][2 * (ni & 1)],
                                   bf[ni >> 1][2 * (ni & 1) + 1]);
        }
    }
    cp_async_wait<0>();

    const bool pair = (p.N & 1) == 0;
#pragma unroll
    for (int mi = 0; mi < 4; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int m = m0 + wm * 64 + mi * 16 + g8 + 8 * h;
                const int n = n0 + wn * 32 + ni * 8 + 2 * t4;
                if (m >= p.M || n >= p.N) continue;
                const float v0 = acc[mi][ni][2 * h], v1 = acc[mi][ni][2 * h + 1];
                const size_t o = static_cast<size_t>(m) * p.N + n;
                if (p.out_mode == kOutBf16) {
                    __nv_bfloat16* c = static_cast<__nv_bfloat16*>(p.out);
                    if (pair && n + 1 < p.N) {
                        *reinterpret_cast<uint32_t*>(c + o) = pack_bf16x2(v0, v1);
                    } else {
                        c[o] = __float2bfloat16_rn(v0);
                        if (n + 1 < p.N) c[o + 1] = __float2bfloat16_rn(v1);
                    }
                } else {
                    float* c = static_cast<float*>(p.out) + static_cast<size_t>(part) * p.M * p.N;
                    if (pair && n + 1 < p.N) {
                        *reinterpret_cast<float2*>(c + o) = make_float2(v0, v1);
                    } else {
                        c[o] = v0;
                        if (n + 1 < p.N) c[o + 1] = v1;
                    }
                }
            }
}

}  // namespace

int launch_gemm(const void* A, const void* W, void* out, int out_mode, int M, int N, int K,
                int split, void* stream) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        GB_SMEM);
    });
    if (attr_err != cudaSuccess) return attr_err;
    GemmParams p;
    p.A = static_cast<const uint16_t*>(A);
    p.W = static_cast<const uint16_t*>(W);
    p.out = out;
    p.M = M;
    p.N = N;
    p.K = K;
    p.split = split;
    p.out_mode = out_mode;
    cudaLaunchConfig_t cfg = {};
    LaunchAttrs la;
    apply_pdl(cfg, la);
    cfg.gridDim = dim3((N + GB_N - 1) / GB_N, (M + GB_M - 1) / GB_M, split);
    cfg.blockDim = dim3(GB_THREADS, 1, 1);
    cfg.dynamicSmemBytes = GB_SMEM;
    cfg.stream = static_cast<cudaStream_t>(stream);
    return cudaLaunchKernelEx(&cfg, gemm_kernel, p);
}

}  // namespace qmm
