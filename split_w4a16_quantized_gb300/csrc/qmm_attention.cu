// Split-KV decode attention for GB300 ("Optimize Prefill vs Decode Kernels",
// Required reasoning process, steps 4 and 5, Kernel design rules, and
// Correctness requirements): one query token per sequence attends to its KV
// history.  The history of each (sequence, KV head) is cut into S splits;
// each split's CTA computes a partial softmax state in FP32 -- the running
// maximum m, the sum l of the exponentials and the unnormalized output o --
// and a second kernel merges the states with the log-sum-exp correction.
// With S = 1 the CTA writes O.
//
// Layout: q BF16 [B, Hq, D]; K, V BF16 [B, Hkv, Lmax, D] (head-major, so a
// split's rows are contiguous); O BF16 [B, Hq, D].  Query head h reads KV
// head h / QG, QG = Hq / Hkv (grouped-query attention): one CTA serves the QG
// query heads of its KV head and reads each K and V row once for all of them.
//
// The op reads every KV byte once and is HBM-bound.  The page's decode
// recipe sizes the MMA's M axis by the query rows and fills its K axis with
// the head dimension, and the warp-level BF16 MMA (m16n8k16, FP32 accumulate)
// is what keeps the
// instruction count per position small enough for the memory stream: the QG
// heads are the M rows (padded to 16), keys and head dims the N and K axes,
// and the score accumulators become the A operand of P.V in registers
// (FlashAttention-2 style).  tcgen05 needs M >= 64, four to sixteen times the
// head count here.
//
// CTA (split s, KV head g, sequence b): 4 compute warps and one copy warp.
//   - The copy warp's lane 0 loads tiles of 64 positions of K and V into a
//     3-stage ring with 2-D TMA copies (boxes of 64 rows x 64 dims, 128-byte
//     swizzle, so the ldmatrix reads below are free of bank conflicts).
//   - Compute warp w takes positions 16w..16w+15 of a tile: S = Q K^T
//     (D/16 k-steps, two n-blocks of 8 positions), scaled by scale*log2(e);
//     positions past the split are masked to -inf; the warp's running max and
//     sum per head are updated (online softmax, exp2); o is rescaled and
//     P V accumulated with P split into two BF16 terms (hi + lo), so the
//     weights enter the product with about 16 bits.
//   - At the end the 4 warps' states are merged in shared memory.
// Every wait is bounded (1 s): a wait that runs out sets the status word and
// the CTA winds down after its copies in flight have landed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "qmm.h"
#include "qmm_device.cuh"
#include "qmm_internal.h"
#include "qmm_sm100.cuh"

namespace qmm {

// 2-D tensor map helper (qmm_w4a16_tc.cu)
bool encode_2d(CUtensorMap* map, CUtensorMapDataType type, const void* ptr, uint64_t rows,
               uint64_t cols, int elem, uint32_t box_rows, uint32_t box_cols,
               CUtensorMapSwizzle swizzle);

namespace {

constexpr int kTileKeys = 64;                          // positions per stage
constexpr int kAttnWarps = 4;                          // compute warps
constexpr int kKeysPerWarp = kTileKeys / kAttnWarps;   // 16
constexpr int kAttnStages = 3;
constexpr int kAttnThreads = 32 * (kAttnWarps + 1);    // + the copy warp
constexpr int kBox = 64 * 128;                         // one TMA box: 64 rows x 128 bytes

template <int D>
struct AttnCfg {
    static_assert(D == 64 || D == 128, "head dim");
    static constexpr int BOXES = D / 64;        // 64-dim boxes per tile
    static constexpr int TILE = BOXES * kBox;   // one K (or V) tile
    static constexpr int STAGE = 2 * TILE;      // K tile, then V tile
};

struct AttnParams {
    const __nv_bfloat16* q;
    const int* lens;
    __nv_bfloat16* O;
    float* pm;      // [B, Hq, S] partial maxima (scaled scores, log2 units)
    float* pl;      // [B, Hq, S] partial sums of exp2(score - m)
    float* po;      // [B, Hq, S, D] partial unnormalized outputs
    int* status;
    int Hq, Hkv, Lmax, S, chunk;  // chunk: positions per split, a multiple of 64
    float qscale;                 // scale * log2(e)
};

// Byte offset in a tile of the 16-byte chunk holding dims [d, d + 8) of row r:
// box d / 64, 128-byte rows, chunk (d % 64) / 8 swizzled with r % 8.
__device__ __forceinline__ uint32_t tile_off(int r, int d) {
    return static_cast<uint32_t>((d >> 6) * kBox + r * 128 + ((((d & 63) >> 3) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t r[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

template <int QG, int D>
struct AttnSmem {
    uint64_t full[kAttnStages];
    uint64_t empty[kAttnStages];
    float wm[kAttnWarps][QG];
    float wl[kAttnWarps][QG];
};

template <int QG, int D>
__global__ void __launch_bounds__(kAttnThreads, 2)
    attn_split_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const AttnParams p) {
    using C = AttnCfg<D>;
    using Sm = AttnSmem<QG, D>;
    constexpr int KS = D / 16;     // k-steps of S = Q K^T
    constexpr int NB = D / 8;      // n-blocks of P V
    extern __shared__ uint8_t attn_smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(attn_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Sm& sm = *reinterpret_cast<Sm*>(ring + kAttnStages * C::STAGE);
    __shared__ int abort_flag;
    volatile int* abort = &abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    pdl_trigger();
    if (tid == 0) {
        abort_flag = 0;
        for (int i = 0; i < kAttnStages; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], kAttnWarps);
        }
        mbar_fence_init();
        tma_prefetch_map(&kmap);
        tma_prefetch_map(&vmap);
    }
    pdl_wait();
    __syncthreads();
    int len = p.lens[b];
    len = len < 0 ? 0 : (len > p.Lmax ? p.Lmax : len);
    const int l0 = s * p.chunk;
    const int l1 = l0 + p.chunk < len ? l0 + p.chunk : len;
    const int ntiles = l1 > l0 ? (l1 - l0 + kTileKeys - 1) / kTileKeys : 0;
    const int row0 = (b * p.Hkv + g) * p.Lmax + l0;  // first row of the split

    if (warp == kAttnWarps) {
        // ---- copy warp ----
        if (lane == 0) {
            int t = 0;
            for (; t < ntiles; ++t) {
                const int st = t % kAttnStages;
                if (t >= kAttnStages &&
                    !mbar_wait(&sm.empty[st], ((t / kAttnStages) & 1) ^ 1, abort, p.status))
                    break;
                uint8_t* dst = ring + st * C::STAGE;
                const int y = row0 + t * kTileKeys;
                // the compute warps read the stage with ordinary loads
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(&sm.full[st], C::STAGE);
#pragma unroll
                for (int x = 0; x < C::BOXES; ++x) {
                    tma_load_2d(dst + x * kBox, &kmap, &sm.full[st], x * 64, y);
                    tma_load_2d(dst + C::TILE + x * kBox, &vmap, &sm.full[st], x * 64, y);
                }
            }
            if (*abort) {  // let the copies in flight land before the CTA exits
                for (int j = t > kAttnStages ? t - kAttnStages : 0; j < t; ++j)
                    mbar_wait(&sm.full[j % kAttnStages], (j / kAttnStages) & 1, nullptr,
                              p.status);
            }
        }
    } else {
        // ---- compute warps ----
        const int gr = lane >> 2, tq = lane & 3;  // fragment row (head), column pair
        // A operand of S: rows = heads (QG of 16 used), k = head dims
        uint32_t qa[KS][2];
        {
            const __nv_bfloat16* qv =
                p.q + (static_cast<size_t>(b) * p.Hq + g * QG + (gr < QG ? gr : 0)) * D;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const uint32_t lo = *reinterpret_cast<const uint32_t*>(qv + ks * 16 + 2 * tq);
                const uint32_t hi = *reinterpret_cast<const uint32_t*>(qv + ks * 16 + 8 + 2 * tq);
                qa[ks][0] = gr < QG ? lo : 0u;
                qa[ks][1] = gr < QG ? hi : 0u;
            }
        }
        float o[NB][4];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int i = 0; i < 4; ++i) o[nb][i] = 0.f;
        float m_run = -INFINITY, l_run = 0.f;  // of head `gr` (rows < QG)
        const uint32_t ring_a = smem_addr(ring);
        // ldmatrix row addresses: matrix j = lane / 8, row lane % 8
        const int mj = lane >> 3, mr = lane & 7;
        for (int t = 0; t < ntiles; ++t) {
            const int st = t % kAttnStages;
            if (!mbar_wait_warp(&sm.full[st], (t / kAttnStages) & 1, abort, p.status)) break;
            const int keys = l1 - l0 - t * kTileKeys < kTileKeys ? l1 - l0 - t * kTileKeys
                                                                  : kTileKeys;
            const int kb = warp * kKeysPerWarp;        // the warp's first position in the tile
            const int valid = keys - kb;
            if (valid > 0) {
                const uint32_t kt = ring_a + st * C::STAGE;
                const uint32_t vt = kt + C::TILE;
                // S = Q K^T for positions kb..kb+15: matrices (keys j/2, dims j%2)
                float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    uint32_t kf[4];
                    ldmatrix_x4(kf, kt + tile_off(kb + (mj >> 1) * 8 + mr, ks * 16 + (mj & 1) * 8));
                    const uint32_t a[4] = {qa[ks][0], 0u, qa[ks][1], 0u};
                    mma_bf16_16816(sc[0], a, kf[0], kf[1]);
                    mma_bf16_16816(sc[1], a, kf[2], kf[3]);
                }
                // online softmax of row `gr` over the 16 positions
                float x[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int pos = kb + (e >> 1) * 8 + 2 * tq + (e & 1);
                    const float v = sc[e >> 1][e & 1] * p.qscale;
                    x[e] = pos - kb < valid ? v : -INFINITY;
                }
                float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float mn = fmaxf(m_run, mx);
                const float corr = exp2f(m_run - mn);
                float pw[4], rs = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    pw[e] = exp2f(x[e] - mn);
                    rs += pw[e];
                }
                rs += __shfl_xor_sync(0xffffffffu, rs, 1);
                rs += __shfl_xor_sync(0xffffffffu, rs, 2);
                l_run = l_run * corr + rs;
                m_run = mn;
                // P as A operand (rows = heads, k = positions), two BF16 terms
                uint32_t ph[4], pl[4];
                {
                    const uint32_t h0 = pack_bf16x2(pw[0], pw[1]);
                    const uint32_t h1 = pack_bf16x2(pw[2], pw[3]);
                    float r[4];
                    r[0] = pw[0] - __uint_as_float(h0 << 16);
                    r[1] = pw[1] - __uint_as_float(h0 & 0xFFFF0000u);
                    r[2] = pw[2] - __uint_as_float(h1 << 16);
                    r[3] = pw[3] - __uint_as_float(h1 & 0xFFFF0000u);
                    ph[0] = h0; ph[1] = 0u; ph[2] = h1; ph[3] = 0u;
                    pl[0] = pack_bf16x2(r[0], r[1]); pl[1] = 0u;
                    pl[2] = pack_bf16x2(r[2], r[3]); pl[3] = 0u;
                }
                // o = o * corr + P V: matrices (keys j%2, dims j/2), transposed
#pragma unroll
                for (int db = 0; db < NB / 2; ++db) {
                    uint32_t vf[4];
                    ldmatrix_x4_trans(vf, vt + tile_off(kb + (mj & 1) * 8 + mr, db * 16 + (mj >> 1) * 8));
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        float* acc = o[2 * db + h];
                        acc[0] *= corr;
                        acc[1] *= corr;
                        mma_bf16_16816(acc, ph, vf[2 * h], vf[2 * h + 1]);
                        mma_bf16_16816(acc, pl, vf[2 * h], vf[2 * h + 1]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[st]);
        }
        // ---- merge the warps' states (the stage ring is free now) ----
        asm volatile("bar.sync 1, %0;\n" ::"n"(32 * kAttnWarps) : "memory");
        float* wo = reinterpret_cast<float*>(ring);  // [warp][QG][D]
        if (gr < QG) {
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
                wo[(warp * QG + gr) * D + nb * 8 + 2 * tq] = o[nb][0];
                wo[(warp * QG + gr) * D + nb * 8 + 2 * tq + 1] = o[nb][1];
            }
            if (tq == 0) {
                sm.wm[warp][gr] = m_run;
                sm.wl[warp][gr] = l_run;
            }
        }
        asm volatile("bar.sync 1, %0;\n" ::"n"(32 * kAttnWarps) : "memory");
        if (!*abort) {
            for (int e = tid; e < QG * D; e += 32 * kAttnWarps) {
                const int h = e / D, d = e % D;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, sm.wm[w][h]);
                float num = 0.f, den = 0.f;
                if (M != -INFINITY) {
#pragma unroll
                    for (int w = 0; w < kAttnWarps; ++w) {
                        const float f = exp2f(sm.wm[w][h] - M);
                        num = fmaf(f, wo[(w * QG + h) * D + d], num);
                        den = fmaf(f, sm.wl[w][h], den);
                    }
                }
                const size_t bh = static_cast<size_t>(b) * p.Hq + g * QG + h;
                if (p.S == 1) {
                    p.O[bh * D + d] = __float2bfloat16_rn(num / den);
                } else {
                    const size_t ps = bh * p.S + s;
                    p.po[ps * D + d] = num;
                    if (d == 0) {
                        p.pm[ps] = M;
                        p.pl[ps] = den;
                    }
                }
            }
        }
    }
    __syncthreads();
}

// O[b, h, :] = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s, M = max_s m_s,
// in ascending s; one block per (b, h), one thread per dim.
template <int D>
__global__ void __launch_bounds__(D) attn_merge_kernel(const float* __restrict__ pm,
                                                       const float* __restrict__ pl,
                                                       const float* __restrict__ po, int S,
                                                       __nv_bfloat16* __restrict__ O) {
    pdl_trigger();
    pdl_wait();
    const size_t bh = blockIdx.x;
    const int d = threadIdx.x;
    float M = -INFINITY;
    for (int s = 0; s < S; ++s) M = fmaxf(M, pm[bh * S + s]);
    float num = 0.f, den = 0.f;
    for (int s = 0; s < S; ++s) {
        const float m = pm[bh * S + s];
        if (m == -INFINITY) continue;  // an empty split
        const float f = exp2f(m - M);
        num = fmaf(f, po[(bh * S + s) * D + d], num);
        den = fmaf(f, pl[bh * S + s], den);
    }
    O[bh * D + d] = __float2bfloat16_rn(num / den);
}

template <int QG, int D>
int launch_attn(const CUtensorMap& kmap, const CUtensorMap& vmap, const AttnParams& p, int B,
                cudaStream_t st) {
    using C = AttnCfg<D>;
    auto kern = attn_split_kernel<QG, D>;
    // stages (1024-aligned for the 128-byte swizzle), then the barriers and
    // the warps' running maxima and sums
    const size_t smem = 1024 + static_cast<size_t>(kAttnStages) * C::STAGE +
                        sizeof(AttnSmem<QG, D>);
    static int ok = -1;
    static std::once_flag once;
    std::call_once(once, [&] {
        ok = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(smem)) == cudaSuccess;
    });
    if (ok != 1) return cudaErrorInvalidValue;
    // the warps' final states reuse the ring
    static_assert(kAttnWarps * QG * D * 4 <= kAttnStages * C::STAGE, "merge buffer");
    cudaLaunchConfig_t cfg = {};
    LaunchAttrs la;
    apply_pdl(cfg, la);
    cfg.gridDim = dim3(p.S, p.Hkv, B);
    cfg.blockDim = dim3(kAttnThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    int rc = cudaLaunchKernelEx(&cfg, kern, kmap, vmap, p);
    if (rc != cudaSuccess || p.S == 1) return rc;
    cudaLaunchConfig_t mc = {};
    LaunchAttrs mla;
    apply_pdl(mc, mla);
    mc.gridDim = dim3(static_cast<unsigned>(B) * p.Hq, 1, 1);
    mc.blockDim = dim3(D, 1, 1);
    mc.stream = st;
    return cudaLaunchKernelEx(&mc, attn_merge_kernel<D>, static_cast<const float*>(p.pm),
                              static_cast<const float*>(p.pl), static_cast<const float*>(p.po),
                              p.S, p.O);
}

template <int D>
int launch_attn_d(const CUtensorMap& kmap, const CUtensorMap& vmap, const AttnParams& p, int B,
                  int QG, cudaStream_t st) {
    switch (QG) {
        case 1: return launch_attn<1, D>(kmap, vmap, p, B, st);
        case 2: return launch_attn<2, D>(kmap, vmap, p, B, st);
        case 4: return launch_attn<4, D>(kmap, vmap, p, B, st);
        case 8: return launch_attn<8, D>(kmap, vmap, p, B, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int launch_decode_attention(const void* q, const void* K, const void* V, const int* lens, void* O,
                            float* ws, int B, int Hq, int Hkv, int Lmax, int D, float scale,
                            int S, void* stream) {
    int* status = tc_status_ptr();
    if (!status) return cudaErrorInvalidSymbol;
    // K and V as 2-D [B*Hkv*Lmax rows, D] with boxes of 64 rows x 64 dims
    const uint64_t rows = static_cast<uint64_t>(B) * Hkv * Lmax;
    CUtensorMap kmap, vmap;
    if (!encode_2d(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, rows, D, 2, 64, 64,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&vmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, V, rows, D, 2, 64, 64,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    AttnParams p;
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.lens = lens;
    p.O = static_cast<__nv_bfloat16*>(O);
    const size_t heads = static_cast<size_t>(B) * Hq * S;
    p.pm = S > 1 ? ws : nullptr;
    p.pl = S > 1 ? ws + heads : nullptr;
    p.po = S > 1 ? ws + 2 * heads : nullptr;
    p.status = status;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.Lmax = Lmax;
    p.S = S;
    const int per = (Lmax + S - 1) / S;
    p.chunk = (per + kTileKeys - 1) / kTileKeys * kTileKeys;
    p.qscale = scale * 1.4426950408889634f;  // log2(e): exp2 of the scaled score
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return D == 128 ? launch_attn_d<128>(kmap, vmap, p, B, Hq / Hkv, st)
                    : launch_attn_d<64>(kmap, vmap, p, B, Hq / Hkv, st);
}

}  // namespace qmm
