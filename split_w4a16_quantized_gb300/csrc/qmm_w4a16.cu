// W4A16-g128 partition / unsplit matmul kernels (sm_103a).
//
// One CTA computes a BM x BN tile of C = A . W^T (BM activation rows, BN
// weight rows = output columns) over one partition of the reduction axis:
// groups [p*gpp, (p+1)*gpp) with gpp = (Kred/128)/split (tiny-llm book,
// "Week 2 Day 7: Split-K Prefill", Task 2: equal partitions on 128-group
// boundaries, grid z = partition); a split that does not divide the group
// count takes near-equal partitions, the first G mod split one group
// longer.  With split = 1 it writes C directly (the
// unsplit control); otherwise it writes its own partial plane [M, Nout] of
// the workspace with no atomics.
//
// Data path per 128-group ("Optimize Prefill vs Decode Kernels", kernel
// design rules: dequant fused into the main loop, 128-bit loads):
//   - the packed weight tile (BN rows x 64 B) and the activation tile
//     (BM rows x 256 B) stream into a STAGES-deep cp.async ring
//     (gpu-kernels-explained, "Split-K, streams and overlap": the load of
//     tile t+1 overlaps the compute of tile t);
//   - the activation tile is re-ordered once per CTA into the k order the
//     weight registers come out in (below) and XOR-swizzled so every 16-byte
//     fragment load is bank-conflict free;
//   - each thread dequantizes its own weight words in registers
//     (qmm_device.cuh: dequant_word) and feeds them as the A operand of
//     mma.sync m16n8k16 (16 weight rows x 16 k) against 8 activation rows;
//     the dequantized weight never touches shared or global memory.
//
// k order inside a 128-group.  Thread t of a quad owns packed words
// 4t..4t+3 of its two weight rows (one 16-byte load).  Word 4t+jj covers
// k0 = 32t + 8jj .. k0+7 and is spent on two MMA k-steps h = 0, 1:
//   step h: fragment slots (2t, 2t+1)   <- nibbles (2h,   2h+4)   of the word
//           fragment slots (2t+8, 2t+9) <- nibbles (2h+1, 2h+5)
// The activation operand must carry the same k in the same slots, so each
// 16-byte activation chunk (a0..a7 = A[m, k0..k0+7]) is stored as the four
// BF16 pairs (a0,a4) (a1,a5) (a2,a6) (a3,a7): one 16-byte shared load then
// yields the B fragments of both k-steps.  The reduction is a sum over k,
// so any k order used identically on both operands gives the same result.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qmm {
namespace {

struct W4Params {
    const uint16_t* A;       // BF16 bits [M, Kred]
    const uint32_t* Wq;      // [Nout, Kred/8]
    const uint16_t* scales;  // BF16 bits [Nout, G]
    const uint16_t* biases;  // BF16 bits [Nout, G]
    void* out;               // BF16 or FP32 planes [split, M, Nout]
    int M, Kred, Nout, G;
    int gpp;     // groups in the longest partition (sizes shared memory)
    int gq, gr;  // G / split, G % split: partition p holds gq + (p < gr) groups
    int out_mode;
};

template <int BM_, int WT_, int NW_, int STAGES_>
struct W4Cfg {
    static constexpr int BM = BM_;         // activation rows per CTA
    static constexpr int WT = WT_;         // 16-row weight tiles per warp
    static constexpr int NW = NW_;         // warps per CTA
    static constexpr int STAGES = STAGES_;
    static constexpr int BN = NW * 16 * WT;
    static constexpr int THREADS = NW * 32;
    static constexpr int W_STAGE = BN * 64;   // packed weight bytes of one group
    static constexpr int A_STAGE = BM * 256;  // activation bytes of one group
    static constexpr int STAGE = W_STAGE + A_STAGE;
    static constexpr int PERM = BM * 256;     // one re-ordered activation tile
    static constexpr int PIPE = STAGES * STAGE + 2 * PERM;
    static constexpr int EPI_LD = BN + 4;     // FP32 epilogue row pitch (floats)
    static constexpr int EPI = BM * EPI_LD * 4;
    static constexpr int FIXED = PIPE > EPI ? PIPE : EPI;
    static_assert(BM % 8 == 0 && STAGES >= 4, "tile");
};

// position of 16-byte chunk c (0..15) of activation row r in the re-ordered tile
__device__ __forceinline__ int perm_chunk(int r, int c) { return c ^ ((c >> 2) & 2) ^ (r & 1); }

template <class C>
__global__ void __launch_bounds__(C::THREADS) w4a16_kernel(const W4Params p) {
    constexpr int BM = C::BM, BN = C::BN, WT = C::WT, NT = BM / 8, STAGES = C::STAGES;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* pipe = smem;
    uint8_t* perm = smem + STAGES * C::STAGE;
    // per-group scales and biases of this CTA's rows: sc[gi * BN + r], bi[...]
    uint16_t* sc = reinterpret_cast<uint16_t*>(smem + C::FIXED);
    uint16_t* bi = sc + p.gpp * BN;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g8 = lane >> 2, t4 = lane & 3;
    const int n0 = blockIdx.x * BN, m0 = blockIdx.y * BM, part = blockIdx.z;
    const int ngrp = p.gq + (part < p.gr ? 1 : 0);
    const int gbeg = part * p.gq + (part < p.gr ? part : p.gr);
    const size_t wrow = static_cast<size_t>(p.Kred) / 8;  // words per weight row
    pdl_trigger();
    pdl_wait();

    auto load_stage = [&](int i, int slot) {
        const int grp = gbeg + i;
        uint8_t* ws = pipe + slot * C::STAGE;
        uint8_t* as = ws + C::W_STAGE;
        for (int c = tid; c < BN * 4; c += C::THREADS) {
            const int r = c >> 2, ch = c & 3, n = n0 + r;
            const bool ok = n < p.Nout;
            const uint32_t* src = p.Wq + static_cast<size_t>(ok ? n : 0) * wrow + grp * 16 + ch * 4;
            cp_async16(smem_addr(ws + r * 64 + ch * 16), src, ok);
        }
        for (int c = tid; c < BM * 16; c += C::THREADS) {
            const int r = c >> 4, ch = c & 15, m = m0 + r;
            const bool ok = m < p.M;
            const uint16_t* src =
                p.A + static_cast<size_t>(ok ? m : 0) * p.Kred + grp * kGroup + ch * 8;
            cp_async16(smem_addr(as + r * 256 + ch * 16), src, ok);
        }
    };

    auto reorder = [&](int slot, int buf) {
        const uint8_t* as = pipe + slot * C::STAGE + C::W_STAGE;
        uint8_t* pb = perm + buf * C::PERM;
        for (int c = tid; c < BM * 16; c += C::THREADS) {
            const int r = c >> 4, ch = c & 15;
            const uint4 v = *reinterpret_cast<const uint4*>(as + r * 256 + ch * 16);
            uint4 o;
            o.x = __byte_perm(v.x, v.z, 0x5410);  // (a0, a4)
            o.y = __byte_perm(v.x, v.z, 0x7632);  // (a1, a5)
            o.z = __byte_perm(v.y, v.w, 0x5410);  // (a2, a6)
            o.w = __byte_perm(v.y, v.w, 0x7632);  // (a3, a7)
            *reinterpret_cast<uint4*>(pb + r * 256 + perm_chunk(r, ch) * 16) = o;
        }
    };

    float acc[WT][NT][4];
#pragma unroll
    for (int a = 0; a < WT; ++a)
#pragma unroll
        for (int b = 0; b < NT; ++b)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[a][b][c] = 0.f;

    auto compute = [&](int slot, int buf, int i) {
        const uint8_t* ws = pipe + slot * C::STAGE;
        const uint8_t* pb = perm + buf * C::PERM;
        uint4 wv[WT][2];
        uint32_t ss[WT][2], bb[WT][2];
#pragma unroll
        for (int wt = 0; wt < WT; ++wt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int R = warp * 16 * WT + wt * 16 + g8 + 8 * h;
                wv[wt][h] = *reinterpret_cast<const uint4*>(ws + R * 64 + t4 * 16);
                ss[wt][h] = bf16_pair(sc[i * BN + R]);
                bb[wt][h] = bf16_pair(bi[i * BN + R]);
            }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            uint32_t w[WT][2][4];
#pragma unroll
            for (int wt = 0; wt < WT; ++wt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t word = jj == 0 ? wv[wt][h].x
                                        : jj == 1 ? wv[wt][h].y
                                        : jj == 2 ? wv[wt][h].z
                                                  : wv[wt][h].w;
                    dequant_word(word, ss[wt][h], bb[wt][h], w[wt][h]);
                }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int r = nt * 8 + g8;
                const uint4 b = *reinterpret_cast<const uint4*>(
                    pb + r * 256 + perm_chunk(r, 4 * t4 + jj) * 16);
#pragma unroll
                for (int wt = 0; wt < WT; ++wt) {
                    const uint32_t a0[4] = {w[wt][0][0], w[wt][1][0], w[wt][0][1], w[wt][1][1]};
                    const uint32_t a1[4] = {w[wt][0][2], w[wt][1][2], w[wt][0][3], w[wt][1][3]};
                    mma_bf16_16816(acc[wt][nt], a0, b.x, b.y);
                    mma_bf16_16816(acc[wt][nt], a1, b.z, b.w);
                }
            }
        }
    };

    // pipeline: commit c carries group c (empty past the end); before
    // iteration i the commits 0..i+1 must have landed.
#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
        if (s < ngrp) load_stage(s, s);
        cp_async_commit();
    }
    // scales and biases of this CTA's rows for every group of the partition,
    // loaded while the first copies are in flight
    for (int t = tid; t < 2 * BN; t += C::THREADS) {
        const int r = t % BN;
        load_group_row(t < BN ? p.scales : p.biases, p.Nout, p.G, n0 + r, gbeg, ngrp,
                       (t < BN ? sc : bi) + r, BN);
    }
    cp_async_wait<STAGES - 2>();
    __syncthreads();
    reorder(0, 0);
    for (int i = 0; i < ngrp; ++i) {
        cp_async_wait<STAGES - 3>();
        __syncthreads();
        if (i + STAGES - 1 < ngrp) load_stage(i + STAGES - 1, (i + STAGES - 1) % STAGES);
        cp_async_commit();
        if (i + 1 < ngrp) reorder((i + 1) % STAGES, (i + 1) & 1);
        compute(i % STAGES, i & 1, i);
    }
    cp_async_wait<0>();
    __syncthreads();

    // epilogue: stage the FP32 tile in shared memory, then 16-byte stores
    float* epi = reinterpret_cast<float*>(smem);
#pragma unroll
    for (int wt = 0; wt < WT; ++wt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int R = warp * 16 * WT + wt * 16 + g8;
            const int mr = nt * 8 + 2 * t4;
            epi[mr * C::EPI_LD + R] = acc[wt][nt][0];
            epi[(mr + 1) * C::EPI_LD + R] = acc[wt][nt][1];
            epi[mr * C::EPI_LD + R + 8] = acc[wt][nt][2];
            epi[(mr + 1) * C::EPI_LD + R + 8] = acc[wt][nt][3];
        }
    __syncthreads();

    const size_t plane = static_cast<size_t>(part) * p.M * p.Nout;
    if (p.out_mode == kOutBf16) {
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + plane;
        const bool vec = (p.Nout & 7) == 0;
        for (int idx = tid; idx < BM * (BN / 8); idx += C::THREADS) {
            const int ml = idx / (BN / 8), nl = (idx - ml * (BN / 8)) * 8;
            const int m = m0 + ml, n = n0 + nl;
            if (m >= p.M || n >= p.Nout) continue;
            const float* e = epi + ml * C::EPI_LD + nl;
            __nv_bfloat16* dst = out + static_cast<size_t>(m) * p.Nout + n;
            if (vec) {
                uint4 v;
                v.x = pack_bf16x2(e[0], e[1]);
                v.y = pack_bf16x2(e[2], e[3]);
                v.z = pack_bf16x2(e[4], e[5]);
                v.w = pack_bf16x2(e[6], e[7]);
                *reinterpret_cast<uint4*>(dst) = v;
            } else {
                for (int v = 0; v < 8 && n + v < p.Nout; ++v) dst[v] = __float2bfloat16_rn(e[v]);
            }
        }
    } else {
        float* out = static_cast<float*>(p.out) + plane;
        const bool vec = (p.Nout & 3) == 0;
        for (int idx = tid; idx < BM * (BN / 4); idx += C::THREADS) {
            const int ml = idx / (BN / 4), nl = (idx - ml * (BN / 4)) * 4;
            const int m = m0 + ml, n = n0 + nl;
            if (m >= p.M || n >= p.Nout) continue;
            const float* e = epi + ml * C::EPI_LD + nl;
            float* dst = out + static_cast<size_t>(m) * p.Nout + n;
            if (vec) {
                *reinterpret_cast<float4*>(dst) = make_float4(e[0], e[1], e[2], e[3]);
            } else {
                for (int v = 0; v < 4 && n + v < p.Nout; ++v) dst[v] = e[v];
            }
        }
    }
}

// Probe kernels: one warp per (16 weight rows, one group).  Lane (g8, t4)
// loads exactly the words the matmul kernels give it and writes every value
// back at the k it stands for.  The dequant probe takes the path the lean
// kernel takes for each scale (dequant_word_subnormal where the scale allows
// it, dequant_word otherwise).  The unpack probe forms each q twice, through
// dequant_word with scale 1 and bias 0 and through dequant_word_subnormal
// with scale 2^-10 (q * 2^-10 is exact), and writes 0xFF where they differ.
__global__ void probe_kernel(const uint32_t* __restrict__ Wq, const uint16_t* __restrict__ scales,
                             const uint16_t* __restrict__ biases, int Nout, int Kred,
                             uint8_t* __restrict__ q_out, __nv_bfloat16* __restrict__ w_out) {
    const int lane = threadIdx.x & 31, g8 = lane >> 2, t4 = lane & 3;
    const int grp = blockIdx.y, G = Kred / kGroup;
    const size_t wrow = static_cast<size_t>(Kred) / 8;
    constexpr uint16_t kTwoPowMinus10 = 0x3A80;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int n = blockIdx.x * 16 + g8 + 8 * h;
        if (n >= Nout) continue;
        const uint4 wv = *reinterpret_cast<const uint4*>(Wq + n * wrow + grp * 16 + t4 * 4);
        uint16_t s = 0, b = 0;
        if (w_out) {
            s = scales[static_cast<size_t>(n) * G + grp];
            b = biases[static_cast<size_t>(n) * G + grp];
        }
        const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            uint32_t w[4], u[4];
            if (w_out) {
                if (scale_subnormal_ok(s))
                    dequant_word_subnormal(words[jj], scale_shifted_pair(s, 133),
                                           scale_shifted_pair(s, 129), bf16_pair(b), w);
                else
                    dequant_word(words[jj], bf16_pair(s), bf16_pair(b), w);
            } else {
                dequant_word(words[jj], kBf16x2One, 0, w);
                dequant_word_subnormal(words[jj], scale_shifted_pair(kTwoPowMinus10, 133),
                                       scale_shifted_pair(kTwoPowMinus10, 129), 0, u);
            }
            const size_t k0 = static_cast<size_t>(n) * Kred + grp * kGroup + 32 * t4 + 8 * jj;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {  // e = 0: nibble i, e = 1: nibble i + 4
                    const uint16_t bits = static_cast<uint16_t>(w[i] >> (16 * e));
                    if (w_out) {
                        w_out[k0 + i + 4 * e] = __ushort_as_bfloat16(bits);
                    } else {
                        const float q1 = __bfloat162float(__ushort_as_bfloat16(bits));
                        const float q2 = __bfloat162float(__ushort_as_bfloat16(
                                             static_cast<uint16_t>(u[i] >> (16 * e)))) * 1024.0f;
                        q_out[k0 + i + 4 * e] = q1 == q2 ? static_cast<uint8_t>(q1) : 0xFFu;
                    }
                }
            }
        }
    }
}

template <class C>
int launch_cfg(const W4Params& p, int split, cudaStream_t stream) {
    auto kern = w4a16_kernel<C>;
    static int limit = -1;
    static std::once_flag once;
    std::call_once(once, [&] { limit = set_max_dynamic_smem(reinterpret_cast<const void*>(kern)); });
    if (limit < 0) return cudaErrorInvalidValue;
    const size_t smem = static_cast<size_t>(C::FIXED) + static_cast<size_t>(C::BN) * p.gpp * 4;
    if (limit < 0 || smem > static_cast<size_t>(limit)) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    LaunchAttrs la;
    apply_pdl(cfg, la);
    cfg.gridDim = dim3((p.Nout + C::BN - 1) / C::BN, (p.M + C::BM - 1) / C::BM, split);
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

// Family table entries (qmm_internal.h: kFamilies) -> kernel configurations.
using Fam0 = W4Cfg<8, 1, 4, 4>;    // M <= 8:  BM 8,  BN 64
using Fam1 = W4Cfg<16, 1, 4, 4>;   // M <= 16: BM 16, BN 64
using Fam2 = W4Cfg<32, 2, 4, 4>;   // M <= 32: BM 32, BN 128
using Fam3 = W4Cfg<64, 1, 8, 4>;   // larger:  BM 64, BN 128
static_assert(Fam0::BM == kMmaFamilies[0].bm && Fam0::BN == kMmaFamilies[0].bn, "family 0");
static_assert(Fam1::BM == kMmaFamilies[1].bm && Fam1::BN == kMmaFamilies[1].bn, "family 1");
static_assert(Fam2::BM == kMmaFamilies[2].bm && Fam2::BN == kMmaFamilies[2].bn, "family 2");
static_assert(Fam3::BM == kMmaFamilies[3].bm && Fam3::BN == kMmaFamilies[3].bn, "family 3");

}  // namespace

int launch_w4a16(const Family& fam, const void* A, const uint32_t* Wq, const void* scales,
                 const void* biases, void* out, int out_mode, int M, int Kred, int Nout,
                 int split, void* stream, void* fused_C, uint32_t* counters) {
    if (fam.kind == kKindTc)
        return launch_w4a16_tc(fam.bm, A, Wq, scales, biases, out, out_mode, M, Kred, Nout, split,
                               stream, fused_C, counters);
    if (fam.kind == kKindLean)
        return launch_w4a16_lean(fam.bm, A, Wq, scales, biases, out, out_mode, M, Kred, Nout,
                                 split, stream, fused_C, counters);
    if (fused_C) return cudaErrorInvalidValue;
    W4Params p;
    p.A = static_cast<const uint16_t*>(A);
    p.Wq = Wq;
    p.scales = static_cast<const uint16_t*>(scales);
    p.biases = static_cast<const uint16_t*>(biases);
    p.out = out;
    p.M = M;
    p.Kred = Kred;
    p.Nout = Nout;
    p.G = Kred / kGroup;
    p.gq = p.G / split;
    p.gr = p.G % split;
    p.gpp = p.gq + (p.gr ? 1 : 0);
    p.out_mode = out_mode;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (fam.bm) {
        case Fam0::BM: return launch_cfg<Fam0>(p, split, st);
        case Fam1::BM: return launch_cfg<Fam1>(p, split, st);
        case Fam2::BM: return launch_cfg<Fam2>(p, split, st);
        default: return launch_cfg<Fam3>(p, split, st);
    }
}

static int launch_probe(const uint32_t* Wq, const void* scales, const void* biases, int Nout,
                        int Kred, uint8_t* q, void* w, void* stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((Nout + 15) / 16, Kred / kGroup, 1);
    cfg.blockDim = dim3(32, 1, 1);
    cfg.stream = static_cast<cudaStream_t>(stream);
    return cudaLaunchKernelEx(&cfg, probe_kernel, Wq, static_cast<const uint16_t*>(scales),
                              static_cast<const uint16_t*>(biases), Nout, Kred, q,
                              static_cast<__nv_bfloat16*>(w));
}

int launch_unpack_probe(const uint32_t* Wq, int Nout, int Kred, uint8_t* q, void* stream) {
    return launch_probe(Wq, nullptr, nullptr, Nout, Kred, q, nullptr, stream);
}

int launch_dequant_probe(const uint32_t* Wq, const void* scales, const void* biases, int Nout,
                         int Kred, void* w, void* stream) {
    return launch_probe(Wq, scales, biases, Nout, Kred, nullptr, w, stream);
}

}  // namespace qmm
