// W4A16-g128 partition / unsplit matmul on the 5th-generation tensor cores
// (tcgen05, sm_103a).
//
// A CTA owns 128 weight rows (output columns n0..n0+127) x BNA activation
// rows (m0..m0+BNA-1) over one partition of the reduction axis (tiny-llm
// book, "Week 2 Day 7: Split-K Prefill", Task 2: grid z = partition, equal
// partitions on 128-group boundaries, each writes its own partial plane, no
// atomics).  A split that does not divide the group count takes near-equal
// partitions, the first G mod split one group longer.  The product is
// computed transposed, C^T tile = W . A^T:
//   - MMA A operand = dequantized weights, 128 rows x 16 k, held in TENSOR
//     MEMORY (lane = weight row).  The weights go packed HBM -> shared memory
//     (TMA) -> registers (unpack + dequant) -> tensor memory (tcgen05.st);
//     BF16 weights never travel through shared memory, whose bandwidth a
//     dequantized operand would otherwise exhaust at HBM rate.
//   - MMA B operand = activations, BNA rows x 16 k, loaded by TMA into
//     128-byte-swizzled shared memory (K-major).
//   - D = FP32 accumulators in tensor memory, 128 lanes x BNA columns each.
// Warp roles (16 warps):
//   warp 0      TMA producer (one thread): packed weights into a deep ring
//               the dequantizers release on read, activation tiles into a
//               ring the MMAs release;
//   warps 1..N  MMA issuers (N = 3, 2 or 1 by tile width), each owning every
//               N-th group and its own accumulator; warp 1 also allocates
//               tensor memory.  An issuing thread spends tens of nanoseconds
//               per tcgen05.mma, so narrow tiles need several issuers; the
//               accumulators are added in a fixed order in the epilogue, so
//               results stay deterministic;
//   warps 4-15  three dequantizer sets of four warps (warp w serves tensor
//               memory lanes 32*(w%4).. and every third group), then the
//               epilogue.  A weight row's group is dequantized with one BF16
//               fused multiply-add per pair of weights where its scale allows
//               (dequant_row_group_sub, tiles up to 128 rows), else with two.
// Every mbarrier wait is bounded (qmm_sm100.cuh): a wait that runs out sets
// the status word, the CTA stops issuing work, waits (bounded) for what is in
// flight, frees its tensor memory and exits.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
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

// rank-dimensional tiled map (dims[0] innermost; strides in bytes of dims 1..)
bool encode_tiled(CUtensorMap* map, CUtensorMapDataType type, int rank, const void* ptr,
                  const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                  CUtensorMapSwizzle swizzle) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return fn(map, type, static_cast<cuuint32_t>(rank), const_cast<void*>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
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

constexpr int kWRows = 128;            // weight rows per CTA (MMA M)
constexpr int kWGroup = kWRows * 64;   // packed weight bytes of one group
constexpr int kWBox = 2 * kWGroup;     // one weight copy: 128 rows x two groups
constexpr int kMaxWStages = 16;
constexpr int kMaxActStages = 16;
constexpr int kMaxAStages = 8;
constexpr int kCtlWarps = 4;           // producer, MMA issuers, allocator

// Ring position of group i: stage j = i / gps, slot j % n, phase (j / n) & 1.
// The divisions use multiply-high by a host-computed reciprocal (exact for
// the small j of one partition), so the control warps -- which share their
// schedulers with busy dequantizer warps -- spend few instructions per group.
struct Ring {
    int n;          // stages
    uint32_t magic; // ceil(2^32 / n)
    int gps_log2;   // groups per stage = 1 << gps_log2
};
__device__ __forceinline__ void ring_pos(const Ring& r, int i, int& slot, uint32_t& phase,
                                         int& within) {
    const uint32_t j = static_cast<uint32_t>(i) >> r.gps_log2;
    const uint32_t q = __umulhi(j, r.magic);
    slot = static_cast<int>(j - q * r.n);
    phase = q & 1u;
    within = i & ((1 << r.gps_log2) - 1);
}

struct TcParams {
    const uint16_t* scales;
    const uint16_t* biases;
    void* out;
    int* status;
    int M, Kred, Nout, G, out_mode;
    int gpp;        // groups in the longest partition (sizes the rings)
    int split;      // partitions of the reduction axis
    int gq, gr;     // G / split, G % split: partition p holds gq + (p < gr) groups
    int weights_static;  // 1: only the activation copies wait for earlier kernels
    int fused;           // 1: the last CTA of an output tile adds its planes into C
    void* C;             // BF16 [M, Nout] (fused reduce)
    uint32_t* counters;  // one per output tile (fused reduce), zero between calls
    int tma_store;  // 1: the output tile leaves through a TMA store of a staged tile
    int cluster;    // 1: the tile's partitions are one cluster and add their staged
                    //    partial tiles through distributed shared memory into C
    Ring wr, ar;    // weight ring, activation ring (same groups per stage)
};

constexpr int ct_gcd(int a, int b) { return b == 0 ? a : ct_gcd(b, a % b); }

template <int BNA>
struct TcCfg {
    static_assert(BNA % 16 == 0 && BNA >= 16 && BNA <= 256, "MMA N");
    static constexpr int ACT_BOX = BNA * 128;       // one 64-k activation chunk
    static constexpr int ACT_GROUP = 2 * ACT_BOX;   // one 128-group
    // MMA issuers, each with its own accumulator: an issuing thread spends
    // tens of nanoseconds per tcgen05.mma, about the tensor time of an N = 128
    // MMA, so tiles up to N = 128 spread the issue over threads
    static constexpr int NACC = BNA <= 32 ? 3 : BNA <= 128 ? 2 : 1;
    // dequantizer warp sets of four warps (one per tensor-memory lane
    // quarter); wide tiles spend more tensor time per group, so two sets keep
    // up and leave tensor memory for two-deep A buffers per set
    static constexpr int DSETS = BNA <= 64 ? 3 : 2;
    static constexpr int THREADS = 32 * (kCtlWarps + 4 * DSETS);
    static constexpr int DCOLS = NACC * BNA;
    // tensor memory: accumulators in [0, DCOLS), then A buffers of 64 columns
    // (one 128-group of weights: 128 lanes x 128 k BF16)
    static constexpr int ACOL = DCOLS <= 64 ? 64 : (DCOLS + 63) / 64 * 64;
    // Group i goes to A buffer i % A_STAGES, dequantizer set i % DSETS and
    // issuer i % NACC.  A_STAGES is a multiple of lcm(DSETS, NACC), so every
    // buffer has one writing set and one issuer, each of which passes every
    // lap of its barriers: a parity wait is then never satisfied by a
    // completion two laps old, which a buffer shared round-robin between sets
    // would allow.
    static constexpr int A_LCM = DSETS / ct_gcd(DSETS, NACC) * NACC;
    static constexpr int A_AVAIL = (512 - ACOL) / 64 < 6 ? (512 - ACOL) / 64 : 6;
    static constexpr int A_STAGES = A_AVAIL / A_LCM * A_LCM;
    static constexpr int TMEM_COLS = 512;
    static constexpr uint32_t IDESC = idesc_bf16_f32(kWRows, BNA);
    // groups per TMA stage: one copy of several groups amortizes the
    // producer's barrier work over more bytes
    // (weight stages of four groups: the producer's proxy fence and copy
    // are paid once per four groups; activation stages are as small as the
    // activation ring's depth needs.  The 256-row tile is the exception: its
    // activations are 64 KB a group against 8 KB of weights, so its weight
    // stages hold two groups and the shared memory goes to a third
    // activation stage)
    static constexpr int WGPS_LOG2 = BNA == 256 ? 1 : 2;
    static constexpr int WGPS = 1 << WGPS_LOG2;
    static constexpr int AGPS_LOG2 = BNA <= 32 ? 2 : BNA <= 64 ? 1 : 0;
    static constexpr int AGPS = 1 << AGPS_LOG2;
    static constexpr int W_STAGE = WGPS * kWGroup;
    static constexpr int ACT_STAGE = AGPS * ACT_GROUP;
    static_assert(A_STAGES >= DSETS && A_STAGES <= kMaxAStages && A_STAGES % A_LCM == 0,
                  "A ring");
    static_assert(NACC <= kCtlWarps - 1, "issuer warps");
};

// pair (q[2c], q[2c+1]) of a packed word as BF16 (128 + q): byte c of x holds
// both nibbles; byte c of x >> 4 has the odd one in its low nibble.
__device__ __forceinline__ uint32_t natural_pair(uint32_t x, uint32_t x4, uint32_t sel) {
    return nibbles_to_bf16x2_biased(__byte_perm(x, x4, sel));
}

// 64 BF16 pairs of one weight row and group, in k order (pair c = k 2c, 2c+1),
// with one fused multiply-add per pair: each half keeps only its nibble, which
// then reads as the BF16 subnormal q * 2^-133, and s133 is the scale times
// 2^133 (scale_shifted_pair), so the FMA forms q * scale + bias with a single
// rounding -- the value dequant_row_group forms in two steps.  For scales that
// scale_subnormal_ok accepts.
__device__ __forceinline__ void dequant_row_group_sub(const uint4 wv[4], uint32_t s133,
                                                      uint32_t bb, uint32_t out[64]) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const uint32_t x = j % 4 == 0 ? wv[j / 4].x : j % 4 == 1 ? wv[j / 4].y
                         : j % 4 == 2 ? wv[j / 4].z : wv[j / 4].w;
        const uint32_t x4 = x >> 4;
        const uint32_t sel[4] = {0x4400u, 0x5511u, 0x6622u, 0x7733u};
#pragma unroll
        for (int c = 0; c < 4; ++c)
            out[4 * j + c] = fma_bf16x2(__byte_perm(x, x4, sel[c]) & 0x000F000Fu, s133, bb);
    }
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

// A ring of n stages of gps groups each, its groups dealt round-robin to
// `users` consumers (dequantizer sets or MMA issuers), waits by parity: a
// consumer's wait on lap L of a slot is sound only if it also waited on lap
// L - 1 of that slot.  That holds when every stage holds a group of every
// consumer, or when n * gps is a multiple of the consumer count (the stage
// one lap back then holds the same consumers' groups).
__host__ __device__ constexpr bool ring_laps_ok(int n, int gps, int users) {
    return gps >= users || (n * gps) % users == 0;
}

// Shared-memory carve-up of one CTA (base 1024-aligned).
struct TcSmem {
    uint8_t* act;       // ar.n x ACT_STAGE
    uint8_t* w;         // wr.n x W_STAGE
    uint64_t* w_full;   // [kMaxWStages]
    uint64_t* w_empty;
    uint64_t* act_full; // [kMaxActStages]
    uint64_t* act_empty;
    uint64_t* a_full;   // [kMaxAStages]
    uint64_t* a_empty;
    uint64_t* acc_full;
    uint32_t* tmem_slot;
};

__host__ __device__ constexpr size_t tc_bar_bytes() {
    return (2 * kMaxWStages + 2 * kMaxActStages + 2 * kMaxAStages + 1) * 8 + 16;
}

template <int BNA>
__device__ __forceinline__ TcSmem carve(uint8_t* base, const TcParams& p) {
    using C = TcCfg<BNA>;
    TcSmem s;
    s.act = base;
    s.w = s.act + p.ar.n * C::ACT_STAGE;
    uint64_t* b = reinterpret_cast<uint64_t*>(s.w + p.wr.n * C::W_STAGE);
    s.w_full = b;
    s.w_empty = b + kMaxWStages;
    s.act_full = b + 2 * kMaxWStages;
    s.act_empty = s.act_full + kMaxActStages;
    s.a_full = s.act_empty + kMaxActStages;
    s.a_empty = s.a_full + kMaxAStages;
    s.acc_full = s.a_empty + kMaxAStages;
    s.tmem_slot = reinterpret_cast<uint32_t*>(s.acc_full + 1);
    return s;
}

// Producer (one thread): per weight stage, two 2-D TMA copies of two groups
// each (128 rows x 128 bytes, the 128-byte swizzle) into the weight ring
// (released by the dequantizers as soon as they have read it) and, per AGPS
// groups, one copy of the matching activation chunks into the activation ring
// (released by the MMA commits).  Both rings are polled without blocking, so
// neither waits behind the other.  Weight rows of 128 bytes halve the TMA
// requests of 64-byte rows; a box that runs past the end of a weight row is
// zero-filled.  The partition holds gpp groups from group gbeg on.
template <int BNA>
__device__ __forceinline__ void tc_producer(const TcSmem& sm, const TcParams& p,
                                            const CUtensorMap* wmap, const CUtensorMap* amap,
                                            const CUtensorMap* amap_1, int n0, int m0, int gbeg,
                                            int gpp, volatile int* abort) {
    using C = TcCfg<BNA>;
    const int nw = (gpp + C::WGPS - 1) >> C::WGPS_LOG2;
    const int na = (gpp + C::AGPS - 1) >> C::AGPS_LOG2;
    // a last activation stage of fewer than AGPS groups is filled one group
    // at a time through the one-group map; a last weight stage of one or two
    // groups takes one two-group box
    constexpr int kBoxes = C::WGPS / 2;  // two-group boxes per weight stage
    const int wtail = gpp & (C::WGPS - 1), atail = gpp & (C::AGPS - 1);
    const int alast = atail ? na - 1 : na;
    const int wlast_boxes = wtail == 0 ? kBoxes : (wtail + 1) >> 1;
    int jw = 0, ja = 0, sw = 0, sa = 0;
    uint32_t pw = 0, pa = 0;
    auto issue_w = [&]() {
        // the dequantizers read this stage with ordinary loads
        fence_proxy_async_smem();
        const int boxes = jw == nw - 1 ? wlast_boxes : kBoxes;
        const int x = (gbeg + jw * C::WGPS) * 16;  // 32-bit words
        mbar_arrive_expect_tx(&sm.w_full[sw], boxes * kWBox);
        tma_load_2d(sm.w + sw * C::W_STAGE, wmap, &sm.w_full[sw], x, n0);
        if (boxes == 2)
            tma_load_2d(sm.w + sw * C::W_STAGE + kWBox, wmap, &sm.w_full[sw], x + 32, n0);
        ++jw;
        if (++sw == p.wr.n) { sw = 0; pw ^= 1; }
    };
    if (p.weights_static) {
        // static weights: every weight slot is filled (and dequantized by the
        // sets) before the wait for the earlier kernels; only the activation
        // copies come after it
        while (jw < nw && jw < p.wr.n) issue_w();
        pdl_wait();
    }
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t spin = 0; jw < nw || ja < na; ++spin) {
        bool progress = false;
        if (jw < nw && mbar_probe(&sm.w_empty[sw], pw ^ 1)) {
            issue_w();
            progress = true;
        }
        if (ja < na && mbar_probe(&sm.act_empty[sa], pa ^ 1)) {
            const int g = gbeg + ja * C::AGPS;
            uint8_t* dst = sm.act + sa * C::ACT_STAGE;
            if (ja == alast) {
                mbar_arrive_expect_tx(&sm.act_full[sa], atail * C::ACT_GROUP);
                for (int t = 0; t < atail; ++t)
                    tma_load_3d(dst + t * C::ACT_GROUP, amap_1, &sm.act_full[sa], 0, m0,
                                (g + t) * 2);
            } else {
                mbar_arrive_expect_tx(&sm.act_full[sa], C::ACT_STAGE);
                tma_load_3d(dst, amap, &sm.act_full[sa], 0, m0, g * 2);
            }
            ++ja;
            if (++sa == p.ar.n) { sa = 0; pa ^= 1; }
            progress = true;
        }
        if (!progress && (spin & 255u) == 0) {
            if (*abort) break;
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                *abort = 1;
                atomicExch(p.status, kStatusTimeout);
                break;
            }
        }
    }
    if (*abort) {  // let copies in flight land before the CTA exits
        for (int j = jw > p.wr.n ? jw - p.wr.n : 0; j < jw; ++j)
            mbar_wait(&sm.w_full[j % p.wr.n], (j / p.wr.n) & 1, nullptr, p.status);
        for (int j = ja > p.ar.n ? ja - p.ar.n : 0; j < ja; ++j)
            mbar_wait(&sm.act_full[j % p.ar.n], (j / p.ar.n) & 1, nullptr, p.status);
    }
}

// MMA issuer c (one thread): groups c, c + NACC, ... into accumulator c.
template <int BNA>
__device__ __forceinline__ void tc_issuer(const TcSmem& sm, const TcParams& p, uint32_t tmem,
                                          int c, int gpp, volatile int* abort) {
    using C = TcCfg<BNA>;
    const uint32_t d_tm = tmem + c * BNA;
    for (int i = c; i < gpp; i += C::NACC) {
        int sa, within;
        uint32_t ph;
        ring_pos(p.ar, i, sa, ph, within);
        const int ab = i % C::A_STAGES;
        if (!mbar_wait(&sm.act_full[sa], ph, abort, p.status)) break;
        if (!mbar_wait(&sm.a_full[ab], (i / C::A_STAGES) & 1, abort, p.status)) break;
        tc_fence_after();
        const uint32_t a_tm = tmem + C::ACOL + ab * 64;
        const uint64_t b0 =
            sdesc_kmajor_sw128(smem_addr(sm.act + sa * C::ACT_STAGE + within * C::ACT_GROUP));
        const uint32_t acc = i != c;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // k step of 16: +32 bytes in the swizzle atom
            umma_bf16_tmem_a(d_tm, a_tm + kk * 8,
                             b0 + ((((kk >> 2) * C::ACT_BOX) + (kk & 3) * 32) >> 4), C::IDESC,
                             acc | (kk != 0));
        umma_commit(&sm.act_empty[sa]);
        umma_commit(&sm.a_empty[ab]);
    }
    umma_commit(sm.acc_full);
}

// Dequantizer warp of lane quarter `quarter` in set `set`: groups set,
// set + DSETS, ...; weight row = 32 * quarter + lane.
template <int BNA>
__device__ __forceinline__ void tc_dequant(const TcSmem& sm, const TcParams& p, uint32_t tmem,
                                           int quarter, int set, int lane, int n0, int gbeg,
                                           int gpp, volatile int* abort) {
    using C = TcCfg<BNA>;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    // this row's scale and bias, fetched one of the set's groups ahead so the
    // load overlaps the previous group (rows past Nout dequantize to zero)
    const bool live = n0 + row < p.Nout;
    const size_t gp = static_cast<size_t>(live ? n0 + row : 0) * p.G + gbeg;
    uint16_t s_next = 0, b_next = 0;
    if (live && set < gpp) {
        s_next = __ldg(p.scales + gp + set);
        b_next = __ldg(p.biases + gp + set);
    }
    for (int i = set; i < gpp; i += C::DSETS) {
        const uint16_t s_cur = s_next, b_cur = b_next;
        if (live && i + C::DSETS < gpp) {
            s_next = __ldg(p.scales + gp + i + C::DSETS);
            b_next = __ldg(p.biases + gp + i + C::DSETS);
        }
        int sw, within;
        uint32_t ph;
        ring_pos(p.wr, i, sw, ph, within);
        const int ab = i % C::A_STAGES;
        if (!mbar_wait_warp(&sm.w_full[sw], ph, abort, p.status)) break;
        // box `within / 2`, row of 128 bytes, 16-byte chunks 4*(within % 2) ..
        // +3 under the 128-byte swizzle (chunk k of row r at k ^ (r % 8))
        const uint8_t* wr = sm.w + sw * C::W_STAGE + (within >> 1) * kWBox + row * 128;
        uint4 wv[4];
#pragma unroll
        for (int c = 0; c < 4; ++c)
            wv[c] = *reinterpret_cast<const uint4*>(
                wr + ((((within & 1) << 2) + c) ^ (row & 7)) * 16);
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.w_empty[sw]);
        uint32_t w[64];
        // the one-FMA form where the scale allows, up to 128-row tiles (at the
        // 256-row tile it measured slower: down at M = 2048, 106 against 102.5 us)
        if (BNA <= 128 && scale_subnormal_ok(s_cur))
            dequant_row_group_sub(wv, scale_shifted_pair(s_cur, 133), bf16_pair(b_cur), w);
        else
            dequant_row_group(wv, bf16_pair(s_cur), bf16_pair(b_cur), w);
        if (!mbar_wait_warp(&sm.a_empty[ab], ((i / C::A_STAGES) & 1) ^ 1, abort, p.status)) break;
        // the stores below must follow the MMAs that read this buffer before
        tc_fence_after();
        const uint32_t ta = tmem + lane_base + C::ACOL + ab * 64;
        tmem_st16(ta + 0, w);
        tmem_st16(ta + 16, w + 16);
        tmem_st16(ta + 32, w + 32);
        tmem_st16(ta + 48, w + 48);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.a_full[ab]);
    }
}

// Fused reduce of one output tile by its last-arriving CTA: C[m, n] = BF16 of
// the FP32 sum of the split planes in ascending order (the same arithmetic as
// the separate reduce kernel, so the same bits).  Threads take items of eight
// consecutive outputs; two items' loads of four planes each are in flight at
// once, kept raw until the adds.  Not inlined: its registers stay out of the
// main loop's allocation.
template <typename T>
struct Raw8p;
template <>
struct Raw8p<__nv_bfloat16> {
    uint4 u;
    __device__ __forceinline__ void load(const __nv_bfloat16* p) {
        u = __ldcg(reinterpret_cast<const uint4*>(p));
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
struct Raw8p<float> {
    float4 a, b;
    __device__ __forceinline__ void load(const float* p) {
        a = __ldcg(reinterpret_cast<const float4*>(p));
        b = __ldcg(reinterpret_cast<const float4*>(p) + 1);
    }
    __device__ __forceinline__ void add_to(float acc[8]) const {
        acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
        acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
    }
};
__device__ __forceinline__ float plane_load(const __nv_bfloat16* p) { return __bfloat162float(__ldcg(p)); }
__device__ __forceinline__ float plane_load(const float* p) { return __ldcg(p); }

template <typename T>
__device__ __noinline__ void reduce_tile(const T* planes, __nv_bfloat16* C, int M, int Nout,
                                         int split, int m0, int rows, int n0, int cols, int t,
                                         int nthreads) {
    const size_t plane = static_cast<size_t>(M) * Nout;
    if (Nout % 8 == 0) {  // cols is then a multiple of 8 and items are 16-byte aligned
        const int per_row = cols / 8;
        const int items = rows * per_row;
        for (int i0 = t; i0 < items; i0 += 2 * nthreads) {
            float acc[2][8];
            size_t off[2];
            bool live[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int i = i0 + u * nthreads;
                live[u] = i < items;
                const int ii = live[u] ? i : 0;
                off[u] = static_cast<size_t>(m0 + ii / per_row) * Nout + n0 + (ii % per_row) * 8;
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[u][j] = 0.f;
            }
            for (int p0 = 0; p0 < split; p0 += 4) {
                Raw8p<T> r[4][2];
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int u = 0; u < 2; ++u)
                        if (live[u] && p0 + q < split) r[q][u].load(planes + (p0 + q) * plane + off[u]);
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int u = 0; u < 2; ++u)
                        if (live[u] && p0 + q < split) r[q][u].add_to(acc[u]);
            }
#pragma unroll
            for (int u = 0; u < 2; ++u)
                if (live[u]) {
                    uint4 o;
                    o.x = pack_bf16x2(acc[u][0], acc[u][1]);
                    o.y = pack_bf16x2(acc[u][2], acc[u][3]);
                    o.z = pack_bf16x2(acc[u][4], acc[u][5]);
                    o.w = pack_bf16x2(acc[u][6], acc[u][7]);
                    *reinterpret_cast<uint4*>(C + off[u]) = o;
                }
        }
    } else {
        const int items = rows * cols;
        for (int i = t; i < items; i += nthreads) {
            const size_t o = static_cast<size_t>(m0 + i / cols) * Nout + n0 + i % cols;
            float acc = 0.f;
            for (int p = 0; p < split; ++p) acc += plane_load(planes + p * plane + o);
            C[o] = __float2bfloat16_rn(acc);
        }
    }
}

// ---- cluster reduce (QMM_REDUCE_CLUSTER) --------------------------------------
//
// The split partitions of one output tile run as one thread-block cluster.
// Each CTA stages its partial tile in shared memory as [m][n] in the partial
// type -- BF16-rounded like a plane, or FP32 -- and after a cluster barrier
// CTA r adds rows [r * per, (r + 1) * per) of every partition's staged tile,
// read through distributed shared memory in ascending partition order, in
// FP32, and rounds once into C: the reduce kernel's arithmetic, without the
// planes in global memory or a second launch (tiny-llm "Week 2 Day 7", Task 4
// adds the planes in FP32 in partition order).  A second cluster barrier
// keeps every staged tile alive until all partners have read it.
template <int BNA>
__device__ __forceinline__ void cluster_reduce_tile(const uint8_t* staged, const TcParams& p, int n0,
                                                    int m0, int t, int nthreads) {
    cluster_add_tile(staged, kWRows, p.out_mode == kOutF32, p.M - m0 < BNA ? p.M - m0 : BNA,
                     p.Nout - n0 < kWRows ? p.Nout - n0 : kWRows, p.split,
                     static_cast<__nv_bfloat16*>(p.C) + static_cast<size_t>(m0) * p.Nout + n0,
                     p.Nout, t, nthreads);
}

// Epilogue of one warp: columns (activation rows) in 16-column chunks c with
// c % DSETS == set; the used accumulators are added in a fixed order.  With
// p.tma_store the tile is staged in shared memory as [m][n] (the activation
// ring, idle once every MMA has completed) and leaves in one TMA store, which
// also clips rows past M and columns past Nout; otherwise each thread stores
// its column's values directly.
template <int BNA>
__device__ __forceinline__ void tc_epilogue(const TcSmem& sm, const TcParams& p, uint32_t tmem,
                                            const CUtensorMap* omap, int quarter, int set,
                                            int lane, int n0, int m0, int part, int gpp,
                                            volatile int* abort) {
    using C = TcCfg<BNA>;
    const bool ok = mbar_wait_warp(sm.acc_full, 0, abort, p.status);
    if (p.weights_static) pdl_wait();  // outputs: earlier kernels may read the planes
    if (ok) {
        tc_fence_after();
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const int r = quarter * 32 + lane;  // row of the weight tile
        const int n = n0 + r;
        const int nacc = gpp < C::NACC ? gpp : C::NACC;  // accumulators that received groups
        const size_t plane = static_cast<size_t>(part) * p.M * p.Nout;
        for (int c = set; c < BNA / 16; c += C::DSETS) {
            uint32_t d[16];
            tmem_ld16(tmem + lane_base + c * 16, d);
            tmem_ld_wait();
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(d[j]);
            for (int a = 1; a < nacc; ++a) {
                tmem_ld16(tmem + lane_base + a * BNA + c * 16, d);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] += __uint_as_float(d[j]);
            }
            if (p.tma_store || p.cluster) {
                if (p.out_mode == kOutBf16) {
                    __nv_bfloat16* t = reinterpret_cast<__nv_bfloat16*>(sm.act);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        t[(c * 16 + j) * kWRows + r] = __float2bfloat16_rn(v[j]);
                } else {
                    float* t = reinterpret_cast<float*>(sm.act);
#pragma unroll
                    for (int j = 0; j < 16; ++j) t[(c * 16 + j) * kWRows + r] = v[j];
                }
                continue;
            }
            if (n >= p.Nout) continue;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int m = m0 + c * 16 + j;
                if (m < p.M) {
                    const size_t o = plane + static_cast<size_t>(m) * p.Nout + n;
                    if (p.out_mode == kOutBf16)
                        static_cast<__nv_bfloat16*>(p.out)[o] = __float2bfloat16_rn(v[j]);
                    else
                        static_cast<float*>(p.out)[o] = v[j];
                }
            }
        }
    }
    if (p.fused) {
        // Count this CTA's plane in.  Every epilogue thread's plane stores are
        // made visible (fence) before the elected thread's increment; the
        // CTA that brings the count to the split adds the tile's planes.  A CTA
        // whose wait ran out still counts in (its planes are invalid, and so is
        // C, which the status word reports), so the counter always returns to
        // zero.
        __shared__ int last;
        __threadfence();
        asm volatile("bar.sync 3, %0;\n" ::"n"(128 * C::DSETS) : "memory");
        if (set == 0 && quarter == 0 && lane == 0) {
            const unsigned tile = static_cast<unsigned>(m0 / BNA) * ((p.Nout + kWRows - 1) / kWRows) +
                                  static_cast<unsigned>(n0 / kWRows);
            const unsigned prev = atomicAdd(&p.counters[tile], 1u);
            last = prev == static_cast<unsigned>(p.split) - 1;
            if (last) {
                p.counters[tile] = 0;
                __threadfence();
            }
        }
        asm volatile("bar.sync 3, %0;\n" ::"n"(128 * C::DSETS) : "memory");
        if (last) {
            const int rows = p.M - m0 < BNA ? p.M - m0 : BNA;
            const int cols = p.Nout - n0 < kWRows ? p.Nout - n0 : kWRows;
            const int t = (set * 4 + quarter) * 32 + lane;
            if (p.out_mode == kOutBf16)
                reduce_tile(static_cast<const __nv_bfloat16*>(p.out),
                            static_cast<__nv_bfloat16*>(p.C), p.M, p.Nout, p.split, m0, rows,
                            n0, cols, t, 128 * C::DSETS);
            else
                reduce_tile(static_cast<const float*>(p.out), static_cast<__nv_bfloat16*>(p.C),
                            p.M, p.Nout, p.split, m0, rows, n0, cols, t, 128 * C::DSETS);
        }
    }
    if (p.tma_store) {
        // every epilogue warp reaches this barrier, with or without a tile
        fence_proxy_async_smem();
        asm volatile("bar.sync 3, %0;\n" ::"n"(128 * C::DSETS) : "memory");
        if (ok && !*abort && set == 0 && quarter == 0 && lane == 0) {
            tma_store_3d(omap, sm.act, n0, m0, part);
            tma_store_commit();
            tma_store_wait_read();
        }
    }
}

// One CTA: the output tile (n0.., m0..) over partition `part` of the call
// described by p and its tensor maps.
template <int BNA>
__device__ __forceinline__ void tc_cta(const TcParams& p, const CUtensorMap* wmap_,
                                       const CUtensorMap* amap_, const CUtensorMap* amap_1_,
                                       const CUtensorMap* omap_, int n0, int m0, int part) {
    const CUtensorMap& wmap = *wmap_;
    const CUtensorMap& amap = *amap_;
    const CUtensorMap& amap_1 = *amap_1_;
    const CUtensorMap& omap = *omap_;
    using C = TcCfg<BNA>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const TcSmem sm = carve<BNA>(base, p);
    __shared__ int abort_flag;
    volatile int* abort = &abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // partition `part`: groups [gbeg, gbeg + gpp), the first G mod split
    // partitions one group longer
    const int gpp = p.gq + (part < p.gr ? 1 : 0);
    const int gbeg = part * p.gq + (part < p.gr ? part : p.gr);

    pdl_trigger();
    if (tid == 0) {
        abort_flag = 0;
        for (int s = 0; s < p.wr.n; ++s) {
            mbar_init(&sm.w_full[s], 1);
            mbar_init(&sm.w_empty[s], 4 * C::WGPS);  // four dequant warps per group
        }
        for (int s = 0; s < p.ar.n; ++s) {
            mbar_init(&sm.act_full[s], 1);
            mbar_init(&sm.act_empty[s], C::AGPS);  // one issuer commit per group
        }
        for (int b = 0; b < C::A_STAGES; ++b) {
            mbar_init(&sm.a_full[b], 4);
            mbar_init(&sm.a_empty[b], 1);
        }
        mbar_init(sm.acc_full, C::NACC);
        mbar_fence_init();
        tma_prefetch_map(&wmap);
        tma_prefetch_map(&amap);
    }
    if (warp == 0 && !p.weights_static) {
        // The packed weights are a read-only input: this CTA's share is pulled
        // into L2 while the kernels before it on the stream finish.  L2 is the
        // point of coherence, so the loads after the wait below still see
        // anything those kernels wrote.
        const int nbox = (gpp + 1) >> 1;
        for (int j = lane; j < nbox; j += 32) tma_prefetch_l2_2d(&wmap, (gbeg + 2 * j) * 16, n0);
    }
    if (warp == 1) {  // tensor memory is not global memory: allocated before the wait
        tmem_alloc(sm.tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    // Global memory that earlier kernels on the stream may write is read (and
    // outputs are written) only after the dependency wait.  With static
    // weights only the activation copies (the producer) and the epilogue wait.
    if (!p.weights_static) pdl_wait();
    __syncthreads();  // barriers initialized; the producer starts at once
    uint32_t tmem = 0;
    // warp 1's tensor-memory address reaches the issuers and dequantizers
    // through named barrier 2
    constexpr int kTmemBarThreads = 32 * C::NACC + 32 * 4 * C::DSETS;

    if (warp == 0) {
        if (lane == 0)
            tc_producer<BNA>(sm, p, &wmap, &amap, &amap_1, n0, m0, gbeg, gpp, abort);
    } else if (warp <= C::NACC) {
        tc_fence_before();
        asm volatile("bar.sync 2, %0;\n" ::"n"(kTmemBarThreads) : "memory");
        tc_fence_after();
        tmem = *sm.tmem_slot;
        if (lane == 0) tc_issuer<BNA>(sm, p, tmem, warp - 1, gpp, abort);
    } else if (warp >= kCtlWarps) {
        tc_fence_before();
        asm volatile("bar.sync 2, %0;\n" ::"n"(kTmemBarThreads) : "memory");
        tc_fence_after();
        tmem = *sm.tmem_slot;
        const int quarter = warp & 3, set = (warp - kCtlWarps) >> 2;
        tc_dequant<BNA>(sm, p, tmem, quarter, set, lane, n0, gbeg, gpp, abort);
        tc_epilogue<BNA>(sm, p, tmem, &omap, quarter, set, lane, n0, m0, part, gpp, abort);
    }

    // ---- teardown: every MMA has finished before tensor memory is freed ----
    tc_fence_before();
    __syncthreads();
    if (p.cluster) {
        // every thread of every partition's CTA passes both barriers, also
        // after a wait ran out (C is then invalid, as the status word says)
        cluster_barrier();  // every partner's partial tile is staged
        cluster_reduce_tile<BNA>(sm.act, p, n0, m0, tid, C::THREADS);
        cluster_barrier();  // every partner has read this CTA's tile
    }
    if (warp == 1) {
        if (lane == 0 && *abort) mbar_wait(sm.acc_full, 0, nullptr, p.status);
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int BNA>
__global__ void __launch_bounds__(TcCfg<BNA>::THREADS, 1)
    w4a16_tc_kernel(const __grid_constant__ CUtensorMap wmap,
                    const __grid_constant__ CUtensorMap amap,
                    const __grid_constant__ CUtensorMap amap_1,
                    const __grid_constant__ CUtensorMap omap, const TcParams p) {
    tc_cta<BNA>(p, &wmap, &amap, &amap_1, &omap, blockIdx.x * kWRows, blockIdx.y * BNA,
                blockIdx.z);
}

// Several independent calls of one tile width in one launch: the CTAs of call
// c are the linear block indices [cta_begin, next call's cta_begin), in the
// order (column tile, row tile, partition) of a single call's grid.  Each CTA
// copies its call's parameters to shared memory and runs the same CTA body.
struct TcCall {
    CUtensorMap wmap, amap, amap_1, omap;
    TcParams p;
    int n_tiles, m_tiles;
    int cta_begin;
};
struct TcGroup {
    int ncalls;
    TcCall call[kMaxGroupCalls];
};

template <int BNA>
__global__ void __launch_bounds__(TcCfg<BNA>::THREADS, 1)
    w4a16_tc_group_kernel(const __grid_constant__ TcGroup g) {
    static_assert(sizeof(TcParams) % 4 == 0, "parameter copy");
    __shared__ TcParams sp;
    int c = 0;
    while (c + 1 < g.ncalls && static_cast<int>(blockIdx.x) >= g.call[c + 1].cta_begin) ++c;
    const TcCall& call = g.call[c];
    if (threadIdx.x < sizeof(TcParams) / 4)
        reinterpret_cast<int*>(&sp)[threadIdx.x] =
            reinterpret_cast<const int*>(&call.p)[threadIdx.x];
    __syncthreads();
    int t = static_cast<int>(blockIdx.x) - call.cta_begin;
    const int nx = t % call.n_tiles;
    t /= call.n_tiles;
    const int my = t % call.m_tiles;
    tc_cta<BNA>(sp, &call.wmap, &call.amap, &call.amap_1, &call.omap, nx * kWRows, my * BNA,
                t / call.m_tiles);
}

// ---- persistent grouped kernel ---------------------------------------------
//
// One CTA per SM walks a list of output tiles ("items") of the calls in a
// group.  Item k is the k-th CTA of the one-CTA-per-tile grouped grid (calls
// longest partition first), and CTA b of P takes items b, 2P-1-b, 2P+b, ...:
// a snake over rounds of P items, so every CTA draws one item from each band
// of the longest-first list.  The prologue (barriers, tensor memory,
// descriptor prefetch, the call table) runs once per CTA, and the producer
// streams the next item's weights and activations while the current one
// drains.
//
// Groups are numbered by one counter across the CTA's items: group g goes to
// A buffer g % A_STAGES, dequantizer set g % DSETS and issuer g % NACC, as in
// one tile.  Each item's groups fill its own ring stages, so an item's last
// weight or activation stage may be short; the producer counts the absent
// positions into that stage's release barrier when it issues the copy.  A
// short stage lacks some consumers, which then skip that lap of its slot; the
// parity waits stay sound because every consumer first passes the item's
// accumulator hand-off (the epilogue waits for all of the item's MMAs, the
// issuers wait for the epilogue), by which time every stage of the item has
// landed.  Full stages hold a group of every consumer (WGPS >= DSETS,
// AGPS >= NACC or one-group stages on a ring whose depth is a multiple of
// NACC).  The epilogue adds the accumulators in the item's own order
// (accumulator of local group 0 first), so each output equals the
// one-CTA-per-tile kernel's bit for bit.  Output tiles leave by direct
// stores: the activation ring is no longer idle when an epilogue runs.

// The per-call fields the roles read, cached in shared memory at CTA start
// (reads of the launch's call table in parameter space at every item boundary
// would wait on the constant cache).
struct TcpCall {
    const uint16_t* scales;
    const uint16_t* biases;
    void* out;
    int cta_begin, n_tiles, m_tiles, gq, gr, M, Nout, G, out_mode;
};

struct TcpItem {
    int call;        // index into the launch's call table
    int n0, m0, part;
    int gbeg, gpp;   // reduction groups [gbeg, gbeg + gpp)
};

__device__ __forceinline__ int tcp_item_index(int round, int b, int P) {
    return round * P + ((round & 1) ? P - 1 - b : b);
}

// Item of this CTA in round `round`; false once the list is exhausted.
template <int BNA>
__device__ __forceinline__ bool tcp_item(const TcpCall* sc, int ncalls, int total, int round,
                                         TcpItem& it) {
    const int k = tcp_item_index(round, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x));
    if (k >= total) return false;
    int c = 0;
    while (c + 1 < ncalls && k >= sc[c + 1].cta_begin) ++c;
    const TcpCall& call = sc[c];
    int t = k - call.cta_begin;
    const int nx = t % call.n_tiles;
    t /= call.n_tiles;
    const int my = t % call.m_tiles;
    const int part = t / call.m_tiles;
    it.call = c;
    it.n0 = nx * kWRows;
    it.m0 = my * BNA;
    it.part = part;
    it.gpp = call.gq + (part < call.gr ? 1 : 0);
    it.gbeg = part * call.gq + (part < call.gr ? part : call.gr);
    return true;
}

// Slot and phase of global stage j of a ring.
__device__ __forceinline__ void ring_stage(const Ring& r, int j, int& slot, uint32_t& phase) {
    const uint32_t q = __umulhi(static_cast<uint32_t>(j), r.magic);
    slot = j - static_cast<int>(q) * r.n;
    phase = q & 1u;
}

struct TcpSmem : TcSmem {
    uint64_t* acc_empty;  // the epilogue has read the accumulators out
    uint64_t* drain;      // every MMA of the CTA has completed
    uint64_t* deq_done;   // every dequantizer warp has left its loop
};

template <int BNA>
__device__ __forceinline__ TcpSmem carve_p(uint8_t* base, const TcParams& p) {
    TcpSmem s;
    static_cast<TcSmem&>(s) = carve<BNA>(base, p);
    s.acc_empty = s.acc_full + 1;
    s.drain = s.acc_full + 2;
    s.deq_done = s.acc_full + 3;
    s.tmem_slot = reinterpret_cast<uint32_t*>(s.acc_full + 4);
    return s;
}

__device__ __forceinline__ void mbar_arrive_n(uint64_t* bar, uint32_t n) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_addr(bar)), "r"(n)
                 : "memory");
}

// Producer (one thread): the weight and activation stages of the CTA's items
// in order, each ring polled without blocking as in the one-tile producer.
// An item's last stage may be short: only its groups are copied, and the
// absent positions are counted into the stage's release barrier at once.
template <int BNA>
__device__ __forceinline__ void tcp_producer(const TcpSmem& sm, const TcGroup& g,
                                             const TcpCall* sc, int ncalls, int total,
                                             volatile int* abort) {
    using C = TcCfg<BNA>;
    const Ring wr = g.call[0].p.wr, ar = g.call[0].p.ar;
    int* status = g.call[0].p.status;
    const bool wstatic = g.call[0].p.weights_static != 0;
    TcpItem iw, ia;
    int rw = 0, ra = 0, jw = 0, ja = 0;  // rounds and stages within the items
    int nw = 0, na = 0;                  // stages issued (global)
    int sw = 0, sa = 0;
    uint32_t pw = 0, pa = 0;
    bool wlive = tcp_item<BNA>(sc, ncalls, total, 0, iw);
    bool alive = wlive;
    ia = iw;
    auto issue_w = [&]() {
        const CUtensorMap* map = &g.call[iw.call].wmap;
        fence_proxy_async_smem();  // the dequantizers read the slot with ordinary loads
        const int left = iw.gpp - jw * C::WGPS;
        const int real = left < C::WGPS ? left : C::WGPS;
        const int boxes = (real + 1) >> 1;
        const int x = (iw.gbeg + jw * C::WGPS) * 16;  // 32-bit words
        if (real < C::WGPS) mbar_arrive_n(&sm.w_empty[sw], 4 * (C::WGPS - real));
        mbar_arrive_expect_tx(&sm.w_full[sw], boxes * kWBox);
        tma_load_2d(sm.w + sw * C::W_STAGE, map, &sm.w_full[sw], x, iw.n0);
        if (boxes == 2)
            tma_load_2d(sm.w + sw * C::W_STAGE + kWBox, map, &sm.w_full[sw], x + 32, iw.n0);
        ++nw;
        if (++sw == wr.n) { sw = 0; pw ^= 1; }
        if (++jw * C::WGPS >= iw.gpp) {
            jw = 0;
            wlive = tcp_item<BNA>(sc, ncalls, total, ++rw, iw);
        }
    };
    auto issue_a = [&]() {
        const TcCall& call = g.call[ia.call];
        const int left = ia.gpp - ja * C::AGPS;
        const int real = left < C::AGPS ? left : C::AGPS;
        const int g0 = ia.gbeg + ja * C::AGPS;
        uint8_t* dst = sm.act + sa * C::ACT_STAGE;
        if (real == C::AGPS) {
            mbar_arrive_expect_tx(&sm.act_full[sa], C::ACT_STAGE);
            tma_load_3d(dst, &call.amap, &sm.act_full[sa], 0, ia.m0, g0 * 2);
        } else {  // a short last stage: one-group copies
            mbar_arrive_n(&sm.act_empty[sa], C::AGPS - real);
            mbar_arrive_expect_tx(&sm.act_full[sa], real * C::ACT_GROUP);
            for (int t = 0; t < real; ++t)
                tma_load_3d(dst + t * C::ACT_GROUP, &call.amap_1, &sm.act_full[sa], 0, ia.m0,
                            (g0 + t) * 2);
        }
        ++na;
        if (++sa == ar.n) { sa = 0; pa ^= 1; }
        if (++ja * C::AGPS >= ia.gpp) {
            ja = 0;
            alive = tcp_item<BNA>(sc, ncalls, total, ++ra, ia);
        }
    };
    if (wstatic) {
        // static weights: the first lap of weight slots is filled before the
        // wait for the earlier kernels; only the activation copies wait
        while (wlive && nw < wr.n) issue_w();
        pdl_wait();
    }
    // a wait ends in an abort only after kWaitLimitNs without any progress
    unsigned long long t0 = globaltimer_ns();
    bool restamp = false;
    for (uint32_t spin = 0; wlive || alive; ++spin) {
        bool progress = false;
        if (wlive && mbar_probe(&sm.w_empty[sw], pw ^ 1)) {
            issue_w();
            progress = true;
        }
        if (alive && mbar_probe(&sm.act_empty[sa], pa ^ 1)) {
            issue_a();
            progress = true;
        }
        if (progress) {
            restamp = true;
        } else if ((spin & 255u) == 0) {
            if (*abort) break;
            const unsigned long long now = globaltimer_ns();
            if (restamp) {
                t0 = now;
                restamp = false;
            } else if (now - t0 > kWaitLimitNs) {
                *abort = 1;
                atomicExch(status, kStatusTimeout);
                break;
            }
        }
    }
    if (*abort) {  // let copies in flight land before the CTA exits
        for (int j = nw > wr.n ? nw - wr.n : 0; j < nw; ++j)
            mbar_wait(&sm.w_full[j % wr.n], (j / wr.n) & 1, nullptr, status);
        for (int j = na > ar.n ? na - ar.n : 0; j < na; ++j)
            mbar_wait(&sm.act_full[j % ar.n], (j / ar.n) & 1, nullptr, status);
    }
}

// MMA issuer c (one thread): of every item, the groups whose global index is
// c mod NACC, into accumulator c; the first one of an item starts the
// accumulator.  Before an item's groups it waits for the previous item's
// epilogue to have read the accumulators out.
template <int BNA>
__device__ __forceinline__ void tcp_issuer(const TcpSmem& sm, const TcGroup& g,
                                           const TcpCall* sc, int ncalls, int total,
                                           uint32_t tmem, int c, volatile int* abort) {
    using C = TcCfg<BNA>;
    const Ring ar = g.call[0].p.ar;
    int* status = g.call[0].p.status;
    const uint32_t d_tm = tmem + c * BNA;
    TcpItem it;
    int g0 = 0, abase = 0;  // first global group and activation stage of the item
    bool ok = true;
    for (int r = 0; ok && tcp_item<BNA>(sc, ncalls, total, r, it); ++r) {
        if (r > 0) {
            if (!mbar_wait(sm.acc_empty, (r - 1) & 1, abort, status)) break;
            tc_fence_after();
        }
        const int first = ((c - g0) % C::NACC + C::NACC) % C::NACC;
        for (int i = first; i < it.gpp; i += C::NACC) {
            const int gg = g0 + i;
            int sa;
            uint32_t ph;
            ring_stage(ar, abase + (i >> C::AGPS_LOG2), sa, ph);
            const int within = i & (C::AGPS - 1);
            const int ab = gg % C::A_STAGES;
            if (!mbar_wait(&sm.act_full[sa], ph, abort, status) ||
                !mbar_wait(&sm.a_full[ab], (gg / C::A_STAGES) & 1, abort, status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t a_tm = tmem + C::ACOL + ab * 64;
            const uint64_t b0 = sdesc_kmajor_sw128(
                smem_addr(sm.act + sa * C::ACT_STAGE + within * C::ACT_GROUP));
            const uint32_t acc = i != first;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)  // k step of 16: +32 bytes in the swizzle atom
                umma_bf16_tmem_a(d_tm, a_tm + kk * 8,
                                 b0 + ((((kk >> 2) * C::ACT_BOX) + (kk & 3) * 32) >> 4),
                                 C::IDESC, acc | (kk != 0));
            umma_commit(&sm.act_empty[sa]);
            umma_commit(&sm.a_empty[ab]);
        }
        if (!ok) break;
        umma_commit(sm.acc_full);
        g0 += it.gpp;
        abase += (it.gpp + C::AGPS - 1) >> C::AGPS_LOG2;
    }
    umma_commit(sm.drain);
}

// The scale and bias of a dequantizer thread's next group, which may lie in a
// later item: fetched one of the set's groups ahead, so the load overlaps the
// previous group (and an epilogue, across items).
template <int BNA>
struct TcpAhead {
    int round, g0, i, gpp;  // the item's round and first global group, the local group
    int call;               // the item's call (-1 once the list is exhausted)
    long long row;          // element offset of the row at the item's first group, -1 past Nout
    uint16_t s, b;
    __device__ __forceinline__ void item(const TcpCall* sc, int ncalls, int total, int r,
                                         int wrow) {
        TcpItem it;
        round = r;
        if (!tcp_item<BNA>(sc, ncalls, total, r, it)) {
            call = -1;
            return;
        }
        call = it.call;
        gpp = it.gpp;
        const int n = it.n0 + wrow;
        row = n < sc[call].Nout ? static_cast<long long>(n) * sc[call].G + it.gbeg : -1;
    }
    __device__ __forceinline__ void load(const TcpCall* sc) {
        s = b = 0;
        if (call < 0 || row < 0) return;
        s = __ldg(sc[call].scales + row + i);
        b = __ldg(sc[call].biases + row + i);
    }
    // the set's first group at local index >= from, in this item or a later one
    __device__ __forceinline__ void seek(const TcpCall* sc, int ncalls, int total, int set,
                                         int from, int wrow) {
        using C = TcCfg<BNA>;
        i = from + ((set - (g0 + from)) % C::DSETS + C::DSETS) % C::DSETS;
        while (call >= 0 && i >= gpp) {
            g0 += gpp;
            item(sc, ncalls, total, round + 1, wrow);
            i = ((set - g0) % C::DSETS + C::DSETS) % C::DSETS;
        }
    }
};

// Epilogue of item `r` by one dequantizer warp: columns (activation rows) in
// 16-column chunks c with c % DSETS == set, the accumulators that received
// groups added in the item's order, then direct stores of the warp's output
// column; finally the warp hands the accumulators back to the issuers.
template <int BNA>
__device__ __forceinline__ void tcp_epilogue(const TcpSmem& sm, const TcpCall& call,
                                             const TcpItem& it, int r, int g0, uint32_t tmem,
                                             int quarter, int set, int lane, bool wstatic,
                                             int* status, volatile int* abort) {
    using C = TcCfg<BNA>;
    const bool ok = mbar_wait_warp(sm.acc_full, r & 1, abort, status);
    if (wstatic) pdl_wait();  // outputs: earlier kernels may read the planes
    if (ok) {
        tc_fence_after();
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const int n = it.n0 + quarter * 32 + lane;
        const int nacc = it.gpp < C::NACC ? it.gpp : C::NACC;
        const size_t plane = static_cast<size_t>(it.part) * call.M * call.Nout;
        for (int c = set; c < BNA / 16; c += C::DSETS) {
            float v[16];
#pragma unroll
            for (int a = 0; a < C::NACC; ++a) {
                if (a >= nacc) break;  // warp-uniform
                uint32_t d[16];
                tmem_ld16(tmem + lane_base + ((g0 + a) % C::NACC) * BNA + c * 16, d);
                tmem_ld_wait();
                if (a == 0) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(d[j]);
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] += __uint_as_float(d[j]);
                }
            }
            const int m = it.m0 + c * 16;
            if (n >= call.Nout || m >= call.M) continue;
            const int rows = call.M - m < 16 ? call.M - m : 16;
            const size_t o = plane + static_cast<size_t>(m) * call.Nout + n;
            if (call.out_mode == kOutBf16) {
                __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(call.out) + o;
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (j < rows) dst[static_cast<size_t>(j) * call.Nout] = __float2bfloat16_rn(v[j]);
            } else {
                float* dst = static_cast<float*>(call.out) + o;
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (j < rows) dst[static_cast<size_t>(j) * call.Nout] = v[j];
            }
        }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.acc_empty);
}

// Dequantizer warp of lane quarter `quarter` in set `set`: of every item, the
// groups whose global index is set mod DSETS (weight row 32 * quarter + lane),
// then the item's epilogue.
template <int BNA>
__device__ __forceinline__ void tcp_dequant(const TcpSmem& sm, const TcGroup& g,
                                            const TcpCall* sc, int ncalls, int total,
                                            uint32_t tmem, int quarter, int set, int lane,
                                            volatile int* abort) {
    using C = TcCfg<BNA>;
    const Ring wr = g.call[0].p.wr;
    int* status = g.call[0].p.status;
    const bool wstatic = g.call[0].p.weights_static != 0;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    TcpAhead<BNA> ahead;
    ahead.g0 = 0;
    ahead.item(sc, ncalls, total, 0, row);
    ahead.seek(sc, ncalls, total, set, 0, row);
    ahead.load(sc);
    TcpItem it;
    int g0 = 0, wbase = 0;  // first global group and weight stage of the item
    bool ok = true;
    for (int r = 0; ok && tcp_item<BNA>(sc, ncalls, total, r, it); ++r) {
        const int first = ((set - g0) % C::DSETS + C::DSETS) % C::DSETS;
        for (int i = first; i < it.gpp; i += C::DSETS) {
            const int gg = g0 + i;
            const uint16_t s_cur = ahead.s, b_cur = ahead.b;
            ahead.seek(sc, ncalls, total, set, ahead.i + C::DSETS, row);
            ahead.load(sc);
            int sw;
            uint32_t ph;
            ring_stage(wr, wbase + (i >> C::WGPS_LOG2), sw, ph);
            const int within = i & (C::WGPS - 1);
            const int ab = gg % C::A_STAGES;
            if (!mbar_wait_warp(&sm.w_full[sw], ph, abort, status)) {
                ok = false;
                break;
            }
            // box `within / 2`, row of 128 bytes, 16-byte chunks 4*(within % 2) ..
            // +3 under the 128-byte swizzle (chunk k of row r at k ^ (r % 8))
            const uint8_t* wrow = sm.w + sw * C::W_STAGE + (within >> 1) * kWBox + row * 128;
            uint4 wv[4];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                wv[c] = *reinterpret_cast<const uint4*>(
                    wrow + ((((within & 1) << 2) + c) ^ (row & 7)) * 16);
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.w_empty[sw]);
            uint32_t w[64];
            if (scale_subnormal_ok(s_cur))
                dequant_row_group_sub(wv, scale_shifted_pair(s_cur, 133), bf16_pair(b_cur), w);
            else
                dequant_row_group(wv, bf16_pair(s_cur), bf16_pair(b_cur), w);
            if (!mbar_wait_warp(&sm.a_empty[ab], ((gg / C::A_STAGES) & 1) ^ 1, abort, status)) {
                ok = false;
                break;
            }
            // the stores below must follow the MMAs that read this buffer before
            tc_fence_after();
            const uint32_t ta = tmem + lane_base + C::ACOL + ab * 64;
            tmem_st16(ta + 0, w);
            tmem_st16(ta + 16, w + 16);
            tmem_st16(ta + 32, w + 32);
            tmem_st16(ta + 48, w + 48);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.a_full[ab]);
        }
        if (!ok) break;
        tcp_epilogue<BNA>(sm, sc[it.call], it, r, g0, tmem, quarter, set, lane, wstatic, status,
                          abort);
        g0 += it.gpp;
        wbase += (it.gpp + C::WGPS - 1) >> C::WGPS_LOG2;
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.deq_done);
}

template <int BNA>
__global__ void __launch_bounds__(TcCfg<BNA>::THREADS, 1)
    w4a16_tc_persist_kernel(const __grid_constant__ TcGroup g, int total) {
    using C = TcCfg<BNA>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const TcParams& p0 = g.call[0].p;
    const TcpSmem sm = carve_p<BNA>(base, p0);
    __shared__ TcpCall sc[kMaxGroupCalls];
    __shared__ int abort_flag;
    volatile int* abort = &abort_flag;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ncalls = g.ncalls;

    pdl_trigger();
    if (tid == 0) {
        abort_flag = 0;
        for (int s = 0; s < p0.wr.n; ++s) {
            mbar_init(&sm.w_full[s], 1);
            mbar_init(&sm.w_empty[s], 4 * C::WGPS);  // four dequant warps per group
        }
        for (int s = 0; s < p0.ar.n; ++s) {
            mbar_init(&sm.act_full[s], 1);
            mbar_init(&sm.act_empty[s], C::AGPS);  // one issuer commit per group
        }
        for (int b = 0; b < C::A_STAGES; ++b) {
            mbar_init(&sm.a_full[b], 4);
            mbar_init(&sm.a_empty[b], 1);
        }
        mbar_init(sm.acc_full, C::NACC);
        mbar_init(sm.acc_empty, 4 * C::DSETS);  // every epilogue warp
        mbar_init(sm.drain, C::NACC);
        mbar_init(sm.deq_done, 4 * C::DSETS);
        mbar_fence_init();
    }
    if (warp == 0 && lane < ncalls) {  // the call table, and its tensor maps prefetched
        const TcCall& call = g.call[lane];
        TcpCall& t = sc[lane];
        t.scales = call.p.scales;
        t.biases = call.p.biases;
        t.out = call.p.out;
        t.cta_begin = call.cta_begin;
        t.n_tiles = call.n_tiles;
        t.m_tiles = call.m_tiles;
        t.gq = call.p.gq;
        t.gr = call.p.gr;
        t.M = call.p.M;
        t.Nout = call.p.Nout;
        t.G = call.p.G;
        t.out_mode = call.p.out_mode;
        tma_prefetch_map(&call.wmap);
        tma_prefetch_map(&call.amap);
        tma_prefetch_map(&call.amap_1);
    }
    if (warp == 1) {  // tensor memory is not global memory: allocated before the wait
        tmem_alloc(sm.tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    if (!p0.weights_static) pdl_wait();
    __syncthreads();  // barriers and call table ready; the producer starts at once
    uint32_t tmem = 0;
    constexpr int kTmemBarThreads = 32 * C::NACC + 32 * 4 * C::DSETS;

    if (warp == 0) {
        if (lane == 0) tcp_producer<BNA>(sm, g, sc, ncalls, total, abort);
    } else if (warp <= C::NACC) {
        tc_fence_before();
        asm volatile("bar.sync 2, %0;\n" ::"n"(kTmemBarThreads) : "memory");
        tc_fence_after();
        tmem = *sm.tmem_slot;
        if (lane == 0) tcp_issuer<BNA>(sm, g, sc, ncalls, total, tmem, warp - 1, abort);
    } else if (warp >= kCtlWarps) {
        tc_fence_before();
        asm volatile("bar.sync 2, %0;\n" ::"n"(kTmemBarThreads) : "memory");
        tc_fence_after();
        tmem = *sm.tmem_slot;
        tcp_dequant<BNA>(sm, g, sc, ncalls, total, tmem, warp & 3, (warp - kCtlWarps) >> 2,
                         lane, abort);
    }

    // ---- teardown: tensor memory is freed once every MMA has completed and
    // every dequantizer warp (the epilogues' reads) has left its loop ----
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        if (lane == 0) {
            mbar_wait(sm.drain, 0, nullptr, p0.status);
            mbar_wait(sm.deq_done, 0, nullptr, p0.status);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// The pipeline shape of one launch: per-tile constants of TcCfg<BNA> and the
// ring depths chosen for a partition of gpp groups under a dynamic shared
// memory limit.  Ring depths (stages of WGPS / AGPS groups): the activation
// ring is shallow, its stages come from L2; the weight ring carries the HBM
// stream and takes the rest of shared memory.  Both depths keep every slot's
// consumers passing every lap (ring_laps_ok).  The persistent schedule keeps
// two activation stages, so the weight ring can hold the next item's first
// groups while the current item drains.  Returns false if nothing fits.
template <int BNA>
bool tc_pipeline(int gpp, long limit, TcPipeline* out, bool persistent = false) {
    using C = TcCfg<BNA>;
    const size_t fixed = 1024 + tc_bar_bytes() + 128;
    const int nst = (gpp + C::AGPS - 1) / C::AGPS;
    int ast = BNA <= 128 ? 4 : 3;
    // weight stages at least: three of four groups, or two of two
    const int wmin = C::WGPS >= 4 ? 3 : 2;
    if (ast > nst + 1) ast = nst + 1 < 2 ? 2 : nst + 1;
    if (persistent) ast = 2;
    int wst = 0;
    for (; ast >= 2; --ast) {
        if (!ring_laps_ok(ast, C::AGPS, C::NACC)) continue;
        const long room = limit - static_cast<long>(fixed) - static_cast<long>(ast) * C::ACT_STAGE;
        wst = room > 0 ? static_cast<int>(room / C::W_STAGE) : 0;
        if (wst > kMaxWStages) wst = kMaxWStages;
        while (wst > 0 && !ring_laps_ok(wst, C::WGPS, C::DSETS)) --wst;
        if (wst >= wmin) break;
    }
    if (ast < 2 || wst < wmin) return false;
    out->nacc = C::NACC;
    out->dsets = C::DSETS;
    out->a_stages = C::A_STAGES;
    out->wgps = C::WGPS;
    out->agps = C::AGPS;
    out->act_stages = ast;
    out->w_stages = wst;
    out->threads = C::THREADS;
    out->smem = fixed + static_cast<size_t>(ast) * C::ACT_STAGE +
                static_cast<size_t>(wst) * C::W_STAGE;
    return true;
}

// Parameters and tensor maps of one call, for a launch whose rings pl describes.
template <int BNA>
bool setup_call(const void* A, const uint32_t* Wq, const void* scales, const void* biases,
                void* out, int out_mode, int M, int Kred, int Nout, int split, void* fused_C,
                uint32_t* counters, const TcPipeline& pl, int* status, TcParams* pp,
                CUtensorMap* wmap, CUtensorMap* amap, CUtensorMap* amap_1, CUtensorMap* omap) {
    using C = TcCfg<BNA>;
    TcParams& p = *pp;
    p.scales = static_cast<const uint16_t*>(scales);
    p.biases = static_cast<const uint16_t*>(biases);
    p.out = out;
    p.status = status;
    p.M = M;
    p.Kred = Kred;
    p.Nout = Nout;
    p.G = Kred / kGroup;
    p.split = split;
    p.gq = p.G / split;
    p.gr = p.G % split;
    p.gpp = p.gq + (p.gr ? 1 : 0);
    p.out_mode = out_mode;
    p.weights_static = weights_static() && pdl_enabled() ? 1 : 0;
    p.fused = fused_C != nullptr && counters != nullptr && split > 1 ? 1 : 0;
    p.C = fused_C;
    p.counters = counters;
    p.cluster = 0;
    // a partition whose last activation stage holds fewer than AGPS groups
    // fills it through a one-group map
    const bool atails = p.gq % C::AGPS != 0 || (p.gr && (p.gq + 1) % C::AGPS != 0);
    const int ast = pl.act_stages, wst = pl.w_stages;
    auto ring = [](int n, int gps_log2) {
        Ring r;
        r.n = n;
        r.magic = static_cast<uint32_t>((0x100000000ull + n - 1) / n);
        r.gps_log2 = gps_log2;
        return r;
    };
    p.wr = ring(wst, C::WGPS_LOG2);
    p.ar = ring(ast, C::AGPS_LOG2);

    // weights as 2-D [Nout][Kred/8 words] with boxes of 128 rows x 32 words (two
    // groups, 128-byte swizzle); activations as [64-k chunk][row][64] boxes of
    // 2*AGPS chunks x BNA rows (128-byte swizzle, the MMA's K-major layout).
    // The one-group map (box of one group) fills short last stages.
    {
        const cuuint64_t adims[3] = {64, static_cast<cuuint64_t>(M),
                                     static_cast<cuuint64_t>(Kred / 64)};
        const cuuint64_t astr[2] = {static_cast<cuuint64_t>(Kred) * 2, 128};
        auto aenc = [&](CUtensorMap* m, int groups) {
            const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(BNA),
                                       static_cast<cuuint32_t>(2 * groups)};
            return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, A, adims, astr, box,
                                CU_TENSOR_MAP_SWIZZLE_128B);
        };
        if (!encode_2d(wmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, Wq, Nout, Kred / 8, 4, kWRows, 32,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
            !aenc(amap, C::AGPS))
            return false;
        if (atails ? !aenc(amap_1, 1) : false) return false;
        if (!atails) *amap_1 = *amap;
    }
    // output planes [split][M][Nout] as a 3-D map with a [BNA][128] box; a TMA
    // store needs 16-byte row pitch, and the staged tile must fit the ring
    *omap = *wmap;
    {
        const int elem = out_mode == kOutBf16 ? 2 : 4;
        const size_t tile = static_cast<size_t>(BNA) * kWRows * elem;
        // (the fused reduce reads planes that other CTAs wrote, so its plane
        // stores stay in the generic proxy)
        p.tma_store = !p.fused && (static_cast<size_t>(Nout) * elem) % 16 == 0 &&
                      tile <= static_cast<size_t>(ast) * C::ACT_STAGE;
        if (p.tma_store) {
            const cuuint64_t odims[3] = {static_cast<cuuint64_t>(Nout), static_cast<cuuint64_t>(M),
                                         static_cast<cuuint64_t>(split)};
            const cuuint64_t ostr[2] = {static_cast<cuuint64_t>(Nout) * elem,
                                        static_cast<cuuint64_t>(M) * Nout * elem};
            const cuuint32_t obox[3] = {kWRows, static_cast<cuuint32_t>(BNA), 1};
            if (!encode_tiled(omap,
                              out_mode == kOutBf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                              3, out, odims, ostr, obox, CU_TENSOR_MAP_SWIZZLE_NONE))
                return false;
        }
    }
    return true;
}

template <int BNA>
int launch_tc(const void* A, const uint32_t* Wq, const void* scales, const void* biases,
              void* out, int out_mode, int M, int Kred, int Nout, int split, void* fused_C,
              uint32_t* counters, cudaStream_t st) {
    using C = TcCfg<BNA>;
    auto kern = w4a16_tc_kernel<BNA>;
    static int limit = -1;
    static std::once_flag once;
    std::call_once(once, [&] { limit = set_max_dynamic_smem(reinterpret_cast<const void*>(kern)); });
    if (limit < 0) return cudaErrorInvalidValue;
    int* status = tc_status_ptr();
    if (!status) return cudaErrorInvalidSymbol;
    const int G = Kred / kGroup;
    TcPipeline pl;
    if (!tc_pipeline<BNA>(G / split + (G % split ? 1 : 0), limit, &pl)) return cudaErrorInvalidValue;
    TcParams p;
    CUtensorMap wmap, amap, amap_1, omap;
    if (!setup_call<BNA>(A, Wq, scales, biases, out, out_mode, M, Kred, Nout, split, fused_C,
                         counters, pl, status, &p, &wmap, &amap, &amap_1, &omap))
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    LaunchAttrs la;
    apply_pdl(cfg, la);
    cfg.gridDim = dim3((Nout + kWRows - 1) / kWRows, (M + BNA - 1) / BNA, split);
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, kern, wmap, amap, amap_1, omap, p);
}

// The call with the cluster reduce: grid z = partition, cluster (1, 1, split),
// C written by the partitions' cluster.  cudaErrorNotSupported (nothing
// launched) when the partial tile cannot be staged in the activation ring or
// the device cannot hold every cluster of the call at once (a partial wave
// of clusters would cost more than the reduce kernel it replaces).
template <int BNA>
int launch_tc_cluster(const void* A, const uint32_t* Wq, const void* scales, const void* biases,
                      void* C, int out_mode, int M, int Kred, int Nout, int split,
                      cudaStream_t st) {
    using Cf = TcCfg<BNA>;
    if (split < 2 || split > 16) return cudaErrorNotSupported;
    auto kern = w4a16_tc_kernel<BNA>;
    static int limit = -1;
    static std::once_flag once;
    std::call_once(once, [&] {
        limit = set_max_dynamic_smem(reinterpret_cast<const void*>(kern));
        if (limit >= 0 && cudaFuncSetAttribute(reinterpret_cast<const void*>(kern),
                                               cudaFuncAttributeNonPortableClusterSizeAllowed,
                                               1) != cudaSuccess)
            limit = -1;
    });
    if (limit < 0) return cudaErrorNotSupported;
    int* status = tc_status_ptr();
    if (!status) return cudaErrorInvalidSymbol;
    const int G = Kred / kGroup;
    TcPipeline pl;
    if (!tc_pipeline<BNA>(G / split + (G % split ? 1 : 0), limit, &pl)) return cudaErrorNotSupported;
    const size_t tile = static_cast<size_t>(BNA) * kWRows * (out_mode == kOutBf16 ? 2 : 4);
    if (tile > static_cast<size_t>(pl.act_stages) * Cf::ACT_STAGE) return cudaErrorNotSupported;
    TcParams p;
    CUtensorMap wmap, amap, amap_1, omap;
    if (!setup_call<BNA>(A, Wq, scales, biases, C, out_mode, M, Kred, Nout, split, nullptr,
                         nullptr, pl, status, &p, &wmap, &amap, &amap_1, &omap))
        return cudaErrorInvalidValue;
    p.cluster = 1;
    p.tma_store = 0;
    p.C = C;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attrs[2];
    int na = 0;
    attrs[na].id = cudaLaunchAttributeClusterDimension;
    attrs[na].val.clusterDim.x = 1;
    attrs[na].val.clusterDim.y = 1;
    attrs[na].val.clusterDim.z = static_cast<unsigned>(split);
    ++na;
    if (pdl_enabled()) {
        attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    const int ntile_n = (Nout + kWRows - 1) / kWRows, ntile_m = (M + BNA - 1) / BNA;
    cfg.gridDim = dim3(ntile_n, ntile_m, split);
    cfg.blockDim = dim3(Cf::THREADS, 1, 1);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = st;
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    // clusters the device holds at once, per (split, shared memory), queried once
    static std::mutex mu;
    static int cache_key[32][2];
    static int cache_val[32];
    static int cache_n = 0;
    int active = -1;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < cache_n; ++i)
            if (cache_key[i][0] == split && cache_key[i][1] == static_cast<int>(pl.smem))
                active = cache_val[i];
        if (active < 0) {
            if (cudaOccupancyMaxActiveClusters(&active, kern, &cfg) != cudaSuccess) {
                cudaGetLastError();  // a refused query is not the caller's error
                active = 0;
            }
            if (cache_n < 32) {
                cache_key[cache_n][0] = split;
                cache_key[cache_n][1] = static_cast<int>(pl.smem);
                cache_val[cache_n++] = active;
            }
        }
    }
    if (active < ntile_n * ntile_m) return cudaErrorNotSupported;
    return cudaLaunchKernelEx(&cfg, kern, wmap, amap, amap_1, omap, p);
}

// Up to kMaxGroupCalls calls of tile width BNA in one launch.  The rings are
// sized for the longest partition of any call; ring depth changes neither the
// groups an accumulator receives nor their order, so every call's result is
// the one its own launch gives.
template <int BNA>
int launch_tc_group(const GroupCall* calls, int n, cudaStream_t st) {
    using C = TcCfg<BNA>;
    if (n < 1 || n > kMaxGroupCalls) return cudaErrorInvalidValue;
    auto kern = w4a16_tc_group_kernel<BNA>;
    static int limit = -1;
    static std::once_flag once;
    std::call_once(once, [&] { limit = set_max_dynamic_smem(reinterpret_cast<const void*>(kern)); });
    if (limit < 0) return cudaErrorInvalidValue;
    int* status = tc_status_ptr();
    if (!status) return cudaErrorInvalidSymbol;
    int gpp_max = 1;
    for (int i = 0; i < n; ++i) {
        const int G = calls[i].Kred / kGroup;
        gpp_max = std::max(gpp_max, G / calls[i].split + (G % calls[i].split ? 1 : 0));
    }
    TcPipeline pl;
    if (!tc_pipeline<BNA>(gpp_max, limit, &pl)) return cudaErrorInvalidValue;
    static TcGroup g;  // large: built on the host once per launch, under a lock
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    g.ncalls = n;
    long long ctas = 0;
    for (int i = 0; i < n; ++i) {
        const GroupCall& c = calls[i];
        TcCall& tc = g.call[i];
        if (!setup_call<BNA>(c.A, c.Wq, c.scales, c.biases, c.out, c.out_mode, c.M, c.Kred, c.Nout,
                             c.split, nullptr, nullptr, pl, status, &tc.p, &tc.wmap, &tc.amap,
                             &tc.amap_1, &tc.omap))
            return cudaErrorInvalidValue;
        tc.n_tiles = (c.Nout + kWRows - 1) / kWRows;
        tc.m_tiles = (c.M + BNA - 1) / BNA;
        tc.cta_begin = static_cast<int>(ctas);
        ctas += static_cast<long long>(tc.n_tiles) * tc.m_tiles * c.split;
        if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
    }
    cudaLaunchConfig_t cfg = {};
    LaunchAttrs la;
    apply_pdl(cfg, la);
    cfg.gridDim = dim3(static_cast<unsigned>(ctas), 1, 1);
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, kern, g);
}


// The persistent schedule of a group: the same call table as the one-CTA-per-
// tile launch, min(tiles, SMs) CTAs, outputs stored directly.
template <int BNA>
int launch_tc_persist(const GroupCall* calls, int n, cudaStream_t st) {
    using C = TcCfg<BNA>;
    if (n < 1 || n > kMaxGroupCalls) return cudaErrorInvalidValue;
    auto kern = w4a16_tc_persist_kernel<BNA>;
    static int limit = -1;
    static std::once_flag once;
    std::call_once(once, [&] { limit = set_max_dynamic_smem(reinterpret_cast<const void*>(kern)); });
    if (limit < 0) return cudaErrorInvalidValue;
    int* status = tc_status_ptr();
    if (!status) return cudaErrorInvalidSymbol;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        return cudaErrorInvalidValue;
    int gpp_max = 1;
    for (int i = 0; i < n; ++i) {
        const int G = calls[i].Kred / kGroup;
        gpp_max = std::max(gpp_max, G / calls[i].split + (G % calls[i].split ? 1 : 0));
    }
    TcPipeline pl;
    if (!tc_pipeline<BNA>(gpp_max, limit, &pl, true)) return cudaErrorInvalidValue;
    static TcGroup g;  // large: built on the host once per launch, under a lock
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    g.ncalls = n;
    long long ctas = 0;
    for (int i = 0; i < n; ++i) {
        const GroupCall& c = calls[i];
        TcCall& tc = g.call[i];
        if (!setup_call<BNA>(c.A, c.Wq, c.scales, c.biases, c.out, c.out_mode, c.M, c.Kred, c.Nout,
                             c.split, nullptr, nullptr, pl, status, &tc.p, &tc.wmap, &tc.amap,
                             &tc.amap_1, &tc.omap))
            return cudaErrorInvalidValue;
        tc.p.tma_store = 0;
        tc.n_tiles = (c.Nout + kWRows - 1) / kWRows;
        tc.m_tiles = (c.M + BNA - 1) / BNA;
        tc.cta_begin = static_cast<int>(ctas);
        ctas += static_cast<long long>(tc.n_tiles) * tc.m_tiles * c.split;
        if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
    }
    cudaLaunchConfig_t cfg = {};
    LaunchAttrs la;
    apply_pdl(cfg, la);
    cfg.gridDim = dim3(static_cast<unsigned>(std::min<long long>(ctas, sms)), 1, 1);
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, kern, g, static_cast<int>(ctas));
}

}  // namespace

int tc_pipeline_config(int bm, int gpp, long smem_limit, TcPipeline* out, bool persistent) {
    if (gpp < 1 || !out) return -1;
    switch (bm) {
        case 16: return tc_pipeline<16>(gpp, smem_limit, out, persistent) ? 0 : 1;
        case 32: return tc_pipeline<32>(gpp, smem_limit, out, persistent) ? 0 : 1;
        case 64: return tc_pipeline<64>(gpp, smem_limit, out, persistent) ? 0 : 1;
        case 128: return tc_pipeline<128>(gpp, smem_limit, out, persistent) ? 0 : 1;
        case 256: return tc_pipeline<256>(gpp, smem_limit, out, persistent) ? 0 : 1;
        default: return -1;
    }
}

int launch_w4a16_tc(int bm, const void* A, const uint32_t* Wq, const void* scales,
                    const void* biases, void* out, int out_mode, int M, int Kred, int Nout,
                    int split, void* stream, void* fused_C, uint32_t* counters) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (bm) {
        case 16: return launch_tc<16>(A, Wq, scales, biases, out, out_mode, M, Kred, Nout, split, fused_C, counters, st);
        case 32: return launch_tc<32>(A, Wq, scales, biases, out, out_mode, M, Kred, Nout, split, fused_C, counters, st);
        case 64: return launch_tc<64>(A, Wq, scales, biases, out, out_mode, M, Kred, Nout, split, fused_C, counters, st);
        case 128: return launch_tc<128>(A, Wq, scales, biases, out, out_mode, M, Kred, Nout, split, fused_C, counters, st);
        case 256: return launch_tc<256>(A, Wq, scales, biases, out, out_mode, M, Kred, Nout, split, fused_C, counters, st);
        default: return cudaErrorInvalidValue;
    }
}

int launch_w4a16_tc_cluster(int bm, const void* A, const uint32_t* Wq, const void* scales,
                            const void* biases, void* C, int out_mode, int M, int Kred, int Nout,
                            int split, void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (bm) {
        case 16: return launch_tc_cluster<16>(A, Wq, scales, biases, C, out_mode, M, Kred, Nout, split, st);
        case 32: return launch_tc_cluster<32>(A, Wq, scales, biases, C, out_mode, M, Kred, Nout, split, st);
        case 64: return launch_tc_cluster<64>(A, Wq, scales, biases, C, out_mode, M, Kred, Nout, split, st);
        case 128: return launch_tc_cluster<128>(A, Wq, scales, biases, C, out_mode, M, Kred, Nout, split, st);
        case 256: return launch_tc_cluster<256>(A, Wq, scales, biases, C, out_mode, M, Kred, Nout, split, st);
        default: return cudaErrorNotSupported;
    }
}

int launch_w4a16_tc_group(int bm, const GroupCall* calls, int n, void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // The persistent schedule serves tiles of up to 64 activation rows.  Wider
    // tiles keep one CTA per tile: their epilogues are long, and without an
    // idle ring to stage the tile in, the persistent epilogue stores directly;
    // tensor memory has no room to double-buffer their accumulators; and
    // their activation stages (32-64 KB a group, from L2) need the deeper
    // activation ring.  Measured on the Qwen3-4B projections, 7 calls per
    // group: M = 32 13 % faster, M = 128 6 % and M = 2048 16 % slower.
    if (grouped_persistent() && bm <= 64) {
        switch (bm) {
            case 16: return launch_tc_persist<16>(calls, n, st);
            case 32: return launch_tc_persist<32>(calls, n, st);
            case 64: return launch_tc_persist<64>(calls, n, st);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (bm) {
        case 16: return launch_tc_group<16>(calls, n, st);
        case 32: return launch_tc_group<32>(calls, n, st);
        case 64: return launch_tc_group<64>(calls, n, st);
        case 128: return launch_tc_group<128>(calls, n, st);
        case 256: return launch_tc_group<256>(calls, n, st);
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
