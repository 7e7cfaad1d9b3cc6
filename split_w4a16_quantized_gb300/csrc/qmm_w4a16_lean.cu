// Lean W4A16-g128 partition / unsplit kernel for few activation rows (M <= 32).
//
// Same contract as the other partition kernels (tiny-llm book, "Week 2 Day
// 7: Split-K Prefill", Task 2): grid y = partition, partition p holds
// gq + (p < gr) groups from group p*gq + min(p, gr); split 1 writes C, a
// larger split writes the CTA's tile of partial plane p with no atomics.
//
// At these M a call streams its packed weights once and does little else
// ("Optimize Prefill vs Decode Kernels": decode matmuls are weight-bound and
// should reach most of the HBM bandwidth), so the kernel keeps the fixed
// cost of a call small and the weight stream busy:
//   - a CTA is BN = 16 * RB * WR weight rows (all M activation rows, BM = 8,
//     16 or 32) and WR * WK warps: WR row slices of RB 16-row blocks times WK
//     k slices.  Its shared memory and registers leave room for 512 threads
//     of CTAs on an SM, so several CTAs share an SM and the next call's CTAs
//     can become resident while this call drains (programmatic dependent
//     launch);
//   - weights stream through a ring in shared memory that is private to
//     each thread: every thread copies its own rows' 16-byte chunks of a
//     group with cp.async, WS - 1 groups ahead of the one it computes, and
//     waits for them with cp.async.wait_group -- no barrier, since nobody
//     else reads them.  The bytes in flight wait in shared memory, not in
//     registers.  With the
//     static-weights promise the first copies are issued before the
//     dependency wait; otherwise the CTA's weight lines are prefetched into
//     L2 there (L2 is the point of coherence, so this is safe even if an
//     earlier kernel writes them).  A copy engine is not used for weights: a
//     tile of one group is 64 rows of 64 bytes, and per-row requests of that
//     size kept the copy engine, not the memory, busy;
//   - the CTA's scales and biases are staged in shared memory in one round
//     trip at the start (before the dependency wait with the static-weights
//     promise, else prefetched into L2 before it), so no group waits on them;
//   - activations (read by every warp) come in by TMA, one box of WK groups
//     x BM rows per ring stage, 128-byte swizzled;
//   - warp w owns RB 16-row weight blocks (row slice w / WK) and every
//     WK-th group of the partition (k slice w % WK); it dequantizes its
//     weight words in registers straight into mma.sync m16n8k16 A fragments
//     (weights as the 16-row operand, activations as the 8-column one) -- the
//     legacy MMA is enough here, the weights' bytes are the bound;
//   - the WK k slices' FP32 tiles are added in shared memory in a fixed
//     order, so the result does not depend on timing.
//
// k order.  Thread (g, t) of a warp (g = lane / 4, t = lane % 4) loads the
// 16-byte chunk t of its rows' 64-byte group (packed words 4t..4t+3, k =
// 32t .. 32t+31).  Word 4t+u covers k0 = 32t + 8u .. k0+7 and feeds two MMA
// k-steps: slots (2t, 2t+1) take nibbles (0, 4) then (2, 6), slots (2t+8,
// 2t+9) nibbles (1, 5) then (3, 7).  The activation operand carries the same
// k in the same slots: the thread reads the 16-byte chunk A[m, k0..k0+7] and
// pairs its BF16 values (a0,a4) (a1,a5) (a2,a6) (a3,a7) with byte permutes.
// At step j a thread takes word u = j, except that threads t = 2, 3 take
// u = j ^ 2: then the eight threads of a shared-memory phase read eight
// distinct 16-byte bank groups of the swizzled activation tile.  The
// reduction is a sum over k, so any order a thread uses identically on both
// operands gives the same product.
//
// Dequantization: dequant_word_subnormal (one BF16 fused multiply-add per
// two weights, exact for scales in [2^-126, 2^-5) and zero) when every scale
// a warp needs for a group allows it, else dequant_word; both give
// BF16(scale * q + bias) with one rounding.
//
// Every wait is bounded (mbar_wait): a wait that runs out sets the status
// word, the CTA stops, waits (bounded) for the copies it has in flight and
// exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "qmm_device.cuh"
#include "qmm_internal.h"
#include "qmm_sm100.cuh"

namespace qmm {

bool encode_tiled(CUtensorMap* map, CUtensorMapDataType type, int rank, const void* ptr,
                  const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                  CUtensorMapSwizzle swizzle);

namespace {

constexpr int kThreadsPerSm = 512;         // resident lean threads an SM is sized for
constexpr int kSmemPerSm = 227 << 10;

template <int NT_, int WR_, int WK_, int RB_>
struct LeanCfg {
    static constexpr int NT = NT_, WR = WR_, WK = WK_, RB = RB_;
    static constexpr int BM = 8 * NT;                 // activation rows
    static constexpr int BN = 16 * RB * WR;           // weight rows
    static constexpr int WARPS = WR * WK;
    static constexpr int THREADS = 32 * WARPS;
    static constexpr int MIN_CTAS = kThreadsPerSm / THREADS;  // per SM
    static constexpr int AG = WK;                     // groups per activation stage
    static_assert(AG == WK, "step i of every warp takes activation stage i");
    static constexpr int HALF = BM * 128;             // one 64-k half-group of BM rows
    static constexpr int STAGE = 2 * AG * HALF;       // one TMA box
    static constexpr int WCH = 2 * RB;                // 16-byte weight chunks a thread copies per group
    static constexpr int WS = NT == 4 ? 2 : 4;        // weight ring depth (groups per thread)
    static constexpr int WRING = WS * WCH * THREADS * 16;
    static constexpr int BUDGET = kSmemPerSm / MIN_CTAS - 4096;  // both rings
    static constexpr int NA_MAX = (BUDGET - WRING) / STAGE;
    static constexpr int EPI_LD = BN + 4;             // FP32 epilogue row pitch (floats)
    static constexpr int EPI = WK * BM * EPI_LD * 4;
    static constexpr int STG = BM * BN * 4;           // cluster reduce: the staged partial tile
    static_assert(STAGE % 1024 == 0, "swizzled stages start on 1024-byte boundaries");
    static_assert(NA_MAX >= 2, "ring depth");
};

struct LeanParams {
    const uint32_t* Wq;      // [Nout, Kred/8]
    const uint16_t* scales;  // BF16 bits [Nout, G]
    const uint16_t* biases;
    void* out;               // C (split 1) or the planes [split, M, Nout]
    __nv_bfloat16* C;        // fused reduce: the final output
    uint32_t* counters;      // fused reduce: one per row tile, zero between calls
    int* status;
    int M, Kred, Nout, G;
    int gq, gr, gpp;         // G / split, G % split, longest partition
    int split, out_mode, fused, wstatic;
    int na;                  // activation ring stages
    int ring_bytes;          // shared memory of the activation ring (and epilogue buffer)
    int cluster;             // 1: the partitions of a column tile are one cluster and add
                             //    their staged partial tiles into C (cluster reduce)
};

// Per-thread view of the CTA: row slice rs, k slice ks, lane (g, t).
template <class Cfg>
struct Lane {
    int tid, lane, ks, rs, g, t, n0;
    __device__ __forceinline__ Lane(int n0_) : tid(threadIdx.x), lane(threadIdx.x & 31), n0(n0_) {
        const int warp = tid >> 5;
        ks = warp % Cfg::WK;
        rs = warp / Cfg::WK;
        g = lane >> 2;
        t = lane & 3;
    }
    // weight row of block rb, half h (rows g and g + 8 of the block)
    __device__ __forceinline__ int row(int rb, int h) const {
        return n0 + (rs * Cfg::RB + rb) * 16 + g + 8 * h;
    }
};

// This thread's weight chunks: chunk k = 2*rb + h is row L.row(rb, h), bytes
// 16t..16t+15 of each group; rows past Nout are zero-filled.  Sources and
// ring positions are formed once per CTA, so a group's copies cost one address
// add each.  Layout [slot][k][thread] keeps every 16-byte access of a warp
// conflict free.
template <class Cfg>
struct WeightCopies {
    static constexpr uint32_t SLOT_BYTES = Cfg::WCH * Cfg::THREADS * 16;
    const uint32_t* src[Cfg::RB][2];  // the row's words 4t.. of group 0
    uint32_t dst[Cfg::RB][2];         // the chunk's position in slot 0
    bool ok[Cfg::RB][2];
    __device__ __forceinline__ WeightCopies(const uint8_t* wring, const LeanParams& p,
                                            const Lane<Cfg>& L) {
        const size_t wrow = static_cast<size_t>(p.Kred) / 8;
#pragma unroll
        for (int rb = 0; rb < Cfg::RB; ++rb)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int n = L.row(rb, h);
                ok[rb][h] = n < p.Nout;
                src[rb][h] = p.Wq + static_cast<size_t>(ok[rb][h] ? n : 0) * wrow + L.t * 4;
                dst[rb][h] = smem_addr(wring + ((2 * rb + h) * Cfg::THREADS + L.tid) * 16);
            }
    }
    // copy group `grp` (absolute) into ring slot `slot`
    __device__ __forceinline__ void copy(int slot, int grp) const {
#pragma unroll
        for (int rb = 0; rb < Cfg::RB; ++rb)
#pragma unroll
            for (int h = 0; h < 2; ++h)
                cp_async16(dst[rb][h] + slot * SLOT_BYTES, src[rb][h] + grp * 16, ok[rb][h]);
    }
};

// Read slot `slot` back; threads t >= 2 swap words (0,1) with (2,3) (see the
// k order above).
template <class Cfg>
__device__ __forceinline__ void read_weights(uint4 (&w)[Cfg::RB][2], const uint8_t* wring,
                                             int slot, const Lane<Cfg>& L) {
#pragma unroll
    for (int rb = 0; rb < Cfg::RB; ++rb)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint4 v = *reinterpret_cast<const uint4*>(
                wring + ((slot * Cfg::WCH + 2 * rb + h) * Cfg::THREADS + L.tid) * 16);
            w[rb][h] = L.t >= 2 ? make_uint4(v.z, v.w, v.x, v.y) : v;
        }
}

// One group of one warp: the group's two activation halves start at act0 /
// act1 (BM rows of 128 swizzled bytes each).
template <class Cfg, bool SUB>
__device__ __forceinline__ void lean_group(const uint8_t* act0, const uint8_t* act1,
                                           const uint4 (&wv)[Cfg::RB][2],
                                           const uint32_t (&c0)[Cfg::RB][2],
                                           const uint32_t (&c1)[Cfg::RB][2],
                                           const uint32_t (&cb)[Cfg::RB][2], int g, int t,
                                           float (&acc)[Cfg::RB][Cfg::NT][4]) {
    const uint8_t* half = t >= 2 ? act1 : act0;
    const int sw = 2 * (t >> 1);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        // this k chunk of every weight row of the warp, dequantized
        uint32_t d[Cfg::RB][2][4];
#pragma unroll
        for (int rb = 0; rb < Cfg::RB; ++rb)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t word = j == 0 ? wv[rb][h].x : j == 1 ? wv[rb][h].y
                                    : j == 2 ? wv[rb][h].z : wv[rb][h].w;
                if (SUB)
                    dequant_word_subnormal(word, c0[rb][h], c1[rb][h], cb[rb][h], d[rb][h]);
                else
                    dequant_word(word, c0[rb][h], cb[rb][h], d[rb][h]);
            }
        // chunk 4t + u of the group, u = j ^ sw: in its half, chunk 4(t & 1) + u,
        // stored at position (chunk ^ row) of the row's 128 bytes
        const int c = 4 * (t & 1) + (j ^ sw);
#pragma unroll
        for (int nt = 0; nt < Cfg::NT; ++nt) {
            const uint4 v = *reinterpret_cast<const uint4*>(half + (nt * 8 + g) * 128 +
                                                            ((c ^ g) << 4));
            const uint32_t b0 = __byte_perm(v.x, v.z, 0x5410);  // (a0, a4)
            const uint32_t b1 = __byte_perm(v.x, v.z, 0x7632);  // (a1, a5)
            const uint32_t b2 = __byte_perm(v.y, v.w, 0x5410);  // (a2, a6)
            const uint32_t b3 = __byte_perm(v.y, v.w, 0x7632);  // (a3, a7)
#pragma unroll
            for (int rb = 0; rb < Cfg::RB; ++rb) {
                const uint32_t a0[4] = {d[rb][0][0], d[rb][1][0], d[rb][0][1], d[rb][1][1]};
                const uint32_t a1[4] = {d[rb][0][2], d[rb][1][2], d[rb][0][3], d[rb][1][3]};
                mma_bf16_16816(acc[rb][nt], a0, b0, b1);
                mma_bf16_16816(acc[rb][nt], a1, b2, b3);
            }
        }
    }
}

// Shared state of one CTA.
struct LeanShared {
    uint8_t* ring;
    uint64_t* full;
    uint64_t* empty;
    int* abort;
    int* issued;  // activation stages issued so far (thread 0)
};

// Scales of the CTA's groups, in place in shared memory ([group][row]): a group
// whose every row's scale suits the one-FMA dequant (scale_subnormal_ok) gets
// its scales as scale * 2^133 (the halves scale_shifted_pair forms), and
// gbad[group] = 0; any other group keeps its raw scales for dequant_word and
// gets gbad[group] = 1.  gbad must be zero beforehand; all threads call this,
// and a barrier must follow before the scales are read.
template <class Cfg>
__device__ __forceinline__ void prepare_scales(uint16_t* sc, uint8_t* gbad, int gpp) {
    for (int i = threadIdx.x; i < gpp * Cfg::BN; i += Cfg::THREADS)
        if (!scale_subnormal_ok(sc[i])) gbad[i / Cfg::BN] = 1;
    __syncthreads();
    for (int i = threadIdx.x; i < gpp * Cfg::BN; i += Cfg::THREADS)
        if (!gbad[i / Cfg::BN]) sc[i] = static_cast<uint16_t>(scale_shifted_pair(sc[i], 133));
}

// Step st of one warp: its group gi = ks + WK * st, whose weights are in slot
// wslot of the thread's ring (landed); activation stage st sits in ring slot
// `slot` with parity `phase`; the CTA's scales (prepared) and biases are in
// sc / bi ([group][row]).  Returns false if a wait ran out.  Releases the
// activation stage (every warp takes one group of each stage); thread 0 then
// refills the slot with stage st + na once every warp has released it.
template <class Cfg>
__device__ __forceinline__ bool lean_step(const LeanShared& sh, const CUtensorMap* amap,
                                          const LeanParams& p, const Lane<Cfg>& L, int gbeg,
                                          int nst, int st, int slot, uint32_t phase,
                                          const uint8_t* wring, int wslot, const uint16_t* sc,
                                          const uint16_t* bi, const uint8_t* gbad,
                                          float (&acc)[Cfg::RB][Cfg::NT][4]) {
    const int na = p.na;
    const int gi = L.ks + Cfg::WK * st;
    if (!mbar_wait_warp(&sh.full[slot], phase, sh.abort, p.status)) return false;
    uint4 wv[Cfg::RB][2];
    read_weights<Cfg>(wv, wring, wslot, L);
    uint32_t c0[Cfg::RB][2], c1[Cfg::RB][2], cb[Cfg::RB][2];
#pragma unroll
    for (int rb = 0; rb < Cfg::RB; ++rb)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int R = L.row(rb, h) - L.n0;
            c0[rb][h] = bf16_pair(sc[gi * Cfg::BN + R]);
            cb[rb][h] = bf16_pair(bi[gi * Cfg::BN + R]);
        }
    const uint8_t* act0 = sh.ring + slot * Cfg::STAGE + (2 * L.ks) * Cfg::HALF;
    const uint8_t* act1 = act0 + Cfg::HALF;
    if (gbad[gi] == 0) {
        // c0 holds scale * 2^133; scale * 2^129 is 4 exponent steps lower,
        // except for a zero scale (either sign), which stays as it is
#pragma unroll
        for (int rb = 0; rb < Cfg::RB; ++rb)
#pragma unroll
            for (int h = 0; h < 2; ++h)
                c1[rb][h] = (c0[rb][h] & 0x7FFFu) ? c0[rb][h] - 0x02000200u : c0[rb][h];
        lean_group<Cfg, true>(act0, act1, wv, c0, c1, cb, L.g, L.t, acc);
    } else {
#pragma unroll
        for (int rb = 0; rb < Cfg::RB; ++rb)
#pragma unroll
            for (int h = 0; h < 2; ++h) c1[rb][h] = 0;
        lean_group<Cfg, false>(act0, act1, wv, c0, c1, cb, L.g, L.t, acc);
    }
    __syncwarp();
    if (L.lane == 0) mbar_arrive(&sh.empty[slot]);
    if (L.tid == 0 && st + na < nst) {
        if (mbar_wait(&sh.empty[slot], phase, sh.abort, p.status)) {
            fence_proxy_async_smem();  // the stage was read with ordinary loads
            mbar_arrive_expect_tx(&sh.full[slot], Cfg::STAGE);
            tma_load_3d(sh.ring + slot * Cfg::STAGE, amap, &sh.full[slot], 0, 0,
                        (gbeg + (st + na) * Cfg::AG) * 2);
            *sh.issued = st + na + 1;
        }
    }
    return !__any_sync(0xffffffffu, *static_cast<volatile int*>(sh.abort) != 0);
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, Cfg::MIN_CTAS)
    w4a16_lean_kernel(const __grid_constant__ CUtensorMap amap, const LeanParams p) {
    constexpr int BM = Cfg::BM, BN = Cfg::BN, RB = Cfg::RB, NT = Cfg::NT, WK = Cfg::WK;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int na = p.na;
    uint8_t* wring = ring + p.ring_bytes;  // [WS][WCH][THREADS] x 16 bytes
    uint16_t* sc = reinterpret_cast<uint16_t*>(wring + Cfg::WRING);  // [group][BN]
    uint16_t* bi = sc + p.gpp * BN;
    uint64_t* full = reinterpret_cast<uint64_t*>(bi + p.gpp * BN);
    uint64_t* empty = full + na;
    uint8_t* gbad = reinterpret_cast<uint8_t*>(empty + na);  // [group]: raw scales
    __shared__ int abort_flag;
    __shared__ int last_flag;
    __shared__ int issued;

    const int part = blockIdx.y, n0 = blockIdx.x * BN;
    const Lane<Cfg> L(n0);
    const int tid = L.tid;
    const int ngrp = p.gq + (part < p.gr ? 1 : 0);
    const int gbeg = part * p.gq + (part < p.gr ? part : p.gr);
    const int nst = (ngrp + Cfg::AG - 1) / Cfg::AG;
    const LeanShared sh{ring, full, empty, &abort_flag, &issued};
    const WeightCopies<Cfg> wc(wring, p, L);
    for (int g = tid; g < ngrp; g += Cfg::THREADS) gbad[g] = 0;

    if (tid == 0) {
        for (int s = 0; s < na; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], Cfg::WARPS);
        }
        abort_flag = 0;
        issued = 0;
        mbar_fence_init();
        tma_prefetch_map(&amap);
    }
    pdl_trigger();
    // this warp's groups are ks, ks + WK, ...; its i-th group goes to ring slot
    // i % WS, and copy commit i carries it (empty commits keep the count)
    const int nmine = ngrp > L.ks ? (ngrp - L.ks + WK - 1) / WK : 0;
    auto issue = [&](int i) {
        if (i < nmine) wc.copy(i % Cfg::WS, gbeg + L.ks + WK * i);
        cp_async_commit();
    };
    auto load_scales = [&] {
        for (int i = tid; i < 2 * BN; i += Cfg::THREADS) {
            const int r = i % BN;
            load_group_row(i < BN ? p.scales : p.biases, p.Nout, p.G, n0 + r, gbeg, ngrp,
                           (i < BN ? sc : bi) + r, BN);
        }
    };
    if (p.wstatic) {
        // weights (packed words, scales and biases) are not written by earlier
        // kernels: start their copies and loads before the wait
        for (int i = 0; i < Cfg::WS - 1; ++i) issue(i);
        load_scales();
    } else {
        // weights are read-only inputs: bring this CTA's weight, scale and bias
        // lines into L2 while the previous kernel finishes
        const uint8_t* wq = reinterpret_cast<const uint8_t*>(p.Wq);
        const int len = ngrp * 64;
        for (int i = tid; i < BN * 4; i += Cfg::THREADS) {
            const int n = n0 + i / 4;
            if (n >= p.Nout) continue;
            const uint8_t* row = wq + static_cast<size_t>(n) * (p.Kred / 2) + static_cast<size_t>(gbeg) * 64;
            for (int off = (i & 3) * 128; off < len + 128; off += 512)
                prefetch_l2(row + (off < len ? off : len - 1));
        }
        for (int i = tid; i < 2 * BN; i += Cfg::THREADS) {
            const int n = n0 + i % BN;
            if (n >= p.Nout) continue;
            const uint16_t* row = (i < BN ? p.scales : p.biases) + static_cast<size_t>(n) * p.G + gbeg;
            prefetch_l2(row);
            prefetch_l2(row + ngrp - 1);
        }
    }
    __syncthreads();  // barriers initialised (and with the promise, scales loaded)
    if (p.wstatic) prepare_scales<Cfg>(sc, gbad, ngrp);
    pdl_wait();
    if (!p.wstatic) {
        for (int i = 0; i < Cfg::WS - 1; ++i) issue(i);
        load_scales();
    }
    if (tid == 0) {
        const int first = nst < na ? nst : na;
        for (int s = 0; s < first; ++s) {
            mbar_arrive_expect_tx(&full[s], Cfg::STAGE);
            tma_load_3d(ring + s * Cfg::STAGE, &amap, &full[s], 0, 0, (gbeg + s * Cfg::AG) * 2);
        }
        issued = first;
    }
    __syncthreads();  // scales and biases in shared memory
    if (!p.wstatic) {
        prepare_scales<Cfg>(sc, gbad, ngrp);
        __syncthreads();
    }

    float acc[RB][NT][4];
#pragma unroll
    for (int rb = 0; rb < RB; ++rb)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[rb][nt][c] = 0.f;

    // step i takes activation stage i (AG == WK: one group of every warp)
    int slot = 0;
    uint32_t phase = 0;
    for (int i = 0; i < nmine; ++i) {
        issue(i + Cfg::WS - 1);  // the slot of group i - 1 was read last iteration
        cp_async_wait<Cfg::WS - 1>();  // this thread's copies of group i have landed
        if (!lean_step<Cfg>(sh, &amap, p, L, gbeg, nst, i, slot, phase, wring, i % Cfg::WS, sc,
                            bi, gbad, acc))
            break;
        if (++slot == na) {
            slot = 0;
            phase ^= 1;
        }
    }
    cp_async_wait<0>();

    // every activation box issued must land before the ring is reused or the
    // CTA exits: they all have unless a wait ran out
    __syncthreads();
    if (tid == 0 && abort_flag) {
        const int n = issued;
        for (int st = n > na ? n - na : 0; st < n; ++st)
            mbar_wait(&full[st % na], (st / na) & 1, nullptr, p.status);
    }

    // ---- epilogue: add the k slices in order, store the tile ----------------
    __syncthreads();  // the ring becomes the buffer
    float* red = reinterpret_cast<float*>(ring);  // [WK][BM][EPI_LD]
#pragma unroll
    for (int rb = 0; rb < RB; ++rb)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int R = (L.rs * RB + rb) * 16 + L.g;
            const int mr = nt * 8 + 2 * L.t;
            float* r0 = red + (L.ks * BM + mr) * Cfg::EPI_LD;
            r0[R] = acc[rb][nt][0];
            r0[Cfg::EPI_LD + R] = acc[rb][nt][1];
            r0[R + 8] = acc[rb][nt][2];
            r0[Cfg::EPI_LD + R + 8] = acc[rb][nt][3];
        }
    __syncthreads();

    const size_t plane = static_cast<size_t>(part) * p.M * p.Nout;
    const bool vec8 = (p.Nout & 7) == 0;
    for (int it = tid; it < BM * (BN / 8); it += Cfg::THREADS) {
        const int m = it / (BN / 8), c = it % (BN / 8);
        const int n = n0 + c * 8;
        if (m >= p.M || n >= p.Nout) continue;
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = 0.f;
#pragma unroll
        for (int k = 0; k < WK; ++k) {
            const float4* src = reinterpret_cast<const float4*>(red + (k * BM + m) * Cfg::EPI_LD + c * 8);
            const float4 x = src[0], y = src[1];
            v[0] += x.x; v[1] += x.y; v[2] += x.z; v[3] += x.w;
            v[4] += y.x; v[5] += y.y; v[6] += y.z; v[7] += y.w;
        }
        if (p.cluster) {
            // the partition's tile, rounded as its plane would be, stays on chip
            uint8_t* stg = ring + Cfg::EPI;
            if (p.out_mode == kOutBf16) {
                uint4 w;
                w.x = pack_bf16x2(v[0], v[1]);
                w.y = pack_bf16x2(v[2], v[3]);
                w.z = pack_bf16x2(v[4], v[5]);
                w.w = pack_bf16x2(v[6], v[7]);
                *reinterpret_cast<uint4*>(stg + (m * BN + c * 8) * 2) = w;
            } else {
                float4* dst = reinterpret_cast<float4*>(stg + (m * BN + c * 8) * 4);
                dst[0] = make_float4(v[0], v[1], v[2], v[3]);
                dst[1] = make_float4(v[4], v[5], v[6], v[7]);
            }
            continue;
        }
        const size_t o = plane + static_cast<size_t>(m) * p.Nout + n;
        if (p.out_mode == kOutBf16) {
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + o;
            if (vec8) {
                uint4 w;
                w.x = pack_bf16x2(v[0], v[1]);
                w.y = pack_bf16x2(v[2], v[3]);
                w.z = pack_bf16x2(v[4], v[5]);
                w.w = pack_bf16x2(v[6], v[7]);
                *reinterpret_cast<uint4*>(dst) = w;
            } else {
                for (int j = 0; j < 8 && n + j < p.Nout; ++j) dst[j] = __float2bfloat16_rn(v[j]);
            }
        } else {
            float* dst = static_cast<float*>(p.out) + o;
            if (vec8) {
                reinterpret_cast<float4*>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
                reinterpret_cast<float4*>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
            } else {
                for (int j = 0; j < 8 && n + j < p.Nout; ++j) dst[j] = v[j];
            }
        }
    }

    if (p.cluster) {
        // every thread of every partition's CTA passes both barriers, also
        // after a wait ran out (C is then invalid, as the status word says)
        cluster_barrier();  // every partner's partial tile is staged
        cluster_add_tile(ring + Cfg::EPI, BN, p.out_mode == kOutF32, p.M,
                         p.Nout - n0 < BN ? p.Nout - n0 : BN, p.split, p.C + n0, p.Nout, tid,
                         Cfg::THREADS);
        cluster_barrier();  // every partner has read this CTA's tile
        return;
    }

    if (p.fused) {
        // Count this CTA's plane in; the CTA that brings the tile's count to
        // the split adds the planes in ascending order in FP32 and rounds
        // once, as the reduce kernel does.  A CTA whose wait ran out still
        // counts in (its plane is invalid, and so is C, which the status
        // word reports), so the counter always returns to zero.
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            const unsigned prev = atomicAdd(&p.counters[blockIdx.x], 1u);
            last_flag = prev == static_cast<unsigned>(p.split) - 1;
            if (last_flag) {
                p.counters[blockIdx.x] = 0;
                __threadfence();
            }
        }
        __syncthreads();
        if (last_flag) {
            const size_t pl = static_cast<size_t>(p.M) * p.Nout;
            for (int it = tid; it < p.M * (BN / 8); it += Cfg::THREADS) {
                const int m = it / (BN / 8), c = it % (BN / 8);
                const int n = n0 + c * 8;
                if (n >= p.Nout) continue;
                const size_t o = static_cast<size_t>(m) * p.Nout + n;
                const int cols = p.Nout - n < 8 ? p.Nout - n : 8;
                float v[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) v[j] = 0.f;
                for (int q = 0; q < p.split; ++q) {
                    if (p.out_mode == kOutBf16) {
                        const __nv_bfloat16* s = static_cast<const __nv_bfloat16*>(p.out) + q * pl + o;
                        if (cols == 8 && vec8) {
                            const uint4 u = __ldcg(reinterpret_cast<const uint4*>(s));
                            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                v[2 * j] += __uint_as_float(w[j] << 16);
                                v[2 * j + 1] += __uint_as_float(w[j] & 0xFFFF0000u);
                            }
                        } else {
                            for (int j = 0; j < cols; ++j) v[j] += __bfloat162float(__ldcg(s + j));
                        }
                    } else {
                        const float* s = static_cast<const float*>(p.out) + q * pl + o;
                        if (cols == 8 && vec8) {
                            const float4 x = __ldcg(reinterpret_cast<const float4*>(s));
                            const float4 y = __ldcg(reinterpret_cast<const float4*>(s) + 1);
                            v[0] += x.x; v[1] += x.y; v[2] += x.z; v[3] += x.w;
                            v[4] += y.x; v[5] += y.y; v[6] += y.z; v[7] += y.w;
                        } else {
                            for (int j = 0; j < cols; ++j) v[j] += __ldcg(s + j);
                        }
                    }
                }
                __nv_bfloat16* dst = p.C + o;
                if (cols == 8 && vec8) {
                    uint4 w;
                    w.x = pack_bf16x2(v[0], v[1]);
                    w.y = pack_bf16x2(v[2], v[3]);
                    w.z = pack_bf16x2(v[4], v[5]);
                    w.w = pack_bf16x2(v[6], v[7]);
                    *reinterpret_cast<uint4*>(dst) = w;
                } else {
                    for (int j = 0; j < cols; ++j) dst[j] = __float2bfloat16_rn(v[j]);
                }
            }
        }
    }
}

template <class Cfg>
int launch_cfg(const LeanParams& p0, const void* A, int split, cudaStream_t stream) {
    auto kern = w4a16_lean_kernel<Cfg>;
    static int limit = -1;
    static std::once_flag once;
    std::call_once(once, [&] {
        limit = set_max_dynamic_smem(reinterpret_cast<const void*>(kern));
        if (limit >= 0 && cudaFuncSetAttribute(reinterpret_cast<const void*>(kern),
                                               cudaFuncAttributeNonPortableClusterSizeAllowed,
                                               1) != cudaSuccess)
            limit = -1;
    });
    if (limit < 0) return p0.cluster ? cudaErrorNotSupported : cudaErrorInvalidValue;
    LeanParams p = p0;
    const int nst = (p.gpp + Cfg::AG - 1) / Cfg::AG;
    p.na = nst < Cfg::NA_MAX ? nst : Cfg::NA_MAX;
    const int epi = Cfg::EPI + Cfg::STG;
    const int ring = p.na * Cfg::STAGE > epi ? p.na * Cfg::STAGE : epi;
    p.ring_bytes = (ring + 1023) / 1024 * 1024;
    const size_t smem = 1024 + static_cast<size_t>(p.ring_bytes) + Cfg::WRING +
                        static_cast<size_t>(p.gpp) * Cfg::BN * 4 + static_cast<size_t>(p.na) * 16 +
                        (static_cast<size_t>(p.gpp) + 15) / 16 * 16;
    if (smem > static_cast<size_t>(limit)) return cudaErrorInvalidValue;
    // activations as [64-k half][row][64] boxes of 2 * AG halves x BM rows
    // (rows past M read as zeros), 128-byte swizzle
    CUtensorMap amap;
    const cuuint64_t adims[3] = {64, static_cast<cuuint64_t>(p.M),
                                 static_cast<cuuint64_t>(p.Kred / 64)};
    const cuuint64_t astr[2] = {static_cast<cuuint64_t>(p.Kred) * 2, 128};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(Cfg::BM), 2 * Cfg::AG};
    if (!encode_tiled(&amap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, A, adims, astr, box,
                      CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    LaunchAttrs la;
    apply_pdl(cfg, la);
    cfg.gridDim = dim3((p.Nout + Cfg::BN - 1) / Cfg::BN, split, 1);
    cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    if (!p.cluster) return cudaLaunchKernelEx(&cfg, kern, amap, p);
    // cluster reduce: the split partitions of a column tile form one cluster;
    // taken only if the device holds every cluster of the call at once
    if (split < 2 || split > 16) return cudaErrorNotSupported;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    attrs[na].id = cudaLaunchAttributeClusterDimension;
    attrs[na].val.clusterDim.x = 1;
    attrs[na].val.clusterDim.y = static_cast<unsigned>(split);
    attrs[na].val.clusterDim.z = 1;
    ++na;
    if (cfg.numAttrs) attrs[na++] = la.attr[0];
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
            if (cache_key[i][0] == split && cache_key[i][1] == static_cast<int>(smem))
                active = cache_val[i];
        if (active < 0) {
            if (cudaOccupancyMaxActiveClusters(&active, kern, &cfg) != cudaSuccess) {
                cudaGetLastError();  // a refused query is not the caller's error
                active = 0;
            }
            if (cache_n < 32) {
                cache_key[cache_n][0] = split;
                cache_key[cache_n][1] = static_cast<int>(smem);
                cache_val[cache_n++] = active;
            }
        }
    }
    if (active < static_cast<int>(cfg.gridDim.x)) return cudaErrorNotSupported;
    return cudaLaunchKernelEx(&cfg, kern, amap, p);
}

// Configurations by activation tile width (kLeanFamilies: bm, bn and CTAs
// per SM must agree).
using Lean8 = LeanCfg<1, 2, 4, 1>;
using Lean16 = LeanCfg<2, 2, 4, 1>;
using Lean32 = LeanCfg<4, 2, 4, 1>;
static_assert(Lean8::BM == kLeanFamilies[0].bm && Lean8::BN == kLeanFamilies[0].bn &&
                  Lean8::MIN_CTAS == kLeanFamilies[0].ctas_per_sm, "lean family 0");
static_assert(Lean16::BM == kLeanFamilies[1].bm && Lean16::BN == kLeanFamilies[1].bn &&
                  Lean16::MIN_CTAS == kLeanFamilies[1].ctas_per_sm, "lean family 1");
static_assert(Lean32::BM == kLeanFamilies[2].bm && Lean32::BN == kLeanFamilies[2].bn &&
                  Lean32::MIN_CTAS == kLeanFamilies[2].ctas_per_sm, "lean family 2");

}  // namespace

namespace {
int launch_lean(int bm, const void* A, const uint32_t* Wq, const void* scales,
                const void* biases, void* out, int out_mode, int M, int Kred, int Nout,
                int split, void* stream, void* fused_C, uint32_t* counters, bool cluster);
}  // namespace

int launch_w4a16_lean(int bm, const void* A, const uint32_t* Wq, const void* scales,
                      const void* biases, void* out, int out_mode, int M, int Kred, int Nout,
                      int split, void* stream, void* fused_C, uint32_t* counters) {
    return launch_lean(bm, A, Wq, scales, biases, out, out_mode, M, Kred, Nout, split, stream,
                       fused_C, counters, false);
}

int launch_w4a16_lean_cluster(int bm, const void* A, const uint32_t* Wq, const void* scales,
                              const void* biases, void* C, int out_mode, int M, int Kred,
                              int Nout, int split, void* stream) {
    return launch_lean(bm, A, Wq, scales, biases, C, out_mode, M, Kred, Nout, split, stream, C,
                       nullptr, true);
}

namespace {
int launch_lean(int bm, const void* A, const uint32_t* Wq, const void* scales,
                const void* biases, void* out, int out_mode, int M, int Kred, int Nout,
                int split, void* stream, void* fused_C, uint32_t* counters, bool cluster) {
    if (M > bm || split < 1) return cluster ? cudaErrorNotSupported : cudaErrorInvalidValue;
    LeanParams p = {};
    p.Wq = Wq;
    p.scales = static_cast<const uint16_t*>(scales);
    p.biases = static_cast<const uint16_t*>(biases);
    p.out = out;
    p.C = static_cast<__nv_bfloat16*>(fused_C);
    p.counters = counters;
    p.status = tc_status_ptr();
    if (!p.status) return cudaErrorInvalidValue;
    p.M = M;
    p.Kred = Kred;
    p.Nout = Nout;
    p.G = Kred / kGroup;
    p.gq = p.G / split;
    p.gr = p.G % split;
    p.gpp = p.gq + (p.gr ? 1 : 0);
    p.split = split;
    p.out_mode = out_mode;
    p.fused = fused_C != nullptr && counters != nullptr && split > 1 ? 1 : 0;
    p.cluster = cluster ? 1 : 0;
    p.wstatic = weights_static() && pdl_enabled() ? 1 : 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (bm) {
        case 8: return launch_cfg<Lean8>(p, A, split, st);
        case 16: return launch_cfg<Lean16>(p, A, split, st);
        case 32: return launch_cfg<Lean32>(p, A, split, st);
        default: return cluster ? cudaErrorNotSupported : cudaErrorInvalidValue;
    }
}
}  // namespace

}  // namespace qmm
