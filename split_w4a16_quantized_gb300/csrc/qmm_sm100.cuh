// Blackwell (sm_100 family, built for sm_103a) primitives in inline PTX:
// mbarriers with bounded waits, TMA tile loads, tensor-memory allocation,
// tcgen05.mma with the A operand in tensor memory, and tcgen05 loads/stores.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "qmm_device.cuh"

namespace qmm {

// Every wait in the tcgen05 kernels gives up after this many nanoseconds,
// records the failure in the status word and lets the kernel wind down.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s

// Kernel status word (device memory); nonzero = a wait timed out.
enum KernelStatus { kStatusOk = 0, kStatusTimeout = 1 };

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- mbarrier ---------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Non-blocking probe: has the phase of `parity` completed?  (try_wait may
// suspend the thread for a while when the phase is still open, which would
// stall a thread that polls several barriers.)
__device__ __forceinline__ bool mbar_probe(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of `parity` to complete.  Returns false (and sets
// *status) if it has not after kWaitLimitNs, or -- when abort is not null --
// as soon as another thread of the CTA has given up (*abort set).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          int* status) {
    if (mbar_test(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_test(bar, parity)) return true;
        if ((i & 255u) == 0) {
            if (abort && *abort) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                if (abort) *abort = 1;
                atomicExch(status, kStatusTimeout);
                return false;
            }
        }
    }
}
// The same wait taken by a whole warp; the result is the same in every lane.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity,
                                               volatile int* abort, int* status) {
    const bool ok = mbar_wait(bar, parity, abort, status);
    return __all_sync(0xffffffffu, ok);
}

// ---- TMA ----------------------------------------------------------------------

// Orders the shared-memory accesses that happen before this point in the
// generic proxy (ordinary loads and stores, including other threads' accesses
// made visible through an mbarrier) before the async-proxy accesses this
// thread issues next (TMA).  A stage read with ordinary loads needs it before
// TMA refills the stage: the mbarrier hand-off alone does not order the two
// proxies.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// Prefetch of a 3-D tile into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int c0, int c1,
                                                   int c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];\n" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}
// Prefetch of a 2-D tile into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int c0, int c1) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];\n" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1)
                 : "memory");
}
// Prefetch of the cache line holding *ptr into L2.
__device__ __forceinline__ void prefetch_l2(const void* ptr) {
    asm volatile("prefetch.global.L2 [%0];\n" ::"l"(ptr));
}
// 2-D tile load into shared memory; completion counted on `bar` in bytes.
// c0 is the innermost coordinate (elements).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];\n" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_addr(bar))
        : "memory");
}

// Contiguous global -> shared copy of `bytes` (a multiple of 16; both
// addresses 16-byte aligned), completion counted on `bar` in bytes.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Named barrier `id` over `threads` threads (whole warps).
__device__ __forceinline__ void named_bar_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(threads) : "memory");
}

// 3-D tile load (c0 innermost), completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
        : "memory");
}

// 3-D tile store from shared memory (c0 innermost); bulk-group completion.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0,
                                             int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];\n" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(src))
        : "memory");
}
__device__ __forceinline__ void tma_store_commit() {
    asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
}
// Wait until the committed stores have read their shared-memory source (the
// global writes complete with the grid, before any dependent grid runs).
__device__ __forceinline__ void tma_store_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
}

// ---- tensor memory ------------------------------------------------------------

// Whole warp: allocate ncols (power of two >= 32) columns; address -> *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                     smem_addr(slot)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

// D[tmem] (+)= A[tmem] * B[smem], kind::f16 (BF16 inputs, FP32 accumulate).
__device__ __forceinline__ void umma_bf16_tmem_a(uint32_t d, uint32_t a, uint64_t bdesc,
                                                 uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
        "r"(a), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on `bar` when every MMA issued so far by this thread is done.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
            smem_addr(bar))
        : "memory");
}

// Instruction descriptor of kind::f16: BF16 A and B, FP32 D, both K-major,
// M x N tile (M in 64/128, N a multiple of 16 up to 256).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4)                              // D format: F32
           | (1u << 7)                            // A format: BF16
           | (1u << 10)                           // B format: BF16
           | (static_cast<uint32_t>(N >> 3) << 17)
           | (static_cast<uint32_t>(M >> 4) << 24);
}

// Shared-memory matrix descriptor, K-major with the 128-byte swizzle: rows of
// 128 bytes, 8-row core groups 1024 bytes apart; the tile starts 1024-aligned
// (an in-atom k offset is added to the start address).
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t saddr) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu)  // start address
           | (static_cast<uint64_t>(1) << 16)               // leading byte offset (unused)
           | (static_cast<uint64_t>(1024 >> 4) << 32)       // stride byte offset
           | (static_cast<uint64_t>(1) << 46)               // descriptor version
           | (static_cast<uint64_t>(2) << 61);              // 128-byte swizzle
}

// 32 lanes x 16 columns of 32 bits: thread i of the warp <-> lane (base + i).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t v[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16};\n" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t v[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15}, [%16];\n"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
          "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}


// ---- thread-block clusters ----------------------------------------------------

// Barrier over every thread of the cluster, ordering shared-memory writes
// before it (release) against reads after it (acquire) across the cluster.
__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_map(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
__device__ __forceinline__ uint4 cluster_ld16(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}


// The cluster reduce of one output tile: `split` partners (cluster ranks
// 0..split-1) each staged their partial tile of rows x cols at `staged`
// ([row][pitch] elements, BF16 or FP32 when f32); this CTA adds its share of
// the rows -- rank r takes rows [r * per, (r + 1) * per), per = ceil(rows /
// split) -- over every partner in ascending rank order in FP32, rounds once
// and stores into C (row-major, leading dimension ldc, already offset to the
// tile).  Called by nthreads threads with index t, between two
// cluster_barrier()s.
static __device__ __noinline__ void cluster_add_tile(const void* staged, int pitch, bool f32, int rows,
                                              int cols, int split, __nv_bfloat16* C, int ldc,
                                              int t, int nthreads) {
    const int rank = static_cast<int>(cluster_rank());
    const int per = (rows + split - 1) / split;
    const int r0 = rank * per, r1 = r0 + per < rows ? r0 + per : rows;
    const int chunks = pitch / 8;
    const uint32_t base = smem_addr(staged);
    for (int it = t; it < (r1 > r0 ? r1 - r0 : 0) * chunks; it += nthreads) {
        const int m = r0 + it / chunks, c8 = (it % chunks) * 8;
        if (c8 >= cols) continue;
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = 0.f;
        const uint32_t off = static_cast<uint32_t>(m * pitch + c8) * (f32 ? 4u : 2u);
        for (int q = 0; q < split; ++q) {
            const uint32_t a = cluster_map(base + off, static_cast<uint32_t>(q));
            if (f32) {
                const uint4 x = cluster_ld16(a), y = cluster_ld16(a + 16);
                v[0] += __uint_as_float(x.x); v[1] += __uint_as_float(x.y);
                v[2] += __uint_as_float(x.z); v[3] += __uint_as_float(x.w);
                v[4] += __uint_as_float(y.x); v[5] += __uint_as_float(y.y);
                v[6] += __uint_as_float(y.z); v[7] += __uint_as_float(y.w);
            } else {
                const uint4 x = cluster_ld16(a);
                const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    v[2 * j] += __uint_as_float(w[j] << 16);
                    v[2 * j + 1] += __uint_as_float(w[j] & 0xFFFF0000u);
                }
            }
        }
        __nv_bfloat16* dst = C + static_cast<size_t>(m) * ldc + c8;
        if ((ldc & 7) == 0 && c8 + 8 <= cols) {
            uint4 o;
            o.x = pack_bf16x2(v[0], v[1]);
            o.y = pack_bf16x2(v[2], v[3]);
            o.z = pack_bf16x2(v[4], v[5]);
            o.w = pack_bf16x2(v[6], v[7]);
            *reinterpret_cast<uint4*>(dst) = o;
        } else {
            for (int j = 0; j < 8 && c8 + j < cols; ++j) dst[j] = __float2bfloat16_rn(v[j]);
        }
    }
}

}  // namespace qmm
