// Device helpers shared by the libqmm kernels (inline PTX for sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace qmm {

// Programmatic dependent launch.  pdl_trigger lets the next kernel on the
// stream begin launching (its blocks run up to their own pdl_wait);
// pdl_wait blocks until the kernels before this one on the stream have
// completed and their memory writes are visible.  Without the launch
// attribute both are no-ops.
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte asynchronous global->shared copy; pred == false fills 16 zero bytes
// (src-size 0) and reads nothing from src.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool pred) {
    const int n = pred ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// d = a * b + c on two BF16 lanes, one rounding to nearest even (fused).
__device__ __forceinline__ uint32_t fma_bf16x2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;\n" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// (x & 0x000F000F) | 0x43004300: the nibbles at bits 0..3 and 16..19 of x
// become the BF16 pair (128 + lo, 128 + hi).  128 = 0x4300 has a unit last
// mantissa place, so OR-ing a 4-bit integer into the mantissa adds it exactly.
__device__ __forceinline__ uint32_t nibbles_to_bf16x2_biased(uint32_t x) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;\n" : "=r"(r) : "r"(x), "n"(0x000F000F), "n"(0x43004300));
    return r;
}

constexpr uint32_t kBf16x2One = 0x3F803F80u;     // (1.0, 1.0)
constexpr uint32_t kBf16x2Neg128 = 0xC300C300u;  // (-128, -128)

// Dequantize one packed word (eight 4-bit q, low nibble first) with the
// group's scale and bias, each replicated in both halves of ss / bb.
// out[i] holds the BF16 pair (w(nibble i), w(nibble i + 4)), i = 0..3.
// Each w is BF16(scale * q + bias) with a single rounding: q is formed
// exactly as (128 + q) - 128, and the fused multiply-add rounds once.
__device__ __forceinline__ void dequant_word(uint32_t word, uint32_t ss, uint32_t bb,
                                             uint32_t out[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t biased = nibbles_to_bf16x2_biased(word >> (4 * i));
        const uint32_t q = fma_bf16x2(biased, kBf16x2One, kBf16x2Neg128);
        out[i] = fma_bf16x2(q, ss, bb);
    }
}

// Dequantization with one fused multiply-add per pair of weights.
//
// A BF16 whose exponent field is zero is subnormal: bits m (7-bit mantissa)
// stand for m * 2^-133.  A nibble q masked into bits 0..3 of a half is thus
// the exact value q * 2^-133, and a nibble left in bits 4..7 is q * 2^-129
// (for q >= 8 bit 7 is the exponent's lowest bit, and the normal number
// 2^-126 + (q - 8) * 2^-129 is again q * 2^-129: the subnormal range joins
// the normal one without a gap).  With the scale pre-multiplied by the
// matching power of two -- an exact exponent shift -- one fused BF16
// multiply-add gives q * scale + bias with a single rounding, the value the
// two-step dequant_word forms.
//
// The shifted scale is exact only for a normal scale whose exponent leaves
// room for +133: biased exponent 1..121, i.e. 2^-126 <= |scale| < 2^-5, or a
// zero scale (left as it is).  scale_subnormal_ok tells which; a group with
// any other scale takes dequant_word.
__device__ __forceinline__ bool scale_subnormal_ok(uint16_t s) {
    const uint32_t e = (s >> 7) & 0xFFu;
    return (s & 0x7FFFu) == 0 || (e >= 1 && e <= 121);
}
// scale * 2^k as BF16 bits replicated in both halves (k = 129 or 133; the
// scale satisfies scale_subnormal_ok)
__device__ __forceinline__ uint32_t scale_shifted_pair(uint16_t s, uint32_t k) {
    const uint32_t v = (s & 0x7FFFu) == 0 ? s : s + (k << 7);
    return (v & 0xFFFFu) * 0x00010001u;
}
// out[i] holds the BF16 pair (w(nibble i), w(nibble i + 4)), i = 0..3, as
// dequant_word lays them out; s133 / s129 are scale_shifted_pair(scale, 133 /
// 129), bb the bias pair.
__device__ __forceinline__ void dequant_word_subnormal(uint32_t word, uint32_t s133, uint32_t s129,
                                                       uint32_t bb, uint32_t out[4]) {
    const uint32_t w8 = word >> 8;
    out[0] = fma_bf16x2(word & 0x000F000Fu, s133, bb);
    out[1] = fma_bf16x2(word & 0x00F000F0u, s129, bb);
    out[2] = fma_bf16x2(w8 & 0x000F000Fu, s133, bb);
    out[3] = fma_bf16x2(w8 & 0x00F000F0u, s129, bb);
}

// scale and bias BF16 bit patterns replicated into both halves of a pair
__device__ __forceinline__ uint32_t bf16_pair(uint16_t v) {
    return static_cast<uint32_t>(v) * 0x00010001u;
}

// Copy one row of a per-group parameter array (scales or biases, BF16
// [Nout, G], 16-byte-aligned base) for groups [gbeg, gbeg + gpp) into
// dst[gi * stride].  The row's values are contiguous, so they are fetched as
// whole 16-byte chunks (up to eight loads in flight per thread, one memory
// round trip per 64 groups) and unpacked in registers; a chunk that would
// cross the end of the array is read element by element.  Rows at or past
// Nout get zeros.
__device__ __forceinline__ void load_group_row(const uint16_t* __restrict__ src, int Nout, int G,
                                               int n, int gbeg, int gpp, uint16_t* dst,
                                               int stride) {
    if (n >= Nout) {
        for (int gi = 0; gi < gpp; ++gi) dst[gi * stride] = 0;
        return;
    }
    const size_t total = static_cast<size_t>(Nout) * G;
    const size_t e0 = static_cast<size_t>(n) * G + gbeg;
    const size_t a0 = e0 & ~static_cast<size_t>(7);
    const int off = static_cast<int>(e0 - a0);
    const int nch = (off + gpp + 7) >> 3;
    for (int c0 = 0; c0 < nch; c0 += 8) {
        uint4 v[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const size_t e = a0 + static_cast<size_t>(c0 + c) * 8;
            if (c0 + c < nch && e + 8 <= total) {
                v[c] = __ldg(reinterpret_cast<const uint4*>(src + e));
            } else if (c0 + c < nch) {
                uint16_t t[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) t[j] = e + j < total ? __ldg(src + e + j) : 0;
                v[c] = make_uint4(t[0] | (t[1] << 16), t[2] | (t[3] << 16), t[4] | (t[5] << 16),
                                  t[6] | (t[7] << 16));
            }
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            if (c0 + c >= nch) break;
            const uint32_t w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int gi = (c0 + c) * 8 + j - off;
                if (gi >= 0 && gi < gpp)
                    dst[gi * stride] = static_cast<uint16_t>(w[j >> 1] >> (16 * (j & 1)));
            }
        }
    }
}

// m16n8k16 BF16 MMA with FP32 accumulate: d += a (16x16, row) * b (16x8, col).
// It reads and writes registers only, so the asm is not volatile: the
// compiler may interleave independent MMAs with other work to hide their
// latency (a volatile asm would keep every MMA in source order).
__device__ __forceinline__ void mma_bf16_16816(float d[4], const uint32_t a[4], uint32_t b0,
                                               uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t r[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

}  // namespace qmm
