// Internal declarations shared by the host dispatcher and the kernels of
// libqmm (not part of the C ABI).
#pragma once

#include <cstddef>
#include <cstdint>

namespace qmm {

constexpr int kGroup = 128;  // quantization group length along the reduction axis

// W4A16 kernel families, picked by the number of activation rows M.
// BM = activation rows per CTA, BN = weight rows (output columns) per CTA.
struct Family {
    int max_m;  // family serves M <= max_m (the last one serves every larger M)
    int bm;
    int bn;
};

// Keep in step with the template instantiations in qmm_w4a16.cu.
constexpr Family kFamilies[] = {
    {8, 8, 64},
    {16, 16, 64},
    {32, 32, 128},
    {1 << 30, 64, 128},
};
constexpr int kNumFamilies = sizeof(kFamilies) / sizeof(kFamilies[0]);

inline int family_index(int M) {
    for (int i = 0; i < kNumFamilies - 1; ++i)
        if (M <= kFamilies[i].max_m) return i;
    return kNumFamilies - 1;
}

// GB300 preset tuning constants: target = kTargetPerSm * SMs CTAs, cap.
constexpr int kTargetPerSm = 2;
constexpr int kCap = 16;
constexpr int kDecodeMaxM = 8;      // M <= this keeps >= kDecodeMinK reduction elements per split
constexpr int kDecodeMinK = 512;

enum OutMode { kOutBf16 = 0, kOutF32 = 1 };

// Kernel launchers (qmm_w4a16.cu, qmm_reduce.cu, qmm_gemm.cu).  They assume
// validated arguments and return the cudaError_t of the launch as int.
int launch_w4a16(int family, const void* A, const uint32_t* Wq, const void* scales,
                 const void* biases, void* out, int out_mode, int M, int Kred, int Nout,
                 int split, void* stream);
int launch_reduce(const void* partials, int partial_dtype, int split, int M, int Nout, void* C,
                  void* stream);
int launch_gemm(const void* A, const void* W, void* out, int out_mode, int M, int N, int K,
                int split, void* stream);
int launch_unpack_probe(const uint32_t* Wq, int Nout, int Kred, uint8_t* q, void* stream);
int launch_dequant_probe(const uint32_t* Wq, const void* scales, const void* biases, int Nout,
                         int Kred, void* w, void* stream);

}  // namespace qmm
