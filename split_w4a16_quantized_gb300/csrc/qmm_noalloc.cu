// Allocation-free variant of qmm_w4a16_g128.
//
// Some callers cannot allocate device memory at the point where they run the
// matmul, for example code running inside a custom allocator, or an engine
// that forbids allocation after start-up.  This entry point takes only the
// inputs and C.  It keeps the split-K partial planes in a fixed-size buffer
// that is part of the library's own device image, a file-scope __device__
// array that a device holds for as long as the module stays loaded there.
// Host code cannot use the array's name as a device address, so the first
// call on each device looks the address up with cudaGetSymbolAddress (with
// that device current) and remembers it.  Nothing here calls an allocator.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "qmm.h"
#include "qmm_internal.h"

namespace qmm {
namespace {

constexpr size_t kStaticScratchBytes = static_cast<size_t>(8) << 20;  // 8 MiB

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Device address of g_static_scratch on the current device, or null on error.
// The address is looked up once per device and kept: after cudaDeviceReset the
// module is loaded afresh and the kept address is no longer valid.
void* scratch_on_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return nullptr;
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

}  // namespace
}  // namespace qmm

extern "C" {

size_t qmm_static_scratch_bytes(void) { return qmm::kStaticScratchBytes; }

int qmm_w4a16_g128_noalloc(const void* A, const uint32_t* Wq, const void* scales,
                           const void* biases, void* C, int M, int Kred, int Nout, int split_req,
                           const qmm_policy* pol, int partial_dtype, void* stream,
                           int* split_used) {
    // the checks of qmm_w4a16_g128, in its order, so both return the same codes
    if (!A || !Wq || !scales || !biases || !C || M < 1 || Nout < 1 ||
        (split_req < 0 && split_req != QMM_SPLIT_PLANNED))
        return QMM_EINVAL;
    if (partial_dtype != QMM_PARTIAL_BF16 && partial_dtype != QMM_PARTIAL_F32) return QMM_EINVAL;
    if (pol && !qmm::policy_valid(pol)) return QMM_EINVAL;
    if (Kred < 128 || Kred % 128) return QMM_ESHAPE;
    if (!qmm::aligned16(A) || !qmm::aligned16(Wq) || !qmm::aligned16(C) || !qmm::aligned16(scales) ||
        !qmm::aligned16(biases))
        return QMM_EALIGN;
    int rc = qmm::device_check();
    if (rc != QMM_OK) return rc;
    if (split_req == QMM_SPLIT_PLANNED) {
        // the group plan's split for this call alone, as qmm_w4a16_g128 takes it
        const int shape[3] = {M, Kred, Nout};
        rc = qmm_group_plan(shape, 1, 0, partial_dtype, &split_req);
        if (rc != QMM_OK) return rc;
    }
    // the split this call will use, to size its partial planes
    int split = 1;
    rc = qmm::choose_split(M, Kred, Nout, split_req, pol, &split);
    if (rc != QMM_OK) return rc;
    // the last QMM_FUSED_COUNTER_BYTES (and 256 bytes of slack) are kept for
    // the fused reduce's counters in every mode, so no planes ever land there
    // and the counters stay zero from the module's load on
    const size_t planes = static_cast<size_t>(split) * static_cast<size_t>(M) *
                          static_cast<size_t>(Nout) * (partial_dtype == QMM_PARTIAL_F32 ? 4 : 2);
    if (split > 1 && (planes + 255) / 256 * 256 + 256 + QMM_FUSED_COUNTER_BYTES >
                         qmm::kStaticScratchBytes)
        return QMM_EWORKSPACE;
    void* scratch = qmm::scratch_on_current_device();
    if (!scratch) return QMM_ECUDA;
    return qmm_w4a16_g128(A, Wq, scales, biases, C, M, Kred, Nout, split, pol, scratch,
                          qmm::kStaticScratchBytes, partial_dtype, stream, split_used);
}

}  // extern "C"
