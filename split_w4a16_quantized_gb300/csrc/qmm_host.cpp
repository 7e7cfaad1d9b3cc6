// Host side of libqmm: argument checks, the occupancy split plan and the
// dispatch of the W4A16 matmul, the reduce and the dense split-K GEMM.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <queue>
#include <vector>

#include "qmm.h"
#include "qmm_internal.h"

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool policy_ok(const qmm_policy* p) { return qmm::policy_valid(p); }

int device_sms(int* sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QMM_ENODEV;
    if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return QMM_ENODEV;
    return QMM_OK;
}

int check_device() { return qmm::device_check(); }

// The CUDA error behind this thread's latest QMM_ECUDA (qmm_last_cuda_error).
thread_local int tl_cuda_error = cudaSuccess;

// Launches go through cudaLaunchKernelEx, which reports its own error; the
// caller's pending CUDA error state is left alone.
int launched(int err) {
    if (err == cudaSuccess) return QMM_OK;
    tl_cuda_error = err;
    return QMM_ECUDA;
}

size_t partial_elem_bytes(int dtype) { return dtype == QMM_PARTIAL_F32 ? 4 : 2; }

// Fused reduce: one 32-bit counter per output tile in a fixed area at the end
// of the caller's workspace (the last kFusedCounterBytes, 256-byte aligned),
// so a workspace reused across shapes keeps its counters in one place.
size_t fused_tiles(const qmm::Family& f, int M, int Nout) {
    return static_cast<size_t>((M + f.bm - 1) / f.bm) * static_cast<size_t>((Nout + f.bn - 1) / f.bn);
}
uint32_t* fused_counters(void* workspace, size_t ws_bytes) {
    const uintptr_t end = reinterpret_cast<uintptr_t>(workspace) + ws_bytes;
    return reinterpret_cast<uint32_t*>((end - QMM_FUSED_COUNTER_BYTES) & ~static_cast<uintptr_t>(255));
}
bool fused_applies(const qmm::Family& f, int M, int Nout, int split) {
    return qmm::reduce_fused() && (f.kind == qmm::kKindTc || f.kind == qmm::kKindLean) && split > 1 &&
           fused_tiles(f, M, Nout) * sizeof(uint32_t) <= QMM_FUSED_COUNTER_BYTES;
}

std::atomic<int> g_kernels{QMM_KERNELS_DEFAULT};
std::atomic<int> g_pdl{1};
std::atomic<int> g_wstatic{0};
std::atomic<int> g_reduce{QMM_REDUCE_KERNEL};
std::atomic<int> g_partitions{QMM_PARTITIONS_EQUAL};
std::atomic<int> g_grouped{QMM_GROUPED_PERSISTENT};
std::atomic<int> g_group_plan{QMM_GROUP_PLAN_CALLS};

// Per-call options (qmm_options): the *_ex entry points install theirs for
// the duration of the call on the calling thread; every switch accessor
// reads a field that is not QMM_OPT_DEFAULT from there, else the
// process-wide value.
thread_local const qmm_options* tl_options = nullptr;

struct OptionsScope {
    const qmm_options* prev;
    explicit OptionsScope(const qmm_options* o) : prev(tl_options) { tl_options = o; }
    ~OptionsScope() { tl_options = prev; }
    OptionsScope(const OptionsScope&) = delete;
    OptionsScope& operator=(const OptionsScope&) = delete;
};

int setting(int qmm_options::*field, const std::atomic<int>& global) {
    if (tl_options && tl_options->*field != QMM_OPT_DEFAULT) return tl_options->*field;
    return global.load(std::memory_order_relaxed);
}

bool in_range(int v, int lo, int hi) { return v == QMM_OPT_DEFAULT || (v >= lo && v <= hi); }

bool options_valid(const qmm_options* o) {
    return !o || (in_range(o->kernels, QMM_KERNELS_DEFAULT, QMM_KERNELS_LEAN) &&
                  in_range(o->partitions, QMM_PARTITIONS_EQUAL, QMM_PARTITIONS_NEAR_EQUAL) &&
                  in_range(o->reduce, QMM_REDUCE_KERNEL, QMM_REDUCE_CLUSTER) &&
                  in_range(o->weights_static, 0, 1) && in_range(o->pdl, 0, 1) &&
                  in_range(o->grouped_schedule, QMM_GROUPED_TILES, QMM_GROUPED_PERSISTENT) &&
                  in_range(o->group_plan, QMM_GROUP_PLAN_CALLS, QMM_GROUP_PLAN_GROUP));
}

// a split the current partition rule accepts for G groups (grid z <= 65535)
bool split_fits(int64_t G, int64_t split) {
    if (split < 1 || split > G || split > 65535) return false;
    return qmm::partitions_near_equal() || G % split == 0;
}

// the three bounds of the occupancy rule: min(cap, floor(target/base),
// floor(Kred/min_k)); pol and the shape already checked
int64_t plan_bound(int M, int Kred, int Nout, const qmm_policy* pol) {
    const int64_t base = ceil_div(M, pol->bm) * ceil_div(Nout, pol->bn);
    int64_t bound = pol->cap;
    if (pol->target_blocks / base < bound) bound = pol->target_blocks / base;
    if (Kred / pol->min_k_per_split < bound) bound = Kred / pol->min_k_per_split;
    return bound;
}

template <size_t N>
const qmm::Family& pick(const qmm::Family (&table)[N], int M) {
    for (size_t i = 0; i + 1 < N; ++i)
        if (M <= table[i].max_m) return table[i];
    return table[N - 1];
}

}  // namespace

namespace qmm {

bool policy_valid(const qmm_policy* p) {
    return p && p->bm >= 1 && p->bn >= 1 && p->cap >= 1 && p->target_blocks >= 0 &&
           p->min_k_per_split >= kGroup && p->min_k_per_split % kGroup == 0;
}

int device_check() {
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QMM_ENODEV;
    // Bind the device's primary context to the calling thread: the tensor-map
    // encoder is a driver call, and a thread that has made no runtime call
    // yet has no current context for it.
    if (cudaSetDevice(dev) != cudaSuccess) return QMM_ENODEV;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return QMM_ENODEV;
    return (major == 10 && minor == 3) ? QMM_OK : QMM_ENODEV;
}

const Family& family_for(int M) {
    switch (setting(&qmm_options::kernels, g_kernels)) {
        case QMM_KERNELS_MMA_SYNC: return pick(kMmaFamilies, M);
        case QMM_KERNELS_TCGEN05: return pick(kTcFamilies, M);
        case QMM_KERNELS_LEAN: return pick(kLeanTable, M);
        default: return pick(kDefaultFamilies, M);
    }
}

bool family_shares_launch(const Family& f) { return f.kind == kKindTc; }

bool pdl_enabled() { return setting(&qmm_options::pdl, g_pdl) != 0; }

bool weights_static() { return setting(&qmm_options::weights_static, g_wstatic) != 0; }

bool reduce_fused() { return setting(&qmm_options::reduce, g_reduce) == QMM_REDUCE_FUSED; }

bool reduce_cluster() { return setting(&qmm_options::reduce, g_reduce) == QMM_REDUCE_CLUSTER; }

bool partitions_near_equal() {
    return setting(&qmm_options::partitions, g_partitions) == QMM_PARTITIONS_NEAR_EQUAL;
}

bool grouped_persistent() {
    return setting(&qmm_options::grouped_schedule, g_grouped) == QMM_GROUPED_PERSISTENT;
}

int choose_split(int M, int Kred, int Nout, int split_req, const qmm_policy* pol, int* split,
                 int num_sms) {
    if (split_req == 0) {
        qmm_policy local;
        if (!pol) {
            const int rc = qmm_policy_preset(QMM_PRESET_GB300, M, num_sms, &local);
            if (rc != QMM_OK) return rc;
            pol = &local;
        }
        return partitions_near_equal() ? qmm_splitk_plan_near_equal(M, Kred, Nout, pol, split)
                                       : qmm_splitk_plan(M, Kred, Nout, pol, split);
    }
    if (!split_fits(Kred / kGroup, split_req)) return QMM_ESHAPE;
    *split = split_req;
    return QMM_OK;
}

bool gemm_uses_tc() { return setting(&qmm_options::kernels, g_kernels) != QMM_KERNELS_MMA_SYNC; }

int smem_optin_bytes() {
    static int limit = -1;
    static std::once_flag once;
    std::call_once(once, [] {
        int dev = 0, v = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess)
            limit = v;
    });
    return limit;
}

int set_max_dynamic_smem(const void* kernel) {
    const int limit = smem_optin_bytes();
    cudaFuncAttributes fa;
    if (limit < 0 || cudaFuncGetAttributes(&fa, kernel) != cudaSuccess) return -1;
    const int dyn = limit - static_cast<int>(fa.sharedSizeBytes);
    if (dyn <= 0 ||
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn) != cudaSuccess)
        return -1;
    return dyn;
}

}  // namespace qmm

extern "C" {

int qmm_set_kernels(int which) {
    if (which != QMM_KERNELS_DEFAULT && which != QMM_KERNELS_MMA_SYNC &&
        which != QMM_KERNELS_TCGEN05 && which != QMM_KERNELS_LEAN)
        return QMM_EINVAL;
    return g_kernels.exchange(which);
}

int qmm_set_pdl(int enable) { return g_pdl.exchange(enable ? 1 : 0); }

int qmm_set_weights_static(int enable) { return g_wstatic.exchange(enable ? 1 : 0); }

int qmm_set_reduce(int mode) {
    if (mode != QMM_REDUCE_KERNEL && mode != QMM_REDUCE_FUSED && mode != QMM_REDUCE_CLUSTER)
        return QMM_EINVAL;
    return g_reduce.exchange(mode);
}

int qmm_set_partitions(int mode) {
    if (mode != QMM_PARTITIONS_EQUAL && mode != QMM_PARTITIONS_NEAR_EQUAL) return QMM_EINVAL;
    return g_partitions.exchange(mode);
}

int qmm_wait_timeout_probe(void* stream) {
    int rc = check_device();
    if (rc != QMM_OK) return rc;
    return launched(qmm::launch_wait_probe(stream));
}

namespace {
// the group plan's splits (defined with the grouped call below)
int group_plan_shapes(const int* shapes, int n, int num_sms, int partial_dtype,
                      std::vector<int>* splits);
int launch_group(const qmm_group_call* calls, int n, const std::vector<int>& splits,
                 const std::vector<size_t>& offsets, void* workspace, int partial_dtype,
                 void* stream);
// QMM_SPLIT_BALANCED's plan (defined with the group plan below)
int balanced_plan(int M, int Kred, int Nout, int num_sms, int partial_dtype, int* head,
                  int* s_tail, int* s_plain, int* narrow);
const qmm::Family* narrower_tile(const qmm::Family& f);
size_t balanced_bytes(int M, int Nout, int head, int s_tail, int partial_dtype);
}  // namespace

int qmm_set_group_plan(int mode) {
    if (mode != QMM_GROUP_PLAN_CALLS && mode != QMM_GROUP_PLAN_GROUP) return QMM_EINVAL;
    return g_group_plan.exchange(mode);
}

int qmm_group_plan(const int* shapes, int n, int num_sms, int partial_dtype, int* splits) {
    if (!splits) return QMM_EINVAL;
    std::vector<int> out;
    const int rc = group_plan_shapes(shapes, n, num_sms, partial_dtype, &out);
    if (rc != QMM_OK) return rc;
    std::copy(out.begin(), out.end(), splits);
    return QMM_OK;
}

int qmm_set_grouped_schedule(int mode) {
    if (mode != QMM_GROUPED_TILES && mode != QMM_GROUPED_PERSISTENT) return QMM_EINVAL;
    return g_grouped.exchange(mode);
}

int qmm_kernel_status(int* status, int clear) {
    if (!status) return QMM_EINVAL;
    int rc = check_device();
    if (rc != QMM_OK) return rc;
    return qmm::read_tc_status(status, clear != 0) == cudaSuccess ? QMM_OK : QMM_ECUDA;
}

void qmm_options_init(qmm_options* opt) {
    if (!opt) return;
    *opt = qmm_options{QMM_OPT_DEFAULT, QMM_OPT_DEFAULT, QMM_OPT_DEFAULT, QMM_OPT_DEFAULT,
                       QMM_OPT_DEFAULT, QMM_OPT_DEFAULT, QMM_OPT_DEFAULT};
}

int qmm_w4a16_g128_ex(const void* A, const uint32_t* Wq, const void* scales, const void* biases,
                      void* C, int M, int Kred, int Nout, int split_req, const qmm_policy* pol,
                      void* workspace, size_t ws_bytes, int partial_dtype, void* stream,
                      int* split_used, const qmm_options* opt) {
    if (!options_valid(opt)) return QMM_EINVAL;
    const OptionsScope scope(opt);
    return qmm_w4a16_g128(A, Wq, scales, biases, C, M, Kred, Nout, split_req, pol, workspace,
                          ws_bytes, partial_dtype, stream, split_used);
}

size_t qmm_splitk_workspace_bytes_ex(int M, int Nout, int split, int partial_dtype,
                                     const qmm_options* opt) {
    if (!options_valid(opt)) return 0;
    const OptionsScope scope(opt);
    return qmm_splitk_workspace_bytes(M, Nout, split, partial_dtype);
}

int qmm_call_plan(int M, int Kred, int Nout, int split_req, const qmm_policy* pol,
                  int partial_dtype, int num_sms, const qmm_options* opt, int* split, int* bm,
                  int* bn, int* head_rows) {
    if (!options_valid(opt) || !split || M < 1 || Nout < 1 ||
        (split_req < 0 && split_req != QMM_SPLIT_PLANNED && split_req != QMM_SPLIT_BALANCED))
        return QMM_EINVAL;
    if (partial_dtype != QMM_PARTIAL_BF16 && partial_dtype != QMM_PARTIAL_F32) return QMM_EINVAL;
    if (pol && !policy_ok(pol)) return QMM_EINVAL;
    if (Kred < qmm::kGroup || Kred % qmm::kGroup) return QMM_ESHAPE;
    const OptionsScope scope(opt);
    const qmm::Family& f = qmm::family_for(M);
    if (bm) *bm = f.bm;
    if (bn) *bn = f.bn;
    if (head_rows) *head_rows = 0;
    if (split_req == QMM_SPLIT_BALANCED) {
        int head = 0, s_tail = 1, s_plain = 1, narrow = 0;
        const int rc = balanced_plan(M, Kred, Nout, num_sms, partial_dtype, &head, &s_tail,
                                     &s_plain, &narrow);
        if (rc != QMM_OK) return rc;
        if (head > 0) {
            *split = s_tail;
            if (head_rows) *head_rows = head;
            return QMM_OK;
        }
        if (narrow) {
            const qmm::Family* g = narrower_tile(f);
            if (bm) *bm = g->bm;
            if (bn) *bn = g->bn;
            *split = s_plain;
            return QMM_OK;
        }
        split_req = s_plain;
    }
    if (split_req == QMM_SPLIT_PLANNED) {
        const int shape[3] = {M, Kred, Nout};
        std::vector<int> planned;
        const int rc = group_plan_shapes(shape, 1, num_sms, partial_dtype, &planned);
        if (rc != QMM_OK) return rc;
        split_req = planned[0];
    }
    return qmm::choose_split(M, Kred, Nout, split_req, pol, split, num_sms);
}

size_t qmm_call_workspace_bytes(int M, int Kred, int Nout, int split_req, const qmm_policy* pol,
                                int partial_dtype, int num_sms, const qmm_options* opt) {
    int split = 1, head = 0;
    if (qmm_call_plan(M, Kred, Nout, split_req, pol, partial_dtype, num_sms, opt, &split, nullptr,
                      nullptr, &head) != QMM_OK)
        return 0;
    const OptionsScope scope(opt);
    if (head > 0) return balanced_bytes(M, Nout, head, split, partial_dtype);
    return qmm_splitk_workspace_bytes(M, Nout, split, partial_dtype);
}

size_t qmm_group_workspace_bytes_ex(const qmm_group_call* calls, int n, int partial_dtype,
                                    const qmm_options* opt) {
    if (!options_valid(opt)) return 0;
    const OptionsScope scope(opt);
    return qmm_group_workspace_bytes(calls, n, partial_dtype);
}

int qmm_w4a16_g128_grouped_ex(const qmm_group_call* calls, int n, void* workspace,
                              size_t ws_bytes, int partial_dtype, void* stream, int* splits_used,
                              const qmm_options* opt) {
    if (!options_valid(opt)) return QMM_EINVAL;
    const OptionsScope scope(opt);
    return qmm_w4a16_g128_grouped(calls, n, workspace, ws_bytes, partial_dtype, stream,
                                  splits_used);
}

const char* qmm_last_cuda_error(void) {
    return cudaGetErrorName(static_cast<cudaError_t>(tl_cuda_error));
}

const char* qmm_strerror(int code) {
    switch (code) {
        case QMM_OK: return "ok";
        case QMM_EINVAL: return "invalid argument";
        case QMM_ESHAPE: return "unsupported shape or split";
        case QMM_EWORKSPACE: return "workspace missing or too small";
        case QMM_ECUDA: return "CUDA launch or runtime error";
        case QMM_EALIGN: return "misaligned pointer";
        case QMM_ENODEV: return "no usable CUDA device (compute capability 10.3 required)";
        default: return "unknown error";
    }
}

int qmm_kernel_grouped(int M) {
    if (M < 1) return QMM_EINVAL;
    return qmm::family_shares_launch(qmm::family_for(M)) ? 1 : 0;
}

int qmm_kernel_tile(int M, int* bm, int* bn) {
    if (M < 1 || !bm || !bn) return QMM_EINVAL;
    const qmm::Family& f = qmm::family_for(M);
    *bm = f.bm;
    *bn = f.bn;
    return QMM_OK;
}

int qmm_policy_preset(int which, int M, int num_sms, qmm_policy* out) {
    if (!out) return QMM_EINVAL;
    if (which == QMM_PRESET_PAGES) {
        // tiny-llm split-K chapter, Task 3: 32x32 tiles, ~320 threadgroups, cap 16
        *out = qmm_policy{32, 32, 320, 16, qmm::kGroup};
        return QMM_OK;
    }
    if (which != QMM_PRESET_GB300 || M < 1) return QMM_EINVAL;
    if (num_sms <= 0) {
        int rc = device_sms(&num_sms);
        if (rc != QMM_OK) return rc;
    }
    const qmm::Family& f = qmm::family_for(M);
    *out = qmm_policy{f.bm, f.bn, f.ctas_per_sm * num_sms, qmm::kCap,
                      M <= qmm::kDecodeMaxM ? qmm::kDecodeMinK : qmm::kGroup};
    return QMM_OK;
}

// The split is the largest divisor of G = Kred/128 that stays within the
// three bounds (cap, target/base, Kred/min_k).  Stepping a candidate down by
// one until it divides G, as the chapter words it, ends on that divisor.
int qmm_splitk_plan(int M, int Kred, int Nout, const qmm_policy* pol, int* split_out) {
    if (!split_out || !policy_ok(pol) || M < 1 || Nout < 1) return QMM_EINVAL;
    if (Kred < qmm::kGroup || Kred % qmm::kGroup) return QMM_ESHAPE;
    const int64_t G = Kred / qmm::kGroup;
    const int64_t bound = plan_bound(M, Kred, Nout, pol);
    int best = 1;
    for (int64_t d = 2; d <= bound && d <= G; ++d)
        if (G % d == 0) best = static_cast<int>(d);
    *split_out = best;
    return QMM_OK;
}

// The same three bounds with no divisibility step.  A partition's work is set
// by the longest one, ceil(G/s) groups, which no split within the bound takes
// below ceil(G/bound); the plan is the fewest partitions that reach it, since
// more would only add partial planes.  floor(Kred/min_k) <= G, so every
// partition keeps at least one group.
int qmm_splitk_plan_near_equal(int M, int Kred, int Nout, const qmm_policy* pol, int* split_out) {
    if (!split_out || !policy_ok(pol) || M < 1 || Nout < 1) return QMM_EINVAL;
    if (Kred < qmm::kGroup || Kred % qmm::kGroup) return QMM_ESHAPE;
    const int64_t G = Kred / qmm::kGroup;
    const int64_t bound = plan_bound(M, Kred, Nout, pol);
    if (bound <= 1) {
        *split_out = 1;
        return QMM_OK;
    }
    const int64_t longest = ceil_div(G, bound);
    *split_out = static_cast<int>(ceil_div(G, longest));
    return QMM_OK;
}

size_t qmm_splitk_workspace_bytes(int M, int Nout, int split, int partial_dtype) {
    if (M < 1 || Nout < 1 || split < 1) return 0;
    if (partial_dtype != QMM_PARTIAL_BF16 && partial_dtype != QMM_PARTIAL_F32) return 0;
    if (split == 1) return 0;
    const size_t planes = static_cast<size_t>(split) * static_cast<size_t>(M) *
                          static_cast<size_t>(Nout) * partial_elem_bytes(partial_dtype);
    if (!fused_applies(qmm::family_for(M), M, Nout, split)) return planes;
    // planes, then the fixed counter area (with 256 bytes of alignment slack)
    return (planes + 255) / 256 * 256 + 256 + QMM_FUSED_COUNTER_BYTES;
}

size_t qmm_gemm_workspace_bytes(int M, int N, int split) {
    if (M < 1 || N < 1 || split <= 1) return 0;
    return static_cast<size_t>(split) * static_cast<size_t>(M) * static_cast<size_t>(N) * 4;
}

int qmm_splitk_reduce(const void* partials, int partial_dtype, int split, int M, int Nout,
                      void* C, void* stream) {
    if (!partials || !C || split < 1 || M < 1 || Nout < 1) return QMM_EINVAL;
    if (partial_dtype != QMM_PARTIAL_BF16 && partial_dtype != QMM_PARTIAL_F32) return QMM_EINVAL;
    if (!aligned(partials, 16) || !aligned(C, 16)) return QMM_EALIGN;
    int rc = check_device();
    if (rc != QMM_OK) return rc;
    return launched(qmm::launch_reduce(partials, partial_dtype, split, M, Nout, C, stream));
}

int qmm_w4a16_g128(const void* A, const uint32_t* Wq, const void* scales, const void* biases,
                   void* C, int M, int Kred, int Nout, int split_req, const qmm_policy* pol,
                   void* workspace, size_t ws_bytes, int partial_dtype, void* stream,
                   int* split_used) {
    if (!A || !Wq || !scales || !biases || !C || M < 1 || Nout < 1 ||
        (split_req < 0 && split_req != QMM_SPLIT_PLANNED && split_req != QMM_SPLIT_BALANCED))
        return QMM_EINVAL;
    if (partial_dtype != QMM_PARTIAL_BF16 && partial_dtype != QMM_PARTIAL_F32) return QMM_EINVAL;
    if (pol && !policy_ok(pol)) return QMM_EINVAL;
    if (Kred < qmm::kGroup || Kred % qmm::kGroup) return QMM_ESHAPE;
    if (!aligned(A, 16) || !aligned(Wq, 16) || !aligned(C, 16) || !aligned(scales, 16) ||
        !aligned(biases, 16))
        return QMM_EALIGN;
    qmm::Family fam = qmm::family_for(M);
    if (ceil_div(M, fam.bm) > 65535) return QMM_ESHAPE;
    int rc = check_device();
    if (rc != QMM_OK) return rc;
    if (split_req == QMM_SPLIT_BALANCED) {
        int head = 0, s_tail = 1, s_plain = 1, narrow = 0;
        rc = balanced_plan(M, Kred, Nout, 0, partial_dtype, &head, &s_tail, &s_plain, &narrow);
        if (rc != QMM_OK) return rc;
        if (head > 0) {
            // rows [0, head) unsplit and [head, M) at s_tail, in one partition
            // launch (two calls of the grouped path on the two row ranges)
            const size_t need = balanced_bytes(M, Nout, head, s_tail, partial_dtype);
            if (need > 0) {
                if (!workspace || ws_bytes < need) return QMM_EWORKSPACE;
                if (!aligned(workspace, 16)) return QMM_EALIGN;
            }
            const qmm_group_call calls[2] = {
                {A, Wq, scales, biases, C, head, Kred, Nout},
                {static_cast<const uint8_t*>(A) + static_cast<size_t>(head) * Kred * 2, Wq, scales,
                 biases, static_cast<uint8_t*>(C) + static_cast<size_t>(head) * Nout * 2, M - head,
                 Kred, Nout}};
            rc = launch_group(calls, 2, {1, s_tail}, {0, 0}, workspace, partial_dtype, stream);
            if (rc == QMM_OK && split_used) *split_used = s_tail;
            return rc;
        }
        if (narrow) {  // the narrower tile at its own split
            fam = *narrower_tile(fam);
            if (ceil_div(M, fam.bm) > 65535) return QMM_ESHAPE;
        }
        split_req = s_plain;  // no cut pays: the planned split
    }
    if (split_req == QMM_SPLIT_PLANNED) {
        const int shape[3] = {M, Kred, Nout};
        std::vector<int> planned;
        rc = group_plan_shapes(shape, 1, 0, partial_dtype, &planned);
        if (rc != QMM_OK) return rc;
        split_req = planned[0];
    }

    int split = 1;
    rc = qmm::choose_split(M, Kred, Nout, split_req, pol, &split);
    if (rc != QMM_OK) return rc;

    if (split == 1) {
        rc = launched(qmm::launch_w4a16(fam, A, Wq, scales, biases, C, qmm::kOutBf16, M, Kred,
                                        Nout, 1, stream));
    } else {
        const size_t need = qmm_splitk_workspace_bytes(M, Nout, split, partial_dtype);
        if (!workspace || ws_bytes < need) return QMM_EWORKSPACE;
        if (!aligned(workspace, 16)) return QMM_EALIGN;
        const int mode = partial_dtype == QMM_PARTIAL_F32 ? qmm::kOutF32 : qmm::kOutBf16;
        int ce = cudaErrorNotSupported;
        // one launch: the tile's partitions add their partial tiles in a cluster
        if (qmm::reduce_cluster() && fam.kind == qmm::kKindTc)
            ce = qmm::launch_w4a16_tc_cluster(fam.bm, A, Wq, scales, biases, C, mode, M, Kred,
                                              Nout, split, stream);
        else if (qmm::reduce_cluster() && fam.kind == qmm::kKindLean)
            ce = qmm::launch_w4a16_lean_cluster(fam.bm, A, Wq, scales, biases, C, mode, M, Kred,
                                                Nout, split, stream);
        if (ce != cudaErrorNotSupported) {
            rc = launched(ce);
        } else if (fused_applies(fam, M, Nout, split)) {
            // one launch: the last CTA of each output tile adds the planes
            rc = launched(qmm::launch_w4a16(fam, A, Wq, scales, biases, workspace, mode, M, Kred,
                                            Nout, split, stream, C,
                                            fused_counters(workspace, ws_bytes)));
        } else {
            rc = launched(qmm::launch_w4a16(fam, A, Wq, scales, biases, workspace, mode, M, Kred,
                                            Nout, split, stream));
            if (rc == QMM_OK)
                rc = launched(qmm::launch_reduce(workspace, partial_dtype, split, M, Nout, C, stream));
        }
    }
    if (rc == QMM_OK && split_used) *split_used = split;
    return rc;
}

int qmm_w4a16_g128_partition(const void* A, const uint32_t* Wq, const void* scales,
                             const void* biases, void* partials, size_t partials_bytes, int M,
                             int Kred, int Nout, int split, int partial_dtype, void* stream) {
    if (!A || !Wq || !scales || !biases || !partials || M < 1 || Nout < 1 || split < 1)
        return QMM_EINVAL;
    if (partial_dtype != QMM_PARTIAL_BF16 && partial_dtype != QMM_PARTIAL_F32) return QMM_EINVAL;
    if (Kred < qmm::kGroup || Kred % qmm::kGroup) return QMM_ESHAPE;
    if (!split_fits(Kred / qmm::kGroup, split)) return QMM_ESHAPE;
    if (!aligned(A, 16) || !aligned(Wq, 16) || !aligned(partials, 16) || !aligned(scales, 16) ||
        !aligned(biases, 16))
        return QMM_EALIGN;
    const qmm::Family fam = qmm::family_for(M);
    if (ceil_div(M, fam.bm) > 65535) return QMM_ESHAPE;
    const size_t need = static_cast<size_t>(split) * static_cast<size_t>(M) *
                        static_cast<size_t>(Nout) * partial_elem_bytes(partial_dtype);
    if (partials_bytes < need) return QMM_EWORKSPACE;
    int rc = check_device();
    if (rc != QMM_OK) return rc;
    const int mode = partial_dtype == QMM_PARTIAL_F32 ? qmm::kOutF32 : qmm::kOutBf16;
    return launched(qmm::launch_w4a16(fam, A, Wq, scales, biases, partials, mode, M, Kred, Nout,
                                      split, stream));
}

namespace {

// Checks one grouped call like qmm_w4a16_g128 checks its arguments (host only).
int check_group_call(const qmm_group_call& c) {
    if (!c.A || !c.Wq || !c.scales || !c.biases || !c.C || c.M < 1 || c.Nout < 1)
        return QMM_EINVAL;
    if (c.Kred < qmm::kGroup || c.Kred % qmm::kGroup) return QMM_ESHAPE;
    if (!aligned(c.A, 16) || !aligned(c.Wq, 16) || !aligned(c.C, 16) || !aligned(c.scales, 16) ||
        !aligned(c.biases, 16))
        return QMM_EALIGN;
    if (ceil_div(c.M, qmm::family_for(c.M).bm) > 65535) return QMM_ESHAPE;
    return QMM_OK;
}

// ---- group plan (qmm_set_group_plan) ----------------------------------------
//
// Splits sized for a group's launch rather than for each call alone.  The
// calls of one tile width share a launch; its time is estimated as a
// longest-first list schedule of the CTA tiles on the SMs (a tile costs
// kPlanTileUs plus its partition's groups at plan_group_us) plus the partial
// planes written and read back (kPlanPlaneBytesPerUs).  Starting from every
// call unsplit, the call with the longest partition (lowest index on ties)
// takes its next valid split while that lowers the estimate.  The constants
// are tuning parameters fitted to this library's kernels on GB300, as the
// chapter's 320 and 16 are for its kernels.
constexpr double kPlanTileUs = 3.0;
constexpr double kPlanPlaneBytesPerUs = 3.0e6;
constexpr int64_t kPlanMaxTiles = 1 << 16;  // larger launches keep each call's own split

double plan_group_us(int bm) { return bm <= 32 ? 0.40 : bm <= 64 ? 0.45 : bm <= 128 ? 0.55 : 0.60; }

struct PlanCall {
    int M, Kred, Nout, G, smax;
    int64_t tiles;
};

// Estimated time of one launch with splits s; false if it has too many tiles.
bool plan_cost(const std::vector<PlanCall>& c, const std::vector<int>& s, int bm, int sms,
               int elem, double* cost) {
    struct Cls {
        double d;
        int64_t k;
    };
    std::vector<Cls> cls;
    int64_t tiles = 0;
    double planes = 0.0;
    for (size_t i = 0; i < c.size(); ++i) {
        const int len = (c[i].G + s[i] - 1) / s[i];
        cls.push_back({kPlanTileUs + len * plan_group_us(bm), c[i].tiles * s[i]});
        tiles += c[i].tiles * s[i];
        if (s[i] > 1)
            planes += static_cast<double>(s[i]) * c[i].M * c[i].Nout * 2 * elem / kPlanPlaneBytesPerUs;
    }
    if (tiles > kPlanMaxTiles) return false;
    std::stable_sort(cls.begin(), cls.end(), [](const Cls& a, const Cls& b) { return a.d > b.d; });
    std::priority_queue<double, std::vector<double>, std::greater<double>> load;
    for (int i = 0; i < sms; ++i) load.push(0.0);
    double span = 0.0;
    for (const Cls& k : cls)
        for (int64_t j = 0; j < k.k; ++j) {
            const double l = load.top() + k.d;
            load.pop();
            load.push(l);
            span = std::max(span, l);
        }
    *cost = span + planes;
    return true;
}

// The group plan of shapes (M, Kred, Nout) into splits: per tile width, the
// greedy descent above.  A move that would take the launch over kPlanMaxTiles
// is not made; a launch over it with every call unsplit keeps each call's own
// policy split.
int group_plan(const std::vector<PlanCall>& calls, int sms, int elem, std::vector<int>* splits) {
    splits->assign(calls.size(), 1);
    std::vector<int> widths;
    for (const PlanCall& c : calls) {
        const int bm = qmm::family_for(c.M).bm;
        if (std::find(widths.begin(), widths.end(), bm) == widths.end()) widths.push_back(bm);
    }
    for (int bm : widths) {
        std::vector<size_t> idx;
        std::vector<PlanCall> part;
        for (size_t i = 0; i < calls.size(); ++i)
            if (qmm::family_for(calls[i].M).bm == bm) {
                idx.push_back(i);
                part.push_back(calls[i]);
            }
        std::vector<int> s(part.size(), 1);
        double cost = 0.0;
        // calls of a family the grouped call runs one launch each keep their
        // own policy split, as they would alone
        const bool shared = qmm::family_shares_launch(qmm::family_for(part[0].M));
        bool fits = shared && plan_cost(part, s, bm, sms, elem, &cost);
        while (fits) {
            size_t top = 0;
            for (size_t i = 1; i < part.size(); ++i)
                if ((part[i].G + s[i] - 1) / s[i] > (part[top].G + s[top] - 1) / s[top]) top = i;
            int next = s[top] + 1;
            while (next <= part[top].smax && !split_fits(part[top].G, next)) ++next;
            if (next > part[top].smax) break;
            std::vector<int> t = s;
            t[top] = next;
            double c2 = 0.0;
            // a move over kPlanMaxTiles is not made
            if (!plan_cost(part, t, bm, sms, elem, &c2) || !(c2 < cost)) break;
            s = t;
            cost = c2;
        }
        for (size_t i = 0; i < part.size(); ++i) {
            int split = s[i];
            if (!fits) {  // own launches, or too many tiles to plan: the call's own policy split
                qmm_policy pol;
                int rc = qmm_policy_preset(QMM_PRESET_GB300, part[i].M, sms, &pol);
                if (rc == QMM_OK)
                    rc = qmm::partitions_near_equal()
                             ? qmm_splitk_plan_near_equal(part[i].M, part[i].Kred, part[i].Nout,
                                                          &pol, &split)
                             : qmm_splitk_plan(part[i].M, part[i].Kred, part[i].Nout, &pol, &split);
                if (rc != QMM_OK) return rc;
            }
            (*splits)[idx[i]] = split;
        }
    }
    return QMM_OK;
}

int group_plan_shapes(const int* shapes, int n, int num_sms, int partial_dtype,
                      std::vector<int>* splits) {
    if (!shapes || n < 1) return QMM_EINVAL;
    if (partial_dtype != QMM_PARTIAL_BF16 && partial_dtype != QMM_PARTIAL_F32) return QMM_EINVAL;
    if (num_sms <= 0) {
        const int rc = device_sms(&num_sms);
        if (rc != QMM_OK) return rc;
    }
    std::vector<PlanCall> calls;
    for (int i = 0; i < n; ++i) {
        const int M = shapes[3 * i], Kred = shapes[3 * i + 1], Nout = shapes[3 * i + 2];
        if (M < 1 || Nout < 1) return QMM_EINVAL;
        if (Kred < qmm::kGroup || Kred % qmm::kGroup) return QMM_ESHAPE;
        const qmm::Family& f = qmm::family_for(M);
        const int G = Kred / qmm::kGroup;
        const int min_k = M <= qmm::kDecodeMaxM ? qmm::kDecodeMinK : qmm::kGroup;
        const int smax = std::min(std::min(qmm::kCap, G), std::max(1, Kred / min_k));
        calls.push_back({M, Kred, Nout, G, smax, ceil_div(M, f.bm) * ceil_div(Nout, f.bn)});
    }
    // plans are cached: a model step issues the same group again and again
    struct Entry {
        std::vector<int> key, splits;
    };
    static std::mutex mu;
    static std::vector<Entry> cache;
    std::vector<int> key(shapes, shapes + 3 * n);
    key.push_back(num_sms);
    key.push_back(partial_dtype);
    key.push_back(qmm::partitions_near_equal() ? 1 : 0);
    key.push_back(setting(&qmm_options::kernels, g_kernels));
    {
        std::lock_guard<std::mutex> lock(mu);
        for (const Entry& e : cache)
            if (e.key == key) {
                *splits = e.splits;
                return QMM_OK;
            }
    }
    const int rc = group_plan(calls, num_sms, static_cast<int>(partial_elem_bytes(partial_dtype)),
                              splits);
    if (rc != QMM_OK) return rc;
    std::lock_guard<std::mutex> lock(mu);
    if (cache.size() >= 16) cache.erase(cache.begin());
    cache.push_back({key, *splits});
    return QMM_OK;
}

// ---- balanced split (QMM_SPLIT_BALANCED) ------------------------------------
//
// gpu-kernels-explained, "Split-K, streams and overlap" (Stream-K): a grid
// whose tiles leave a partial last wave idles most SMs while that wave runs.
// At tile granularity the fix is the data-parallel + split-K hybrid: the
// row tiles that fill whole waves run unsplit, and only the rows of the
// partial wave are split, so their shorter CTAs spread over every SM as the
// full-wave CTAs finish.  Both row ranges go into one partition launch
// (longest CTAs first) and the tail's planes into one reduce.  The tail's
// split is the one with the lowest estimate of the group plan's cost model;
// the cut is taken only if that estimate beats the planned split's.  Rows
// [0, head) get exactly the unsplit kernel's result and rows [head, M) that
// of a call on those rows at the tail's split (the same tiles, k order and
// rounding).
// Estimated time of a call whose CTAs fit one wave (tile rows bm, split s):
// the partition's groups at the tile's time per group, plus, when split, the
// reduce launch and the partial planes written and read back.  The times per
// group are those of a CTA of the 128- and 256-row tcgen05 tiles at
// M = 129..2048 on GB300 (tuning parameters, like the group plan's).
constexpr double kReduceLaunchUs = 2.5;
double one_wave_us(int bm, int64_t G, int s, int M, int Nout, int elem) {
    const double group = bm <= 128 ? 0.48 : 0.78;
    double t = static_cast<double>((G + s - 1) / s) * group;
    if (s > 1)
        t += kReduceLaunchUs + 2.0 * s * M * static_cast<double>(Nout) * elem / kPlanPlaneBytesPerUs;
    return t;
}

const qmm::Family* narrower_tile(const qmm::Family& f) {
    if (f.kind != qmm::kKindTc || f.bm <= 128) return nullptr;
    const qmm::Family& g = qmm::family_for(f.bm / 2);
    return g.kind == qmm::kKindTc && g.bm == f.bm / 2 ? &g : nullptr;
}

int balanced_plan(int M, int Kred, int Nout, int num_sms, int partial_dtype, int* head,
                  int* s_tail, int* s_plain, int* narrow) {
    const int shape[3] = {M, Kred, Nout};
    std::vector<int> planned;
    int rc = group_plan_shapes(shape, 1, num_sms, partial_dtype, &planned);
    if (rc != QMM_OK) return rc;
    if (num_sms <= 0) {
        rc = device_sms(&num_sms);
        if (rc != QMM_OK) return rc;
    }
    *s_plain = *s_tail = planned[0];
    *head = 0;
    *narrow = 0;
    const qmm::Family& f = qmm::family_for(M);
    if (!qmm::family_shares_launch(f)) return QMM_OK;
    const int64_t rt = ceil_div(M, f.bm), ct = ceil_div(Nout, f.bn), tiles = rt * ct;
    if (tiles <= num_sms) {
        // No full wave, so no cut.  The next narrower tile has about twice
        // the tiles: at its own policy split it is taken if that split is no
        // larger, its CTAs still fit one wave, and the estimate above favours
        // it.  Its CTAs dequantize twice the weights per multiply-add, which
        // a lower split (fewer planes, or no reduce launch) must pay for.
        const qmm::Family* g = narrower_tile(f);
        if (!g) return QMM_OK;
        qmm_policy pol;
        int s = 0;
        rc = qmm_policy_preset(QMM_PRESET_GB300, g->bm, num_sms, &pol);
        if (rc == QMM_OK)
            rc = qmm::partitions_near_equal() ? qmm_splitk_plan_near_equal(M, Kred, Nout, &pol, &s)
                                              : qmm_splitk_plan(M, Kred, Nout, &pol, &s);
        if (rc != QMM_OK) return rc;
        const int64_t narrow_ctas = ceil_div(M, g->bm) * ceil_div(Nout, g->bn) * s;
        const int G = Kred / qmm::kGroup;
        const int elem = static_cast<int>(partial_elem_bytes(partial_dtype));
        if (s <= *s_plain && narrow_ctas <= num_sms &&
            one_wave_us(g->bm, G, s, M, Nout, elem) < one_wave_us(f.bm, G, *s_plain, M, Nout, elem)) {
            *narrow = 1;
            *s_plain = *s_tail = s;
        }
        return QMM_OK;
    }
    if (tiles % num_sms == 0) return QMM_OK;
    const int64_t h = tiles / num_sms * num_sms / ct;  // row tiles that fit the full waves
    if (h < 1 || h >= rt) return QMM_OK;
    const int m1 = static_cast<int>(h * f.bm);
    if (qmm::family_for(M - m1).bm != f.bm) return QMM_OK;  // the tail must share the launch
    const int G = Kred / qmm::kGroup;
    const int smax = std::min(qmm::kCap, G);
    const int elem = static_cast<int>(partial_elem_bytes(partial_dtype));
    const std::vector<PlanCall> whole = {{M, Kred, Nout, G, smax, tiles}};
    const std::vector<PlanCall> cut = {{m1, Kred, Nout, G, smax, h * ct},
                                       {M - m1, Kred, Nout, G, smax, (rt - h) * ct}};
    double best = 0.0;
    if (!plan_cost(whole, {*s_plain}, f.bm, num_sms, elem, &best)) return QMM_OK;
    int best_s = 0;
    for (int s = 1; s <= smax; ++s) {
        double c = 0.0;
        if (split_fits(G, s) && plan_cost(cut, {1, s}, f.bm, num_sms, elem, &c) && c < best) {
            best = c;
            best_s = s;
        }
    }
    if (best_s > 0) {
        *head = m1;
        *s_tail = best_s;
    }
    return QMM_OK;
}

size_t balanced_bytes(int M, int Nout, int head, int s_tail, int partial_dtype) {
    if (s_tail <= 1) return 0;
    return static_cast<size_t>(s_tail) * static_cast<size_t>(M - head) * static_cast<size_t>(Nout) *
           partial_elem_bytes(partial_dtype);
}

// Every call's arguments, then its split and the offset of its planes in the
// workspace (256-byte aligned); *ws_need receives the total.
int plan_group(const qmm_group_call* calls, int n, int partial_dtype, std::vector<int>* splits,
               std::vector<size_t>* offsets, size_t* ws_need) {
    if (!calls || n < 1) return QMM_EINVAL;
    if (partial_dtype != QMM_PARTIAL_BF16 && partial_dtype != QMM_PARTIAL_F32) return QMM_EINVAL;
    for (int i = 0; i < n; ++i) {
        const int rc = check_group_call(calls[i]);
        if (rc != QMM_OK) return rc;
    }
    splits->assign(static_cast<size_t>(n), 1);
    offsets->assign(static_cast<size_t>(n), 0);
    if (setting(&qmm_options::group_plan, g_group_plan) == QMM_GROUP_PLAN_GROUP) {
        std::vector<int> shapes;
        for (int i = 0; i < n; ++i) {
            shapes.push_back(calls[i].M);
            shapes.push_back(calls[i].Kred);
            shapes.push_back(calls[i].Nout);
        }
        const int rc = group_plan_shapes(shapes.data(), n, 0, partial_dtype, splits);
        if (rc != QMM_OK) return rc;
    }
    size_t off = 0;
    for (int i = 0; i < n; ++i) {
        const qmm_group_call& c = calls[i];
        int& s = (*splits)[static_cast<size_t>(i)];
        if (setting(&qmm_options::group_plan, g_group_plan) != QMM_GROUP_PLAN_GROUP) {
            const int rc = qmm::choose_split(c.M, c.Kred, c.Nout, 0, nullptr, &s);
            if (rc != QMM_OK) return rc;
        }
        if (s > 1) {
            (*offsets)[static_cast<size_t>(i)] = off;
            const size_t planes = static_cast<size_t>(s) * static_cast<size_t>(c.M) *
                                  static_cast<size_t>(c.Nout) * partial_elem_bytes(partial_dtype);
            off += (planes + 255) / 256 * 256;
        }
    }
    *ws_need = off;
    return QMM_OK;
}

}  // namespace

size_t qmm_group_workspace_bytes(const qmm_group_call* calls, int n, int partial_dtype) {
    std::vector<int> splits;
    std::vector<size_t> offsets;
    size_t need = 0;
    if (plan_group(calls, n, partial_dtype, &splits, &offsets, &need) != QMM_OK) return 0;
    return need;
}

int qmm_w4a16_g128_grouped(const qmm_group_call* calls, int n, void* workspace, size_t ws_bytes,
                           int partial_dtype, void* stream, int* splits_used) {
    std::vector<int> splits;
    std::vector<size_t> offsets;
    size_t need = 0;
    int rc = plan_group(calls, n, partial_dtype, &splits, &offsets, &need);
    if (rc != QMM_OK) return rc;
    if (need > 0) {
        if (!workspace || ws_bytes < need) return QMM_EWORKSPACE;
        if (!aligned(workspace, 16)) return QMM_EALIGN;
    }
    rc = check_device();
    if (rc != QMM_OK) return rc;
    rc = launch_group(calls, n, splits, offsets, workspace, partial_dtype, stream);
    if (rc == QMM_OK && splits_used)
        for (int i = 0; i < n; ++i) splits_used[i] = splits[i];
    return rc;
}

}  // extern "C"

namespace {

// The launches of n checked calls at the given splits, the planes of call i
// at workspace + offsets[i]: the tcgen05 calls of one tile width share a
// partition launch, the others run one by one, and one reduce launch adds
// the planes of up to kMaxGroupCalls split calls.
int launch_group(const qmm_group_call* calls, int n, const std::vector<int>& splits,
                 const std::vector<size_t>& offsets, void* workspace, int partial_dtype,
                 void* stream) {
    int rc = QMM_OK;
    const int mode = partial_dtype == QMM_PARTIAL_F32 ? qmm::kOutF32 : qmm::kOutBf16;
    auto out_of = [&](int i) -> void* {
        return splits[i] > 1 ? static_cast<uint8_t*>(workspace) + offsets[i] : calls[i].C;
    };
    // partition launches: tcgen05 calls bucketed by tile width, up to
    // kMaxGroupCalls per launch; mma.sync calls one by one.  Within a launch
    // the calls with the longest partitions come first: blocks are dispatched
    // in index order, so the long CTAs start early and the short ones fill in
    // behind them (longest-first list scheduling) instead of leaving a tail.
    std::vector<int> order(static_cast<size_t>(n));
    for (int i = 0; i < n; ++i) order[i] = i;
    auto longest = [&](int i) {
        const int G = calls[i].Kred / qmm::kGroup;
        return G / splits[i] + (G % splits[i] ? 1 : 0);
    };
    std::stable_sort(order.begin(), order.end(),
                     [&](int a, int b) { return longest(a) > longest(b); });
    std::vector<qmm::GroupCall> bucket;
    for (const int bm : {16, 32, 64, 128, 256}) {
        bucket.clear();
        for (const int i : order) {
            if (rc != QMM_OK) break;
            const qmm::Family fam = qmm::family_for(calls[i].M);
            if (fam.kind != qmm::kKindTc || fam.bm != bm) continue;
            const qmm_group_call& c = calls[i];
            bucket.push_back({c.A, c.Wq, c.scales, c.biases, out_of(i),
                              splits[i] > 1 ? mode : static_cast<int>(qmm::kOutBf16), c.M, c.Kred,
                              c.Nout, splits[i]});
            if (static_cast<int>(bucket.size()) == qmm::kMaxGroupCalls) {
                rc = launched(qmm::launch_w4a16_tc_group(bm, bucket.data(),
                                                         static_cast<int>(bucket.size()), stream));
                bucket.clear();
            }
        }
        if (rc == QMM_OK && !bucket.empty())
            rc = launched(qmm::launch_w4a16_tc_group(bm, bucket.data(),
                                                     static_cast<int>(bucket.size()), stream));
        if (rc != QMM_OK) return rc;
    }
    for (int i = 0; i < n && rc == QMM_OK; ++i) {
        const qmm::Family fam = qmm::family_for(calls[i].M);
        if (fam.kind == qmm::kKindTc) continue;
        const qmm_group_call& c = calls[i];
        rc = launched(qmm::launch_w4a16(fam, c.A, c.Wq, c.scales, c.biases, out_of(i),
                                        splits[i] > 1 ? mode : qmm::kOutBf16, c.M, c.Kred, c.Nout,
                                        splits[i], stream));
    }
    // the planes of every split call, one reduce launch per kMaxGroupCalls
    std::vector<qmm::ReduceCall> red;
    for (int i = 0; i < n && rc == QMM_OK; ++i) {
        if (splits[i] <= 1) continue;
        red.push_back({out_of(i), calls[i].C, splits[i], calls[i].M, calls[i].Nout});
        if (static_cast<int>(red.size()) == qmm::kMaxGroupCalls) {
            rc = launched(qmm::launch_reduce_group(red.data(), static_cast<int>(red.size()),
                                                   partial_dtype, stream));
            red.clear();
        }
    }
    if (rc == QMM_OK && !red.empty())
        rc = launched(qmm::launch_reduce_group(red.data(), static_cast<int>(red.size()),
                                               partial_dtype, stream));
    return rc;
}

}  // namespace

extern "C" {

int qmm_gemm_bf16_splitk(const void* A, const void* W, void* C, int M, int N, int K, int split,
                         void* workspace, size_t ws_bytes, void* stream) {
    if (!A || !W || !C || M < 1 || N < 1 || K < 1 || split < 1) return QMM_EINVAL;
    if (K % 64 || split > K / 64 || split > 65535) return QMM_ESHAPE;
    if (ceil_div(M, 128) > 65535) return QMM_ESHAPE;
    if (!aligned(A, 16) || !aligned(W, 16) || !aligned(C, 16)) return QMM_EALIGN;
    int rc = check_device();
    if (rc != QMM_OK) return rc;
    if (split == 1)
        return launched(qmm::gemm_uses_tc()
                            ? qmm::launch_gemm_tc(A, W, C, qmm::kOutBf16, M, N, K, 1, stream)
                            : qmm::launch_gemm(A, W, C, qmm::kOutBf16, M, N, K, 1, stream));
    if (!workspace || ws_bytes < qmm_gemm_workspace_bytes(M, N, split)) return QMM_EWORKSPACE;
    if (!aligned(workspace, 16)) return QMM_EALIGN;
    rc = launched(qmm::gemm_uses_tc()
                      ? qmm::launch_gemm_tc(A, W, workspace, qmm::kOutF32, M, N, K, split, stream)
                      : qmm::launch_gemm(A, W, workspace, qmm::kOutF32, M, N, K, split, stream));
    if (rc == QMM_OK)
        rc = launched(qmm::launch_reduce(workspace, QMM_PARTIAL_F32, split, M, N, C, stream));
    return rc;
}

int qmm_decode_attention_splits(int B, int Hq, int Hkv, int Lmax, int num_sms, int* splits) {
    if (!splits || B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || Lmax < 1) return QMM_EINVAL;
    if (num_sms <= 0) {
        const int rc = device_sms(&num_sms);
        if (rc != QMM_OK) return rc;
    }
    // grid target: two waves of the kernel's two resident CTAs per SM, the
    // page's "2-4 blocks per SM"; a mix of sequence lengths balances better
    // over more than one wave
    constexpr int kBlocksPerSm = 4;
    const int64_t work = static_cast<int64_t>(B) * Hkv;
    const int64_t target = static_cast<int64_t>(num_sms) * kBlocksPerSm;
    int64_t S = ceil_div(target, work);
    int64_t cap = Lmax / 512;
    if (cap < 1) cap = 1;
    if (S > cap) S = cap;
    *splits = static_cast<int>(S < 1 ? 1 : S);
    return QMM_OK;
}

size_t qmm_decode_attention_workspace_bytes(int B, int Hq, int D, int splits) {
    if (B < 1 || Hq < 1 || D < 1 || splits <= 1) return 0;
    return static_cast<size_t>(B) * Hq * splits * (D + 2) * sizeof(float);
}

int qmm_decode_attention(const void* q, const void* K, const void* V, const int* lens, void* O,
                         int B, int Hq, int Hkv, int Lmax, int D, float scale, int splits_req,
                         void* workspace, size_t ws_bytes, void* stream, int* splits_used) {
    if (!q || !K || !V || !lens || !O || B < 1 || Hq < 1 || Hkv < 1 || Lmax < 1 ||
        splits_req < 0 || Hq % Hkv)
        return QMM_EINVAL;
    const int qg = Hq / Hkv;
    if ((D != 64 && D != 128) || (qg != 1 && qg != 2 && qg != 4 && qg != 8)) return QMM_ESHAPE;
    if (B > 65535 || Hkv > 65535 || splits_req > 65535 ||
        static_cast<int64_t>(B) * Hq > 0x7fffffffLL)
        return QMM_ESHAPE;
    if (!aligned(q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) ||
        !aligned(lens, 4))
        return QMM_EALIGN;
    int rc = check_device();
    if (rc != QMM_OK) return rc;
    int S = splits_req;
    if (S == 0) {
        rc = qmm_decode_attention_splits(B, Hq, Hkv, Lmax, 0, &S);
        if (rc != QMM_OK) return rc;
    }
    if (S > 1) {
        if (!workspace || ws_bytes < qmm_decode_attention_workspace_bytes(B, Hq, D, S))
            return QMM_EWORKSPACE;
        if (!aligned(workspace, 16)) return QMM_EALIGN;
    }
    const float sc = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(D));
    rc = launched(qmm::launch_decode_attention(q, K, V, lens, O, static_cast<float*>(workspace), B,
                                               Hq, Hkv, Lmax, D, sc, S, stream));
    if (rc == QMM_OK && splits_used) *splits_used = S;
    return rc;
}

static int pipeline_config(int bm, int gpp, int smem_limit, int* out, bool persistent) {
    if (!out || gpp < 1 || smem_limit < 1) return QMM_EINVAL;
    qmm::TcPipeline pl;
    const int rc = qmm::tc_pipeline_config(bm, gpp, smem_limit, &pl, persistent);
    if (rc < 0) return QMM_EINVAL;
    if (rc > 0) return QMM_ESHAPE;
    const int v[9] = {pl.nacc, pl.dsets, pl.a_stages, pl.wgps, pl.agps, pl.act_stages,
                      pl.w_stages, pl.threads, static_cast<int>(pl.smem)};
    for (int i = 0; i < 9; ++i) out[i] = v[i];
    return QMM_OK;
}

int qmm_tc_pipeline_config(int bm, int gpp, int smem_limit, int* out) {
    return pipeline_config(bm, gpp, smem_limit, out, false);
}

int qmm_tc_persistent_pipeline_config(int bm, int gpp, int smem_limit, int* out) {
    return pipeline_config(bm, gpp, smem_limit, out, true);
}

int qmm_unpack_probe(const uint32_t* Wq, int Nout, int Kred, uint8_t* q, void* stream) {
    if (!Wq || !q || Nout < 1) return QMM_EINVAL;
    if (Kred < qmm::kGroup || Kred % qmm::kGroup) return QMM_ESHAPE;
    if (!aligned(Wq, 16) || !aligned(q, 16)) return QMM_EALIGN;
    int rc = check_device();
    if (rc != QMM_OK) return rc;
    return launched(qmm::launch_unpack_probe(Wq, Nout, Kred, q, stream));
}

int qmm_dequant_probe(const uint32_t* Wq, const void* scales, const void* biases, int Nout,
                      int Kred, void* w, void* stream) {
    if (!Wq || !scales || !biases || !w || Nout < 1) return QMM_EINVAL;
    if (Kred < qmm::kGroup || Kred % qmm::kGroup) return QMM_ESHAPE;
    if (!aligned(Wq, 16) || !aligned(w, 16) || !aligned(scales, 2) || !aligned(biases, 2))
        return QMM_EALIGN;
    int rc = check_device();
    if (rc != QMM_OK) return rc;
    return launched(qmm::launch_dequant_probe(Wq, scales, biases, Nout, Kred, w, stream));
}

}  // extern "C"
