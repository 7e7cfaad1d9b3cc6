// Streaming host activations through the W4A16 matmul: copy in, compute and
// copy out of successive chunks on three streams, with a fixed number of
// device buffers (gpu-kernels-explained, "Split-K, streams and overlap":
// first Concept section, and Maths, Overlap), and the schedule model of that
// pipeline for planning.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>
#include <vector>

#include "qmm.h"
#include "qmm_internal.h"

namespace {

constexpr int kMaxDevices = 64;

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Events for the executor's cross-stream waits, created once per device and
// handed out per call.  An event may be recorded again while earlier work
// that waits on it is still queued: a wait binds to the record current when
// the wait is enqueued.
std::mutex g_ev_mu;
std::vector<cudaEvent_t> g_ev_free[kMaxDevices];

int acquire_events(int dev, size_t k, std::vector<cudaEvent_t>* out) {
    std::lock_guard<std::mutex> lock(g_ev_mu);
    auto& pool = g_ev_free[dev];
    while (pool.size() < k) {
        cudaEvent_t e;
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return QMM_ECUDA;
        pool.push_back(e);
    }
    out->assign(pool.end() - static_cast<std::ptrdiff_t>(k), pool.end());
    pool.resize(pool.size() - k);
    return QMM_OK;
}

void release_events(int dev, const std::vector<cudaEvent_t>& ev) {
    std::lock_guard<std::mutex> lock(g_ev_mu);
    g_ev_free[dev].insert(g_ev_free[dev].end(), ev.begin(), ev.end());
}

// Checks one chunk's pointers, sizes and alignment the way qmm_w4a16_g128
// checks its arguments (host only, no CUDA call).
int check_call(const qmm_stream_call& c) {
    if (!c.A_host || !c.C_host || !c.Wq || !c.scales || !c.biases || c.M < 1 || c.Nout < 1)
        return QMM_EINVAL;
    if (c.Kred < qmm::kGroup || c.Kred % qmm::kGroup) return QMM_ESHAPE;
    if (!aligned16(c.Wq) || !aligned16(c.scales) || !aligned16(c.biases)) return QMM_EALIGN;
    return QMM_OK;
}

struct Arena {
    size_t a_bytes = 0, c_bytes = 0, ws_bytes = 0;  // per-buffer slots, one workspace
    size_t total(int buffers) const {
        return static_cast<size_t>(buffers) * (align256(a_bytes) + align256(c_bytes)) +
               align256(ws_bytes);
    }
};

// Every chunk's arguments first, then each chunk's split (the policy under
// the current rules, as qmm_w4a16_g128 will take it) and the buffer sizes.
int plan_arena(const qmm_stream_call* calls, int n, Arena* ar, std::vector<int>* splits) {
    for (int i = 0; i < n; ++i) {
        const int rc = check_call(calls[i]);
        if (rc != QMM_OK) return rc;
    }
    splits->assign(static_cast<size_t>(n), 1);
    for (int i = 0; i < n; ++i) {
        const qmm_stream_call& c = calls[i];
        int& split = (*splits)[static_cast<size_t>(i)];
        const int rc = qmm::choose_split(c.M, c.Kred, c.Nout, 0, nullptr, &split);
        if (rc != QMM_OK) return rc;
        ar->a_bytes = std::max(ar->a_bytes, static_cast<size_t>(c.M) * c.Kred * 2);
        ar->c_bytes = std::max(ar->c_bytes, static_cast<size_t>(c.M) * c.Nout * 2);
        ar->ws_bytes = std::max(ar->ws_bytes, qmm_splitk_workspace_bytes(c.M, c.Nout, split,
                                                                         QMM_PARTIAL_BF16));
    }
    return QMM_OK;
}

}  // namespace

extern "C" {

size_t qmm_stream_arena_bytes(const qmm_stream_call* calls, int n, int buffers) {
    if (!calls || n < 1 || buffers < 1) return 0;
    Arena ar;
    std::vector<int> splits;
    if (plan_arena(calls, n, &ar, &splits) != QMM_OK) return 0;
    return ar.total(buffers);
}

int qmm_w4a16_g128_stream(const qmm_stream_call* calls, int n, int buffers, void* arena,
                          size_t arena_bytes, void* stream_in, void* stream_compute,
                          void* stream_out, int* splits_used) {
    if (!calls || n < 1 || buffers < 1 || !arena) return QMM_EINVAL;
    if (reinterpret_cast<uintptr_t>(arena) % 256) return QMM_EALIGN;
    Arena ar;
    std::vector<int> splits;
    int rc = plan_arena(calls, n, &ar, &splits);
    if (rc != QMM_OK) return rc;
    if (arena_bytes < ar.total(buffers)) return QMM_EWORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QMM_ENODEV;

    const int b = std::min(buffers, n);  // buffers past the chunk count stay unused
    const size_t slot = align256(ar.a_bytes) + align256(ar.c_bytes);
    uint8_t* base = static_cast<uint8_t*>(arena);
    void* ws = base + static_cast<size_t>(buffers) * slot;
    auto A_dev = [&](int k) { return static_cast<void*>(base + k * slot); };
    auto C_dev = [&](int k) { return static_cast<void*>(base + k * slot + align256(ar.a_bytes)); };
    cudaStream_t s_in = static_cast<cudaStream_t>(stream_in);
    cudaStream_t s_comp = static_cast<cudaStream_t>(stream_compute);
    cudaStream_t s_out = static_cast<cudaStream_t>(stream_out);

    std::vector<cudaEvent_t> ev;
    rc = acquire_events(dev, static_cast<size_t>(3 * b), &ev);
    if (rc != QMM_OK) return rc;
    cudaEvent_t* loaded = ev.data();
    cudaEvent_t* computed = ev.data() + b;
    cudaEvent_t* stored = ev.data() + 2 * b;
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };
    for (int i = 0; i < n && rc == QMM_OK; ++i) {
        const qmm_stream_call& c = calls[i];
        const int k = i % b;
        const size_t a_bytes = static_cast<size_t>(c.M) * c.Kred * 2;
        const size_t c_bytes = static_cast<size_t>(c.M) * c.Nout * 2;
        // copy in: buffer k is free once chunk i-b's compute has read it
        if (i >= b && !ok(cudaStreamWaitEvent(s_in, computed[k], 0))) rc = QMM_ECUDA;
        if (rc == QMM_OK &&
            (!ok(cudaMemcpyAsync(A_dev(k), c.A_host, a_bytes, cudaMemcpyHostToDevice, s_in)) ||
             !ok(cudaEventRecord(loaded[k], s_in))))
            rc = QMM_ECUDA;
        // compute: after the copy in, and after chunk i-b's copy out has read C
        if (rc == QMM_OK && !ok(cudaStreamWaitEvent(s_comp, loaded[k], 0))) rc = QMM_ECUDA;
        if (rc == QMM_OK && i >= b && !ok(cudaStreamWaitEvent(s_comp, stored[k], 0)))
            rc = QMM_ECUDA;
        if (rc == QMM_OK) {
            int used = 0;
            rc = qmm_w4a16_g128(A_dev(k), c.Wq, c.scales, c.biases, C_dev(k), c.M, c.Kred,
                                c.Nout, 0, nullptr, ws, align256(ar.ws_bytes), QMM_PARTIAL_BF16,
                                s_comp, &used);
            if (rc == QMM_OK && splits_used) splits_used[i] = used;
        }
        if (rc == QMM_OK && !ok(cudaEventRecord(computed[k], s_comp))) rc = QMM_ECUDA;
        // copy out
        if (rc == QMM_OK &&
            (!ok(cudaStreamWaitEvent(s_out, computed[k], 0)) ||
             !ok(cudaMemcpyAsync(c.C_host, C_dev(k), c_bytes, cudaMemcpyDeviceToHost, s_out)) ||
             !ok(cudaEventRecord(stored[k], s_out))))
            rc = QMM_ECUDA;
    }
    release_events(dev, ev);
    return rc;
}

int qmm_overlap_schedule(int n, int buffers, const double* t_load, const double* t_comp,
                         const double* t_store, int out_reuse, double* T, double* events) {
    if (n < 1 || buffers < 1 || !t_load || !t_comp || !t_store || !T) return QMM_EINVAL;
    if (out_reuse != 0 && out_reuse != 1) return QMM_EINVAL;
    for (int i = 0; i < n; ++i)
        if (!(t_load[i] >= 0) || !(t_comp[i] >= 0) || !(t_store[i] >= 0)) return QMM_EINVAL;
    // per chunk: load, compute, store end times; a chunk's start on an engine
    // is the latest end among the chunks it waits for
    std::vector<double> le(static_cast<size_t>(n)), ce(le), se(le);
    for (int i = 0; i < n; ++i) {
        double l0 = i ? le[i - 1] : 0.0;
        if (i >= buffers) l0 = std::max(l0, ce[i - buffers]);
        le[i] = l0 + t_load[i];
        double c0 = le[i];
        if (i) c0 = std::max(c0, ce[i - 1]);
        if (out_reuse && i >= buffers) c0 = std::max(c0, se[i - buffers]);
        ce[i] = c0 + t_comp[i];
        double s0 = ce[i];
        if (i) s0 = std::max(s0, se[i - 1]);
        se[i] = s0 + t_store[i];
        if (events) {
            double* e = events + 6 * static_cast<size_t>(i);
            e[0] = l0;
            e[1] = le[i];
            e[2] = c0;
            e[3] = ce[i];
            e[4] = s0;
            e[5] = se[i];
        }
    }
    *T = se[static_cast<size_t>(n) - 1];
    return QMM_OK;
}

}  // extern "C"
