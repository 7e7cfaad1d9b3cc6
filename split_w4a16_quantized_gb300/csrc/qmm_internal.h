// Internal declarations shared by the host dispatcher and the kernels of
// libqmm (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "qmm.h"

namespace qmm {

constexpr int kGroup = 128;  // quantization group length along the reduction axis

// W4A16 kernel families, picked by the number of activation rows M.
// BM = activation rows per CTA, BN = weight rows (output columns) per CTA.
enum KernelKind { kKindMma = 0, kKindTc = 1, kKindLean = 2 };
struct Family {
    int max_m;  // family serves M <= max_m (the last one serves every larger M)
    int bm;
    int bn;
    int kind;
    int ctas_per_sm;  // CTAs resident per SM (sets the policy's target of one wave)
};

// mma.sync kernels with register dequant (qmm_w4a16.cu); keep in step with
// the template instantiations there.
constexpr Family kMmaFamilies[] = {
    {8, 8, 64, kKindMma, 2},
    {16, 16, 64, kKindMma, 2},
    {32, 32, 128, kKindMma, 2},
    {1 << 30, 64, 128, kKindMma, 2},
};
// tcgen05 kernels, dequantized weights in tensor memory (qmm_w4a16_tc.cu);
// bm is the MMA N (activation rows), bn the MMA M (weight rows).
constexpr Family kTcFamilies[] = {
    {16, 16, 128, kKindTc, 1},
    {32, 32, 128, kKindTc, 1},
    {64, 64, 128, kKindTc, 1},
    {128, 128, 128, kKindTc, 1},
    {1 << 30, 256, 128, kKindTc, 1},
};
// Lean kernels for few activation rows (qmm_w4a16_lean.cu): 32 weight rows
// per CTA, mma.sync with register dequant, two CTAs per SM.
constexpr Family kLeanFamilies[] = {
    {8, 8, 32, kKindLean, 2},
    {16, 16, 32, kKindLean, 2},
    {32, 32, 32, kKindLean, 2},
};
// Lean kernels up to 32 rows, tcgen05 above (QMM_KERNELS_LEAN).
constexpr Family kLeanTable[] = {
    {8, 8, 32, kKindLean, 2},
    {16, 16, 32, kKindLean, 2},
    {32, 32, 32, kKindLean, 2},
    {64, 64, 128, kKindTc, 1},
    {128, 128, 128, kKindTc, 1},
    {1 << 30, 256, 128, kKindTc, 1},
};
// The default table: per M, the family that measured fastest on GB300 over
// the workload's shapes: the lean kernels up to 16 rows, the tcgen05 ones
// from 32 rows (where the legacy MMA rate starts to bound the lean kernel).
constexpr Family kDefaultFamilies[] = {
    {8, 8, 32, kKindLean, 2},
    {16, 16, 32, kKindLean, 2},
    {32, 32, 128, kKindTc, 1},
    {64, 64, 128, kKindTc, 1},
    {128, 128, 128, kKindTc, 1},
    {1 << 30, 256, 128, kKindTc, 1},
};

// A policy the plan accepts (bm, bn, cap >= 1, target >= 0, min_k a
// multiple of 128).
bool policy_valid(const qmm_policy* p);
// QMM_OK if the current device is a compute capability 10.3 GPU, else QMM_ENODEV.
int device_check();

// True if qmm_w4a16_g128_grouped runs the calls of this family in shared
// launches (the tcgen05 families); the others run one launch per call.
bool family_shares_launch(const Family& f);

// Process-wide choice of table (qmm_set_kernels); returns the family for M.
const Family& family_for(int M);

int smem_optin_bytes();

// Raise a kernel's dynamic shared-memory limit to what the device allows next
// to the kernel's own static shared memory; returns that dynamic limit in
// bytes, or -1 on failure.
int set_max_dynamic_smem(const void* kernel);

// Programmatic dependent launch of the library's kernels (qmm_set_pdl).
bool pdl_enabled();
// Weights not written by earlier kernels on the stream (qmm_set_weights_static).
bool weights_static();
// Fused last-CTA reduce of the tcgen05 kernels (qmm_set_reduce).
bool reduce_fused();
// Cluster reduce of the tcgen05 kernels (qmm_set_reduce).
bool reduce_cluster();
// Near-equal partitions for splits that do not divide the groups (qmm_set_partitions).
bool partitions_near_equal();
// Persistent schedule of the grouped call's tcgen05 launches (qmm_set_grouped_schedule).
bool grouped_persistent();
// The split a matmul call dispatches: the policy's (split_req 0, pol NULL =
// the GB300 preset) under the current partition rule, or the forced split if
// that rule accepts it (QMM_ESHAPE otherwise).  Shape and policy checked by
// the caller; returns a QMM_* code.
// num_sms > 0 plans the preset policy for that many SMs instead of the
// current device's.
int choose_split(int M, int Kred, int Nout, int split_req, const qmm_policy* pol, int* split,
                 int num_sms = 0);
struct LaunchAttrs {
    cudaLaunchAttribute attr[1];
};
inline void apply_pdl(cudaLaunchConfig_t& cfg, LaunchAttrs& la) {
    if (!pdl_enabled()) return;
    la.attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    la.attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = la.attr;
    cfg.numAttrs = 1;
}

// GB300 preset tuning constants: target = one wave of the family's CTAs
// (ctas_per_sm * SMs), cap.
constexpr int kCap = 16;
constexpr int kDecodeMaxM = 8;      // M <= this keeps >= kDecodeMinK reduction elements per split
constexpr int kDecodeMinK = 512;

enum OutMode { kOutBf16 = 0, kOutF32 = 1 };

// Kernel launchers (qmm_w4a16.cu, qmm_reduce.cu, qmm_gemm.cu).  They assume
// validated arguments and return the cudaError_t of the launch as int.
// fused_C / counters (tcgen05 and lean families, split > 1): the last CTA of
// each output tile adds the planes into fused_C.
int launch_w4a16(const Family& fam, const void* A, const uint32_t* Wq, const void* scales,
                 const void* biases, void* out, int out_mode, int M, int Kred, int Nout,
                 int split, void* stream, void* fused_C = nullptr, uint32_t* counters = nullptr);
int launch_w4a16_lean(int bm, const void* A, const uint32_t* Wq, const void* scales,
                      const void* biases, void* out, int out_mode, int M, int Kred, int Nout,
                      int split, void* stream, void* fused_C = nullptr,
                      uint32_t* counters = nullptr);

int launch_w4a16_tc(int bm, const void* A, const uint32_t* Wq, const void* scales, const void* biases,
                    void* out, int out_mode, int M, int Kred, int Nout, int split, void* stream,
                    void* fused_C = nullptr, uint32_t* counters = nullptr);
// The call with the cluster reduce (QMM_REDUCE_CLUSTER); cudaErrorNotSupported,
// with nothing launched, where it does not apply (the caller then takes the
// planes and the reduce kernel).
int launch_w4a16_lean_cluster(int bm, const void* A, const uint32_t* Wq, const void* scales,
                              const void* biases, void* C, int out_mode, int M, int Kred,
                              int Nout, int split, void* stream);
int launch_w4a16_tc_cluster(int bm, const void* A, const uint32_t* Wq, const void* scales,
                            const void* biases, void* C, int out_mode, int M, int Kred, int Nout,
                            int split, void* stream);
int read_tc_status(int* out, bool clear);
// Device address of the status word the tcgen05 and attention kernels share.
int* tc_status_ptr();
// One CTA whose bounded wait on a barrier nobody completes runs out
// (qmm_wait_timeout_probe); returns the launch's cudaError_t.
int launch_wait_probe(void* stream);

// Split-KV decode attention (qmm_attention.cu): S splits per (sequence, KV
// head); ws holds the partial states when S > 1 (B*Hq*S*(D+2) floats).
int launch_decode_attention(const void* q, const void* K, const void* V, const int* lens, void* O,
                            float* ws, int B, int Hq, int Hkv, int Lmax, int D, float scale,
                            int S, void* stream);

// Grouped launches: independent calls in one kernel launch (at most
// kMaxGroupCalls per launch; the caller cuts longer lists).
constexpr int kMaxGroupCalls = 16;
struct GroupCall {
    const void* A;
    const uint32_t* Wq;
    const void* scales;
    const void* biases;
    void* out;     // C (split 1) or the call's partial planes
    int out_mode;  // OutMode
    int M, Kred, Nout, split;
};
// One partition launch of the tcgen05 kernel of tile width bm for n calls.
int launch_w4a16_tc_group(int bm, const GroupCall* calls, int n, void* stream);
struct ReduceCall {
    const void* partials;  // [split, M, Nout] planes
    void* C;               // BF16 [M, Nout]
    int split, M, Nout;
};
// One reduce launch for n calls' planes (all of partial_dtype).
int launch_reduce_group(const ReduceCall* calls, int n, int partial_dtype, void* stream);

// Pipeline shape of the tcgen05 W4A16 kernel for one launch.
struct TcPipeline {
    int nacc, dsets, a_stages, wgps, agps, act_stages, w_stages, threads;
    size_t smem;
};
// 0 = ok, 1 = does not fit the shared-memory limit, -1 = bad arguments.
// persistent: the ring shape of the persistent grouped launch (two activation stages).
int tc_pipeline_config(int bm, int gpp, long smem_limit, TcPipeline* out, bool persistent = false);
int launch_reduce(const void* partials, int partial_dtype, int split, int M, int Nout, void* C,
                  void* stream);
int launch_gemm_tc(const void* A, const void* W, void* out, int out_mode, int M, int N, int K,
                   int split, void* stream);
bool gemm_uses_tc();
int launch_gemm(const void* A, const void* W, void* out, int out_mode, int M, int N, int K,
                int split, void* stream);
int launch_unpack_probe(const uint32_t* Wq, int Nout, int Kred, uint8_t* q, void* stream);
int launch_dequant_probe(const uint32_t* Wq, const void* scales, const void* biases, int Nout,
                         int Kred, void* w, void* stream);

}  // namespace qmm
