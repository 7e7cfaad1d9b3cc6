/*
 * qmm.h — C ABI of libqmm: split-K W4A16-g128 projection matmul for GB300
 * (sm_103a), plus the dense BF16 split-K GEMM the same split/reduce scheme
 * is modelled on.
 *
 * Operation (tiny-llm book, "Week 2 Day 7: Split-K Prefill", Why Split the
 * Reduction Dimension?):  C = A . W^T, with
 *   A       BF16 [M, Kred] row-major activations,
 *   W       [Nout, Kred] stored 4-bit affine-quantized in groups of 128 along
 *           the reduction axis (the "w4a16_g128" format):
 *             Wq      uint32 [Nout, Kred/8] row-major; word j of row n holds
 *                     q[n, 8j+i] in bits 4i..4i+3 (low nibble first), q in 0..15
 *             scales  BF16 [Nout, Kred/128] row-major
 *             biases  BF16 [Nout, Kred/128] row-major
 *             w[n, k] = scale[n, k/128] * q[n, k] + bias[n, k/128]
 *   C       BF16 [M, Nout] row-major.
 * The source chapter names the output width K and the reduction length N;
 * this header uses Kred (reduction) and Nout (output width) throughout.
 *
 * Split-K (same chapter, Task 2 and Task 4): the reduction axis is cut into
 * `split` partitions of equal length that start and end on 128-group
 * boundaries; partition p writes its own partial plane [M, Nout] of the
 * workspace (no atomics); a second kernel adds the planes in FP32, in
 * ascending p, and rounds once to BF16.  An opt-in rule
 * (qmm_set_partitions) also takes splits that do not divide the group count,
 * with near-equal partitions.
 *
 * Conventions for every entry point:
 *   - Device pointers are CUDA device memory owned by the caller; the
 *     library never allocates, frees or keeps them.  Host pointers are
 *     marked "host".
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every launch is asynchronous and stream-ordered; no entry
 *     point synchronizes.
 *   - Arguments are checked on the host before any launch; a bad argument
 *     returns an error code and launches nothing.  A launch failure returns
 *     QMM_ECUDA.  Nothing aborts, traps or prints.
 *   - C (and the workspace) must not alias any input.
 *   - Alignment: A, Wq, scales, biases, C, workspace and partial planes
 *     16-byte aligned (QMM_EALIGN otherwise; every allocator hands out at
 *     least that).
 */
#ifndef QMM_H
#define QMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* return codes */
enum {
    QMM_OK = 0,
    QMM_EINVAL = -1,     /* null pointer, non-positive size, unknown enum value */
    QMM_ESHAPE = -2,     /* Kred not a multiple of 128, split the partition rule rejects, size overflow */
    QMM_EWORKSPACE = -3, /* workspace missing or smaller than qmm_splitk_workspace_bytes() */
    QMM_ECUDA = -4,      /* a CUDA call or kernel launch failed */
    QMM_EALIGN = -5,     /* a pointer breaks the alignment rules above */
    QMM_ENODEV = -6      /* no CUDA device, or not compute capability 10.3 */
};

/* partial-plane element type (tiny-llm split-K chapter, Task 2: BF16 planes;
 * an FP32 temporary is the bring-up mode that doubles the partial traffic) */
enum { QMM_PARTIAL_BF16 = 0, QMM_PARTIAL_F32 = 1 };

/* policy presets */
enum { QMM_PRESET_PAGES = 0, QMM_PRESET_GB300 = 1 };

/* Occupancy split policy (tiny-llm split-K chapter, Task 3):
 *   base  = ceil(M/bm) * ceil(Nout/bn)
 *   split = min(cap, floor(target_blocks/base), floor(Kred/min_k_per_split))
 *   then split is lowered until Kred is divisible by split*128;
 *   split <= 1 selects the unsplit kernel.
 * min_k_per_split = 128 is the chapter's rule (its third bound is Kred/128);
 * a larger value keeps at least that many reduction elements per split
 * ("Optimize Prefill vs Decode Kernels", reasoning step 5).  It must be a
 * positive multiple of 128.  bm, bn, cap >= 1; target_blocks >= 0. */
typedef struct {
    int bm;
    int bn;
    int target_blocks;
    int cap;
    int min_k_per_split;
} qmm_policy;

/* Fill *out with a policy preset.
 *   QMM_PRESET_PAGES: the tiny-llm chapter's values (bm = bn = 32,
 *     target_blocks = 320, cap = 16, min_k_per_split = 128); M and num_sms
 *     are ignored.
 *   QMM_PRESET_GB300: bm/bn = the tile of the kernel family this library
 *     dispatches for M (qmm_kernel_tile), target_blocks = a multiple of
 *     num_sms (the chapter calls its 320/16 tuning parameters, not GPU
 *     properties), min_k_per_split = 512 for M <= 8 (decode) else 128.
 *     num_sms <= 0 queries the current CUDA device.
 * Returns QMM_OK, QMM_EINVAL (bad which/M/out) or QMM_ENODEV (query failed).
 * Host only; launches nothing. */
int qmm_policy_preset(int which, int M, int num_sms, qmm_policy *out);

/* Tile (rows of A, rows of W per CTA) of the W4A16 kernel family dispatched
 * for M.  Host only.  Returns QMM_OK or QMM_EINVAL. */
int qmm_kernel_tile(int M, int *bm, int *bn);

/* The occupancy split rule above for one matmul shape.  Pure host function,
 * deterministic, no CUDA calls.  *split_out >= 1 (1 = unsplit).
 * Returns QMM_OK, QMM_EINVAL (null, M/Nout < 1, bad policy fields) or
 * QMM_ESHAPE (Kred not a positive multiple of 128). */
int qmm_splitk_plan(int M, int Kred, int Nout, const qmm_policy *pol, int *split_out);

/* The occupancy rule above without its divisibility step, for near-equal
 * partitions (the longest holds ceil(G/split) of the G = Kred/128 groups):
 *   bound = min(cap, floor(target_blocks/base), floor(Kred/min_k_per_split));
 *   bound <= 1 selects the unsplit kernel; otherwise
 *   longest = ceil(G/bound), the shortest longest partition within the bound,
 *   split = ceil(G/longest), the fewest partitions that reach it (more would
 *   only add partial planes to the reduce).
 * The split the policy takes under QMM_PARTITIONS_NEAR_EQUAL.  It is never
 * smaller than qmm_splitk_plan's and equals it whenever bound divides G.
 * Pure host function; same arguments and returns as qmm_splitk_plan. */
int qmm_splitk_plan_near_equal(int M, int Kred, int Nout, const qmm_policy *pol, int *split_out);

/* Bytes of workspace the split path needs: split*M*Nout*(2 or 4), or 0 when
 * split <= 1; when the fused reduce applies (QMM_REDUCE_FUSED), the planes
 * rounded up to 256 bytes, plus 256, plus QMM_FUSED_COUNTER_BYTES.  Returns 0 for
 * invalid arguments as well. */
size_t qmm_splitk_workspace_bytes(int M, int Nout, int split, int partial_dtype);

/* split_req value of qmm_w4a16_g128: the group plan's split for the call alone. */
#define QMM_SPLIT_PLANNED (-1)
/* split_req value of qmm_w4a16_g128: the balanced split (gpu-kernels-explained,
 * "Split-K, streams and overlap", Stream-K, at tile granularity).  When the
 * call's tiles leave a partial last wave, the row tiles that fill whole waves
 * run unsplit and only the remaining rows are split, in the same partition
 * launch, so the short split CTAs fill the SMs the last wave would leave
 * idle.  When the tiles do not fill one wave and the family's tile has a
 * tcgen05 family of half its rows (the 256-row tile over the 128-row one),
 * the narrower tile is taken at the occupancy rule's split for it
 * (QMM_PRESET_GB300 of that tile) if that split is no larger than
 * QMM_SPLIT_PLANNED's and its CTAs fit one wave: each CTA then has half the
 * multiply-adds, or as many with fewer partial planes.  Otherwise it is
 * QMM_SPLIT_PLANNED. */
#define QMM_SPLIT_BALANCED (-2)

/* C = A . W^T for the W4A16-g128 format (see the top of this header).
 *   split_req  0: split from the policy (qmm_splitk_plan, or
 *              qmm_splitk_plan_near_equal under QMM_PARTITIONS_NEAR_EQUAL);
 *              1: the unsplit kernel (the control, writes C directly);
 *              s > 1: forced split, which must divide Kred/128 under
 *              QMM_PARTITIONS_EQUAL and be at most Kred/128 under
 *              QMM_PARTITIONS_NEAR_EQUAL (QMM_ESHAPE otherwise);
 *              QMM_SPLIT_PLANNED: the split qmm_group_plan gives this call
 *              alone on the current device.  That is the occupancy rule
 *              extended with the group plan's estimate of waves and plane
 *              traffic.  On under-filled calls it equals the policy's split;
 *              past one wave it may split where the policy does not (down at
 *              M = 2048: 2).  Size the workspace with that split.
 *              QMM_SPLIT_BALANCED: rows [0, h) unsplit and rows [h, M) at a
 *              split s, planned with the group plan's estimate on the current
 *              device (qmm_call_plan reports h and s).  Rows [0, h) of C are
 *              bitwise the unsplit call's; rows [h, M) bitwise those of a call
 *              on those rows alone at split s.  The workspace holds the
 *              tail's planes [s, M - h, Nout]; size it with
 *              qmm_call_workspace_bytes.  The reduce is the separate kernel.
 *              Where it takes the narrower tile instead (h = 0), each
 *              128-row slice of C is bitwise that slice called alone at the
 *              same split.
 *   pol        policy used when split_req == 0; NULL = QMM_PRESET_GB300
 *              for this M on the current device.
 *   workspace  device buffer for the partial planes [split, M, Nout] of
 *              partial_dtype; needed only when the split used is > 1, of
 *              at least qmm_splitk_workspace_bytes(M, Nout, split, dtype)
 *              bytes (ws_bytes).  Contents on return are unspecified.
 *   split_used host, nullable: receives the split that was dispatched
 *              (1 = unsplit).
 * Launches one kernel (split 1) or the partition kernel followed by
 * qmm_splitk_reduce's kernel, both on `stream`. */
int qmm_w4a16_g128(const void *A, const uint32_t *Wq, const void *scales, const void *biases,
                   void *C, int M, int Kred, int Nout, int split_req, const qmm_policy *pol,
                   void *workspace, size_t ws_bytes, int partial_dtype, void *stream,
                   int *split_used);

/* The partition kernel of qmm_w4a16_g128 alone (tiny-llm split-K chapter,
 * Task 2: grid z = partition, each partition writes its own plane, no
 * atomics): partials[p, m, n] = round(sum over the groups of partition p of
 * A[m, k] * w[n, k]), FP32 accumulation rounded once to partial_dtype (RNE).
 * Partition p covers groups [p*G/split, (p+1)*G/split), G = Kred/128; under
 * QMM_PARTITIONS_NEAR_EQUAL a split that does not divide G gives partition p
 * floor(G/split) groups, one more for p < G mod split, in order.
 *   split      1 <= split <= G; under QMM_PARTITIONS_EQUAL it must divide G
 *              (QMM_ESHAPE otherwise).  No policy is applied (take it from
 *              the plan of the current rule).
 *   partials   device buffer [split, M, Nout] of partial_dtype, planes
 *              contiguous, of at least split*M*Nout*(2 or 4) bytes
 *              (partials_bytes; QMM_EWORKSPACE when smaller).
 * qmm_w4a16_g128 with a split > 1 is exactly this call followed by
 * qmm_splitk_reduce on the same planes.  One kernel launch on `stream`. */
int qmm_w4a16_g128_partition(const void *A, const uint32_t *Wq, const void *scales,
                             const void *biases, void *partials, size_t partials_bytes, int M,
                             int Kred, int Nout, int split, int partial_dtype, void *stream);

/* C[m, n] = BF16(sum_{p=0}^{split-1} partials[p, m, n]), the sum taken in
 * FP32 in ascending p and rounded once (tiny-llm split-K chapter, Task 4:
 * one reduction thread per output element).  partials is [split, M, Nout]
 * of partial_dtype, planes contiguous.  split >= 1. */
int qmm_splitk_reduce(const void *partials, int partial_dtype, int split, int M, int Nout,
                      void *C, void *stream);

/* Dense BF16 split-K GEMM C = A . W^T, A [M, K] and W [N, K] BF16
 * row-major, C BF16 [M, N] (gpu-kernels-explained, "Split-K, streams and
 * overlap": output tiles of 128 x 128, k cut into `split` slices, partial
 * sums written as FP32 planes and added by a second pass).  k is cut into
 * K/64 tiles; when split does not divide that count the first (K/64 mod
 * split) slices take one extra tile.  K must be a positive multiple of 64,
 * 1 <= split <= K/64.  split = 1 writes C directly; split > 1 needs a
 * workspace of qmm_gemm_workspace_bytes(M, N, split) bytes. */
int qmm_gemm_bf16_splitk(const void *A, const void *W, void *C, int M, int N, int K, int split,
                         void *workspace, size_t ws_bytes, void *stream);
size_t qmm_gemm_workspace_bytes(int M, int N, int split);

/* Test probes of the kernels' weight loader: q[n, k] (uint8 [Nout, Kred])
 * and the dequantized BF16 w[n, k] ([Nout, Kred]) exactly as the matmul
 * kernels form them in registers.  Device buffers, stream-ordered. */
int qmm_unpack_probe(const uint32_t *Wq, int Nout, int Kred, uint8_t *q, void *stream);
int qmm_dequant_probe(const uint32_t *Wq, const void *scales, const void *biases, int Nout,
                      int Kred, void *w, void *stream);

/* Pipeline shape of the tcgen05 W4A16 kernel for a tile of bm activation rows
 * (16, 32, 64, 128 or 256) and a partition of gpp 128-groups, under a dynamic
 * shared-memory limit of smem_limit bytes (the per-block opt-in maximum minus
 * the kernel's static shared memory; 232432 on GB300).  Host only, no CUDA
 * calls: the same computation the launcher makes.  out (host, 9 ints)
 * receives: MMA issuers, dequantizer sets, tensor-memory A buffers, groups
 * per weight stage, groups per activation stage, activation ring stages,
 * weight ring stages, threads per CTA, dynamic shared memory bytes.  The
 * tiny-llm chapter has no counterpart: this call exists so tests can check
 * the pipeline's synchronization rules on the configurations the kernel
 * really uses.  Returns QMM_OK, QMM_EINVAL (bad bm, gpp, limit or null) or
 * QMM_ESHAPE (nothing fits the limit). */
int qmm_tc_pipeline_config(int bm, int gpp, int smem_limit, int *out);

/* The same for the persistent grouped launch (QMM_GROUPED_PERSISTENT), whose
 * rings keep two activation stages and give the rest of shared memory to
 * weight stages; gpp is the longest partition of the launch's calls and
 * smem_limit the opt-in maximum minus that kernel's static shared memory
 * (its call table: 231408 on GB300).  Same outputs and return codes.  The
 * tiny-llm chapter has no counterpart: this call exists so tests can check
 * the persistent pipeline's synchronization on its real configurations. */
int qmm_tc_persistent_pipeline_config(int bm, int gpp, int smem_limit, int *out);

/* Whether qmm_w4a16_g128_grouped runs calls with M activation rows in
 * launches shared with other calls of the same tile width (1: the tcgen05
 * families) or one launch per call (0: the lean and mma.sync families).  The
 * group plan (qmm_group_plan) plans only shared launches; a call that runs
 * alone keeps its single-call policy split.  Follows qmm_set_kernels.
 * QMM_EINVAL for M < 1.  No counterpart on the pages: a query for tests and
 * planning tools. */
int qmm_kernel_grouped(int M);

/* Kernel families used by qmm_w4a16_g128 (process-wide, thread-safe):
 *   QMM_KERNELS_DEFAULT   the tuned table: per M, the family measured fastest
 *                         (lean kernels up to 16 rows, tcgen05 above)
 *   QMM_KERNELS_MMA_SYNC  register-dequant mma.sync kernels for every M
 *   QMM_KERNELS_TCGEN05   tcgen05 kernels (dequantized weights in tensor
 *                         memory) for every M
 *   QMM_KERNELS_LEAN      lean kernels (32 weight rows a CTA, mma.sync,
 *                         weights streamed through per-thread cp.async rings)
 *                         up to 32 rows, tcgen05 above
 * qmm_kernel_tile and the GB300 policy preset follow the choice.  Returns
 * the previous setting, or QMM_EINVAL for an unknown value.  Meant for A/B
 * measurements and tests; the default needs no call. */
enum { QMM_KERNELS_DEFAULT = 0, QMM_KERNELS_MMA_SYNC = 1, QMM_KERNELS_TCGEN05 = 2, QMM_KERNELS_LEAN = 3 };
int qmm_set_kernels(int which);

/* Programmatic dependent launch (on by default): each kernel of the library
 * is launched with programmatic stream serialization, lets the next kernel on
 * the stream start launching early, and reads or writes global memory only
 * after the kernels before it on the stream have completed (griddepcontrol),
 * so stream order is kept while launch latency overlaps.  enable = 0 turns
 * it off (plain stream-ordered launches).  Process-wide; returns the
 * previous setting. */
int qmm_set_pdl(int enable);

/* Where the split planes are added (process-wide, thread-safe):
 *   QMM_REDUCE_KERNEL (default)  the chapter's design (Task 4): the partition
 *       kernel writes the planes and a second kernel, qmm_splitk_reduce's,
 *       adds them.
 *   QMM_REDUCE_FUSED  a one-launch variant of Task 4 for the tcgen05 kernels:
 *       the CTAs of one output tile count themselves in through a 32-bit
 *       counter, and the last to finish adds the tile's planes (FP32,
 *       ascending partition, one cast: the same C bit for bit) and resets the
 *       counter.  The counters live in a fixed area: the last
 *       QMM_FUSED_COUNTER_BYTES of the workspace passed to the call (one per
 *       output tile; calls with more tiles, and the mma.sync family, use the
 *       separate reduce).  qmm_splitk_workspace_bytes includes that area in
 *       this mode.  The counter area must be zero when a workspace is first
 *       used in this mode: zero the workspace once, pass the same workspace
 *       (pointer and size) to every fused call, and zero it again after using
 *       it in QMM_REDUCE_KERNEL mode.  Every call leaves the counters zero,
 *       also when a bounded wait ran out.  Calls that share a workspace must
 *       not overlap on the GPU.
 *   QMM_REDUCE_CLUSTER  a one-launch variant of Task 4 for the tcgen05
 *       kernels that keeps the planes on chip: the split partitions of one
 *       output tile run as one thread-block cluster (up to 16 CTAs), each
 *       stages its partial tile (BF16-rounded, or FP32) in shared memory, and
 *       after a cluster barrier each CTA adds a slice of the tile over every
 *       partition, read through distributed shared memory, in FP32 in
 *       ascending partition order with one cast: the same C bit for bit.  No
 *       plane reaches global memory.  A call whose clusters the device cannot
 *       hold all at once, or whose partial tile does not fit the kernel's
 *       staging area, takes the planes and the reduce kernel as in
 *       QMM_REDUCE_KERNEL; size the workspace as for that mode either way.
 *       Single calls only (the grouped call always uses the reduce kernel).
 * Returns the previous mode, or QMM_EINVAL for an unknown mode. */
#define QMM_FUSED_COUNTER_BYTES 32768
enum { QMM_REDUCE_KERNEL = 0, QMM_REDUCE_FUSED = 1, QMM_REDUCE_CLUSTER = 2 };
int qmm_set_reduce(int mode);

/* Partition rule of the W4A16 calls (process-wide, thread-safe):
 *   QMM_PARTITIONS_EQUAL (default)  the chapter's rule (Task 2, Task 3):
 *       a split divides G = Kred/128, every partition holds G/split groups,
 *       and the policy lowers its split until it divides G
 *       (qmm_splitk_plan).
 *   QMM_PARTITIONS_NEAR_EQUAL  any split 1 <= s <= G.  Partition p holds
 *       floor(G/s) groups, one more for p < G mod s, in order: the cut the
 *       dense GEMM above takes for its k-tiles.  The policy takes
 *       qmm_splitk_plan_near_equal (gpu-kernels-explained, "Split-K, streams
 *       and overlap", Maths: the time falls with the slice length while the
 *       blocks fit one wave).  Down-type shapes (76 groups) then split 7 ways
 *       instead of 4.
 * Applies to qmm_w4a16_g128, qmm_w4a16_g128_partition and
 * qmm_w4a16_g128_noalloc.  With a split that divides G both rules cut the
 * same partitions and give the same bits.  Size workspaces with the split
 * the call will use (qmm_splitk_plan_near_equal's is an upper bound for both
 * rules).  Returns the previous rule, or QMM_EINVAL for an unknown value. */
enum { QMM_PARTITIONS_EQUAL = 0, QMM_PARTITIONS_NEAR_EQUAL = 1 };
int qmm_set_partitions(int mode);

/* Static weights (off by default).  enable = 1 promises that no kernel issued
 * earlier on the same stream writes the packed weights, scales or biases of
 * the matmuls that follow (true of inference weights loaded once).  The
 * tcgen05 partition kernel then loads and dequantizes its first weight stages
 * while the previous kernel on the stream is still running (programmatic
 * dependent launch must be on); only its activation loads and its output
 * writes wait for that kernel.  Weights written by copies or kernels ordered
 * through events or stream synchronization are fine.  The tiny-llm chapter
 * has no counterpart: this is launch-latency overlap on GB300.  Process-wide;
 * returns the previous setting. */
int qmm_set_weights_static(int enable);

/* Status word of the tcgen05 kernels: 0 = ok, 1 = a bounded wait inside a
 * kernel ran out (the kernel stopped early; its output is not valid).
 * Synchronizes with the device (cudaMemcpyFromSymbol); clear != 0 resets the
 * word.  Returns QMM_OK, QMM_EINVAL, QMM_ENODEV or QMM_ECUDA. */
int qmm_kernel_status(int *status, int clear);

/* Test hook for the bounded waits above.  The tiny-llm chapter has no
 * counterpart: this call exists so a test can watch a wait run out on the
 * GPU.  It launches one CTA on `stream` that waits, with the kernels' own
 * bounded wait, on an mbarrier that nothing completes.  After the wait limit
 * (about 1 s) the wait gives up, the status word becomes 1 (as
 * qmm_kernel_status reports it) and the kernel returns; no trap or fault is
 * raised and the context stays usable.  Asynchronous like every launch.
 * Returns QMM_OK, QMM_ENODEV or QMM_ECUDA. */
int qmm_wait_timeout_probe(void *stream);

/* ---- per-call options ------------------------------------------------------
 *
 * The qmm_set_* switches above are process-wide defaults, and some of them
 * change what a call computes (the partition rule and the group plan pick
 * the split, so the result's bits).  A call that passes a qmm_options takes
 * every field that is not QMM_OPT_DEFAULT from it instead, for that call
 * only: two callers in one process (two threads, two libraries) then cannot
 * change each other's results.  Fields and the switch each one overrides:
 *   kernels           QMM_KERNELS_*        qmm_set_kernels
 *   partitions        QMM_PARTITIONS_*     qmm_set_partitions
 *   reduce            QMM_REDUCE_*         qmm_set_reduce
 *   weights_static    0 or 1               qmm_set_weights_static
 *   pdl               0 or 1               qmm_set_pdl
 *   grouped_schedule  QMM_GROUPED_*        qmm_set_grouped_schedule
 *   group_plan        QMM_GROUP_PLAN_*     qmm_set_group_plan
 * A NULL qmm_options means every field QMM_OPT_DEFAULT.  A field outside its
 * range makes the call return QMM_EINVAL (0 from the *_bytes queries) before
 * it checks anything else.  The tiny-llm chapter's single matmul with a
 * use_split_k switch has no process state at all; these calls give the same
 * guarantee for the switches this library adds. */
#define QMM_OPT_DEFAULT (-1)
typedef struct {
    int kernels, partitions, reduce, weights_static, pdl, grouped_schedule, group_plan;
} qmm_options;

/* Every field of *opt set to QMM_OPT_DEFAULT (no-op for NULL). */
void qmm_options_init(qmm_options *opt);

/* qmm_w4a16_g128 under the options (same arguments, codes and results). */
int qmm_w4a16_g128_ex(const void *A, const uint32_t *Wq, const void *scales, const void *biases,
                      void *C, int M, int Kred, int Nout, int split_req, const qmm_policy *pol,
                      void *workspace, size_t ws_bytes, int partial_dtype, void *stream,
                      int *split_used, const qmm_options *opt);

/* qmm_splitk_workspace_bytes under the options (the fused reduce's counter
 * area depends on the reduce mode and the kernel table). */
size_t qmm_splitk_workspace_bytes_ex(int M, int Nout, int split, int partial_dtype,
                                     const qmm_options *opt);

/* What qmm_w4a16_g128_ex would dispatch for this shape, without launching:
 * *split the split (split_req and pol as in qmm_w4a16_g128, QMM_SPLIT_PLANNED
 * and QMM_SPLIT_BALANCED included), *bm / *bn the tile of the kernel that
 * runs (QMM_SPLIT_BALANCED may take a narrower one than the family for M),
 * and *head_rows the rows that QMM_SPLIT_BALANCED runs unsplit (0 when it
 * does not cut the call; *split is then the split of the whole call, else
 * that of rows [*head_rows, M)); the last three are nullable.  num_sms > 0
 * plans for that many SMs; <= 0 queries the current device.  Returns
 * QMM_OK, QMM_EINVAL, QMM_ESHAPE or QMM_ENODEV.  Host only. */
int qmm_call_plan(int M, int Kred, int Nout, int split_req, const qmm_policy *pol,
                  int partial_dtype, int num_sms, const qmm_options *opt, int *split, int *bm,
                  int *bn, int *head_rows);

/* Workspace bytes qmm_w4a16_g128_ex needs for this call as qmm_call_plan
 * plans it (any split_req), or 0 when it needs none or for invalid
 * arguments.  Host only. */
size_t qmm_call_workspace_bytes(int M, int Kred, int Nout, int split_req, const qmm_policy *pol,
                                int partial_dtype, int num_sms, const qmm_options *opt);

/* Static description of a return code. */
const char *qmm_strerror(int code);

/* Name of the CUDA error (cudaGetErrorName) behind the latest QMM_ECUDA that
 * a launch returned on the calling thread ("cudaSuccess" if none has).  A
 * diagnostic with no counterpart on the pages.  Host only. */
const char *qmm_last_cuda_error(void);

/* Allocation-free qmm_w4a16_g128.  The tiny-llm split-K chapter has no
 * counterpart to this call: it exists for callers that cannot allocate
 * device memory where they run the matmul.
 *
 * It computes the same C as qmm_w4a16_g128, with the same arguments
 * (workspace excepted), split rules, alignment rules, kernels and rounding.
 * For equal inputs, split and partial_dtype, the result is bitwise equal.
 * The partial planes live in a fixed buffer of qmm_static_scratch_bytes()
 * (8 MiB), 256-byte aligned, that is a file-scope __device__ array of the
 * library.  The call allocates nothing, neither with cudaMalloc nor any
 * other allocator.
 *   - Set-up: the first call on a device looks the buffer's address up with
 *     cudaGetSymbolAddress, with that device current, and caches it. Make
 *     that first call before any stream capture on the device.  The cached
 *     address does not survive cudaDeviceReset (the module is loaded afresh
 *     and the buffer may move): do not call this entry point on a device
 *     after resetting it.
 *   - Limit: a call whose planes (split * M * Nout * 2 bytes for BF16
 *     partials, * 4 for FP32), rounded up to 256 bytes, exceed
 *     qmm_static_scratch_bytes() - 256 - QMM_FUSED_COUNTER_BYTES returns
 *     QMM_EWORKSPACE and launches nothing (the buffer's last bytes hold the
 *     fused reduce's counters, zero from the start).  The split is the policy's
 *     (split_req = 0), the group plan's (QMM_SPLIT_PLANNED) or the forced
 *     one, as in qmm_w4a16_g128, and the limit applies to the split that
 *     results.  Unsplit calls (split 1) use none of the buffer.
 *     QMM_SPLIT_BALANCED is not taken here (QMM_EINVAL).
 *   - Races: every call on a device shares the one buffer.  Two calls whose
 *     kernels can overlap on the GPU (different streams without ordering
 *     between them) race on it and give undefined results.  Calls ordered
 *     on one stream are safe.
 *   - Nothing has to start at zero: each call's partition kernel writes
 *     every element of the planes it uses before its reduce reads them.
 * Returns the codes of qmm_w4a16_g128, from the same checks in the same
 * order (arguments, policy, shape, alignment, device); QMM_EWORKSPACE then
 * reports planes beyond the buffer, and QMM_ECUDA also covers a failed
 * address lookup. */
int qmm_w4a16_g128_noalloc(const void *A, const uint32_t *Wq, const void *scales,
                           const void *biases, void *C, int M, int Kred, int Nout, int split_req,
                           const qmm_policy *pol, int partial_dtype, void *stream,
                           int *split_used);

/* Size in bytes of the fixed partial-plane buffer of qmm_w4a16_g128_noalloc. */
size_t qmm_static_scratch_bytes(void);

/* ---- several independent calls in few launches ---------------------------
 *
 * gpu-kernels-explained, "Split-K, streams and overlap" (second Concept
 * section): a partial wave leaves SMs idle, and Stream-K balances the work
 * over the SMs instead; "Optimize Prefill vs Decode Kernels" counts some
 * microseconds per launch.  A model
 * step has independent projections (q, k and v of one layer; gate and up)
 * whose calls can share launches: their CTAs fill each other's partial waves
 * and the launch and prologue costs are paid once.
 *
 * One call of a group: the arguments of qmm_w4a16_g128 (device pointers). */
typedef struct {
    const void *A;          /* BF16 [M, Kred] */
    const uint32_t *Wq;     /* [Nout, Kred/8] */
    const void *scales;     /* BF16 [Nout, Kred/128] */
    const void *biases;     /* BF16 [Nout, Kred/128] */
    void *C;                /* BF16 [M, Nout]; no call's C may alias any input or other C */
    int M, Kred, Nout;
} qmm_group_call;

/* Workspace bytes qmm_w4a16_g128_grouped needs: the partial planes of every
 * call whose policy split is > 1, each rounded up to 256 bytes.  0 when no
 * call splits, or for invalid arguments.  Queries the device for the policy
 * (as qmm_policy_preset with num_sms <= 0). */
size_t qmm_group_workspace_bytes(const qmm_group_call *calls, int n, int partial_dtype);

/* The n calls, each with its policy split under the current partition rule
 * (split_req 0 and the GB300 preset of qmm_w4a16_g128), or with the group
 * plan's split under QMM_GROUP_PLAN_GROUP (qmm_set_group_plan), in few launches:
 * the tcgen05 calls of one tile width share one partition launch (up to 16
 * calls per launch), and every split call's planes are added by one reduce
 * launch per 16 split calls.  Calls served by the mma.sync family
 * (qmm_set_kernels) are launched one by one.  The reduce is always the
 * separate kernel (QMM_REDUCE_FUSED does not apply).  Each C is bitwise the C
 * that qmm_w4a16_g128 gives for the call at the same split (its own policy
 * split by default).  The calls must be independent: no
 * call reads another's C.  splits_used (host, nullable, n ints) receives
 * each call's split.  Returns the codes of qmm_w4a16_g128; every call is
 * checked before anything is launched. */
int qmm_w4a16_g128_grouped(const qmm_group_call *calls, int n, void *workspace, size_t ws_bytes,
                           int partial_dtype, void *stream, int *splits_used);

/* qmm_group_workspace_bytes and qmm_w4a16_g128_grouped under per-call
 * options (qmm_options above). */
size_t qmm_group_workspace_bytes_ex(const qmm_group_call *calls, int n, int partial_dtype,
                                    const qmm_options *opt);
int qmm_w4a16_g128_grouped_ex(const qmm_group_call *calls, int n, void *workspace,
                              size_t ws_bytes, int partial_dtype, void *stream, int *splits_used,
                              const qmm_options *opt);

/* Schedule of the grouped call's tcgen05 partition launches (process-wide,
 * thread-safe):
 *   QMM_GROUPED_TILES  one CTA per output tile and partition.
 *   QMM_GROUPED_PERSISTENT (default)  for the launches of tiles up to 64 activation
 *       rows (calls with M <= 64): min(tiles, SMs) CTAs, each walking a list
 *       of the launch's tiles (gpu-kernels-explained, "Split-K, streams and
 *       overlap": a persistent schedule keeps every SM busy rather than
 *       launching one block per tile).  The tiles stay whole.  Each CTA pays
 *       its prologue once, and its copies of the next tile's weights and
 *       activations run while the current tile drains.  Wider tiles keep one
 *       CTA per tile, which measured faster for them.  Each C is bitwise the
 *       C of QMM_GROUPED_TILES (measured on seven projection calls at M = 16,
 *       32 and 64: 13-15 % faster).
 * Returns the previous schedule, or QMM_EINVAL for an unknown value. */
enum { QMM_GROUPED_TILES = 0, QMM_GROUPED_PERSISTENT = 1 };
int qmm_set_grouped_schedule(int mode);

/* Split plan of the grouped call (process-wide, thread-safe):
 *   QMM_GROUP_PLAN_CALLS (default)  each call takes the split qmm_w4a16_g128
 *       would give it alone (the chapter's occupancy policy per call), so each
 *       C is bitwise that call's.
 *   QMM_GROUP_PLAN_GROUP  splits sized for the group (gpu-kernels-explained,
 *       "Split-K, streams and overlap": split only while the SMs would
 *       otherwise idle).  The policy splits every call until it alone fills
 *       the GPU, but a group's calls together already fill it several times,
 *       so those splits only add tiles, each with its fixed cost, and partial
 *       planes.  qmm_group_plan gives the splits.  Each C is bitwise the C of
 *       qmm_w4a16_g128 with split_req = the planned split.
 * qmm_group_workspace_bytes follows the plan in force.  Returns the previous
 * plan, or QMM_EINVAL for an unknown value. */
enum { QMM_GROUP_PLAN_CALLS = 0, QMM_GROUP_PLAN_GROUP = 1 };
int qmm_set_group_plan(int mode);

/* The group plan's splits for n calls of shapes (M, Kred, Nout) (host, 3n
 * ints), without launching anything: per tile width (the calls of one launch),
 * every call starts unsplit, then the call with the longest partition (lowest
 * index on ties) takes its next valid split while that lowers the launch's
 * estimated time.  Valid splits are those of the chapter's rule for a single
 * call: at most 16 and G = Kred/128, at least 512 reduction elements per
 * partition for M <= 8, and dividing G unless QMM_PARTITIONS_NEAR_EQUAL is in
 * force.  The estimate is a longest-first list schedule of the launch's CTA
 * tiles on num_sms SMs plus the partial planes' traffic.  A tile costs 3 us
 * plus 0.40 / 0.45 / 0.55 / 0.60 us per 128-group for tile widths up to
 * 32 / 64 / 128 / more rows.  The planes, written and read back, move at
 * 3 TB/s.  These constants are tuning parameters fitted to this library's
 * kernels on GB300, as the chapter's 320 and 16 are for its kernels.  No
 * move takes a launch over 65536 tiles; a launch over that with every call
 * unsplit keeps each call's own policy split for num_sms.
 * num_sms <= 0 queries the device.  splits (host, n ints) receives the plan.
 * Returns QMM_OK, QMM_EINVAL, QMM_ESHAPE or QMM_ENODEV. */
int qmm_group_plan(const int *shapes, int n, int num_sms, int partial_dtype, int *splits);

/* ---- split-KV decode attention -------------------------------------------
 *
 * "Optimize Prefill vs Decode Kernels" (Required reasoning process, steps 4
 * and 5; Correctness requirements): in decode one query token per sequence
 * attends to its whole KV history, an HBM-bound read of every K and V byte.
 * The history of each (sequence, KV head) is split into S parts (split-KV);
 * each part's partial softmax state -- maximum, sum of exponentials,
 * unnormalized output -- is kept in FP32 and the parts are merged with the
 * log-sum-exp correction.
 *   q     BF16 [B, Hq, D], one query token per sequence
 *   K, V  BF16 [B, Hkv, Lmax, D], head-major (each head's positions contiguous)
 *   lens  device int32 [B]: sequence b uses positions 0 .. lens[b]-1, with
 *         1 <= lens[b] <= Lmax (values outside are clamped into [0, Lmax];
 *         a length of 0 gives NaN outputs for that sequence)
 *   O     BF16 [B, Hq, D]:
 *         O[b,h] = sum_l softmax_l(scale * q[b,h] . K[b,h/QG,l]) V[b,h/QG,l]
 *         with QG = Hq / Hkv query heads per KV head (grouped-query attention)
 * D is 64 or 128; QG is 1, 2, 4 or 8. */

/* The split factor the page prescribes (step 5): S = ceil(num_sms * 4 /
 * (B * Hkv)) -- a grid of 4 blocks per SM, two waves of the kernel's two
 * resident CTAs, within the page's 2-4 -- clamped to [1, max(1,
 * floor(Lmax / 512))] so every split keeps at least 512 positions of the
 * longest sequence.  num_sms <= 0 queries the device.  Returns QMM_OK,
 * QMM_EINVAL or QMM_ENODEV.  Host only. */
int qmm_decode_attention_splits(int B, int Hq, int Hkv, int Lmax, int num_sms, int *splits);

/* Workspace bytes of the partial states for `splits` splits:
 * B * Hq * splits * (D + 2) * 4, or 0 when splits <= 1. */
size_t qmm_decode_attention_workspace_bytes(int B, int Hq, int D, int splits);

/* O = decode attention of q over K, V (above).  splits_req 0 takes
 * qmm_decode_attention_splits; s >= 1 forces s splits (splits past the
 * longest sequence's positions are empty and cost a little).  scale <= 0
 * means 1/sqrt(D).  workspace: device, 16-byte aligned, at least
 * qmm_decode_attention_workspace_bytes bytes when the split used is > 1.
 * One launch (split 1) or the split kernel and the merge kernel on `stream`.
 * splits_used (host, nullable) receives the split.  Returns QMM_OK,
 * QMM_EINVAL (null pointers, sizes < 1, Hq not a multiple of Hkv),
 * QMM_ESHAPE (D not 64 or 128, QG not 1/2/4/8, a grid dimension past 65535,
 * splits_req past 65535), QMM_EALIGN, QMM_EWORKSPACE, QMM_ENODEV or
 * QMM_ECUDA. */
int qmm_decode_attention(const void *q, const void *K, const void *V, const int *lens, void *O,
                         int B, int Hq, int Hkv, int Lmax, int D, float scale, int splits_req,
                         void *workspace, size_t ws_bytes, void *stream, int *splits_used);

/* ---- streaming host activations through the matmul ----------------------
 *
 * gpu-kernels-explained, "Split-K, streams and overlap" (first Concept
 * section; Maths, Overlap): copies and kernels run on separate engines, so a
 * host-to-device copy, a kernel and a device-to-host copy of different chunks
 * can run at once.  With b device buffers, chunk i's copy in waits for chunk
 * i-b's compute to free its buffer; after the pipeline fills it runs at the
 * pace of its slowest engine.
 *
 * One chunk: a W4A16 call whose activations and output live in host memory
 * and whose weights are already on the device. */
typedef struct {
    const void *A_host;     /* host BF16 [M, Kred]; pinned memory to overlap */
    void *C_host;           /* host BF16 [M, Nout]; pinned memory to overlap */
    const uint32_t *Wq;     /* device, as qmm_w4a16_g128 */
    const void *scales;     /* device */
    const void *biases;     /* device */
    int M, Kred, Nout;
} qmm_stream_call;

/* Device bytes qmm_w4a16_g128_stream needs for these calls and `buffers`
 * buffers: per buffer, room for the largest A and C (each rounded up to 256
 * bytes), plus one workspace for the largest split of any call under the
 * current partition rule and reduce mode (computes run one at a time).
 * Returns 0 for invalid arguments.  Host only. */
size_t qmm_stream_arena_bytes(const qmm_stream_call *calls, int n, int buffers);

/* Run n calls as a three-stage pipeline: for chunk i, buffer i % buffers,
 *   stream_in:       wait for chunk i-buffers' compute, copy A_host in;
 *   stream_compute:  wait for that copy and for chunk i-buffers' copy out,
 *                    run qmm_w4a16_g128 (policy split, current rules);
 *   stream_out:      wait for the compute, copy C out to C_host.
 * The waits use events the library creates once per device and reuses.  The
 * streams may be equal (the stages then serialize).  arena: device memory of
 * at least qmm_stream_arena_bytes(calls, n, buffers) bytes (arena_bytes),
 * 256-byte aligned; its contents on return are unspecified (under
 * QMM_REDUCE_FUSED zero it before its first use, as any fused-reduce
 * workspace).  splits_used (host, nullable, n ints) receives each call's
 * split.  Asynchronous: synchronize stream_out before reading C_host.
 * Each call's result is bitwise what qmm_w4a16_g128 gives for it.
 * Returns QMM_OK, QMM_EINVAL (null calls/arena, n < 1, buffers < 1, a chunk
 * with null pointers or bad sizes), QMM_ESHAPE, QMM_EALIGN, QMM_EWORKSPACE
 * (arena too small) or QMM_ECUDA.  Arguments of every chunk are checked
 * before anything is enqueued. */
int qmm_w4a16_g128_stream(const qmm_stream_call *calls, int n, int buffers, void *arena,
                          size_t arena_bytes, void *stream_in, void *stream_compute,
                          void *stream_out, int *splits_used);

/* The schedule model of that pipeline (the Split-K page's, Maths: Overlap),
 * for planning: n chunks with per-chunk engine times t_load[i], t_comp[i],
 * t_store[i] >= 0 (host arrays, any unit).  Each engine takes the chunks in
 * order, one at a time; chunk i's load starts after chunk i-1's load and
 * chunk i-buffers' compute; its compute after its load and chunk i-1's
 * compute (and, with out_reuse = 1, after chunk i-buffers' store, the rule
 * the executor above adds for its output buffers); its store after its
 * compute and chunk i-1's store.  *T receives the end of the last store;
 * events (host, nullable, [n][6]) the start and end of each chunk's load,
 * compute and store.  Returns QMM_OK or QMM_EINVAL.  Host only. */
int qmm_overlap_schedule(int n, int buffers, const double *t_load, const double *t_comp,
                         const double *t_store, int out_reuse, double *T, double *events);

#ifdef __cplusplus
}
#endif

#endif /* QMM_H */
