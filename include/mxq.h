/*
 * mxq — affine group-wise quantized matrix multiply for sm_103a (GB300).
 *
 * The operation (mlxcel issue #1536, Baseline section: weights stored as
 * "affine 4-bit / group 64", activations bf16; issue #1538, 4-bit vs 8-bit
 * section: 8-bit codes are unsigned bytes, and the product accumulates in
 * float at every width):
 *
 *   w^[n, k] = s[n, k/G] * q[n, k] + b[n, k/G]
 *   y[m, n]  = sum_k x[m, k] * w^[n, k]          (fp32 accumulation)
 *
 * G = group_size, the k values that share one scale/bias pair: 64 (the
 * stored format named above), 32 or 128 (issue #1536, Diagnosis item 4: the
 * tile choice there tests group_size <= 64, so the format also comes with
 * other group sizes; 32 and 128 are the sizes on either side of 64).
 *
 * Storage, all row-major and contiguous:
 *   x       bf16   [M, K]            activations
 *   w       uint32 [N, K*bits/32]    packed codes.  4-bit: eight codes per
 *                                    little-endian word, lowest k in the
 *                                    lowest nibble (integer_subbyte<4>, the
 *                                    qmm_naive kernel name in issue #1536's
 *                                    profile table).  8-bit: four codes per
 *                                    word, lowest k in the lowest byte.
 *                                    2-bit: sixteen codes per word, lowest k
 *                                    in the lowest two bits.  3- and 6-bit:
 *                                    the same little-endian bit stream per
 *                                    row, code k in bits [k*b, k*b + b), so
 *                                    a code may straddle two words (the bit
 *                                    width is a parameter of the kernels in
 *                                    issue #1536, Diagnosis item 3).
 *   scales  bf16   [N, K/G]          s per (output row, group of G k)
 *   biases  bf16   [N, K/G]          b per (output row, group of G k)
 *   y       bf16   [M, N]            output, rounded once from fp32 (RNE)
 *
 * All pointers except `stream` are DEVICE pointers owned by the caller; the
 * library allocates nothing and keeps no pointer after a call returns.  All
 * calls are asynchronous on `stream` (a cudaStream_t, NULL = legacy default
 * stream) and return after the launch.  Arguments are checked on the host
 * before anything is launched; a call that returns an error has launched
 * nothing and written nothing.  Inputs must be finite.
 *
 * Device requirement: compute capability 10.3 (sm_103a).
 */
#ifndef MXQ_H
#define MXQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MXQ_OK = 0,
    MXQ_ERR_INVALID_ARG = 1, /* bad size, bits, group size or null pointer   */
    MXQ_ERR_MISALIGNED = 2,  /* x, w or y not 16-byte aligned; or a scale /
                                bias / id pointer not aligned to its type     */
    MXQ_ERR_UNSUPPORTED = 3, /* a valid request this build does not implement */
    MXQ_ERR_ARCH = 4,        /* current device is not compute capability 10.3 */
    MXQ_ERR_CUDA = 5,        /* a CUDA runtime call or launch failed          */
    MXQ_ERR_WORKSPACE = 6,   /* workspace missing or smaller than required    */
    MXQ_ERR_SCRATCH_LIMIT = 7 /* mxq_gather_qmm_noalloc: the request needs more
                                 than MXQ_NOALLOC_SCRATCH_BYTES of scratch      */
} mxq_status;

/* Bits set in *dev_status (device memory, written by the kernels when the
 * caller passes a non-null pointer; the call first stores 0 there).        */
#define MXQ_DEV_BAD_EXPERT_ID   0x1 /* an expert id outside [0, E)             */
#define MXQ_DEV_UNSORTED_IDS    0x2 /* expert ids decrease somewhere           */
#define MXQ_DEV_BAD_ROW_SRC     0x4 /* a row_src entry outside [0, T)          */
#define MXQ_DEV_TIMEOUT         0x8 /* an on-chip pipeline wait gave up; the
                                       output is incomplete                   */

/* Decode GEMV, M = 1 (mlxcel issue #1536, Diagnosis item 3: the qmv kernel;
 * fp32 accumulation at every width is the fix that item names).
 *   x: bf16 [K]; y: bf16 [N]; w, scales, biases as above.
 *   dev_status: device int32 or NULL; receives 0 or MXQ_DEV_TIMEOUT.
 * Requirements: bits in {2, 3, 4, 6, 8}; group_size in {32, 64, 128}; K > 0,
 * K % 64 == 0 and K % group_size == 0 (K % 128 == 0 at 3 bits); N > 0;
 * x, w, y 16-byte aligned; scales, biases 2-byte aligned.  The streaming
 * kernel is used when K % 512 == 0, K <= 20480, K / group_size % 8 == 0 and
 * scales/biases are 16-byte aligned; other shapes take a direct-load kernel
 * (same result rule, different summation order).  The streaming kernel is
 * launched as a
 * programmatic dependent launch: its CTAs may be placed on SMs while the
 * kernel before it on the stream finishes, but they read and write nothing
 * until that kernel has completed, so stream order is kept.                 */
mxq_status mxq_qmv(const void* x, const uint32_t* w, const void* scales, const void* biases,
                   void* y, int K, int N, int bits, int group_size, int32_t* dev_status,
                   void* stream);

/* Decode GEMV for the other operand layout (mlxcel PR #1562, What changed:
 * the grouped GEMM is checked for both operand layouts): w is stored [K, N],
 * row k holding the codes of every output n as the same little-endian bit
 * stream (code n in bits [n*b, n*b + b) of row k), and each group is G
 * consecutive n of one row:
 *   w:      uint32 [K, N*bits/32]
 *   scales, biases: bf16 [K, N/G]
 *   y[n] = sum_k x[k] * (s[k, n/G] * q[k, n] + b[k, n/G])   (fp32 accumulation)
 *   x: bf16 [K]; y: bf16 [N].
 * Requirements: bits in {2, 4, 8} (3 and 6: MXQ_ERR_UNSUPPORTED); group_size
 * in {32, 64, 128}; K > 0; N > 0, N % 64 == 0 and N % group_size == 0;
 * x, w, y 16-byte aligned; scales, biases 2-byte aligned.  `dev_status`
 * (device int32, may be NULL) receives 0.  Up to 8 CTAs of a thread-block
 * cluster split K and add their partials in rank order: deterministic.     */
mxq_status mxq_qmv_kn(const void* x, const uint32_t* w, const void* scales, const void* biases,
                      void* y, int K, int N, int bits, int group_size, int32_t* dev_status,
                      void* stream);

/* Prefill GEMM for the [K, N] operand layout (mlxcel PR #1562, What
 * changed: both operand layouts), w, scales and biases as for mxq_qmv_kn:
 *   y[m, n] = sum_k x[m, k] * (s[k, n/G] * q[k, n] + b[k, n/G])
 *   x: bf16 [M, K]; y: bf16 [M, N].
 * M = 1 runs mxq_qmv_kn (the same operation).  Otherwise the tcgen05 tensor
 * cores: each code word dequantises (one bf16 rounding of s*q + b, as in
 * mxq_qmm) into 8 bf16 contiguous along n, stored as the MMA's MN-major A
 * operand in shared memory; fp32 accumulation in tensor memory.  With fewer
 * tiles than SMs, K is split over up to 8 CTAs of a cluster and the fp32
 * partials are added in a fixed order: deterministic.
 * Requirements: bits in {2, 4, 8} (3 and 6: MXQ_ERR_UNSUPPORTED);
 * group_size in {32, 64, 128}; M > 0; K > 0 (K % 8 == 0 when M > 1); N > 0,
 * N % 64 == 0, N % group_size == 0; x, w, y 16-byte aligned; scales,
 * biases 2-byte aligned.  `dev_status` (device int32, may be NULL) receives
 * 0 or MXQ_DEV_TIMEOUT.                                                     */
mxq_status mxq_qmm_kn(const void* x, const uint32_t* w, const void* scales, const void* biases,
                      void* y, int M, int K, int N, int bits, int group_size,
                      int32_t* dev_status, void* stream);

/* Prefill GEMM, y[M, N] = x[M, K] . w^[N, K]^T (mlxcel issue #1536, Baseline
 * profile table and Diagnosis item 4: the qmm_naive kernel).  M = 1 runs the
 * streaming GEMV of mxq_qmv (the same operation); M = 2 or 3 runs one such
 * GEMV per activation row where the shape allows (fewer rows than a tensor
 * tile's fill is worth).  Otherwise the tcgen05
 * tensor cores: codes are dequantised to bf16 into tensor memory (the MMA's
 * A operand) and the products accumulate in fp32 in tensor memory.  When M
 * and N give fewer 128 x 256 tiles than the GPU has SMs, K is split over up
 * to 8 CTAs of a thread-block cluster and the fp32 partials are added
 * through distributed shared memory in a fixed order; with enough tiles, one
 * persistent CTA per SM walks them.  Either way the result is deterministic
 * for a given shape.
 * Requirements as for mxq_qmv plus M > 0.  `dev_status` (device int32, may
 * be NULL) receives 0 or MXQ_DEV_TIMEOUT.                                   */
mxq_status mxq_qmm(const void* x, const uint32_t* w, const void* scales, const void* biases,
                   void* y, int M, int K, int N, int bits, int group_size, int32_t* dev_status,
                   void* stream);

/* Sorted mixture-of-experts grouped variant (mlxcel PR #1562, Summary: the
 * sorted-MoE prefill path that routes a quantized GatherQMM into a grouped
 * GEMM, B = tokens * top_k rows sorted by expert).
 *   x:          bf16 [T, K]  activation rows
 *   w:          uint32 [E, N, K*bits/32]; scales, biases: bf16 [E, N, K/G]
 *   expert_ids: int32 [B], non-decreasing: expert of sorted row r
 *   row_src:    int32 [B], row of x that feeds sorted row r; NULL means r
 *               (then T must equal B)
 *   y:          bf16 [B, N], in sorted row order
 *   workspace:  device scratch, 256-byte aligned, overwritten by the call:
 *               mxq_gather_workspace_bytes(B, E, K, N) bytes when row_src
 *               is given (it also holds the activation rows in sorted
 *               order), otherwise the smaller mxq_gather_workspace_bytes(B,
 *               E, 0, N) suffices.
 *   dev_status: device int32 or NULL; receives the MXQ_DEV_* bits.
 * Rows whose expert id lies outside [0, E), or whose row_src lies outside
 * [0, T), are skipped and their y rows set to zero.  If the ids are not
 * non-decreasing, nothing is computed, all of y is set to zero and
 * MXQ_DEV_UNSORTED_IDS is reported.  No invalid input makes the kernels
 * read or write out of bounds.
 * Calls with at most 32 rows (a decode step) run one GEMV per row against
 * its expert's matrix (the same result rule, another summation order) and
 * use no workspace memory, though the size check still applies.
 * Larger calls build a tile table on the GPU and run the tensor-core GEMM:
 * at 2 and 4 bits two persistent CTAs per SM take tiles from a counter; at
 * 3, 6 and 8 bits one CTA computes each tile.
 * Requirements: B, E, T, N > 0; K > 0, K % 64 == 0, K % group_size == 0;
 * bits in {2, 3, 4, 6, 8} (K % 128 == 0 at 3 bits); group_size in
 * {32, 64, 128}; x, w, y 16-byte aligned; the rest aligned to type.          */
mxq_status mxq_gather_qmm(const void* x, const uint32_t* w, const void* scales,
                          const void* biases, const int32_t* expert_ids,
                          const int32_t* row_src, void* y, int T, int B, int E, int K, int N,
                          int bits, int group_size, void* workspace, size_t workspace_bytes,
                          int32_t* dev_status, void* stream);

/* The sorted mixture-of-experts grouped GEMM for the [K, N] operand layout
 * (mlxcel PR #1562, What changed: the grouped GEMM is checked against the
 * dense per-expert reference in both operand layouts):
 *   w:      uint32 [E, K, N*bits/32]; scales, biases: bf16 [E, K, N/G]
 *   y[r, n] = sum_k x[src(r), k] * (s_e[k, n/G] * q_e[k, n] + b_e[k, n/G]),
 *             e = expert_ids[r]
 * Every other argument, the workspace (mxq_gather_workspace_bytes) and the
 * handling of invalid ids and rows are as for mxq_gather_qmm.  The call
 * builds the tile table on the GPU (tiles of at most 64 sorted rows of one
 * expert), copies routed rows into sorted order, and runs one CTA per (tile,
 * 128 columns) on the tensor cores, at every B.
 * Requirements: B, E, T > 0; bits in {2, 4, 8} (3 and 6:
 * MXQ_ERR_UNSUPPORTED); group_size in {32, 64, 128}; K > 0, K % 8 == 0;
 * N > 0, N % 64 == 0, N % group_size == 0; alignment as for mxq_gather_qmm. */
mxq_status mxq_gather_qmm_kn(const void* x, const uint32_t* w, const void* scales,
                             const void* biases, const int32_t* expert_ids,
                             const int32_t* row_src, void* y, int T, int B, int E, int K, int N,
                             int bits, int group_size, void* workspace, size_t workspace_bytes,
                             int32_t* dev_status, void* stream);

/* Workspace bytes mxq_gather_qmm (and mxq_gather_qmm_gateup) needs for B
 * rows over E experts with K-wide activation rows routed through row_src
 * (K = 0: no row_src). */
size_t mxq_gather_workspace_bytes(int B, int E, int K, int N);

/* The gate and up projections of a mixture-of-experts layer in one call
 * (mlxcel issue #1538, comment "Correction: MoE decode does not route to
 * qmm_naive": decode steps run fused per-expert gate/up kernels): the same
 * routed activation rows against two expert weight sets of one shape,
 *   y_gate[r, n] = sum_k x[src(r), k] * w^gate_{e(r)}[n, k]
 *   y_up[r, n]   = sum_k x[src(r), k] * w^up_{e(r)}[n, k]
 * with every argument as in mxq_gather_qmm (w_gate/w_up, scales_*,
 * biases_* each [E, N, ...] with the same shape; y_gate, y_up [B, N]; the
 * same workspace size).  No activation function is applied: the pages name
 * none; a caller combines the two outputs.  One launch computes both
 * projections: with at most 32 rows the per-row GEMVs of both sets (grid z
 * = the set); otherwise the routed rows are put in sorted order once and
 * the grouped GEMM takes the tiles of both sets (persistent CTAs at 2 and 4
 * bits, one CTA per tile and set otherwise).  Each output is bit for bit the
 * output mxq_gather_qmm gives for its set.  The status word reports the id
 * and row_src checks and timeouts of either set.                          */
mxq_status mxq_gather_qmm_gateup(const void* x, const uint32_t* w_gate, const void* scales_gate,
                                 const void* biases_gate, const uint32_t* w_up,
                                 const void* scales_up, const void* biases_up,
                                 const int32_t* expert_ids, const int32_t* row_src, void* y_gate,
                                 void* y_up, int T, int B, int E, int K, int N, int bits,
                                 int group_size, void* workspace, size_t workspace_bytes,
                                 int32_t* dev_status, void* stream);

/* Sorted mixture-of-experts GEMM without any allocation: the same operation,
 * arguments, results and checks as mxq_gather_qmm, but the scratch memory
 * comes from one fixed array inside the library instead of a caller-provided
 * workspace.  (The pages that define the operation have no counterpart to
 * this call; it exists for callers that cannot provide device memory.)
 *
 * Who needs it: callers that have no device allocator of their own (plain C
 * hosts), runtimes whose device memory is fully reserved before serving
 * starts, and loops that must not allocate between steps.  Nothing is
 * allocated at call time, by the caller or by the library: the scratch is
 * MXQ_NOALLOC_SCRATCH_BYTES of device memory reserved on each device when
 * the library's device code is loaded there.
 *
 * Limit: a request whose scratch, mxq_gather_workspace_bytes(B, E, K, N)
 * with row_src (or mxq_gather_workspace_bytes(B, E, 0, N) without), exceeds
 * MXQ_NOALLOC_SCRATCH_BYTES returns MXQ_ERR_SCRATCH_LIMIT before anything
 * touches the device.  32 MiB holds, for example, the tile table and the
 * sorted rows of 4584 routed rows of K = 2816.
 *
 * Set-up: the first call on each device looks up the scratch's device
 * address with that device current (this may load the library's device
 * code); make that first call before capturing a stream into a graph.  The
 * address is kept for the life of the process: do not use this entry point
 * on a device after cudaDeviceReset (or any other teardown of its primary
 * context), since the scratch may then live at another address.
 * Nothing in the scratch has to start at zero: every call writes all the
 * scratch it reads.
 *
 * Concurrency: all calls on one device share the scratch.  Two calls whose
 * execution overlaps (different streams, or different threads without
 * ordering between them) race on it and produce wrong results; order them,
 * for example by issuing every call on the same stream.                    */
#define MXQ_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
mxq_status mxq_gather_qmm_noalloc(const void* x, const uint32_t* w, const void* scales,
                                  const void* biases, const int32_t* expert_ids,
                                  const int32_t* row_src, void* y, int T, int B, int E, int K,
                                  int N, int bits, int group_size, int32_t* dev_status,
                                  void* stream);

/* Affine group-wise encoder: the stored format from float weights (the
 * format of mlxcel issue #1536, Baseline section; the affine map read as
 * bias = group minimum, scale = group range / (2^bits - 1)).
 *   w:      float [N, K] row-major (finite), 16-byte aligned
 *   codes:  uint32 [N, K*bits/32], 16-byte aligned (output)
 *   scales, biases: bf16 [N, K/G] (output)
 * Per (row, group of G = group_size): mn, mx = min, max (-0 read as +0);
 * s = bf16(RN(RN(mx - mn) / (2^bits - 1))), b = bf16(mn), rounded to nearest
 * even; q = clamp(rint(RN(RN(w - b) / s)), 0, 2^bits - 1) with the stored
 * bf16 s and b, q = 0 when s == 0.  All decisions in binary32, so the codes
 * are reproducible bit for bit.  Requirements: bits in {2, 3, 4, 6, 8}
 * (K % 128 == 0 at 3 bits);
 * group_size in {32, 64, 128}; K > 0, K % 64 == 0, K % group_size == 0;
 * N > 0.                                                                    */
mxq_status mxq_quantize(const float* w, uint32_t* codes, void* scales, void* biases, int N,
                        int K, int bits, int group_size, void* stream);

/* Static description of a status code. */
const char* mxq_status_string(mxq_status status);

/* Library version, major * 10000 + minor * 100 + patch. */
int mxq_version(void);

/* Testing aid; the pages have no counterpart.  Every on-chip pipeline wait
 * (a warp waiting for a copy, a stage or an accumulator) gives up after a
 * budget of SM clock cycles, after which the kernel winds down, the call's
 * dev_status receives MXQ_DEV_TIMEOUT and the output is incomplete.  This
 * sets that budget for kernels launched from now on by any thread of the
 * process (kernels already launched keep theirs) and returns the budget now
 * in force.  cycles <= 0 restores the default, 2e9 cycles (about one second
 * at 2 GHz); larger values are clamped to it.  The environment variable
 * MXQ_DEBUG_WAIT_BUDGET, read at the first launch, gives the initial value.
 * A CTA's waits for the copies and MMAs it issued itself, before it exits or
 * frees tensor memory, always take the default budget, so a short budget
 * leaves no asynchronous write behind a finished kernel, and a call after it
 * runs normally.                                                             */
long long mxq_debug_set_wait_budget(long long cycles);

#ifdef __cplusplus
}
#endif

#endif /* MXQ_H */
