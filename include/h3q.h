/*
 * h3q.h -- C ABI of the GB300 (sm_103a) W8A8 INT8 projection Linear.
 *
 * The operation is the INT8 projection of the MiniMax-H3 DiT: the Q, K, V,
 * attention-output, FC1 and FC2 Linears at the native hidden width K = 5376
 * (and the FC2 input width 21504), with no K padding and no weight
 * dequantisation.  Sources, by page title and section:
 *   [P1] "feat(mps): support MiniMax-H3 INT8 inference on Apple M5"
 *        (ModelTC/LightX2V pull request #1672): opening description (the
 *        300-Linear dit_proj profile, native K = 5376, no K padding, no weight
 *        dequantisation); Validation (INT8 weights with finite positive FP32
 *        per-channel scales, CPU INT32 references); Summary by CodeRabbit
 *        (activation quantiser with masked tails, exact K tiles).
 *   [P2] "MLX implementation and experiment report" (MiniMax-H3-Image-mlx,
 *        reports/RESULTS.md): What the default preserves (a biased BF16
 *        Linear adds the bias before the single rounding of the output).
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller, except the
 *     host buffers of h3q_linear_w8a8_grouped_host.  The library allocates no
 *     device memory and keeps no per-call state.
 *   - Layouts are dense and row-major with the last dimension contiguous:
 *     activations X [M, K] (tokens x in-features), weights W [N, K]
 *     (out-features x in-features, the nn.Linear layout), outputs [M, N].
 *   - BF16 tensors are passed as uint16_t bit patterns.
 *   - Every base pointer must be 16-byte aligned (vector loads and TMA);
 *     anything else returns H3Q_ERR_MISALIGNED.
 *   - Shapes: M >= 1, N >= 1, 16 <= K <= 133143 and K % 16 == 0.  The K bound
 *     keeps K * 127^2 below 2^31, so the INT32 accumulator cannot overflow;
 *     K % 16 keeps every INT8 row 16-byte aligned.  M <= 2^31 - 65536 and
 *     N <= 65535 * 128 (32-bit tile coordinates); within these, M and N are
 *     arbitrary: ragged tiles are masked.
 *   - Work is enqueued on `stream` and runs asynchronously, except where an
 *     entry point says it synchronises.  Argument errors are returned before
 *     anything is enqueued.  A launch failure returns H3Q_ERR_CUDA; faults of
 *     already-enqueued work surface at the caller's next synchronisation.
 *   - Results are bitwise deterministic run to run.
 *   - An entry point that does not synchronise puts all its work on `stream`,
 *     so it can be captured in a CUDA graph and replayed.
 */
#ifndef H3Q_H
#define H3Q_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum h3q_status {
  H3Q_OK = 0,
  H3Q_ERR_INVALID_ARG = 1,       /* null pointer, bad dtype, workspace too small */
  H3Q_ERR_UNSUPPORTED_SHAPE = 2, /* M, N or K outside the rules above          */
  H3Q_ERR_MISALIGNED = 3,        /* a base pointer not 16-byte aligned          */
  H3Q_ERR_NONFINITE = 4,         /* a weight row holds Inf or NaN               */
  H3Q_ERR_CUDA = 5,              /* a CUDA runtime or launch error              */
  H3Q_ERR_TIMEOUT = 6,           /* a bounded device-side wait gave up          */
  H3Q_ERR_NO_DEVICE = 7          /* no sm_103 device is current                 */
} h3q_status;

typedef enum h3q_dtype {
  H3Q_DTYPE_F32 = 0,
  H3Q_DTYPE_BF16 = 1
} h3q_dtype;

/* Static, human-readable name of a status code (never NULL). */
const char* h3q_status_string(int status);

/* Library ABI version: major * 10000 + minor * 100 + patch. */
int h3q_version(void);

/*
 * A1 -- offline weight quantiser ([P1] Validation; Changes table, "per-row
 * INT8 conversion").  For each output channel n:
 *     a = max_k |W[n,k]|,  s = a / 127 (FP32, round to nearest even),
 *     q[n,k] = clamp(rint(W[n,k] / s), -127, 127)   (FP32 division, ties even),
 * with s = 1 and q = 0 for an all-zero row and s = 2^-149 for a non-zero row
 * whose a / 127 underflows to zero.
 *
 *   w         [N, K] FP32 (w_dtype = H3Q_DTYPE_F32) or BF16 bits (H3Q_DTYPE_BF16)
 *   q_out     [N, K] int8, written
 *   scale_out [N] FP32, written: finite and positive on success
 *
 * Returns H3Q_ERR_NONFINITE if any weight is Inf or NaN (q_out and scale_out
 * are then unspecified).  To check this it copies the N scales to the host and
 * SYNCHRONISES `stream` before returning; it is an offline call.
 */
h3q_status h3q_quantize_weights(const void* w, int w_dtype, int64_t N, int64_t K,
                                int8_t* q_out, float* scale_out, cudaStream_t stream);

/*
 * A2 -- per-token activation quantiser ([P1] Summary by CodeRabbit: the
 * activation quantiser, tails masked).  For each token row m of X, the same
 * rule as A1 over exactly K elements (a row is never padded).
 *
 *   x         [M, K] BF16 bits
 *   q_out     [M, K] int8, written
 *   scale_out [M] FP32, written
 *
 * Non-finite activations are outside the contract: no check is made and the
 * affected rows' results are unspecified (no fault).  The kernel is launched
 * with programmatic dependent launch: its blocks may be scheduled while the
 * previous kernel on `stream` finishes, and wait for that kernel's results
 * before they read x, so stream order is kept.
 */
h3q_status h3q_quantize_act(const uint16_t* x, int64_t M, int64_t K,
                            int8_t* q_out, float* scale_out, cudaStream_t stream);

/*
 * Bytes of device workspace that h3q_linear_w8a8 needs for this shape: the
 * quantised activations re-coded as FP16 (exact: every INT8 value is an FP16
 * value), read by the tensor cores; per 256 tokens the largest sum of squares
 * of a coded row, whole and per quarter of K; a 256-byte status block; per 16
 * weight rows the largest sum of squares, whole and per quarter of K; and a
 * list of the tiles computed in K chunks (about
 * M * 2 * K + 8 * M * N / 32768 + 5 * N / 4 bytes in all).  The caller
 * allocates it; calls that share a workspace must not overlap on the GPU.
 */
size_t h3q_linear_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * A2 + A3 + A4 -- the W8A8 Linear:
 *     acc[m,n] = sum_k qa[m,k] * qw[n,k]                      (exact INT32)
 *     y[m,n]   = BF16_RNE(acc[m,n] * xs[m] * ws[n] + bias[n])  (one rounding)
 * ([P1] Validation, CPU INT32 references; [P2] What the default preserves,
 * bias added before the rounding).  The BF16 result is within one BF16 ulp of
 * that value computed exactly.  The product runs on the FP16 tensor cores as
 * exact integer arithmetic, so acc is the exact INT32 sum: a tile of 256
 * tokens x 256 channels accumulates all of K in FP32 when the largest
 * squared row norms of its INT8 activations and weights multiply to at most
 * 2^48 (every partial sum is then an integer of magnitude <= 2^24, by
 * Cauchy-Schwarz); any other tile drains its FP32 partial sums into INT32
 * every <= 1024 K.
 *
 * Where the activations come from:
 *   x != NULL            BF16 [M, K]; quantised here (A2).  xs is written, and
 *                        xq too unless it is NULL.
 *   x == NULL, xq != NULL  already quantised: xq [M, K] int8 and xs [M] are read.
 *   x == NULL, xq == NULL  reuse: the workspace still holds the coded
 *                        activations of the previous call made with it (same
 *                        M and K, nothing written to it since); xs is read.
 *                        This lets Linears that share an input (Q, K, V)
 *                        quantise it once.
 *
 *   xs         [M] FP32 activation scales (never NULL).
 *   wq, ws     [N, K] int8 weights and [N] FP32 per-channel scales (from A1).
 *   bias       [N] BF16 bits, or NULL for no bias.
 *   y          [M, N] BF16 bits, written; may be NULL if acc_out is not NULL.
 *   acc_out    [M, N] int32 raw accumulators, written; NULL to skip (testing).
 *   workspace  >= h3q_linear_workspace_bytes(M, N, K) bytes, 16-byte aligned.
 *
 * Everything is enqueued on `stream`; the call does not synchronise.  If a
 * bounded device-side wait gives up (it cannot on a healthy GPU), the kernel
 * returns early, leaves the outputs unspecified and sets the workspace's
 * status word: see h3q_workspace_status.
 */
h3q_status h3q_linear_w8a8(const uint16_t* x, int8_t* xq, float* xs,
                           const int8_t* wq, const float* ws, const uint16_t* bias,
                           int64_t M, int64_t N, int64_t K,
                           uint16_t* y, int32_t* acc_out,
                           void* workspace, size_t workspace_bytes,
                           cudaStream_t stream);

/*
 * Bytes of device workspace for h3q_linear_w8a8_grouped with G Linears of
 * this shape (as h3q_linear_workspace_bytes, with the weight norms and the
 * fallback lists once per Linear).  0 if G is outside 1..4.
 */
size_t h3q_linear_grouped_workspace_bytes(int G, int64_t M, int64_t N, int64_t K);

/*
 * A2 + A3 + A4 for G Linears that read the same activations -- the Q, K and
 * V projections of a DiT block ([P1] opening description: the per-block
 * projections of the 300-Linear dit_proj profile, quantised separately, never
 * fused) -- in one pass: A2 once, then the output tiles of all G Linears from
 * one persistent GEMM launch.  Each result is that of h3q_linear_w8a8 with
 * the same operands, bit for bit.
 *
 *   x, xq, xs  as in h3q_linear_w8a8 (quantise, pre-quantised, or reuse).
 *   G          1..4 Linears, all of shape [N, K].
 *   wq, ws, bias, y
 *              host arrays of G device pointers: INT8 weights [N, K], FP32
 *              scales [N], BF16 bias [N] (bias itself, or any entry, may be
 *              NULL), BF16 outputs [M, N] (never NULL).
 *   workspace  >= h3q_linear_grouped_workspace_bytes(G, M, N, K) bytes.
 *
 * Errors as h3q_linear_w8a8; G outside 1..4 or a NULL array or required
 * entry gives H3Q_ERR_INVALID_ARG.  The pointer arrays are read during the
 * call only.  Enqueued on `stream`; does not synchronise.
 */
h3q_status h3q_linear_w8a8_grouped(const uint16_t* x, int8_t* xq, float* xs, int G,
                                   const int8_t* const* wq, const float* const* ws,
                                   const uint16_t* const* bias,
                                   int64_t M, int64_t N, int64_t K,
                                   uint16_t* const* y, void* workspace, size_t workspace_bytes,
                                   cudaStream_t stream);

/*
 * Status of the last h3q_linear_w8a8 that used `workspace` (same M, K):
 * H3Q_OK, or H3Q_ERR_TIMEOUT if one of its bounded device-side waits gave up.
 * SYNCHRONISES `stream` to read the status word.
 */
h3q_status h3q_workspace_status(const void* workspace, int64_t M, int64_t K,
                                cudaStream_t stream);

/*
 * Bytes of device workspace for h3q_linear_w8a8_grouped_host: a grouped
 * workspace for one chunk of min(chunk_rows, M) rows, then one status word
 * per chunk.  0 if G is outside 1..4, a size is < 1, or chunk_rows is not a
 * positive multiple of 16.
 */
size_t h3q_linear_w8a8_grouped_host_workspace_bytes(int G, int64_t M, int64_t N, int64_t K,
                                                    int64_t chunk_rows);

/*
 * The row chunks h3q_linear_w8a8_grouped_host makes of M rows with these
 * chunk_rows and first_rows (0 = the default first chunk): returns how many
 * there are, and writes the first min(count, capacity) chunk sizes to
 * rows_out (which may be NULL).  Returns -1 for arguments the pipeline
 * rejects.  Host-only: touches no device.
 */
int64_t h3q_linear_w8a8_grouped_host_chunks(int64_t M, int64_t chunk_rows, int64_t first_rows,
                                            int64_t* rows_out, int64_t capacity);

/*
 * The grouped Linear (h3q_linear_w8a8_grouped, A2 + A3 + A4 with A2 once)
 * from and to page-locked HOST memory: the one entry point that takes host
 * pointers.  X is uploaded, and the G outputs downloaded, in row chunks that
 * overlap both copy directions with the grouped calls.  The host link is the
 * bound, and the outputs are G times the input, so the first chunks are small
 * and the downloads start early: chunk sizes run first_rows, 2*first_rows, ...
 * up to chunk_rows, then chunk_rows until M is covered.  Each output row is
 * that of h3q_linear_w8a8_grouped on the same operands, bit for bit (the row
 * chunks do not change any row's arithmetic: A2 is per token, and each output
 * element depends on its own token row only).
 *
 *   x_host     [M, K] BF16, page-locked host memory (cudaHostAlloc or
 *              cudaHostRegister); read.
 *   G, wq, ws, bias
 *              as in h3q_linear_w8a8_grouped (device pointers).
 *   y_host     host array of G page-locked host pointers, [M, N] BF16 each;
 *              written.
 *   x_dev      [M, K] BF16 device staging for X; overwritten.
 *   xs         [M] FP32 device; the activation scales are written.
 *   y_dev      host array of G device pointers, [M, N] BF16 each; the
 *              outputs are written there too.  When the G outputs are the
 *              consecutive [M, N] blocks of one [G, M, N] buffer on each side,
 *              a chunk's downloads are one 2D copy, which the link carries
 *              faster (if the runtime refuses that copy, they go one by one).
 *   chunk_rows steady chunk size, a positive multiple of 16.
 *   first_rows first chunk size, a multiple of 16 in [16, chunk_rows];
 *              0 picks chunk_rows / 4 rounded up to a multiple of 16.
 *   workspace  >= h3q_linear_w8a8_grouped_host_workspace_bytes(G, M, N, K,
 *              chunk_rows) bytes of device memory.
 *   stream     the grouped calls run here; the copy streams start after the
 *              work already queued on it.
 *   h2d_stream, d2h_stream
 *              the upload and download streams.  Overlap needs three distinct
 *              streams that do not synchronise with one another (non-blocking
 *              streams); equal streams still give the right result, serially.
 *
 * SYNCHRONISES: returns once y_host holds every output (or, after a failure,
 * once nothing it enqueued is still running).  Returns H3Q_ERR_TIMEOUT if a
 * bounded device-side wait of any chunk gave up; argument errors (including
 * pageable host memory: H3Q_ERR_INVALID_ARG) come before anything is
 * enqueued.  The library keeps a few CUDA events per device across calls
 * (created on first use); calls from several host threads take turns.
 */
h3q_status h3q_linear_w8a8_grouped_host(const uint16_t* x_host, int G, const int8_t* const* wq,
                                        const float* const* ws, const uint16_t* const* bias,
                                        int64_t M, int64_t N, int64_t K,
                                        uint16_t* const* y_host, uint16_t* x_dev, float* xs,
                                        uint16_t* const* y_dev, int64_t chunk_rows,
                                        int64_t first_rows, void* workspace,
                                        size_t workspace_bytes, cudaStream_t stream,
                                        cudaStream_t h2d_stream, cudaStream_t d2h_stream);

/*
 * Diagnostic: how many tiles of 128 tokens x 256 channels the last
 * h3q_linear_w8a8 (or, summed over its Linears, h3q_linear_w8a8_grouped)
 * that used `workspace` (same M, K) computed with K cut into
 * chunks, because the squared-norm bounds did not let one FP32 accumulator
 * hold all of K; the other tiles took the single-accumulator path.  Both
 * paths give the same exact result; the chunked one is slower.  Written to
 * *tiles.  SYNCHRONISES `stream`.
 */
h3q_status h3q_linear_chunked_tiles(const void* workspace, int64_t M, int64_t K,
                                    int64_t* tiles, cudaStream_t stream);

/*
 * Diagnostic: how many tiles of 256 tokens x 256 channels the same call
 * computed with one FP32 accumulator over all of K by way of checkpoints:
 * the whole-K norm bound failed, but the bounds of the four quarters of K
 * ("norm segments") held, and between runs of segments the kernel read the
 * accumulator's largest magnitude and proved that the next run could not
 * carry a partial sum past 2^24.  A tile whose proof fails is also counted
 * by h3q_linear_chunked_tiles (as one or two 128-token tiles): the chunked
 * kernel recomputes it.  Written to *tiles.  SYNCHRONISES `stream`.
 */
h3q_status h3q_linear_checkpointed_tiles(const void* workspace, int64_t M, int64_t K,
                                         int64_t* tiles, cudaStream_t stream);

/*
 * The group-wise affine comparison scheme (weight-only; "MLX implementation and
 * experiment report", Operator tuning: Q8/g64 and Q4/g64 GEMMs; "[feat] Add
 * MiniMax H3 MLX T2VA inference": affine INT8/INT6/INT4 checkpoints).  Not the
 * W8A8 method: the activations stay BF16, and the weights carry a step and an
 * offset per output channel and group of 64 inputs.  Offline quantisation:
 *
 *   w       [N, K] FP32 (w_dtype = H3Q_DTYPE_F32) or BF16 bits, K a multiple of 64
 *   bits    8 (Q8/g64) or 4 (Q4/g64)
 *   q_out   [N, K] unsigned codes in [0, 2^bits - 1], one per byte (4-bit codes
 *           are not packed: the GEMM reads both widths alike)
 *   ab_out  [N, K/64][2] FP32: per group the step a and the offset b, so that
 *           the group's weights are represented by a q + b
 *
 * Per group, with L = 2^bits - 1: b = min, a = (max - min) / L (each an FP32
 * operation, rounded to nearest even; a = 1 for a constant group, the
 * smallest positive FP32 when the quotient underflows), q = clamp(rint((w -
 * b) / a), 0, L).  Returns H3Q_ERR_INVALID_ARG for another bits,
 * H3Q_ERR_NONFINITE if any weight is Inf or NaN, H3Q_ERR_UNSUPPORTED_SHAPE if
 * K is not a multiple of 64.  SYNCHRONISES `stream` (offline call).
 */
h3q_status h3q_quantize_weights_affine(const void* w, int w_dtype, int bits, int64_t N,
                                       int64_t K, uint8_t* q_out, float* ab_out,
                                       cudaStream_t stream);

/*
 * The weight-only Linear of the comparison scheme:
 *   y[m, n] = BF16_RNE( sum_k x[m, k] w^[n, k] + bias[n] ),
 *   w^[n, k] = BF16_RNE( RN_fp32( a q[n, k] + b ) )   (one FP32 FMA, then BF16)
 * with the sum accumulated in FP32 on the tensor cores (order unspecified).
 *
 *   x       [M, K] BF16, K a multiple of 64        (read)
 *   q, ab   as h3q_quantize_weights_affine wrote them (read)
 *   bias    [N] BF16, or NULL                      (read)
 *   y       [M, N] BF16                            (written)
 *   status  one device uint32, zeroed by the call; nonzero after it if a
 *           bounded device-side wait gave up (the outputs are then unspecified)
 *
 * Errors as h3q_linear_w8a8.  Enqueued on `stream`; does not synchronise.
 */
h3q_status h3q_linear_affine_w8(const uint16_t* x, const uint8_t* q, const float* ab,
                                const uint16_t* bias, int64_t M, int64_t N, int64_t K,
                                uint16_t* y, uint32_t* status, cudaStream_t stream);

/*
 * Self-test of the device-side failure path (no counterpart on the pages).
 * Every wait in the library's kernels is bounded: after the limit (2 s) the
 * kernel sets a bit in the call's status word and returns, and the call then
 * reports H3Q_ERR_TIMEOUT through h3q_workspace_status instead of hanging the
 * GPU.  This entry point drives that path on purpose, without a fault: one
 * thread waits with the same helper on an mbarrier that nothing arrives on.
 *   status  one device uint32 (4-byte aligned), zeroed by the call
 * Returns H3Q_ERR_TIMEOUT when the wait gave up and reported it (the expected
 * result; the context stays usable), H3Q_OK if it did not.  SYNCHRONISES
 * `stream`; takes about 2 s.
 */
h3q_status h3q_selftest_bounded_wait(uint32_t* status, cudaStream_t stream);

/*
 * Throughput probe of the one INT8 tensor instruction of sm_103 (no
 * counterpart on the pages; it supplies the denominator of "% of dense INT8
 * peak").  sm_103a has no INT8 tcgen05 MMA, so the part's INT8 tensor rate is
 * that of the warp-level mma.sync m16n8k32 s8 x s8 -> s32.  Every warp of a
 * full grid (4 blocks of 8 warps per SM) runs 8 independent accumulator
 * chains of it for about 40 ms; the launch is timed with CUDA events on
 * `stream`, and 8192 operations per instruction (2 * 16 * 8 * 32) over that
 * time are written to *tops (TOPS, 1e12 operations per second).  Allocates no
 * device memory; SYNCHRONISES `stream`.
 */
h3q_status h3q_probe_mma_s8_tops(double* tops, cudaStream_t stream);

/*
 * Throughput probe of the FP16 tensor instruction the hot GEMM issues (no
 * counterpart on the pages; it supplies the ceiling that the GEMM's
 * tensor-pipe share is read against): tcgen05.mma.cta_group::2.kind::f16,
 * M = N = 256, K = 16, FP32 accumulator in TMEM, B K-major in shared memory
 * with the 128-byte swizzle, and A in TMEM (a_in_smem = 0, the hot kernel's
 * form) or in shared memory (a_in_smem = 1).  One CTA pair per two SMs, as
 * many as can be resident at once, each issuing 65536 MMAs back to back over
 * one resident k-block of small-integer operands (about 4 ms); the launch is
 * timed with CUDA events on `stream`, and 2 * 256 * 256 * 16 operations per
 * MMA over that time are written to *tflops (1e12 per second).
 *
 *   H3Q_ERR_INVALID_ARG  tflops NULL, or a_in_smem not 0 or 1
 *   H3Q_ERR_TIMEOUT      the bounded wait for the MMAs gave up (2 s)
 *
 * Allocates no device memory; SYNCHRONISES `stream`.
 */
h3q_status h3q_probe_mma_f16_pair_tflops(double* tflops, int a_in_smem, cudaStream_t stream);

/*
 * A3 + A4 on the legacy warp-level INT8 tensor instruction (mma.sync
 * m16n8k32 s8 -> s32), exact by construction; the same arithmetic and output
 * as h3q_linear_w8a8 from pre-quantised activations.  Kept as the baseline
 * the tcgen05 path is measured against: on sm_103 this instruction is the
 * only INT8 tensor path, and it is several times slower.
 *
 *   xq [M, K] int8, xs [M] FP32, wq [N, K] int8, ws [N] FP32, bias [N] BF16
 *   or NULL; y [M, N] BF16 and/or acc_out [M, N] int32.  No workspace.
 */
h3q_status h3q_linear_w8a8_mma_sync(const int8_t* xq, const float* xs, const int8_t* wq,
                                    const float* ws, const uint16_t* bias,
                                    int64_t M, int64_t N, int64_t K,
                                    uint16_t* y, int32_t* acc_out, cudaStream_t stream);

/*
 * h3q_linear_w8a8 for callers that cannot allocate device memory (the pages
 * have no counterpart: this is a convenience of this library).  Some callers
 * may not call cudaMalloc at call time -- an inference engine's plugin enqueue
 * that is handed only its input and output buffers, or a serving loop that
 * must not block on, or fail in, the allocator once warmed up.  This entry
 * point allocates nothing: its scratch is a 16 MiB array built into the
 * library, which every GPU that loads the library holds until the process
 * exits.
 *
 * Arguments and results are those of h3q_linear_w8a8, without the workspace,
 * and with x or xq required (there is no reuse of an earlier call's
 * activations).  Shapes whose h3q_linear_workspace_bytes(M, N, K) exceeds
 * 16 MiB (16777216 bytes) are rejected with H3Q_ERR_UNSUPPORTED_SHAPE; at
 * N = K = 5376 that allows M up to 1559 tokens.
 *
 * The first call in a CUDA context looks up the array's device address (with
 * the device current) and keeps it for that context; make that first call
 * before any stream capture.  After cudaDeviceReset the device has a new
 * context, and the next call looks the address up again.  All calls share the
 * one array and each rewrites what it needs of it, so calls whose work
 * overlaps on the GPU (different streams, or concurrent host threads) race
 * and must be serialised by the caller.  Enqueued on `stream`; does not
 * synchronise.  A bounded device-side wait that gives up (it cannot on a
 * healthy GPU) leaves the outputs unspecified and sets the status word in the
 * built-in scratch: read it with h3q_linear_w8a8_noalloc_status.
 */
h3q_status h3q_linear_w8a8_noalloc(const uint16_t* x, int8_t* xq, float* xs,
                                   const int8_t* wq, const float* ws, const uint16_t* bias,
                                   int64_t M, int64_t N, int64_t K,
                                   uint16_t* y, int32_t* acc_out, cudaStream_t stream);

/*
 * Status of the last h3q_linear_w8a8_noalloc on the current device (called
 * with the same M and K, and no other no-alloc call since): H3Q_OK, or
 * H3Q_ERR_TIMEOUT if one of its bounded device-side waits gave up -- what
 * h3q_workspace_status reports for a caller-provided workspace (the pages
 * have no counterpart).  An M and K whose workspace would not fit the built-in
 * scratch even at N = 1 give H3Q_ERR_UNSUPPORTED_SHAPE.  SYNCHRONISES `stream`
 * to read the status word; allocates nothing.
 */
h3q_status h3q_linear_w8a8_noalloc_status(int64_t M, int64_t K, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* H3Q_H */
