/*
 * imp_nvfp4.h -- NVFP4 weight-quantized linear layer for GB300 (sm_103a).
 *
 * The operation: the 4-bit weight-quantized linear layer that dominates the
 * memory-bound decode step of a single-GPU LLM inference engine.  The imp
 * engine README ("How it works": decode is bandwidth-bound, so the weights
 * are stored in 4 bits (NVFP4) and multiplied without being unpacked to 16
 * bits; prefill is compute-bound) and the engineering-log entry "NVFP4 at the
 * bit level" (four bits and two scales) define the format:
 *
 *   W is N rows of K elements.  Each element is an E2M1 code (1 sign, 2
 *   exponent, 1 mantissa bit: magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6), packed two
 *   per byte -- element 2i in the low nibble of byte i of its row.  Every 16
 *   consecutive elements of a row (a block) share one E4M3 scale byte
 *   (OCP FP8 E4M3 "fn": bias 7, max 448, sign bit always 0 here).  The whole
 *   tensor shares one fp32 scale s.  Element value = e2m1 * e4m3 * s.
 *
 * Quantizer recipe (bit-exact, IEEE fp32, every step correctly rounded):
 *   g  = max |x| over the tensor;  s = g / 2688  (2688 = 6 * 448)
 *   per block: a = max |x_j|; u = (a / 6) / s (u = 0 when s = 0);
 *              sb = E4M3(u), round to nearest even, saturating at 448
 *              d  = e4m3(sb) * s
 *              code_j = 0 if d == 0, else sign(x_j) | E2M1(|x_j| / d), round
 *              to nearest even, saturating at 6.
 *
 * Linear layer: Y[M][N] = X[M][K] * W^T, bf16 in and out, fp32 accumulation.
 *   M <= 16 (decode, "1. The big picture", section "Two phases with very
 *   different costs": one token per step, every weight read once): X stays
 *   bf16; y[m][n] = s * sum_b e4m3(sb[n][b]) * sum_{j<16} x[m][16b+j] *
 *   e2m1(c[n][16b+j]).
 *   M > 16 (prefill): X is first quantized with the same recipe (its own
 *   tensor scale s_x) and Y = s_x * s * sum over blocks of the products of
 *   the two block-scaled E2M1 operands, on the block-scaled FP4 tensor cores.
 *   The result is rounded to bf16 with round-to-nearest-even.
 *
 * Conventions for every entry point:
 *   - All buffers are DEVICE memory allocated and owned by the caller.  The
 *     library never allocates, frees or synchronizes.  Between calls it
 *     keeps only host-side caches, guarded for use from several threads:
 *     TMA descriptors keyed by array address and shape, the SM count, a
 *     launch counter, and the device address of the fixed scratch of
 *     imp_nvfp4_quantize_noalloc (per device and context).  Results never
 *     depend on them.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream); all work
 *     is enqueued on it asynchronously.
 *   - The return value reports argument and launch errors only.  A call that
 *     returns anything but IMP_OK has enqueued nothing.
 *   - `dev_status` (device int32, may be NULL) receives data-dependent
 *     conditions found while the kernels run: the kernels OR IMP_DEV_* flags
 *     into it, so the caller zeroes it beforehand and reads it after the
 *     stream synchronizes.  Kernels never trap; every wait inside a kernel is
 *     bounded and sets IMP_DEV_TIMEOUT when it gives up.
 *   - Row-major layouts; all base pointers 16-byte aligned; leading
 *     dimensions (in elements) multiples of 8.
 */
#ifndef IMP_NVFP4_H
#define IMP_NVFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  IMP_OK = 0,
  IMP_ERR_INVALID_ARG = 1,         /* NULL pointer, negative size, rows/K mismatch */
  IMP_ERR_UNSUPPORTED_SHAPE = 2,   /* K not a positive multiple of 64 (16 for quantize) */
  IMP_ERR_MISALIGNED = 3,          /* pointer not 16-byte aligned or ld not a multiple of 8 */
  IMP_ERR_WORKSPACE_TOO_SMALL = 4, /* ws_bytes below the *_workspace_size() figure */
  IMP_ERR_CUDA = 5                 /* a kernel launch failed (cudaGetLastError) */
} imp_status;

/* Flags OR-ed into *dev_status by the kernels. */
enum {
  IMP_DEV_OK = 0,
  IMP_DEV_NONFINITE_INPUT = 1, /* a NaN or Inf in a tensor being quantized; outputs unspecified */
  IMP_DEV_TIMEOUT = 2,         /* a bounded in-kernel wait gave up; outputs unspecified */
  IMP_DEV_RANGE = 4            /* imp_mxfp4_to_nvfp4: a block's scale is too far below the
                                  largest to be exact in NVFP4; outputs unspecified */
};

/* An NVFP4 tensor of `rows` x `K` elements (device pointers, caller-owned):
 *   codes        uint8[rows][K/2]   packed E2M1 codes, low nibble = even element
 *   scales       uint8[rows][K/16]  E4M3 block scales, row-major
 *   tensor_scale float[1]           s = global amax / 2688                        */
typedef struct {
  uint8_t *codes;
  uint8_t *scales;
  float *tensor_scale;
  int64_t rows;
  int64_t K;
} imp_nvfp4_tensor;

/* Bytes of workspace imp_nvfp4_quantize needs for a rows x K tensor
 * (per-CTA partial maxima; no initialization required). */
size_t imp_nvfp4_quantize_workspace_size(int64_t rows, int64_t K);

/* Quantize a bf16 matrix to NVFP4 with the recipe above.
 *   x_bf16    device bf16[rows][ldx]; only the first K columns are read.
 *   rows, K   rows >= 0 (0 writes s = 0 and nothing else; codes and scales
 *             may then be NULL), K > 0, K % 16 == 0.
 *   ldx       row stride of x in elements, ldx >= K, ldx % 8 == 0.
 *   out       out->rows == rows, out->K == K; codes/scales/tensor_scale written.
 *   Bit-exact: codes, scale bytes and s equal the recipe's for every input
 *   without NaN/Inf.  A NaN or Inf sets IMP_DEV_NONFINITE_INPUT.            */
imp_status imp_nvfp4_quantize(const void *x_bf16, int64_t rows, int64_t K, int64_t ldx,
                              const imp_nvfp4_tensor *out, int32_t *dev_status,
                              void *workspace, size_t ws_bytes, void *stream);

/* Allocation-free quantizer (no counterpart in the source pages; an addition
 * of this library).  For callers that may not allocate device memory at the
 * point of the call -- a serving loop that forbids allocation after start-up,
 * code running inside a stream capture, a process whose device memory is one
 * fixed pool -- and so cannot provide imp_nvfp4_quantize's workspace.
 * Same arguments, results and errors as imp_nvfp4_quantize, minus the
 * workspace: the scratch (per-CTA partial maxima, 4 KB) lives in a fixed
 * device array inside the library, which every GPU that loads the library
 * keeps until the process exits.  Sizes whose scratch would exceed that
 * array return IMP_ERR_WORKSPACE_TOO_SMALL (with 4 KB no valid size does).
 *   - Allocates nothing and calls no allocating routine.
 *   - The first call in a device's context looks up the array's device
 *     address (with that device current) and caches it for that context (a
 *     device reset or a new context looks it up again); make that first call
 *     before any stream capture that is to contain later calls.
 *   - All calls share the one array: calls that can run at the same time on
 *     the GPU (different streams, concurrent graphs) race and corrupt each
 *     other's results.  The array needs no clearing: each call overwrites
 *     what it reads.                                                        */
imp_status imp_nvfp4_quantize_noalloc(const void *x_bf16, int64_t rows, int64_t K, int64_t ldx,
                                      const imp_nvfp4_tensor *out, int32_t *dev_status,
                                      void *stream);

/* Bytes of workspace imp_nvfp4_gemm (and imp_nvfp4_gemm_mma) needs for
 * Y[M][N] = X[M][K] W^T.  M <= 16: the FP4 decode path's split X, its
 * partial sums and counters when the shape takes that path
 * (K % 256 == 0, K >= 1024, N >= 128), else 0.  M > 16: the quantized X and
 * X's and W's atom-layout scales.  0 also for shapes no path accepts. */
size_t imp_nvfp4_gemm_workspace_size(int64_t M, int64_t N, int64_t K);

/* An addition of this library (host-side query; the pages have no
 * counterpart), used to count launches and name the weight-streaming kernel.
 * The plan imp_nvfp4_gemm follows for Y[M][N] = X[M][K] W^T on the current
 * device, given a workspace of imp_nvfp4_gemm_workspace_size bytes and
 * 16-byte aligned arrays: returns the number of kernels one call launches
 * (0 if the call rejects the shape) and stores in *kernel (when kernel is not
 * NULL) the static name of the kernel that streams W: "gemv_f4r_kernel" /
 * "gemv_f4_kernel" (FP4 tensor cores, X split per call, inside the kernel
 * or by a split kernel before it), "gemv_tc_kernel"
 * (f16 tensor cores), "gemv_kernel" (CUDA cores) or "gemm_mxf4_kernel"
 * (prefill).  Host only; launches nothing. */
int32_t imp_nvfp4_gemm_plan(int64_t M, int64_t N, int64_t K, const char **kernel);

/* Y = X * W^T.
 *   x_bf16   device bf16[M][ldx], ldx >= K, ldx % 8 == 0.
 *   M        M >= 0 (0 = nothing to do).  M <= 16 takes the decode path,
 *            M > 16 the prefill path (X quantized on device, block-scaled FP4
 *            tensor-core MMA).
 *   K        K > 0, K % 64 == 0, and w->K == K.
 *   w        NVFP4 weight with w->rows = N >= 0 rows (0 = nothing to do).
 *   y_bf16   device bf16[M][ldy], ldy >= N, ldy % 8 == 0; fully overwritten.
 *   workspace  imp_nvfp4_gemm_workspace_size(M, N, K) bytes, 16-byte aligned
 *            (else IMP_ERR_WORKSPACE_TOO_SMALL / IMP_ERR_MISALIGNED); owned by
 *            the caller, needs no clearing (each launch leaves its per-tile
 *            counters at zero, so a captured call replays correctly; only
 *            after a call that reported IMP_DEV_TIMEOUT should it be zeroed
 *            before that call is replayed); calls that may run at the same
 *            time on the GPU need separate workspaces.
 *   Decode shapes: every K up to 61440; beyond that the FP4 path takes
 *   K % 256 == 0 with N >= 128 (other long-K shapes return
 *   IMP_ERR_UNSUPPORTED_SHAPE).  imp_nvfp4_gemm_plan tells which kernel a
 *   shape takes.
 *   Decode (M <= 16) kernels are launched with programmatic dependent launch:
 *   when the previous kernel on the stream allows it (this library's decode
 *   kernels do), the call may start streaming W before that kernel finishes;
 *   X is read only after it completes.  So W must not be written by a kernel
 *   that itself allows early launch (the quantizers here do not).
 *   Accuracy: |y - y_exact| <= 2e-3 * sum_k |x_k w_k| + 1e-5 + 2^-8 |y_exact|
 *   per element, with y_exact the exact product of the operands defined
 *   above; the last term is the rounding of the result to bf16.  Results are
 *   bitwise reproducible from run to run (fixed reduction order).           */
imp_status imp_nvfp4_gemm(const void *x_bf16, int64_t M, int64_t K, int64_t ldx,
                          const imp_nvfp4_tensor *w, void *y_bf16, int64_t ldy,
                          int32_t *dev_status, void *workspace, size_t ws_bytes, void *stream);

/* ---- tensor-core operand layout ("MMA layout") -----------------------------
 * A one-time transform of a weight for the tensor-core kernels; values are
 * unchanged.  It follows "How imp turns a model file into words", part one
 * ("loading the model (happens once)"): the engine converts every weight
 * once at load so that the per-token steps read it in the form its kernels
 * want.  The layout itself is this library's (what the sm_103a tensor-core
 * copies read); the pages do not give one.
 *   Scales: 512-byte atoms, one per 128 rows x 4 blocks (64 elements of K);
 *     row r of the atom at byte 16*(r % 32) + 4*((r / 32) % 4), block j of it
 *     at + j.  Atoms of a 128-row block follow each other along K; row blocks
 *     follow each other.
 *   Codes: 16 KB tiles of 128 rows x 256 elements (128 bytes per row), each
 *     stored as a 128-byte-swizzled operand tile (row rr at rr * 128, its
 *     16-byte unit u at unit u ^ (rr % 8)); tiles run along K (K padded to a
 *     multiple of 256), then down the rows.
 *   Rows are padded to a multiple of 256; padding is zero.
 * An imp_nvfp4_tensor "in MMA layout" has codes and scales in these layouts
 * (rows and K are the logical sizes; the tensor scale is unchanged).       */

/* Bytes of MMA-layout scales / codes for a rows x K tensor (K % 64 == 0). */
size_t imp_nvfp4_mma_scales_size(int64_t rows, int64_t K);
size_t imp_nvfp4_mma_codes_size(int64_t rows, int64_t K);

/* Copy tensor `t` (row-major) into the MMA layout.
 *   t           NVFP4 tensor, rows >= 1, K % 64 == 0.
 *   mma_codes   device buffer of >= imp_nvfp4_mma_codes_size(rows, K) bytes;
 *   mma_scales  device buffer of >= imp_nvfp4_mma_scales_size(rows, K) bytes;
 *               both 16-byte aligned, padding written as 0.  Either may be
 *               NULL (with 0 bytes) to skip that part.                     */
imp_status imp_nvfp4_prepare_mma(const imp_nvfp4_tensor *t, void *mma_codes, size_t codes_bytes,
                                 void *mma_scales, size_t scales_bytes, void *stream);

/* An addition of this library: the prefill path's on-device activation
 * quantizer (the imp README, "How it works": prefill is compute-bound and
 * runs on the 4-bit tensor cores) exposed on its own.
 * Quantize like imp_nvfp4_quantize (bit-identical codes, scale bytes and
 * tensor scale) but write the scales in the MMA (atom) layout, for the X
 * operand of imp_nvfp4_gemm_fp4: out->scales must hold
 * imp_nvfp4_mma_scales_size(rows, K) bytes; codes stay row-major [rows][K/2].
 * K % 64 == 0.                                                             */
imp_status imp_nvfp4_quantize_mma(const void *x_bf16, int64_t rows, int64_t K, int64_t ldx,
                                  const imp_nvfp4_tensor *out, int32_t *dev_status,
                                  void *workspace, size_t ws_bytes, void *stream);

/* An addition of this library, with imp_nvfp4_gemm_fp4 below.
 * Bytes of the optional workspace of imp_nvfp4_gemm_fp4 (on the current
 * device): per-tile counters and one partial 128 x 256 fp32 tile per CTA
 * and split segment (~39 MB on a 152-SM GPU).  0 for invalid sizes.       */
size_t imp_nvfp4_gemm_fp4_workspace_size(int64_t M, int64_t N, int64_t K);

/* An addition of this library: the prefill GEMM step (the imp README
 * feature matrix, "NVFP4 block-scaled ... GEMM/GEMV"; "How it works":
 * prefill is compute-bound) callable without the activation quantizer.
 * Y = Xq * Wq^T, both operands NVFP4: the block-scaled FP4 tensor-core GEMM
 * alone (tcgen05.mma kind::mxf4nvf4, fp32 accumulation in tensor memory),
 * times s_x * s_w, rounded to bf16.
 *   xq  from imp_nvfp4_quantize_mma: M rows (M >= 1), row-major codes,
 *       atom-layout scales, K % 64 == 0;
 *   wq  N rows in MMA layout, wq->K == K;
 *   y   bf16[M][ldy], ldy >= N, ldy % 8 == 0.
 *   workspace  NULL, or imp_nvfp4_gemm_fp4_workspace_size(M, N, K) bytes,
 *       16-byte aligned (else IMP_ERR_WORKSPACE_TOO_SMALL / MISALIGNED),
 *       needing no clearing.  With it the (tile, K step) work is spread
 *       evenly over the SMs (stream-K: tiles split between CTAs are summed
 *       from fp32 partials in K order, so results stay bitwise repeatable);
 *       without it each CTA computes whole 128 x 256 tiles.  The two
 *       schedules round differently (both within the accuracy of
 *       imp_nvfp4_gemm).                                                   */
imp_status imp_nvfp4_gemm_fp4(const imp_nvfp4_tensor *xq, const imp_nvfp4_tensor *wq,
                              void *y_bf16, int64_t ldy, int32_t *dev_status, void *workspace,
                              size_t ws_bytes, void *stream);

/* Y = X * W^T like imp_nvfp4_gemm, with W in MMA layout (the serving form:
 * weights prepared once at load -- "How imp turns a model file into words",
 * part one -- and read as contiguous 16 KB tiles).  An addition of this
 * library in place of an imp_nvfp4_gemm that would look for prepared scales
 * beside the row-major tensor: the caller chooses the form explicitly.  M <= 16 takes the
 * decode path (FP4 tensor cores, X split per call), which needs
 * K % 256 == 0, K >= 1024, N >= 128 (else IMP_ERR_UNSUPPORTED_SHAPE);
 * M > 16 the prefill path.  Workspace: imp_nvfp4_gemm_workspace_size(M, N,
 * K) bytes, 16-byte aligned.  Other arguments and the accuracy are those of
 * imp_nvfp4_gemm.                                                          */
imp_status imp_nvfp4_gemm_mma(const void *x_bf16, int64_t M, int64_t K, int64_t ldx,
                              const imp_nvfp4_tensor *w_mma, void *y_bf16, int64_t ldy,
                              int32_t *dev_status, void *workspace, size_t ws_bytes, void *stream);

/* ---- grouped decode GEMV ---------------------------------------------------
 * One X times several weights of the same K in one call -- a layer's q, k
 * and v projections, or its gate and up projections -- the same products as
 * concatenating the weights along N, except that each weight keeps its own
 * tensor scale and output.  It serves the engine's per-token launch sequence,
 * which is recorded once and replayed ("How imp turns a model file into
 * words", part one; the imp README, "How it works": CUDA graphs replay the
 * decode launches): fewer, larger launches make that sequence shorter.  The
 * grouping is an addition of this library.                                */
#define IMP_NVFP4_MAX_GROUPS 4
typedef struct {
  imp_nvfp4_tensor w;  /* weight g in MMA layout: w.rows = N_g >= 1, w.K == K */
  void *y_bf16;        /* device bf16[M][ldy]: Y_g = X * W_g^T, fully overwritten */
  int64_t ldy;         /* >= N_g, multiple of 8 */
} imp_nvfp4_group;

/* Bytes of workspace imp_nvfp4_gemm_grouped needs (N: the n_groups row
 * counts; 0 for invalid arguments). */
size_t imp_nvfp4_gemm_grouped_workspace_size(int64_t M, int64_t K, const int64_t *N,
                                             int32_t n_groups);

/* Like imp_nvfp4_gemm_plan for a grouped call: kernels launched in total
 * (0: rejected) and, in *kernel, the name of the first weight-streaming
 * kernel.  Host only.                                                      */
int32_t imp_nvfp4_gemm_grouped_plan(int64_t M, int64_t K, const int64_t *N, int32_t n_groups,
                                    const char **kernel);

/* Y_g = X * W_g^T for g < n_groups (1 <= n_groups <= IMP_NVFP4_MAX_GROUPS).
 *   x_bf16, M, K, ldx   as for imp_nvfp4_gemm_mma (M = 0: nothing to do).
 *   1 <= M <= 2, K % 256 == 0 and K >= 1024 (the decode case): one
 *   weight-streaming kernel for all groups, scheduled over the groups'
 *   128-row tiles together (after one split of X, or splitting X itself
 *   when a CTA holds at most six K chunks).  Other shapes (and a tile or K
 *   count that plan cannot hold) run imp_nvfp4_gemm_mma once per group, in
 *   order, on `stream`; a shape it rejects returns
 *   IMP_ERR_UNSUPPORTED_SHAPE before anything is enqueued.
 *   workspace  imp_nvfp4_gemm_grouped_workspace_size bytes, 16-byte aligned.
 *   Accuracy as for imp_nvfp4_gemm; results are bitwise reproducible from
 *   run to run, though the one-pass schedule may sum a tile's K chunks in
 *   another grouping than a call on that weight alone.                     */
imp_status imp_nvfp4_gemm_grouped(const void *x_bf16, int64_t M, int64_t K, int64_t ldx,
                                  const imp_nvfp4_group *groups, int32_t n_groups,
                                  int32_t *dev_status, void *workspace, size_t ws_bytes,
                                  void *stream);

/* ---- decode chain ----------------------------------------------------------------
 * A decode step is a chain of GEMVs in which a call's X is often the
 * previous call's output (a layer's projections one after another, the last
 * layer feeding the LM head).  The engine records that per-token sequence
 * once and replays it ("How imp turns a model file into words", part one;
 * the imp README, "How it works": CUDA graphs replay the decode launches).
 * This call runs up to four such calls ("links") in ONE persistent launch:
 * one CTA per SM streams every link's weight through one pipeline, and only
 * a link whose X is the previous link's output waits for it (a per-link
 * count of finished CTAs in the workspace), so the weight stream does not
 * stop between calls.  One launch instead of a few per call: on launch-
 * bound layers (a 0.6B-class layer's 7 projections as 4 links: 38 us,
 * against 49 us as grouped calls and 35 us as those calls replayed from a
 * CUDA graph) it beats separate calls without a graph; on a 27B-class step
 * it runs within ~1 % of the separate calls (109.5 vs 108.5 us).
 * An addition of this library.                                            */
#define IMP_NVFP4_MAX_CHAIN 4
typedef struct {
  const imp_nvfp4_group *groups; /* 1..IMP_NVFP4_MAX_GROUPS weights of one K (MMA layout),
                                    each with its output, as for imp_nvfp4_gemm_grouped */
  int32_t n_groups;
  const void *x_bf16;            /* device bf16[M][ldx]; NULL: X is the previous link's
                                    groups[0] output (its K must equal that weight's rows) */
  int64_t ldx;                   /* ignored when x_bf16 is NULL */
  int32_t x_swiglu;              /* with x_bf16 NULL: 1 takes X = bf16(silu(g) * u), g and u
                                    the previous link's groups[0] and groups[1] outputs (the
                                    activation of imp_nvfp4_gemm_mma_swiglu); 0 takes g */
} imp_nvfp4_chain_link;

/* Bytes of workspace imp_nvfp4_gemm_chain needs (on the current device;
 * 0 for invalid arguments). */
size_t imp_nvfp4_gemm_chain_workspace_size(int64_t M, const imp_nvfp4_chain_link *links,
                                           int32_t n_links);

/* 1 if imp_nvfp4_gemm_chain runs these links as one persistent launch, 0 if
 * it runs them one grouped call after another (or rejects them).  Host only. */
int32_t imp_nvfp4_gemm_chain_plan(int64_t M, const imp_nvfp4_chain_link *links, int32_t n_links);

/* For each link c in order (1 <= n_links <= IMP_NVFP4_MAX_CHAIN):
 * Y_cg = X_c * W_cg^T for its groups g, with X_c = links[c].x_bf16 or, if
 * that is NULL (c >= 1), the output of links[c-1].groups[0] -- or, with
 * x_swiglu, bf16(silu(that output) * the output of links[c-1].groups[1])
 * (a layer's down projection after its grouped gate and up).
 *   M             M >= 0 (M = 0: nothing to do).
 *   links         host array; weights, outputs and strides as for
 *                 imp_nvfp4_gemm_grouped.  No output may overlap another
 *                 link's output or any link's X (except the NULL form),
 *                 else IMP_ERR_INVALID_ARG: links run concurrently on
 *                 different SMs.
 *   workspace     imp_nvfp4_gemm_chain_workspace_size bytes, 16-byte
 *                 aligned, needing no clearing (the launch's first CTA
 *                 clears its counters and publishes the launch; graph
 *                 replay is fine).  Launches that can run at the same time
 *                 must not share it.
 * 1 <= M <= 2, every K % 256 == 0 and K >= 1024, and a schedule that fits
 * (at most 24 K chunks of 256 per CTA and link): one launch of one CTA per
 * SM, all of which must be resident at once (its CTAs wait for each other):
 * it needs the GPU to itself while it runs -- with another kernel holding
 * SMs for more than a second a wait gives up and sets IMP_DEV_TIMEOUT.
 * Otherwise each link runs as imp_nvfp4_gemm_grouped, in order, on
 * `stream`.  Accuracy as for imp_nvfp4_gemm; results are
 * bitwise reproducible from run to run (each CTA splits its own chunks of X
 * with its own power-of-two prescale, so the roundings can differ from a
 * grouped call's).                                                          */
imp_status imp_nvfp4_gemm_chain(int64_t M, const imp_nvfp4_chain_link *links, int32_t n_links,
                                int32_t *dev_status, void *workspace, size_t ws_bytes,
                                void *stream);

/* ---- fused prefill MLP pieces -------------------------------------------------
 * A layer's MLP ("1. The big picture": the MLP transforms each token's vector
 * on its own) in the Qwen-class models the pages run is gate and up
 * projections, h = silu(gate) * up, then the down projection.  These two
 * calls fuse the activation into the gate/up GEMM's epilogue and fold the
 * global amax of h into it, so the down projection's activation quantizer
 * reads h once instead of twice.  Additions of this library.            */

/* Workspace of imp_nvfp4_gemm_swiglu (X's quantization), 0 if rejected. */
size_t imp_nvfp4_gemm_swiglu_workspace_size(int64_t M, int64_t N, int64_t K);

/* h = silu(X Wg^T) * (X Wu^T) for prefill (M > 16): X quantized on device as
 * in imp_nvfp4_gemm, both products on the block-scaled FP4 tensor cores in
 * one kernel (each 256-row W tile = 128 rows of Wg + the same 128 rows of
 * Wu), silu(v) = v / (1 + e^-v) and the product in fp32, h rounded to bf16.
 *   w_gate, w_up  MMA layout (imp_nvfp4_prepare_mma), same N and K.
 *   h_bf16        device bf16[M][ldh], ldh >= N, ldh % 8 == 0.
 *   h_amax        device uint32, 4-byte aligned: receives the largest |h| as
 *                 bf16 magnitude bits (zeroed by this call), for
 *                 imp_nvfp4_quantize_mma_amax.  A non-finite h sets
 *                 IMP_DEV_NONFINITE_INPUT.
 *   M <= 16 returns IMP_ERR_UNSUPPORTED_SHAPE.  Accuracy: g and u within
 *   the fp32 accumulation of exact products, then the two roundings above. */
imp_status imp_nvfp4_gemm_swiglu(const void *x_bf16, int64_t M, int64_t K, int64_t ldx,
                                 const imp_nvfp4_tensor *w_gate, const imp_nvfp4_tensor *w_up,
                                 void *h_bf16, int64_t ldh, uint32_t *h_amax,
                                 int32_t *dev_status, void *workspace, size_t ws_bytes,
                                 void *stream);

/* The decode counterpart (M <= 16): the down projection of an MLP whose
 * input is the activation of its gate and up outputs,
 *   Y = h * W^T,   h = bf16(silu(gate) * up)   (silu(v) = v / (1 + e^-v),
 * evaluated in fp32 as imp_nvfp4_gemm_swiglu does), with h formed where the
 * decode path's split of X reads it (no separate activation kernel, h is
 * not written).  gate_bf16 and up_bf16: device bf16[M][ld], ld >= K,
 * ld % 8 == 0, 16-byte aligned (the outputs of the layer's gate and up
 * projections, e.g. one imp_nvfp4_gemm_grouped call).  w in MMA layout.
 * The shape must take the FP4 decode path (K % 256 == 0, K >= 1024,
 * N >= 128, M <= 16), else IMP_ERR_UNSUPPORTED_SHAPE.  Workspace as for
 * imp_nvfp4_gemm_mma.  Accuracy: that of imp_nvfp4_gemm on h.  An addition
 * of this library.                                                          */
imp_status imp_nvfp4_gemm_mma_swiglu(const void *gate_bf16, const void *up_bf16, int64_t M,
                                     int64_t K, int64_t ld, const imp_nvfp4_tensor *w_mma,
                                     void *y_bf16, int64_t ldy, int32_t *dev_status,
                                     void *workspace, size_t ws_bytes, void *stream);
/* Kernel launches of imp_nvfp4_gemm_mma_swiglu (0: rejected) and, in
 * *kernel, the weight-streaming kernel.  Host only. */
int32_t imp_nvfp4_gemm_mma_swiglu_plan(int64_t M, int64_t N, int64_t K, const char **kernel);

/* imp_nvfp4_quantize_mma with the global amax already known (bf16 magnitude
 * bits of max|x| in device memory, as imp_nvfp4_gemm_swiglu writes it): the
 * encode pass alone, one read of X.  Bit-identical to imp_nvfp4_quantize_mma
 * when *amax is the true max|x|.  rows >= 1, K % 64 == 0.  dev_status is not
 * written: non-finite values are reported by whoever folded the amax
 * (imp_nvfp4_gemm_swiglu does); a non-finite *amax gives a zero tensor
 * scale and all-zero codes.                                                */
imp_status imp_nvfp4_quantize_mma_amax(const void *x_bf16, int64_t rows, int64_t K, int64_t ldx,
                                       const uint32_t *amax, const imp_nvfp4_tensor *out,
                                       int32_t *dev_status, void *stream);

/* ---- other weight formats ---------------------------------------------------
 * The imp README's feature matrix lists, besides NVFP4 (the primary path),
 * MXFP4 and FP8 E4M3 weights.                                              */

/* MXFP4 tensor (OCP Microscaling Formats v1.0): rows x K elements, K % 32 == 0.
 *   codes   uint8[rows][K/2]   packed E2M1 codes, low nibble = even element
 *   scales  uint8[rows][K/32]  E8M0 block scales: byte b stands for 2^(b - 127) */
typedef struct {
  uint8_t *codes;
  uint8_t *scales;
  int64_t rows;
  int64_t K;
} imp_mxfp4_tensor;

/* Quantize a bf16 matrix to MXFP4 as the MX specification converts: per
 * 32-element block, shared exponent e = floor(log2(block amax)) - 2 clamped
 * to [-127, 127] (an all-zero block takes -127), scale byte e + 127, codes
 * E2M1(x / 2^e) rounded to nearest even and saturating at 6, sign copied
 * from x.  Bit-exact.  rows >= 1, K % 32 == 0, ldx >= K, ldx % 8 == 0; no
 * workspace.  NaN/Inf sets IMP_DEV_NONFINITE_INPUT.                        */
imp_status imp_mxfp4_quantize(const void *x_bf16, int64_t rows, int64_t K, int64_t ldx,
                              const imp_mxfp4_tensor *out, int32_t *dev_status, void *stream);

/* Bytes of workspace imp_mxfp4_to_nvfp4 needs (one scratch word). */
size_t imp_mxfp4_to_nvfp4_workspace_size(void);

/* The same values in NVFP4 form, for the NVFP4 kernels (an addition of this
 * library: MXFP4 weights are served by converting them once at load, like
 * imp_nvfp4_prepare_mma).  Exact: each 16-element half of a block keeps the
 * codes and gets the E4M3 scale 2^(e - t), with the fp32 tensor scale 2^t,
 * t = (the largest e among halves with a nonzero code) - 8; halves whose
 * codes are all zero get scale 0.  Exact whenever every such e is at least
 * t - 9, i.e. no nonzero half sits more than 2^17 below the largest; one
 * that does sets IMP_DEV_RANGE.
 *   in    MXFP4 tensor, rows >= 1, K % 64 == 0.
 *   out   NVFP4 tensor of the same rows and K (row-major layout); out->codes
 *         may equal in->codes (then the codes are not copied).           */
imp_status imp_mxfp4_to_nvfp4(const imp_mxfp4_tensor *in, const imp_nvfp4_tensor *out,
                              int32_t *dev_status, void *workspace, size_t ws_bytes,
                              void *stream);

/* FP8 E4M3 weight tensor: codes uint8[rows][K] (OCP FP8 E4M3 "fn"), one fp32
 * tensor scale s8; element value = e4m3(code) * s8.                        */
typedef struct {
  uint8_t *codes;
  float *tensor_scale;
  int64_t rows;
  int64_t K;
} imp_fp8_tensor;

/* Workspace of imp_fp8_quantize (per-CTA partial maxima). */
size_t imp_fp8_quantize_workspace_size(int64_t rows, int64_t K);

/* Quantize a bf16 matrix to FP8 E4M3 with one tensor scale: s8 = global
 * amax / 448 (fp32 division), code = E4M3(x / s8) rounded to nearest even,
 * saturating at 448, sign copied from x; s8 = 0 gives all codes 0.
 * Bit-exact.  rows >= 1, K % 16 == 0, ldx >= K, ldx % 8 == 0.             */
imp_status imp_fp8_quantize(const void *x_bf16, int64_t rows, int64_t K, int64_t ldx,
                            const imp_fp8_tensor *out, int32_t *dev_status, void *workspace,
                            size_t ws_bytes, void *stream);

/* Workspace of imp_fp8_gemm (0 for shapes it rejects). */
size_t imp_fp8_gemm_workspace_size(int64_t M, int64_t N, int64_t K);

/* Kernels one imp_fp8_gemm call launches (0: rejected) and the name of the
 * weight-streaming kernel.  Host only. */
int32_t imp_fp8_gemm_plan(int64_t M, int64_t N, int64_t K, const char **kernel);

/* Decode GEMV / skinny GEMM on FP8 weights: Y = X * W^T with
 * w[n][k] = e4m3(code) * s8, X bf16, fp32 accumulation, bf16 Y.
 *   1 <= M <= 16 (M = 0: nothing to do); K % 128 == 0, K >= 512; N >= 128.
 *   The weight is fed to the FP8 tensor cores (tcgen05.mma kind::f8f6f4)
 *   unchanged; X is split per call into eight E4M3 components (exact
 *   products, fp32 sums), in passes of two rows of X.
 *   Accuracy and the other conventions as for imp_nvfp4_gemm.             */
imp_status imp_fp8_gemm(const void *x_bf16, int64_t M, int64_t K, int64_t ldx,
                        const imp_fp8_tensor *w, void *y_bf16, int64_t ldy, int32_t *dev_status,
                        void *workspace, size_t ws_bytes, void *stream);

/* Human-readable name of a status code (static storage). */
const char *imp_status_string(imp_status status);

/* Self-test of the in-kernel failure detection: launches one kernel whose
 * single bounded wait (on an mbarrier that nothing arrives at) gives up after
 * the library's wait limit (1 s), ORs IMP_DEV_TIMEOUT into *dev_status and
 * returns -- the same wait every kernel of this library uses on its
 * pipelines.  No fault, trap or hang: the context stays usable.
 *   dev_status  device int32, 4-byte aligned (else IMP_ERR_INVALID_ARG). */
imp_status imp_selftest_bounded_wait(int32_t *dev_status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* IMP_NVFP4_H */
