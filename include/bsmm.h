/*
 * bsmm.h -- block-scaled low-precision matrix multiply for GB300 (sm_103a).
 *
 * C ABI of libbsmm.so.  Plain pointers and sizes only; no C++ or framework
 * types cross this boundary and no exception leaves it.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every data pointer is a DEVICE pointer owned by the caller.  The library
 *    never allocates, frees or keeps device memory of its own, apart from
 *    static device arrays in the loaded module: a 4-byte status word, and the
 *    scratch of bsmm_gemm_noalloc.  Scratch memory a call needs is passed in
 *    as `workspace`; its size comes from the matching *_workspace_size()
 *    query (0 means no workspace is needed).  A workspace holds one call's
 *    scratch until the call's kernels finish: calls that may run at the
 *    same time on the GPU (different streams) need workspaces of their own.
 *  - Every call is asynchronous with respect to the host: it validates its
 *    arguments, enqueues kernels on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream) and returns.  Results are ready when the stream
 *    reaches that point.  Calls are safe to issue from several host threads.
 *  - Every call returns a bsmm_status.  On failure nothing has been enqueued
 *    (argument errors) or the CUDA error is reported (BSMM_ERR_CUDA);
 *    bsmm_last_error() then returns a message for the calling thread.
 *  - Matrices are row-major.  Strides are in elements.  A GEMM operand's
 *    contraction axis K is its innermost (contiguous) axis.  E2M1 codes are
 *    packed two per byte along the contiguous axis, even element in the low
 *    nibble, so a row of K E2M1 codes is K/2 bytes.
 *  - Device pointers given to the GEMMs must be 16-byte aligned.
 *  - A zero-sized problem (M == 0, or B == 0) is BSMM_OK and launches nothing.
 *  - Kernels never spin without bound: every wait inside a kernel gives up
 *    after a limit (bsmm_set_wait_timeout_ns), records the failure in the
 *    device status word and returns.  bsmm_check_device_status() reports it.
 *
 * Sources (the four pages this library implements):
 *  [JAX]  jax.nn.scaled_matmul documentation ("Mathematically" definition,
 *         Parameters, Notes on the cuDNN/Blackwell formats, Examples).
 *  [TT]   TensorTonic, "Int8 Matmul with Per-Channel Scales" (problem
 *         statement, Requirements, Constraints, Examples).
 *  [AB]   atrex-bench operator #002 "block_scaled_mm" (Reference
 *         Implementation, Shapes table, Input Generation).
 *  [NKI]  AWS Neuron NKI "Matmul MXFP8 Backward Kernel API Reference"
 *         (introduction, Parameters, Returns).
 */
#ifndef BSMM_H_
#define BSMM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so this header needs no CUDA
 * headers. */
typedef struct CUstream_st* bsmm_stream_t;

typedef enum bsmm_status {
  BSMM_OK = 0,
  BSMM_ERR_INVALID_ARG = 1,  /* null pointer, bad enum, negative size        */
  BSMM_ERR_SHAPE = 2,        /* sizes inconsistent with each other           */
  BSMM_ERR_ALIGNMENT = 3,    /* pointer or row pitch not 16-byte aligned     */
  BSMM_ERR_UNSUPPORTED = 4,  /* valid request this build has no kernel for   */
  BSMM_ERR_CUDA = 5,         /* a CUDA runtime/driver call failed            */
  BSMM_ERR_TIMEOUT = 6,      /* a bounded in-kernel wait gave up             */
  BSMM_ERR_WORKSPACE = 7     /* workspace missing or smaller than required   */
} bsmm_status;

typedef enum bsmm_dtype {
  BSMM_F32 = 0,   /* binary32                                               */
  BSMM_BF16 = 1,  /* bfloat16                                               */
  BSMM_E4M3 = 2,  /* float8_e4m3fn: bias 7, no Inf, max 448                 */
  BSMM_E5M2 = 3,  /* float8_e5m2:   bias 15, IEEE-like, max 57344           */
  BSMM_E2M1 = 4,  /* float4_e2m1fn: max 6, packed two per byte              */
  BSMM_INT8 = 5   /* signed 8-bit integer codes in [-127, 127]              */
} bsmm_dtype;

typedef enum bsmm_scale_type {
  BSMM_SCALE_F32 = 0,    /* one binary32 per block                           */
  BSMM_SCALE_UE8M0 = 1,  /* one byte per block: 2^(byte-127); 0xFF is NaN   */
  BSMM_SCALE_UE4M3 = 2   /* one byte per block: unsigned E4M3 value          */
} bsmm_scale_type;

/* ------------------------------------------------------------------------ */
/* Library state                                                            */
/* ------------------------------------------------------------------------ */

/* Version as MAJOR*10000 + MINOR*100 + PATCH. */
int bsmm_version(void);

/* Message describing the most recent failure on the calling host thread
 * ("" if none).  The pointer stays valid until the thread's next call. */
const char* bsmm_last_error(void);

/* Limit, in nanoseconds, of every bounded wait inside the library's kernels
 * (default 1e9 = one second).  Applies to launches enqueued afterwards. */
void bsmm_set_wait_timeout_ns(uint64_t ns);

/* Synchronizes `stream`, then reads and clears the device status word of
 * the current device.  Returns BSMM_ERR_TIMEOUT if any kernel gave up a wait
 * since the last check (the kernel's outputs are then undefined, the CUDA
 * context stays usable), BSMM_ERR_CUDA if the stream reported an error, else
 * BSMM_OK.  `*where` (if not NULL) receives the recorded wait-site code. */
bsmm_status bsmm_check_device_status(bsmm_stream_t stream, int* where);

/* Diagnostic with no counterpart on the pages: launches one CTA that waits
 * on an mbarrier nothing ever arrives on, with a limit of `timeout_ns`.  The
 * wait gives up, the kernel records BSMM_ERR_TIMEOUT in the status word and
 * returns.  Used to test the timeout path without faulting a GPU. */
bsmm_status bsmm_selftest_wait_timeout(uint64_t timeout_ns, bsmm_stream_t stream);

/* Diagnostic with no counterpart on the pages.  Every quantizer computes its
 * binary32 quotient x / scale through one correctly rounded reciprocal per
 * block and two exact-remainder correction steps (Markstein's method) instead
 * of a division per element.  This checks that form against the hardware's
 * IEEE division on `pairs` pseudo-random (x, s) pairs generated from `seed`
 * on the GPU (divisors in [2^-80, 2^126), quotients on and next to rounding
 * ties, tiny x), and adds the number of disagreements to the 64-bit counter at
 * the device address `mismatches`, which the caller zeroes.  Asynchronous on
 * `stream`; BSMM_ERR_INVALID_ARG if `mismatches` is NULL. */
bsmm_status bsmm_selftest_quotient(uint64_t pairs, uint64_t seed, uint64_t* mismatches, bsmm_stream_t stream);

/* Per-kernel timing, with no counterpart on the pages (measurement aid).
 * bsmm_trace_start() discards earlier records and turns recording on: from
 * then on every launch of this library's kernels, from any host thread,
 * records a CUDA event before and after itself on its own stream.
 * bsmm_trace_stop() turns recording off; records stay readable until the
 * next start.  bsmm_trace_count() is the number of launches recorded.
 * bsmm_trace_read(i, ...) waits for launch i to finish and gives the
 * kernel's name (a static string, or NULL pointers skipped), its start
 * relative to launch 0's start in milliseconds (0 when launch 0 ran on
 * another device), and its duration in milliseconds.  The events add a few
 * microseconds of host time to each launch and small gaps between kernels;
 * do not trace inside stream capture.  bsmm_trace_read returns
 * BSMM_ERR_INVALID_ARG for an index out of range and BSMM_ERR_CUDA when that
 * launch's events could not be recorded or read. */
bsmm_status bsmm_trace_start(void);
bsmm_status bsmm_trace_stop(void);
int bsmm_trace_count(void);
bsmm_status bsmm_trace_read(int i, const char** name, float* start_ms, float* ms);

/* ------------------------------------------------------------------------ */
/* Quantizer                                                                */
/* ------------------------------------------------------------------------ */

/* Absmax block quantizer.
 *
 * Defined by [AB] Input Generation (binary32 scale = max(absmax/448, 1e-10),
 * codes = E4M3(clamp(x/scale, +-448))) and [TT] problem statement (INT8:
 * scale = absmax/127, all-zero block -> 1, codes = clip(round(x/scale),
 * +-127)).  UE8M0 and UE4M3 scales have no rule on the pages; this library
 * uses: UE8M0 scale = 2^ceil(log2(absmax/qmax)) (exponent clamped to
 * [-127,127]; zero block -> 1), UE4M3 scale = E4M3(absmax/qmax) rounded to
 * nearest (zero block -> 1, a scale rounding to 0 -> 2^-9).  qmax is the
 * code format's largest value: E4M3 448, E5M2 57344, E2M1 6, INT8 127.
 * All arithmetic is binary32; each code comes from the correctly rounded
 * quotient x/scale, as IEEE division gives it (not x*(1/scale) rounded
 * twice; see bsmm_selftest_quotient for how it is computed); rounding is to
 * nearest, ties to even; floating codes saturate.
 * Inputs are taken to be finite: the pages give no rule for NaN or
 * infinity, the library does not look for them, and a block holding one gets
 * unspecified codes and scale.
 *
 *   x        [rows, cols] input, element (r, c) at x[r*ld_x + c]; F32 or BF16.
 *   block_rows x block_cols
 *            block shape.  Supported: 1 x {16,32,64,128}, 1 x cols (one scale
 *            per row), {16,32,64,128} x 1, rows x 1 (one scale per column),
 *            128 x 128.  rows % block_rows == 0 and cols % block_cols == 0.
 *   code_type  E4M3, E5M2, E2M1 or INT8.   scale_type  F32, UE8M0 or UE4M3
 *            (INT8 codes need F32 scales).
 *   transpose_out
 *            0: codes [rows, cols] at codes[r*ld_codes + c] (E2M1: byte
 *               (r*ld_codes + c)/2 holds element c and c+1 of row r; ld_codes
 *               counts elements and must be even), scales
 *               [rows/block_rows, cols/block_cols] row-major, pitch
 *               ld_scales elements.
 *            1: (only for column blocks) codes stored transposed,
 *               [cols, rows] at codes[c*ld_codes + r], scales transposed
 *               [cols/block_cols, rows/block_rows] with pitch ld_scales.
 *   codes    output, 1 byte per code (E2M1: half a byte).
 *   scales   output, 4 bytes (F32) or 1 byte per scale.
 *
 * Errors: BSMM_ERR_INVALID_ARG (null pointer, bad enum), BSMM_ERR_SHAPE
 * (indivisible shape, pitch too small), BSMM_ERR_UNSUPPORTED (other block
 * shapes, transposed row blocks, INT8 with a non-F32 scale). */
bsmm_status bsmm_quantize(const void* x, bsmm_dtype x_type, int64_t rows, int64_t cols,
                          int64_t ld_x, int block_rows, int block_cols, bsmm_dtype code_type,
                          bsmm_scale_type scale_type, int transpose_out, void* codes,
                          int64_t ld_codes, void* scales, int64_t ld_scales,
                          bsmm_stream_t stream);

/* Several independent quantizations in one call: the same results as
 * bsmm_quantize on each job in turn.  block_scaled_mm quantizes a weight
 * matrix per problem in 128 x 128 tiles; a single such matrix of 2048 x 2048
 * is too small to keep the GPU busy, so the 128 x 128 jobs that would run
 * on the tile quantizer share launches (up to 16 jobs a launch, per input
 * type and per divided / power-of-two scale), and every other job runs as
 * bsmm_quantize runs it.
 *
 *   jobs     count job descriptions (host memory, read during the call);
 *            each field means what the bsmm_quantize argument of that name
 *            means.  No job's codes or scales may overlap another job's
 *            input or output: the order of the jobs' launches is unspecified.
 *   count    0 is a no-op.
 *
 * Errors: every job is checked before anything is launched; the first bad
 * job's error is returned, its index leading the bsmm_last_error() message.
 * BSMM_ERR_INVALID_ARG also for count < 0 or a null jobs with count > 0. */
typedef struct bsmm_quantize_job {
  const void* x;
  bsmm_dtype x_type;
  int64_t rows, cols, ld_x;
  int block_rows, block_cols;
  bsmm_dtype code_type;
  bsmm_scale_type scale_type;
  int transpose_out;
  void* codes;
  int64_t ld_codes;
  void* scales;
  int64_t ld_scales;
} bsmm_quantize_job;

bsmm_status bsmm_quantize_batch(const bsmm_quantize_job* jobs, int count, bsmm_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Batched block-scaled GEMM                                                */
/* ------------------------------------------------------------------------ */

/* y[b,m,n] = sum_k (a[b,m,k] * a_scales[b,m,k/bs_a]) * (w[b,n,k] * b_scales[b,n,k/bs_b])
 * with bs_a = K/K_a and bs_b = K/K_b inferred from the scale counts, FP32
 * accumulation ([JAX] "Mathematically" definition and Parameters).
 *
 * Codes: a_type, b_type both in {E4M3, E5M2} (they may differ) or both
 * E2M1; scales UE8M0 or UE4M3; any block sizes bs_a, bs_b.  The tensor cores
 * take ([JAX] Notes, cuDNN on Blackwell):
 *   MXFP8: FP8 codes, UE8M0 scales, blocks that are multiples of 32.
 *   NVFP4: E2M1 codes, UE4M3 scales, blocks that are multiples of 16.
 *   MXFP4: E2M1 codes, UE8M0 scales, blocks that are multiples of 32 (this
 *          kernel needs N * sizeof(y element) % 16 == 0).
 * (a block of several hardware blocks repeats its scale; K must be a
 * multiple of 32).  Every other combination -- e.g. the jax cuDNN example's
 * UE8M0 scales per 16 FP8 elements, or FP8 codes with UE4M3 scales -- runs
 * on a CUDA-core kernel (decode, scale, FP32 FMA; no workspace needed).
 * Other code or scale types return BSMM_ERR_UNSUPPORTED.
 *
 *   a        [B, M, K] codes, contiguous (E2M1: K/2 bytes per row).
 *   b        [B, N, K] codes, contiguous.
 *   a_scales [B, M, K_a] scale bytes, contiguous.  b_scales [B, N, K_b].
 *   y        [B, M, N] output, F32 or BF16 (round to nearest even),
 *            contiguous.
 *   workspace  device scratch of at least bsmm_gemm_workspace_size() bytes
 *            (holds the scales in the tensor-core scale-factor layout).
 *   Pointers 16-byte aligned; E2M1 needs an even K.
 */
size_t bsmm_gemm_workspace_size(int64_t B, int64_t M, int64_t N, int64_t K, bsmm_dtype a_type);

bsmm_status bsmm_gemm(int64_t B, int64_t M, int64_t N, int64_t K,
                      const void* a, bsmm_dtype a_type, const void* b, bsmm_dtype b_type,
                      const void* a_scales, int64_t K_a, const void* b_scales, int64_t K_b,
                      bsmm_scale_type scale_type, void* y, bsmm_dtype y_type,
                      void* workspace, size_t workspace_bytes, bsmm_stream_t stream);

/* No counterpart on the pages: bsmm_gemm for callers that cannot allocate.
 *
 * Some callers cannot call cudaMalloc at all: a plugin running inside a host
 * framework that owns every device allocation and exposes no allocator to
 * it, or a service that forbids device allocations after start-up so that
 * its memory footprint stays fixed.  They cannot provide bsmm_gemm's
 * workspace, so this variant keeps that scratch (the scales rearranged into
 * the tensor-core scale-factor layout) in a static device array inside the
 * library instead: BSMM_NOALLOC_SCRATCH_BYTES bytes, held by every GPU that
 * loads the library until the process exits.
 *
 * Arguments, formats and results are those of bsmm_gemm, without workspace.
 * The call allocates nothing (no cudaMalloc, no cudaFree, no allocating
 * library routine).  Its first call on a device looks up the array's device
 * address once (cudaGetSymbolAddress, with that device current); make that
 * first call before any stream capture.  Every call shares the one array and
 * rewrites all of it that it reads, so consecutive calls on one stream are
 * safe, but calls whose kernels overlap on the GPU (different streams, or
 * different host threads) race on it and give undefined results.
 *
 * Errors: those of bsmm_gemm, and BSMM_ERR_WORKSPACE when the problem needs
 * more than BSMM_NOALLOC_SCRATCH_BYTES of scratch, i.e. when
 * bsmm_gemm_workspace_size(B, M, N, K, a_type) exceeds it (e.g. an MXFP8
 * batch of 8 x 4096 x 4096 x 8192 needs 16 MiB and fits; E2M1 problems need
 * room for NVFP4's replicated B blocks: 8192^3 takes 32 MiB, 16384^3
 * 128 MiB and does not fit). */
#define BSMM_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

bsmm_status bsmm_gemm_noalloc(int64_t B, int64_t M, int64_t N, int64_t K,
                              const void* a, bsmm_dtype a_type, const void* b, bsmm_dtype b_type,
                              const void* a_scales, int64_t K_a, const void* b_scales, int64_t K_b,
                              bsmm_scale_type scale_type, void* y, bsmm_dtype y_type,
                              bsmm_stream_t stream);

/* ------------------------------------------------------------------------ */
/* GEMM with 1 x group_k activation and group_n x group_k weight FP32 scales */
/* ------------------------------------------------------------------------ */

/* y[m,n] = sum_kb a_scales[m,kb] * b_scales[n/group_n,kb] *
 *          sum_{k in block kb} a[m,k] * b[n,k]
 * with FP32 promotion of every K block's partial sum ([AB] Reference
 * Implementation; inputs as produced by [AB] Input Generation).
 *
 *   a        [M, K] E4M3 (or E5M2) codes, contiguous.
 *   b        [N, K] E4M3 (or E5M2) codes, contiguous.
 *   a_scales [M, K/group_k] binary32.   b_scales [N/group_n, K/group_k].
 *   y        [M, N] binary32 output, contiguous.
 *   group_n = group_k = 128 (the pages' only configuration); other values
 *   return BSMM_ERR_UNSUPPORTED.  N % group_n == 0 and K % group_k == 0
 *   (BSMM_ERR_SHAPE otherwise).  M is arbitrary.
 */
bsmm_status bsmm_gemm_grouped(int64_t M, int64_t N, int64_t K, const void* a, bsmm_dtype a_type,
                              const void* b, bsmm_dtype b_type, const float* a_scales,
                              const float* b_scales, int group_n, int group_k, float* y,
                              bsmm_stream_t stream);

/* ------------------------------------------------------------------------ */
/* INT8 per-channel symmetric matmul                                        */
/* ------------------------------------------------------------------------ */

/* [TT] problem statement and Requirements: s_x[b] = max_i |x[b,i]| / 127,
 * s_w[j] = max_i |w[i,j]| / 127 (all-zero row/column -> 1), codes
 * clip(round(v/s), -127, 127), a[b,j] = sum_i x_q[b,i]*w_q[i,j] accumulated
 * exactly in int32, y[b,j] = float32(a[b,j]) * s_x[b] * s_w[j].
 *
 *   x [B, D_in] binary32, w [D_in, D_out] binary32 (both contiguous).
 *   Outputs (contiguous): x_q int8 [B, D_in], x_scales [B], w_q int8
 *   [D_in, D_out] (the page's layout), w_scales [D_out], y [B, D_out].
 *   acc      optional int32 [B, D_out] output of the exact integer sums
 *            (NULL to skip).
 *   workspace  at least bsmm_int8_channel_workspace_size() bytes (holds
 *            K-padded, K-major copies of both operands' codes for the
 *            matmul, and the int32 partial sums of the tiles whose K range
 *            the matmul splits over otherwise idle SMs).
 *   Any D_in >= 1 (the matmul's copies are zero-padded to a multiple of
 *   128).  With B == 0 only w is quantized (w_q,
 *   w_scales); x, x_q, x_scales, y and acc are not touched, and the
 *   workspace needs D_out * 4 bytes (the query returns it).
 * The integer sums are exact for any codes: the matmul runs on the bf16
 * tensor cores (codes and their products are exact there) and adds FP32
 * partials of at most 1024 products, each an exact integer below 2^24, in
 * int32.  Where y or acc cannot be stored through TMA (D_out % 4 != 0, or a
 * base not 16-byte aligned) the warp-level integer MMA computes the sums.
 * On the tensor-core path w's quantization runs beside x's on a stream the
 * library keeps per device: it starts after the work already on `stream`
 * (an event recorded there) and `stream` waits for it before the matmul, so
 * the call stays ordered on `stream` as a whole (CUDA graph capture
 * included).
 */
size_t bsmm_int8_channel_workspace_size(int64_t B, int64_t D_in, int64_t D_out);

bsmm_status bsmm_int8_channel(const float* x, const float* w, int64_t B, int64_t D_in,
                              int64_t D_out, int8_t* x_q, float* x_scales, int8_t* w_q,
                              float* w_scales, float* y, int32_t* acc, void* workspace,
                              size_t workspace_bytes, bsmm_stream_t stream);

/* ------------------------------------------------------------------------ */
/* MXFP8 linear-layer backward                                              */
/* ------------------------------------------------------------------------ */

/* [NKI] introduction: forward Y = X W^T with X [M,K], W [N,K], Y [M,N];
 * backward dX = dY W ([M,K], contraction over N) and dW = dY^T X ([N,K],
 * contraction over M).  Every operand is MXFP8-quantized (UE8M0 scale per 32
 * elements, rule as in bsmm_quantize) along its own contraction axis: dY
 * and W along N for dX; dY and X along M for dW.  fp8_type is E5M2 (the
 * page's default) or E4M3.  Outputs are bfloat16 (round to nearest even).
 *
 *   dY [M, N], W [N, K], X [M, K] bfloat16, contiguous.
 *   dX [M, K], dW [N, K] bfloat16, contiguous.
 *   workspace  at least bsmm_linear_backward_workspace_size() bytes,
 *            256-byte aligned.  The call leaves the four quantized operands
 *            there, in this order, each part starting on a 256-byte boundary:
 *            the codes of dY along N [M, N], then their scales in the atom
 *            layout below (bsmm_scale_atoms_size(1, M, N, fp8_type, UE8M0)
 *            bytes); W^T along N [K, N] and its atoms; dY^T along M [N, M]
 *            and its atoms; X^T along M [K, M] and its atoms.
 *   M, N and K must be multiples of 32.
 */
size_t bsmm_linear_backward_workspace_size(int64_t M, int64_t N, int64_t K);

bsmm_status bsmm_linear_backward(const void* dY, const void* W, const void* X, int64_t M,
                                 int64_t N, int64_t K, bsmm_dtype fp8_type, void* dX, void* dW,
                                 void* workspace, size_t workspace_bytes, bsmm_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Scales in the tensor cores' own layout                                    */
/* ------------------------------------------------------------------------ */

/* [NKI] Parameters: the backward takes optional pre-computed scales for its
 * operands and flags saying that they are pre-swizzled.  Here the swizzled
 * form is the layout in which the tcgen05 block-scaled MMAs take their scale
 * factors, so that quantizers can write it and GEMMs read it in place, with
 * no relayout between them.
 *
 * The atom layout of one GEMM operand of B x R rows x K (the contraction
 * axis), hardware blocks of bs = 32 (UE8M0) or 16 (UE4M3) along K:
 *   - 512-byte atoms [B][RT][KS4]: RT = ceil(R / 256) * 2 row tiles of 128
 *     rows; KS4 = ceil(K / kt) * (kt / bs / 4) atoms per row tile, where
 *     kt = 128 for FP8 codes and 256 for E2M1 (an atom holds 4 blocks).
 *   - The scale of row 128 t + w (0 <= w < 128), block 4 j + i (0 <= i < 4) is
 *     byte (w % 32) * 16 + (w / 32) * 4 + i of atom (b, t, j).
 *   - Rows past R and blocks past K hold the neutral scale (UE8M0 127, which
 *     is 1.0; UE4M3 0).
 * Formats: MXFP8 (E4M3 / E5M2 codes, UE8M0), MXFP4 (E2M1, UE8M0), NVFP4
 * (E2M1, UE4M3).  bsmm_scale_atoms_size returns the bytes (0 for other
 * combinations or empty sizes).
 */
size_t bsmm_scale_atoms_size(int64_t B, int64_t rows, int64_t K, bsmm_dtype code_type,
                             bsmm_scale_type scale_type);

/* Quantize a GEMM operand with its scales written straight into the atom
 * layout (same codes and scale values as bsmm_quantize with blocks of 1 x bs
 * along K).
 *   transpose_in = 0: x [B * rows, K] row-major, contiguous.
 *   transpose_in = 1: x [K, rows] (the operand transposed; B must be 1).
 *   codes [B * rows, K] (E2M1: K / 2 bytes a row, packed as in bsmm_quantize).
 *   atoms  at least bsmm_scale_atoms_size() bytes, 4-byte aligned; the call
 *          writes all of it (padding included).
 * Errors: BSMM_ERR_UNSUPPORTED for other code / scale pairs, BSMM_ERR_SHAPE
 * when K is not a multiple of bs, BSMM_ERR_WORKSPACE when atoms_bytes is too
 * small.
 */
bsmm_status bsmm_quantize_atoms(const void* x, bsmm_dtype x_type, int64_t B, int64_t rows, int64_t K,
                                int transpose_in, bsmm_dtype code_type, bsmm_scale_type scale_type,
                                void* codes, void* atoms, size_t atoms_bytes, bsmm_stream_t stream);

/* bsmm_gemm with both operands' scales in the atom layout (one scale per
 * hardware block).  Same result as bsmm_gemm with the row-major scales they
 * hold.  MXFP8 reads the atoms in place and takes no workspace (NULL, 0);
 * MXFP4 and NVFP4 need bsmm_gemm_workspace_size() bytes, 256-byte aligned, in
 * which the CTA-pair kernel's copy blocks are written from the atoms.
 * Pointers 16-byte aligned; K a multiple of 32.
 */
bsmm_status bsmm_gemm_atoms(int64_t B, int64_t M, int64_t N, int64_t K, const void* a, bsmm_dtype a_type,
                            const void* b, bsmm_dtype b_type, const void* a_atoms, const void* b_atoms,
                            bsmm_scale_type scale_type, void* y, bsmm_dtype y_type, void* workspace,
                            size_t workspace_bytes, bsmm_stream_t stream);

/* [NKI] Parameters (pre-computed scales, pre-swizzled inputs): the backward's
 * two GEMMs from operands already quantized along their contraction axes,
 * MXFP8 with fp8_type codes:
 *   dy_n [M, N] (dY along N),  w_t  [K, N] (W^T along N),
 *   dy_t [N, M] (dY^T along M), x_t [K, M] (X^T along M),
 * each with its UE8M0 scales: row-major [rows][contraction / 32]
 * (scales_are_atoms = 0, as bsmm_quantize writes them) or in the atom layout
 * (scales_are_atoms = 1, as bsmm_quantize_atoms writes them).
 * dX [M, K] = dY W and dW [N, K] = dY^T X, bfloat16.  The workspace is
 * bsmm_linear_backward_quantized_workspace_size() bytes (0 with atoms),
 * 256-byte aligned.  M, N and K multiples of 32; pointers 16-byte aligned.
 */
size_t bsmm_linear_backward_quantized_workspace_size(int64_t M, int64_t N, int64_t K, int scales_are_atoms);

bsmm_status bsmm_linear_backward_quantized(int64_t M, int64_t N, int64_t K, bsmm_dtype fp8_type,
                                           const void* dy_n, const void* dy_n_scales, const void* w_t,
                                           const void* w_t_scales, const void* dy_t, const void* dy_t_scales,
                                           const void* x_t, const void* x_t_scales, int scales_are_atoms,
                                           void* dX, void* dW, void* workspace, size_t workspace_bytes,
                                           bsmm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BSMM_H_ */
