/*
 * fp4lin.h -- C ABI of the GB300 (sm_103a) FP4 quantized linear layer.
 *
 * The method is the quantized linear layer of the FP4 LLM-training framework
 * described on the pages "首个 FP4 精度的大模型训练框架来了，来自微软研究院"
 * (czzqal.com), "Microsoft Research bringt den ersten FP4-Genauigkeitsrahmen
 * für das Training großer Modelle heraus" (topaibox.com) and "Optimizing Large
 * Language Model Training Using FP4 Quantization" (shd-paper.top, abstract).
 *
 * Notation: A is the activation, M x K BF16, row-major (tokens x in-features);
 * W is the weight, K x N BF16, row-major (in-features x out-features);
 * s_A (M) and s_W (N) are fp32 scales; codes are E2M1 (1 sign, 2 exponent,
 * 1 mantissa bit), two per byte, element 2c in the low nibble.
 *
 * Conventions for every call:
 *  - Ownership: the caller owns every buffer.  The library allocates no device
 *    or host memory, frees nothing and never synchronizes, except
 *    fp4_device_status, which synchronizes the given stream.
 *  - Pointers marked "device" must be device (or managed) memory of the
 *    current CUDA device.  Buffers and leading dimensions are in ELEMENTS of
 *    the buffer's type unless the name ends in _bytes.
 *  - Streams: all work is enqueued on `stream` (NULL = legacy default stream).
 *  - Errors: arguments are validated on the host before any launch; a bad
 *    argument returns an error and launches nothing.  A launch failure returns
 *    FP4_ERR_CUDA.  Conditions only the device can see (a bounded wait that ran
 *    out, CSR capacity exceeded) set sticky flags in a device word that
 *    fp4_device_status reads; those calls still return FP4_OK.
 *  - Device: only compute capability 10.3 (GB300, sm_103a) is accepted;
 *    anything else returns FP4_ERR_DEVICE_UNSUPPORTED.
 *  - Per-device state: on its first call on a device the library looks up
 *    device addresses (its status word, the built-in scratch array of
 *    fp4_quantize_cols_noalloc) and sets kernel attributes, and keeps them
 *    for the life of the process.  Do not use the library on a device after
 *    cudaDeviceReset (or any other teardown of that device's primary
 *    context) in the same process: the kept addresses would be stale.
 */
#ifndef FP4LIN_H
#define FP4LIN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* fp4_stream_t; /* same handle as cudaStream_t */

typedef enum fp4_status {
  FP4_OK = 0,
  FP4_ERR_INVALID_ARG = 1,        /* null pointer, bad enum, q outside (0, 1] */
  FP4_ERR_SHAPE = 2,              /* sizes or leading dimensions not supported */
  FP4_ERR_ALIGNMENT = 3,          /* a pointer or leading dimension misaligned */
  FP4_ERR_WORKSPACE = 4,          /* workspace missing or too small */
  FP4_ERR_CAPACITY = 5,           /* nnz capacity below outlier_max_nnz */
  FP4_ERR_TIMEOUT = 6,            /* a device wait ran out (from fp4_device_status) */
  FP4_ERR_DEVICE_UNSUPPORTED = 7, /* current device is not sm_103 */
  FP4_ERR_CUDA = 8,               /* a CUDA runtime / driver call failed */
  FP4_ERR_INTERNAL = 9            /* a device-side consistency check failed */
} fp4_status;

typedef enum fp4_out_type {
  FP4_OUT_BF16 = 0,        /* Y in BF16, round to nearest even */
  FP4_OUT_FP32 = 1,        /* Y in fp32 */
  FP4_OUT_RAW_ACC_FP32 = 2 /* the unscaled FP4 accumulator sum_k qA*qW in fp32; no scales, no compensation */
} fp4_out_type;

/* Element type of the weight gradient written by fp4_linear_wgrad_dge. */
typedef enum fp4_dw_type {
  FP4_DW_FP32 = 0,  /* dW in fp32 */
  FP4_DW_E4M3 = 1   /* E4M3 codes of fl32(dW * scale), one byte each: the FP8 gradient
                       for communication (page "首个 FP4 ...", mixed-precision passage) */
} fp4_dw_type;

/* Sticky device flags reported by fp4_device_status. */
#define FP4_FLAG_TIMEOUT 0x1u  /* an mbarrier wait in a GEMM ran past its limit */
#define FP4_FLAG_CAPACITY 0x2u /* the CSR staging area was too small */
#define FP4_FLAG_INTERNAL 0x4u /* device consistency check failed */

/* Human-readable name of a status code (static string, never NULL). */
const char* fp4_status_string(fp4_status status);

/* Version of this ABI (incremented on any signature change). */
int fp4_abi_version(void);

/* Text of the CUDA error behind the calling thread's most recent FP4_ERR_CUDA
 * from a kernel launch (static string, never NULL). */
const char* fp4_last_cuda_error(void);

/*
 * fp4_quantize_rows -- token-wise (row) absmax quantization of A to E2M1, with
 * an optional fused outlier clamp.
 *
 * Defined by: page "首个 FP4 ..." (czzqal.com), granularity passage (A is
 * quantized per row / token) and quantization passage (scale into the FP4
 * range, round to the nearest FP4 value); page "Microsoft Research bringt ..."
 * (topaibox.com), section "Innovationen in der Vorwärts- und
 * Rückwärtspropagation".  Per row i: x' = clamp_t ? sign(x) min(|x|, *clamp_t) : x;
 * absmax_i = max |x'|; s_A[i] = 6 / absmax_i (one fp32 division; 1 if absmax is
 * 0 or the quotient is not finite); code = E2M1 round-to-nearest-even of the
 * fp32 product x' * s_A[i], saturating at 6, sign kept for values rounding to 0.
 *
 *   A       device, BF16, M x K, row stride lda (elements); 16-byte aligned
 *   M, K    M >= 0; 0 < K <= 16384 and K % 32 == 0
 *   lda     >= K, lda % 8 == 0
 *   clamp_t device fp32 scalar (e.g. t_out of outlier_clamp_quantile) or NULL
 *   codes   device, uint8, M x ldc_bytes, row i holds K/2 bytes; 16-byte aligned
 *   ldc_bytes >= K/2, ldc_bytes % 16 == 0
 *   scales  device, fp32, M
 * Errors: INVALID_ARG, SHAPE, ALIGNMENT, DEVICE_UNSUPPORTED, CUDA.
 */
fp4_status fp4_quantize_rows(const void* A, int64_t M, int64_t K, int64_t lda, const float* clamp_t,
                             uint8_t* codes, int64_t ldc_bytes, float* scales, fp4_stream_t stream);

/*
 * fp4_quantize_cols -- channel-wise (column) absmax quantization of W to
 * E2M1, written K-major (codes_t = packed W^T, N rows of K/2 bytes).
 *
 * Defined by: page "首个 FP4 ..." (czzqal.com), granularity passage (W is
 * quantized per column / channel).  Same rule as fp4_quantize_rows applied to
 * every column j of W: s_W[j] = 6 / max_k |W[k,j]|.
 *
 *   W       device, BF16, K x N, row stride ldw (elements); 16-byte aligned
 *   K, N    K > 0, K % 32 == 0; N > 0, N % 8 == 0
 *   ldw     >= N, ldw % 8 == 0
 *   codes_t device, uint8, N x ldc_bytes; 16-byte aligned; ldc_bytes >= K/2, % 16 == 0
 *   scales  device, fp32, N
 *   workspace device, >= fp4_quantize_cols_workspace(N) bytes, 16-byte aligned;
 *           used as scratch for the column maxima (contents on entry ignored)
 * Errors: INVALID_ARG, SHAPE, ALIGNMENT, WORKSPACE, DEVICE_UNSUPPORTED, CUDA.
 */
size_t fp4_quantize_cols_workspace(int64_t N);
fp4_status fp4_quantize_cols(const void* W, int64_t K, int64_t N, int64_t ldw, uint8_t* codes_t,
                             int64_t ldc_bytes, float* scales, void* workspace, size_t ws_bytes,
                             fp4_stream_t stream);

/*
 * fp4_quantize_cols_noalloc -- fp4_quantize_cols for callers that cannot give
 * the library any scratch memory.
 *
 * There is no counterpart on the pages: this is an interface variant, not part
 * of the method.  Callers that cannot allocate -- code inside a framework that
 * owns every device allocation, real-time paths that must not call cudaMalloc
 * (it can synchronize the device), embedded users with a fixed memory budget --
 * get the same result as fp4_quantize_cols (bit for bit) without a workspace.
 * The column maxima are kept in a fixed device array built into the library
 * (64 Ki entries, 256 KiB, held on every GPU that loads the library until the
 * process exits); N above 65536 returns FP4_ERR_SHAPE.  Arguments, alignment
 * and errors are those of fp4_quantize_cols without the workspace pair.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) and caches it; make that first call outside any
 * stream capture.  All calls share the one array, and each call clears the
 * part it uses before using it, so calls must not overlap on the GPU: two
 * calls in flight at the same time on different streams race on the array.
 * No device or host memory is allocated by this call.
 */
fp4_status fp4_quantize_cols_noalloc(const void* W, int64_t K, int64_t N, int64_t ldw, uint8_t* codes_t,
                                     int64_t ldc_bytes, float* scales, fp4_stream_t stream);

/*
 * outlier_clamp_quantile -- quantile threshold of |A|, clamp, and the sparse
 * compensation matrix dA = A - A_clamped in CSR form.
 *
 * Defined by: page "首个 FP4 ..." (czzqal.com), outlier passage (a quantile
 * search finds the largest-magnitude outliers of A, they are clamped to a
 * threshold giving A_clamped, and a sparse compensation matrix built from A and
 * A_clamped is nonzero only at the clamped positions); page "Microsoft Research
 * bringt ..." (topaibox.com), "Peak-Dämpfung und -Kompensation von Ausreißern".
 * t = the k-th smallest |A| over all M*K elements, k = ceil(q*M*K) (IEEE
 * double, limited to [1, M*K]), no interpolation; clamped entries are those
 * with |A| > t; A_clamped = sign(A) min(|A|, t); dA values = A - sign(A) t in
 * fp32.  Rows ascending, column indices ascending within a row.
 *
 *   A        device, BF16, M x K (row stride lda), 16-byte aligned; 1 <= M*K < 2^32
 *   K        K % 8 == 0, K <= 16384; lda >= K, lda % 8 == 0
 *   q        0 < q <= 1
 *   t_out    device fp32 scalar: t (feed it to fp4_quantize_rows as clamp_t)
 *   row_ptr  device int32, M + 1
 *   col_idx  device int32, nnz_capacity
 *   vals     device fp32, nnz_capacity
 *   nnz_capacity >= outlier_max_nnz(M, K, q) (host-side check, CAPACITY if not)
 *   nnz_out  device int64 scalar: number of entries written (= row_ptr[M]); may be NULL
 *   A_clamped device BF16 M x ldac, or NULL for none; ldac >= K, % 8 == 0
 *   workspace device, >= outlier_clamp_quantile_workspace(M, K, nnz_capacity) bytes,
 *            16-byte aligned; scratch (histogram, counters, CSR staging),
 *            contents on entry ignored
 * outlier_max_nnz returns M*K - k: at most that many entries exceed t.
 * Errors: INVALID_ARG, SHAPE, ALIGNMENT, CAPACITY, WORKSPACE,
 *         DEVICE_UNSUPPORTED, CUDA; device-side INTERNAL flag if the staged
 *         count disagrees with the histogram.
 */
int64_t outlier_max_nnz(int64_t M, int64_t K, double q);
size_t outlier_clamp_quantile_workspace(int64_t M, int64_t K, int64_t nnz_capacity);
fp4_status outlier_clamp_quantile(const void* A, int64_t M, int64_t K, int64_t lda, double q,
                                  float* t_out, int32_t* row_ptr, int32_t* col_idx, float* vals,
                                  int64_t nnz_capacity, int64_t* nnz_out, void* A_clamped,
                                  int64_t ldac, void* workspace, size_t ws_bytes,
                                  fp4_stream_t stream);

/*
 * fp4_quantize_rows_outliers -- outlier_clamp_quantile and
 * fp4_quantize_rows(clamp_t = t) in one call that reads A twice instead of
 * three times: the first pass finds the threshold t, the second clamps,
 * stages the CSR entries of dA and writes the E2M1 codes and row scales of
 * A_clamped from the same registers.
 *
 * Defined by: the passages cited for outlier_clamp_quantile and
 * fp4_quantize_rows (clamping happens before the row quantization, page
 * "首个 FP4 ..." (czzqal.com), outlier and quantization passages).  Outputs are
 * bit-identical to the two separate calls.
 *
 *   A, M, K, lda, q, t_out, row_ptr, col_idx, vals, nnz_capacity, nnz_out,
 *   workspace, ws_bytes   as for outlier_clamp_quantile (no A_clamped output)
 *   codes, ldc_bytes, scales   as for fp4_quantize_rows; K % 32 == 0
 * Both calls' limits apply, in particular K <= 16384.
 * Errors: INVALID_ARG, SHAPE, ALIGNMENT, CAPACITY, WORKSPACE,
 *         DEVICE_UNSUPPORTED, CUDA.
 */
fp4_status fp4_quantize_rows_outliers(const void* A, int64_t M, int64_t K, int64_t lda, double q, uint8_t* codes,
                                      int64_t ldc_bytes, float* scales, float* t_out, int32_t* row_ptr,
                                      int32_t* col_idx, float* vals, int64_t nnz_capacity, int64_t* nnz_out,
                                      void* workspace, size_t ws_bytes, fp4_stream_t stream);

/*
 * fp4_linear_fwd_workspace -- bytes of device workspace that fp4_linear_fwd
 * uses to run the compensation on the tensor cores for an M x K by K x N
 * product (grows as 1 KB per row of M and of N).  0 for invalid shapes.
 * Host-only.  This workspace has no counterpart on the pages: it holds the
 * scaled, split operands of the compensation product described below.
 */
size_t fp4_linear_fwd_workspace(int64_t M, int64_t N, int64_t K);

/*
 * fp4_linear_fwd -- FP4 GEMM on tcgen05 (kind::mxf4, unit block scales) with
 * the row x column scales and the sparse dA*W compensation.
 *
 * Defined by: page "首个 FP4 ..." (czzqal.com), GeMM passage (custom FP4 GEMM
 * kernel, tiled multiply in FP4) and granularity passage (the row / column
 * scales match the GEMM's parallel layout and need no transpose, so they factor
 * out of the K-sum); outlier passage (compensation matrix).
 *   acc[i,j] = sum_k decode(a_codes[i,k]) * decode(w_codes_t[j,k])   (exact in fp32)
 *   Y[i,j]   = acc[i,j] / (s_A[i] s_W[j]) + sum_{e in row i of dA} val[e] * W[col[e], j]
 *
 * How the compensation runs (results agree to fp32 rounding either way):
 *   - workspace given and dA has at most 128 distinct nonzero columns (outlier
 *     channels): the product over those columns runs on the tensor cores as
 *     TF32 MMAs into the same accumulator, with dA s_A and W s_W each split
 *     into two TF32 parts (relative error of each term about 2^-22);
 *   - otherwise (no workspace, or more distinct columns): the epilogue threads
 *     add the sum in fp32, entry by entry in CSR order.
 *
 *   a_codes   device uint8 M x lda_codes_bytes (K-major), 16-byte aligned, lda_codes_bytes % 16 == 0
 *   s_a       device fp32 M
 *   w_codes_t device uint8 N x ldw_codes_bytes (K-major), 16-byte aligned, % 16 == 0
 *   s_w       device fp32 N
 *   M, N, K   M, N >= 1; 32 <= K <= 16384, K % 32 == 0; M, N < 2^31; N % 8 == 0
 *   dA_row_ptr, dA_col, dA_val  device CSR of dA (as from outlier_clamp_quantile),
 *             all three NULL for no compensation; row_ptr starts at 0 and does not
 *             decrease, and entries [0, row_ptr[M]) of dA_col / dA_val are readable
 *             (not checked: it would take a host synchronization); the columns of
 *             a row must be distinct (the epilogue path is fastest when they
 *             ascend); an entry whose column lies outside [0, K) is skipped and
 *             reported as the device-side INTERNAL flag
 *   W         device BF16 K x ldw (the unquantized weight), required iff compensation
 *   Y         device, M x ldy elements of the output type; 16-byte aligned, ldy % 8 == 0
 *   y_type    fp4_out_type
 *   workspace device, 256-byte aligned, ws_bytes >= fp4_linear_fwd_workspace(M, N, K),
 *             or NULL; used only with compensation; must not be shared by calls
 *             that may run at the same time; owned by the caller
 * Errors: INVALID_ARG, SHAPE, ALIGNMENT, WORKSPACE (non-NULL and too small),
 *         DEVICE_UNSUPPORTED, CUDA; device-side TIMEOUT flag if a pipeline wait
 *         runs out (about 1 s); device-side INTERNAL flag for a dA column
 *         outside [0, K) (the entry is skipped, on both compensation paths).
 */
fp4_status fp4_linear_fwd(const uint8_t* a_codes, int64_t lda_codes_bytes, const float* s_a,
                          const uint8_t* w_codes_t, int64_t ldw_codes_bytes, const float* s_w,
                          int64_t M, int64_t N, int64_t K, const int32_t* dA_row_ptr,
                          const int32_t* dA_col, const float* dA_val, const void* W, int64_t ldw,
                          void* Y, int y_type, int64_t ldy, void* workspace, size_t ws_bytes,
                          fp4_stream_t stream);

/*
 * fp4_linear_fwd_dense_workspace -- bytes of device workspace fp4_linear_fwd_dense
 * needs: the fp32 FP4 product (4 M N), the dense three-part split of dA
 * (6 M K), W^T in BF16 (2 N K) and the engine's split-tail area.  0 for
 * invalid shapes (K % 64 != 0) or an unsupported device.  Host-only.
 */
size_t fp4_linear_fwd_dense_workspace(int64_t M, int64_t N, int64_t K);

/*
 * fp4_linear_fwd_dense -- the same result as fp4_linear_fwd with compensation,
 * for a dense dA (a low clamp quantile: every tile of dA holds entries).
 *
 * Defined by: page "Microsoft Research bringt den ersten FP4-Genauigkeits-
 * rahmen ..." (topaibox.com), "Peak-Dämpfung und -Kompensation von
 * Ausreißern" (the clamped A in FP4, the residual dA multiplied in higher
 * precision and added), with the granularity passage of page "首个 FP4 ..."
 * (czzqal.com) for the scales:
 *   Y[i,j] = acc[i,j] / (s_A[i] s_W[j]) + sum_k dA[i,k] W[k,j]
 * How: the FP4 product goes to the workspace in fp32; dA is written densely as
 * BF16 parts per entry whose sum is the fp32 entry exactly -- two (A and
 * -sign(A) t) when the clamp threshold t is given, else three (hi + mid + lo)
 * -- and multiplied by the BF16 W on the BF16 tensor cores (fp32 accumulation
 * in 2048-term chunks, about 2e-6 of the sum of |terms| per output); the sum
 * of the two products is rounded once to the output type.
 * Choose it over fp4_linear_fwd when dA averages tens of entries per row or
 * more (its cost does not depend on nnz); fp4_linear_fwd is faster for a few
 * outlier channels.
 *
 *   arguments as for fp4_linear_fwd, except:
 *   K         64 <= K <= 16384, K % 64 == 0
 *   dA_row_ptr, dA_col, dA_val, W   required
 *   dA_t      device fp32 scalar or NULL: the clamp threshold t that produced dA
 *             (t_out of outlier_clamp_quantile / fp4_quantize_rows_outliers), so
 *             that every value is A - sign(A) t with A and t BF16 values; then
 *             the product runs over 2K instead of 3K.  An entry that breaks this
 *             premise is multiplied as a two-part rounding of its value and
 *             reported as the device-side INTERNAL flag.  4-byte aligned.
 *   y_type    FP4_OUT_BF16 or FP4_OUT_FP32
 *   workspace device, 256-byte aligned, ws_bytes >= fp4_linear_fwd_dense_workspace(M, N, K);
 *             required; must not be shared by calls that may run at the same time
 * Errors: INVALID_ARG, SHAPE, ALIGNMENT, WORKSPACE, DEVICE_UNSUPPORTED, CUDA;
 *         device-side INTERNAL flag for an entry whose column lies outside [0, K)
 *         (the entry is skipped) or that breaks the dA_t premise, TIMEOUT as for
 *         fp4_linear_fwd.
 */
fp4_status fp4_linear_fwd_dense(const uint8_t* a_codes, int64_t lda_codes_bytes, const float* s_a,
                                const uint8_t* w_codes_t, int64_t ldw_codes_bytes, const float* s_w,
                                int64_t M, int64_t N, int64_t K, const int32_t* dA_row_ptr,
                                const int32_t* dA_col, const float* dA_val, const float* dA_t,
                                const void* W, int64_t ldw,
                                void* Y, int y_type, int64_t ldy, void* workspace, size_t ws_bytes,
                                fp4_stream_t stream);

/*
 * fp4_linear_wgrad_dge -- BF16 weight-gradient GEMM on tcgen05 (kind::f16)
 * with the differentiable-gradient-estimator (DGE) factor in the epilogue.
 *
 * Defined by: page "首个 FP4 ..." (czzqal.com), DGE passage (hard quantization
 * forward; in backward a continuous differentiable function refits the
 * quantizer and its derivative gives a correction of the gradient); page
 * "Optimizing Large Language Model Training Using FP4 Quantization", abstract.
 *   G[r,j]  = sum_m A[m,r] dY[m,j]                                  (fp32 accumulate)
 *   x       = |fl32(W[r,j] * s_W[j])|   (the value the column quantizer rounds)
 *   dW[r,j] = G[r,j] * f'(x),  f'(x) = min(clip, (1/k) |u|^(1/k - 1)),
 *             u = 2 (x - lo)/delta - 1 on the E2M1 interval [lo, lo + delta]
 *             holding x (delta 0.5 below 2, 1 below 4, 2 below 6); f' = 1/k for x >= 6.
 *
 *   A   device BF16 M x lda (tokens x in), 16-byte aligned, lda % 8 == 0
 *   dY  device BF16 M x lddy (tokens x out), 16-byte aligned, lddy % 8 == 0
 *   W   device BF16 K x ldw, s_w device fp32 N (from fp4_quantize_cols)
 *   M, N, K  M >= 1; N % 8 == 0; K % 8 == 0; all < 2^31
 *   dge_k > 0, dge_clip > 0
 *   dW  device K x lddw, 16-byte aligned, lddw % 4 == 0, of the element type
 *       dw_type gives; written once per element while other tiles still read
 *       W and s_w, so dW must not alias A, dY, W or s_w
 *   dw_type   FP4_DW_FP32, or FP4_DW_E4M3: the page says gradients are
 *       communicated in FP8 and names neither the variant nor the scaling;
 *       the reading taken is E4M3 (bias 7, 3 mantissa bits, largest finite
 *       448) with one per-tensor scale: dW8[r,j] = E4M3(fl32(dW[r,j] * scale)),
 *       round half to the even mantissa, magnitudes past 448 saturate to 448,
 *       a value that rounds to zero keeps its sign; dW ~ decode(dW8) / scale
 *   dw_scale  E4M3 only: device fp32 scalar, the per-tensor scale (read on the
 *       device, so it may be produced by an earlier kernel); NULL for fp32
 *   dw_amax   E4M3 only: device fp32 scalar, set to max |dW| over the whole
 *       gradient (before scaling; zeroed on the stream first, then raised with
 *       atomics), e.g. to derive the next step's scale 448 / amax; must not
 *       overlap dW; NULL for fp32
 *   workspace  device, 256-byte aligned, ws_bytes >= fp4_linear_wgrad_dge_workspace(M, N, K),
 *       or NULL.  With it, a last wave of tiles that would leave at least half
 *       of the SM pairs idle is computed as two halves of the token range on
 *       two pairs, combined through the workspace (the result is the same
 *       whichever half finishes first).  Must not be shared by calls that may
 *       run at the same time; owned by the caller.
 * Errors: INVALID_ARG (also: an unknown dw_type, E4M3 without dw_scale or
 *         dw_amax, dw_amax inside dW), SHAPE, ALIGNMENT (also: dw_scale or
 *         dw_amax not 4-byte aligned), WORKSPACE (non-NULL and too small),
 *         DEVICE_UNSUPPORTED, CUDA; device-side TIMEOUT flag as for fp4_linear_fwd.
 */
fp4_status fp4_linear_wgrad_dge(const void* A, int64_t lda, const void* dY, int64_t lddy, const void* W,
                                int64_t ldw, const float* s_w, int64_t M, int64_t N, int64_t K,
                                float dge_k, float dge_clip, void* dW, int dw_type, int64_t lddw,
                                const float* dw_scale, float* dw_amax,
                                void* workspace, size_t ws_bytes, fp4_stream_t stream);

/*
 * fp4_linear_wgrad_dge_workspace -- bytes of workspace fp4_linear_wgrad_dge
 * uses for these sizes on the current device (0: it never splits a tile, and
 * a NULL workspace is as good).  Returns 0 for non-positive sizes or an
 * unsupported device.
 */
size_t fp4_linear_wgrad_dge_workspace(int64_t M, int64_t N, int64_t K);

/*
 * fp4_linear_dgrad -- BF16 input-gradient GEMM on tcgen05 (kind::f16):
 *   dX[m,k] = sum_n dY[m,n] W[k,n]        (fp32 accumulate; dX = dY W^T)
 *
 * Not on the pages: they give the forward pass and the DGE weight gradient
 * (page "首个 FP4 ...", czzqal.com, DGE passage) but not the input gradient.
 * This is the chain rule of Y = A W, the plainest reading that closes the
 * linear's backward: the same BF16 engine as fp4_linear_wgrad_dge, with the
 * BF16 W the caller passes (the unquantized weight, as the compensation uses).
 * The reduction over N runs in 2048-element chunks summed in fp32 registers.
 *
 *   dY  device BF16 M x lddy (tokens x out), 16-byte aligned, lddy % 8 == 0
 *   W   device BF16 K x ldw (in x out), 16-byte aligned, ldw % 8 == 0
 *   M, N, K  M >= 1; N, K >= 8; N % 8 == 0; K % 8 == 0; all < 2^31
 *   dX  device M x lddx (tokens x in) of dx_type, 16-byte aligned, lddx % 8 == 0,
 *       lddx >= K; must not alias dY or W
 *   dx_type  FP4_OUT_BF16 (round to nearest even) or FP4_OUT_FP32
 *   workspace  device, 256-byte aligned, ws_bytes >= fp4_linear_dgrad_workspace(M, N, K),
 *       or NULL: the split tail of fp4_linear_wgrad_dge, over the N range
 * Errors: INVALID_ARG (null pointer, other dx_type), SHAPE, ALIGNMENT,
 *         WORKSPACE (non-NULL and too small), DEVICE_UNSUPPORTED, CUDA;
 *         device-side TIMEOUT flag as for fp4_linear_fwd.
 */
fp4_status fp4_linear_dgrad(const void* dY, int64_t lddy, const void* W, int64_t ldw, int64_t M,
                            int64_t N, int64_t K, void* dX, int dx_type, int64_t lddx,
                            void* workspace, size_t ws_bytes, fp4_stream_t stream);

/*
 * fp4_linear_dgrad_workspace -- bytes of workspace fp4_linear_dgrad uses for
 * these sizes on the current device (0 when it never splits a tile).
 */
size_t fp4_linear_dgrad_workspace(int64_t M, int64_t N, int64_t K);

/*
 * fp4_device_status -- synchronize `stream`, then return the sticky device
 * flags (FP4_FLAG_*) of the current device in *flags_out and clear them.
 * The return value is FP4_ERR_TIMEOUT / FP4_ERR_CAPACITY / FP4_ERR_INTERNAL
 * for the first flag set in that order, FP4_OK if none, FP4_ERR_CUDA if the
 * synchronization failed.  flags_out may be NULL.
 */
fp4_status fp4_device_status(fp4_stream_t stream, uint32_t* flags_out);

/*
 * fp4_selftest_bounded_wait -- launch one CTA that waits on an mbarrier which
 * nothing ever completes, with a limit of timeout_us microseconds (1..10^6).
 * The wait gives up, the kernel sets FP4_FLAG_TIMEOUT and returns; the
 * context stays usable.  Exercises the bounded-wait path of the GEMM
 * pipelines without a fault.  Errors: INVALID_ARG, DEVICE_UNSUPPORTED, CUDA.
 */
fp4_status fp4_selftest_bounded_wait(uint32_t timeout_us, fp4_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FP4LIN_H */
