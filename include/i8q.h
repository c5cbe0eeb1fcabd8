/*
 * i8q.h -- C ABI of libi8q.so, a single-GPU (sm_103a) engine for linear int8
 * quantization and the quantized matrix products it feeds.
 *
 * Conventions for every entry point below
 *  - Status: functions returning int give I8Q_OK (0) on success or a negative
 *    I8Q_ERR_* code.  The text of the most recent error on the calling host
 *    thread is returned by i8q_last_error().  Arguments are validated on the
 *    host before anything is launched; a rejected call launches nothing and
 *    writes nothing.
 *  - Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *    default stream).  Calls are asynchronous on that stream unless stated.
 *  - Pointers: tensor arguments are DEVICE pointers unless stated.  The
 *    caller owns every tensor, every workspace and the stream; a context owns
 *    only the internal buffers it allocates.  Tensors are dense and
 *    row-major (C order) with the shapes given; no aliasing between inputs
 *    and outputs.
 *  - Exactness: integer results (quantized tensors, int32 accumulators) are
 *    bit-exact.  Float epilogues evaluate each operation once, in fp32,
 *    rounding to nearest even, in the order the operator text gives (no
 *    fused multiply-add); fp32->bf16 rounds to nearest even.
 *
 * Sources, by page title and section:
 *  [DQIP] Simd, "SynetDynamicQuantizedInnerProduct16b": Detailed Description
 *         (algorithm listing; typeA/typeB/typeC and avoidOverflow paragraph)
 *         and the member documentation of Init, Enable, InternalBufferSize,
 *         ExternalBufferSize, Info, SetParams, Forward, Clear.
 *  [QL]   ONNX Runtime contrib schemas, "QuantizeLinear" ver 1.
 *  [DQL]  ONNX Runtime contrib schemas, "DequantizeLinear" ver 1.
 *  [QLC]  onnx-light docs, "QLinearConv" (since version 10): inputs, bias
 *         rule, type constraints.
 *  [LSTM] ONNX Runtime contrib schemas, "DynamicQuantizeLSTM": attributes,
 *         inputs X, W, R, B, initial_h, initial_c, W/R scale and zero point,
 *         outputs Y, Y_h, Y_c.
 *  [QG]   ONNX Runtime contrib schemas, "QGemm": inputs A, a_scale,
 *         a_zero_point, B, b_scale, b_zero_point, C, y_scale, y_zero_point;
 *         attributes transA, transB, alpha.
 *  [MITF] ONNX Runtime contrib schemas, "MatMulIntegerToFloat" and
 *         "DynamicQuantizeMatMul": inputs A, B, a_scale, b_scale,
 *         a_zero_point, b_zero_point, bias.
 *  [QEW]  ONNX Runtime contrib schemas, "MulInteger", "QLinearAdd",
 *         "QLinearMul" (doc formulas, Numpy-style broadcasting),
 *         "QLinearLeakyRelu", "QLinearSigmoid" (doc strings).
 */
#ifndef I8Q_H
#define I8Q_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define I8Q_OK 0
#define I8Q_ERR_INVALID_ARG (-1)    /* bad pointer, size, type or combination */
#define I8Q_ERR_UNSUPPORTED (-2)    /* valid operator input this build does not run */
#define I8Q_ERR_NOT_INITIALIZED (-3) /* context missing, or SetParams not yet called */
#define I8Q_ERR_ALLOC (-4)          /* device allocation failed */
#define I8Q_ERR_CUDA (-5)           /* a CUDA runtime/driver call failed */
#define I8Q_ERR_DEVICE_TIMEOUT (-6) /* a bounded device-side wait gave up */

/* ---- element types ----------------------------------------------------- */
#define I8Q_F32 0
#define I8Q_BF16 1
#define I8Q_S8 2
#define I8Q_U8 3
#define I8Q_S32 4

/* ---- activations applied after the bias ([DQIP] Forward) --------------- */
#define I8Q_ACT_IDENTITY 0
#define I8Q_ACT_RELU 1
#define I8Q_ACT_GELU 2 /* 0.5*x*(1+erf(x/sqrt(2))), fp32 */

/* ---- QuantizeLinear / DequantizeLinear axis ------------------------------ */
#define I8Q_NO_AXIS INT32_MIN /* no 'axis' attribute: per-tensor parameters */

/* ---- LSTM direction ------------------------------------------------------ */
#define I8Q_LSTM_FORWARD 0
#define I8Q_LSTM_REVERSE 1
#define I8Q_LSTM_BIDIRECTIONAL 2

/* ---- LSTM activation functions ("activations" attribute) ----------------
 * The ONNX LSTM operator's list, in its order.  Each is its operator's
 * formula in fp32 with one rounding per operation; exp, expm1, log1p, tanh
 * and sigmoid are fixed operation sequences (the library's own, not the
 * platform's math library), so results are reproducible bit for bit:
 *   RELU max(0,x); TANH; SIGMOID 1/(1+e^-x); AFFINE a*x+b;
 *   LEAKY_RELU x>=0 ? x : a*x; THRESHOLDED_RELU x>a ? x : 0;
 *   SCALED_TANH a*tanh(b*x); HARD_SIGMOID min(max(a*x+b,0),1);
 *   ELU x>=0 ? x : a*(e^x-1); SOFTSIGN x/(1+|x|); SOFTPLUS log(1+e^x). */
#define I8Q_LSTM_ACT_RELU 0
#define I8Q_LSTM_ACT_TANH 1
#define I8Q_LSTM_ACT_SIGMOID 2
#define I8Q_LSTM_ACT_AFFINE 3
#define I8Q_LSTM_ACT_LEAKY_RELU 4
#define I8Q_LSTM_ACT_THRESHOLDED_RELU 5
#define I8Q_LSTM_ACT_SCALED_TANH 6
#define I8Q_LSTM_ACT_HARD_SIGMOID 7
#define I8Q_LSTM_ACT_ELU 8
#define I8Q_LSTM_ACT_SOFTSIGN 9
#define I8Q_LSTM_ACT_SOFTPLUS 10

/* Text of the last error raised on this host thread ("" if none).  The
 * pointer stays valid until the next call on this thread. */
const char* i8q_last_error(void);

/* Library version string, e.g. "i8q 0.1 sm_103a". */
const char* i8q_version(void);

/* ========================================================================
 * Dynamic quantized inner product [DQIP]
 *
 *   A[i,k] -> uA[i,k], scaleA[i], zeroA[i]   (uint8, per row)
 *   B[k,j] -> iB[k,j], scaleB[j]             (int8, per column; or given)
 *   sum    = sum_k (uA[i,k] - zeroA[i]) * iB[k,j]          (exact int32)
 *   C[i,j] = ConvertToTypeC(Activate(sum * scaleA[i] * scaleB[j] + bias[j]))
 *
 * Row quantization of A (the page names only its outputs): per row,
 * mn = min(0, min A), mx = max(0, max A), scaleA = (mx - mn) / 255,
 * zeroA = saturate_u8(rint(-mn / scaleA)), uA = saturate_u8(rint(A / scaleA)
 * + zeroA); an all-zero row takes scaleA = 1, zeroA = 0.
 * Column quantization of fp32/bf16 B: scaleB = max|B[:,j]| / 127 (or / 63
 * with avoidOverflow, range [-64,63]), iB = saturate(rint(B / scaleB)); an
 * all-zero column takes scaleB = 1.  rint rounds half to even.
 * Layouts: A is M x K, B is K x N, C is M x N, all row-major.
 * ====================================================================== */
typedef struct i8q_qgemm_ctx i8q_qgemm_ctx;

/* Init [DQIP]: create (*ctx == NULL) or re-initialize (*ctx != NULL) a
 * context on the current CUDA device.  An existing context is recreated only
 * when any argument differs from its own (sizes, types, constB, bias flag,
 * activation, avoidOverflow); otherwise it is kept with its parameters.
 *   typeA: I8Q_F32 | I8Q_BF16.  typeC: I8Q_F32 | I8Q_BF16.
 *   typeB: I8Q_F32 | I8Q_S8 (constB only) when constB; I8Q_F32 | I8Q_BF16
 *          when B is given to every Forward.
 *   activation: I8Q_ACT_*.  avoidOverflow is ignored when typeB is I8Q_S8.
 *   M, N, K >= 1 and K <= 65536 (so every int32 sum is exact).
 * Synchronous.  Errors: INVALID_ARG, UNSUPPORTED, ALLOC, CUDA; on error
 * *ctx is left as it was. */
int i8q_qgemm_dyn_init(i8q_qgemm_ctx** ctx, size_t M, size_t N, size_t K, int typeA, int typeB,
                       int typeC, int constB, int bias, int activation, int avoidOverflow);

/* Enable [DQIP]: 1 if ctx exists and Forward can be called (for constB,
 * SetParams has been called), else 0. */
int i8q_qgemm_dyn_enabled(const i8q_qgemm_ctx* ctx);

/* InternalBufferSize [DQIP]: bytes of device memory the context owns:
 * quantized B (int8 and the bf16 operand copy), column sums, B scales, bias,
 * activation parameters and the fallback scratch used when Forward gets
 * buf == NULL.  0 for a NULL ctx. */
size_t i8q_qgemm_dyn_internal_buffer_size(const i8q_qgemm_ctx* ctx);

/* ExternalBufferSize [DQIP]: bytes of the caller's scratch `buf` for
 * Forward: the quantized copy of A (uint8 and its bf16 operand copy),
 * scaleA, zeroA and, for non-constant B, its quantized copy, scales and
 * column sums.  0 for a NULL ctx. */
size_t i8q_qgemm_dyn_external_buffer_size(const i8q_qgemm_ctx* ctx);

/* Info [DQIP]: short description of the selected implementation (device
 * architecture and algorithm).  Owned by ctx, valid until the next call of
 * this function or i8q_qgemm_dyn_clear; NULL for a NULL ctx. */
const char* i8q_qgemm_dyn_info(i8q_qgemm_ctx* ctx);

/* SetParams [DQIP]: store weights, bias and activation parameters.
 *   weight: K x N, fp32 (typeB F32, quantized here per column) or int8
 *           (typeB S8, stored as given).  Required when constB; ignored
 *           (may be NULL) otherwise.
 *   scale:  N fp32 per-column scales; required when typeB is S8, else
 *           ignored.
 *   bias:   N fp32, or NULL for zeros (also ignored when Init had bias = 0).
 *   params: activation parameters, or NULL (none of I8Q_ACT_* takes any).
 * Pointers may be host or device memory (copied with cudaMemcpyDefault).
 * Synchronous: returns after the copy-in and weight preparation finished.
 * Errors: NOT_INITIALIZED, INVALID_ARG, CUDA. */
int i8q_qgemm_dyn_set_params(i8q_qgemm_ctx* ctx, const void* weight, const float* scale,
                             const float* bias, const float* params, void* stream);

/* Forward [DQIP]: C = dynamic quantized product of A and B.
 *   A: M x K of typeA.  B: K x N of typeB, or NULL when constB.
 *   buf: device scratch of at least i8q_qgemm_dyn_external_buffer_size
 *        bytes, 256-byte aligned, or NULL to use the context's own.
 *   C: M x N of typeC.
 * A, B and C are device pointers.  Asynchronous on stream; concurrent
 * Forward calls on one context must use distinct buf (a NULL buf is shared).
 * Errors: NOT_INITIALIZED, INVALID_ARG, CUDA. */
int i8q_qgemm_dyn_forward(i8q_qgemm_ctx* ctx, const void* A, const void* B, void* buf, void* C,
                          void* stream);

/* Same as Forward, but A and C are HOST pointers (pinned for asynchronous
 * copies, or pageable): A is copied to context-owned device staging memory,
 * the product runs, and C is copied back; returns after C is in host
 * memory.  Work already queued on `stream` runs first.  With M >= 2048 the
 * call is pipelined over up to 8 row chunks (rows are independent: A is
 * quantized per row and B is constant) on streams owned by the context, so
 * one chunk's upload, another's product and a third's download overlap;
 * results are those of Forward, bit for bit.  Not on the pages: it is the
 * whole host-to-host path of Forward for callers that keep their tensors in
 * host memory.  B must be NULL (constB contexts).  Calls on one context must
 * not overlap. */
int i8q_qgemm_dyn_forward_host(i8q_qgemm_ctx* ctx, const void* A_host, void* C_host, void* stream);

/* Test hook, not on the pages: run Forward's quantization and integer
 * product, and write the exact int32 sums sum_k (uA - zeroA) * iB (M x N)
 * to acc instead of the float epilogue.  Same arguments as Forward. */
int i8q_qgemm_dyn_forward_s32(i8q_qgemm_ctx* ctx, const void* A, const void* B, void* buf,
                              int32_t* acc, void* stream);

/* Test hook, not on the pages: device addresses, inside `buf` (or the
 * context's fallback scratch when buf is NULL), of the quantized A written
 * by the last Forward: uA (M x K uint8, row stride *lda bytes), scaleA (M
 * fp32) and zeroA (M int32).  Any output pointer may be NULL. */
int i8q_qgemm_dyn_buf_views(i8q_qgemm_ctx* ctx, void* buf, uint8_t** uA, size_t* lda, float** scaleA,
                            int32_t** zeroA);

/* Test hook, not on the pages: device addresses of the quantized B --
 * the stored constant B, or the B the last Forward quantized into `buf`
 * (or the fallback scratch when buf is NULL) -- transposed to N rows of K
 * codes (row stride *ldb elements): *iBt as int8 and *iBt_bf16 as bf16
 * holding the same integers, either set to NULL when that copy is not kept
 * (a non-constant B keeps only the copy its product reads); its N fp32
 * scales and N int32 column sums.  Any output pointer may be NULL. */
int i8q_qgemm_dyn_weight_views(i8q_qgemm_ctx* ctx, void* buf, int8_t** iBt, void** iBt_bf16, size_t* ldb,
                               float** scaleB, int32_t** colsum);

/* Clear [DQIP]: release the context and everything it owns; *ctx = NULL.
 * Synchronizes the device first.  NULL or *ctx == NULL is a no-op. */
void i8q_qgemm_dyn_clear(i8q_qgemm_ctx** ctx);

/* Allocation-free dynamic quantized inner product.  The pages have no
 * counterpart: it exists for callers that may not allocate device memory --
 * code running inside a host application that owns all device memory
 * through its own pool (a plugin, for instance), or code that cannot take
 * cudaMalloc/cudaFree's possible device synchronization -- and so can
 * neither create a context nor pass a scratch buffer of their own.
 *
 * Same result as a context with constB, typeB = I8Q_S8 (B given already
 * quantized, with its per-column scales) followed by Forward:
 *   A: M x K (typeA F32|BF16); B: K x N int8 row-major; scaleB: N fp32;
 *   bias: N fp32 or NULL; activation: I8Q_ACT_*; C: M x N (typeC F32|BF16).
 * All device pointers.  Every intermediate (uint8 A with its row scales and
 * zero points, B transposed with its column sums) lives in one file-scope
 * device array of I8Q_QGEMM_STATIC_SCRATCH_BYTES (32 MiB), held by every GPU
 * that loads the library until the process exits; sizes whose
 * i8q_qgemm_dyn_static_scratch_bytes exceed it are rejected with
 * I8Q_ERR_UNSUPPORTED.  The call allocates nothing.  The first call on each
 * device looks up the array's device address (cudaGetSymbolAddress) with
 * that device current; make that first call before any stream capture.
 * All calls share the one array: calls that overlap on the GPU (other
 * streams, other host threads) race and corrupt each other's results.
 * Asynchronous on stream. */
#define I8Q_QGEMM_STATIC_SCRATCH_BYTES ((size_t)32 << 20)
int i8q_qgemm_dyn_static(size_t M, size_t N, size_t K, int typeA, const void* A, const int8_t* B,
                         const float* scaleB, const float* bias, int activation, int typeC, void* C,
                         void* stream);

/* Bytes of the static array i8q_qgemm_dyn_static uses for these sizes. */
size_t i8q_qgemm_dyn_static_scratch_bytes(size_t M, size_t N, size_t K);

/* Size of the static array (I8Q_QGEMM_STATIC_SCRATCH_BYTES). */
size_t i8q_qgemm_dyn_static_scratch_capacity(void);

/* ========================================================================
 * QuantizeLinear [QL] and DequantizeLinear [DQL]
 *
 * x has `rank` dims given by the HOST array `shape` (rank 0..8).  Per-tensor
 * (axis == I8Q_NO_AXIS): n_scale == 1.  Per-axis: axis in [-rank, rank-1]
 * and n_scale == shape[axis].  Scale and zero point are device arrays of
 * n_scale entries; the zero point has the quantized type.
 * ====================================================================== */

/* QuantizeLinear [QL]: y = saturate(rint(x / y_scale) + y_zero_point),
 * rint = round half to even, saturating to [0,255] (ytype I8Q_U8) or
 * [-128,127] (I8Q_S8).  x: fp32.  y: same shape, ytype.  Scales must be
 * finite and nonzero for defined results. */
int i8q_quantize_linear(const float* x, const int64_t* shape, int rank, int axis, const float* y_scale,
                        const void* y_zero_point, size_t n_scale, int ytype, void* y, void* stream);

/* DequantizeLinear [DQL]: y = (x - x_zero_point) * x_scale, fp32 output.
 * x: xtype I8Q_U8 or I8Q_S8. */
int i8q_dequantize_linear(const void* x, int xtype, const int64_t* shape, int rank, int axis,
                          const float* x_scale, const void* x_zero_point, size_t n_scale, float* y,
                          void* stream);

/* ========================================================================
 * QLinearConv [QLC], 2-D, NCHW
 *
 *   acc = sum_{c in group, kh, kw} (x - x_zero_point) * (w - w_zero_point[m])
 *         (a position outside x holds real 0, i.e. x_zero_point)
 *   acc += B[m]   (int32 bias, scale x_scale*w_scale[m], zero point 0)
 *   y = saturate(rint(((float)acc * (x_scale * w_scale[m])) / y_scale) + y_zero_point)
 * The page gives no requantization formula; this is DequantizeLinear of the
 * accumulator followed by QuantizeLinear with (y_scale, y_zero_point).
 *   x: xtype (U8|S8) [N, C, H, W].  w: wtype (U8|S8) [M, C/group, kH, kW].
 *   w_scale / w_zero_point: n_w == 1 (per tensor) or n_w == M entries
 *   (device; the zero point has type wtype).  B: int32 [M] or NULL.
 *   pads {top, left, bottom, right} >= 0; strides, dilations {h, w} >= 1;
 *   C == w.shape[1] * group, M % group == 0.
 *   y: ytype (U8|S8) [N, M, OH, OW], OH = (H + pt + pb - dh*(kH-1) - 1)/sh + 1.
 * workspace: device scratch of at least i8q_qlinearconv_workspace_size
 * bytes (may be NULL when that size is 0), 256-byte aligned. */
int i8q_qlinearconv(const void* x, int xtype, const int64_t* xshape, float x_scale, int x_zero_point,
                    const void* w, int wtype, const int64_t* wshape, const float* w_scale,
                    const void* w_zero_point, size_t n_w, float y_scale, int y_zero_point,
                    const int32_t* B, const int64_t* pads, const int64_t* strides,
                    const int64_t* dilations, int64_t group, void* y, int ytype, void* workspace,
                    size_t ws_bytes, void* stream);

/* Scratch bytes i8q_qlinearconv needs for these shapes (host arrays as in
 * i8q_qlinearconv).  Returns 0 on invalid shapes. */
size_t i8q_qlinearconv_workspace_size(const int64_t* xshape, const int64_t* wshape, const int64_t* pads,
                                      const int64_t* strides, const int64_t* dilations, int64_t group);

/* ========================================================================
 * QGemm [QG] (ONNX Runtime contrib schemas, "QGemm", inputs A .. y_zero_point
 * and attributes transA, transB, alpha):
 *   acc[i,j] = sum_k (A[i,k] - a_zero_point) * (B[k,j] - b_zero_point[j])
 *   acc += C[i,j]            (int32; scale alpha * a_scale * b_scale, zp 0)
 *   y = (float)acc * ((alpha * a_scale) * b_scale[j])
 *   quantized output: y = saturate(rint(y / y_scale) + y_zero_point)
 * The schema gives C the scale alpha / beta * a_scale * b_scale but defines
 * no beta; it is read as 1.  The rescale is DequantizeLinear of the integer
 * sum, then QuantizeLinear (the schema gives no formula).
 *   A: device, atype (U8|S8) codes, (M, K) row-major, or (K, M) if transA.
 *   a_scale, a_zero_point: per-tensor scalars (host values); a_zero_point
 *   within A's range.
 *   B: device, btype (U8|S8) codes, (K, N) row-major, or (N, K) if transB.
 *   b_scale: device fp32, n_b == 1 (per tensor) or N (per column) entries.
 *   b_zero_point: device, btype, n_b entries, or NULL (zero).
 *   C: device int32 (c_rows, c_cols) row-major with c_rows in {1, M} and
 *   c_cols in {1, N}, broadcast to (M, N); or NULL.
 *   quantize_y == 0: Y is fp32 (M, N).  Otherwise Y holds ytype (U8|S8)
 *   codes with y_scale / y_zero_point (host values).
 *   workspace: device scratch of at least i8q_qgemm_workspace_size bytes,
 *   256-byte aligned (the centred bf16 operands, their sums and the column
 *   parameters); the caller owns it and all tensors.
 * Errors: INVALID_ARG (types, ranges, shapes, workspace), UNSUPPORTED
 * (K > 65536), CUDA. */
int i8q_qgemm(const void* A, int atype, int transA, int64_t M, int64_t K, float a_scale, int a_zero_point,
              const void* B, int btype, int transB, int64_t N, const float* b_scale, const void* b_zero_point,
              size_t n_b, const int32_t* C, int64_t c_rows, int64_t c_cols, float alpha, int quantize_y,
              float y_scale, int y_zero_point, int ytype, void* Y, void* workspace, size_t ws_bytes, void* stream);

/* Scratch bytes i8q_qgemm needs for M x N x K (0 for sizes below 1). */
size_t i8q_qgemm_workspace_size(int64_t M, int64_t N, int64_t K);

/* ========================================================================
 * MatMulIntegerToFloat [MITF]:
 *   acc[i,j] = sum_k (A[i,k] - a_zero_point[i]) * (B[k,j] - b_zero_point[j])
 *   Y[i,j]   = (float)acc * (a_scale[i] * b_scale[j]) + bias[j]
 *   A: device, atype (U8|S8) codes (M, K) row-major (the leading dimensions
 *   of an N-dimensional A flattened into M).  B: device, btype (U8|S8)
 *   (K, N) row-major.
 *   a_scale: device fp32, n_a == 1 (per tensor) or M (per row of A) entries;
 *   a_zero_point: device, atype, n_a entries, or NULL (zero).  The schema
 *   repeats B's "per-column" sentence for A; a scale per summation index
 *   cannot leave the integer sum, so A's parameters are read as per tensor
 *   or per row.
 *   b_scale: device fp32, n_b == 1 or N entries; b_zero_point: device,
 *   btype, n_b entries, or NULL.  bias: device fp32 [N] or NULL.
 *   Y: device fp32 (M, N).
 *   workspace: at least i8q_matmul_integer_workspace_size bytes, 256-byte
 *   aligned.
 * Errors: INVALID_ARG, UNSUPPORTED (K > 65536), CUDA. */
int i8q_matmul_integer_to_float(const void* A, int atype, int64_t M, int64_t K, const void* B, int btype, int64_t N,
                                const float* a_scale, const void* a_zero_point, size_t n_a, const float* b_scale,
                                const void* b_zero_point, size_t n_b, const float* bias, float* Y, void* workspace,
                                size_t ws_bytes, void* stream);

/* DynamicQuantizeMatMul [MITF]: fp32 A (M, K) is quantized to uint8 per
 * tensor (the schema names no method; the formula is that of a row of the
 * dynamic inner product applied to the whole tensor: range widened to
 * contain 0, scale = (max - min) / 255, zero point = saturate(rint(-min /
 * scale)), codes = saturate(rint(A / scale) + zero point)), then
 * MatMulIntegerToFloat with B's parameters as above.  a_scale_out (device
 * fp32, 1 entry) and a_zero_point_out (device uint8, 1 entry) receive the
 * computed parameters when not NULL.  Same workspace as
 * i8q_matmul_integer_to_float. */
int i8q_dynamic_quantize_matmul(const float* A, int64_t M, int64_t K, const void* B, int btype, int64_t N,
                                const float* b_scale, const void* b_zero_point, size_t n_b, const float* bias,
                                float* Y, float* a_scale_out, uint8_t* a_zero_point_out, void* workspace,
                                size_t ws_bytes, void* stream);

/* Scratch bytes of i8q_matmul_integer_to_float / i8q_dynamic_quantize_matmul
 * for M x N x K (0 for sizes below 1). */
size_t i8q_matmul_integer_workspace_size(int64_t M, int64_t N, int64_t K);

/* ========================================================================
 * Quantized elementwise operators [QEW].  Scales and zero points are
 * per-tensor scalars (host values); zero points lie in their type's range.
 * A and B broadcast Numpy-style (shapes right-aligned, size-1 dimensions
 * repeat; ranks 0..8); the caller allocates C with the broadcast shape,
 * row-major.  A, B, C, X, Y are device pointers.  Errors: INVALID_ARG. */
#define I8Q_QLINEAR_ADD 0
#define I8Q_QLINEAR_MUL 1
#define I8Q_QLINEAR_LEAKY_RELU 0
#define I8Q_QLINEAR_SIGMOID 1

/* QLinearAdd / QLinearMul, A, B and C all of qtype (U8|S8):
 *   add: C = (A_scale * (A - A_zp) + B_scale * (B - B_zp)) / C_scale + C_zp
 *   mul: C = ((A - A_zp) * (B - B_zp)) * (A_scale * B_scale) / C_scale + C_zp
 * evaluated in the order written (fp32, each operation rounded once), then
 * round half to even and saturation.  Large outputs go through the table of
 * all 256 x 256 codes; the library keeps up to 16 such tables (64 KB each,
 * in static device memory of each GPU that loads it) for parameter sets
 * seen before, and computes the table inside the call otherwise. */
int i8q_qlinear_binary(int op, const void* A, const int64_t* a_shape, int a_rank, float a_scale, int a_zero_point,
                       const void* B, const int64_t* b_shape, int b_rank, float b_scale, int b_zero_point,
                       float c_scale, int c_zero_point, int qtype, void* C, void* stream);

/* MulInteger: C (int32) = (A - A_zp) * (B - B_zp); atype, btype U8|S8. */
int i8q_mul_integer(const void* A, int atype, const int64_t* a_shape, int a_rank, int a_zero_point, const void* B,
                    int btype, const int64_t* b_shape, int b_rank, int b_zero_point, int32_t* C, void* stream);

/* QLinearLeakyRelu (alpha used) / QLinearSigmoid on n codes of qtype:
 *   d = (x - x_zp) * x_scale;  f = alpha * d if d < 0 else d  |  1 / (1 + exp(-d))
 *   y = saturate(rint(f / y_scale) + y_zp).
 * The sigmoid is the library's fixed-sequence fp32 function (see
 * I8Q_LSTM_ACT_SIGMOID), so the codes do not depend on a math library. */
int i8q_qlinear_unary(int op, const void* X, int64_t n, int qtype, float x_scale, int x_zero_point, float y_scale,
                      int y_zero_point, float alpha, void* Y, void* stream);

/* ========================================================================
 * DynamicQuantizeLSTM [LSTM]: int8 W and R with per-channel (or
 * per-direction) scales and zero point 0, fp32 X, default activations
 * (sigmoid for i, o, f; tanh for the cell candidate and the output), gate
 * column order i, o, f, c; no peepholes, no sequence_lens, no clip,
 * input_forget = 0.  X and each step's hidden state are quantized per row
 * to uint8 exactly as A of the dynamic quantized inner product.
 *   Per direction d and step t (t runs T-1..0 for the reverse direction):
 *   Gx = X_t W[d] (dequantized), Gh = h_{t-1} R[d] (dequantized),
 *   g = ((Gx + Gh) + Wb) + Rb; i,o,f = sigmoid; ct = tanh;
 *   c = f*c_{t-1} + i*ct; h = o*tanh(c).
 *   X [T, batch, input]; W [D, input, 4H]; R [D, H, 4H] (int8);
 *   W_scale, R_scale: n == D (per direction) or D*4H (per channel) fp32;
 *   W_zero_point, R_zero_point: int8, n entries, all zero, or NULL;
 *   Bias [D, 8H] or NULL; h0, c0 [D, batch, H] or NULL (zeros);
 *   Y [T, D, batch, H], Y_h, Y_c [D, batch, H]; any output may be NULL.
 *   D = 2 for I8Q_LSTM_BIDIRECTIONAL, else 1.
 * Nonzero zero points are taken as in i8q_dq_lstm_forward_ex.
 * workspace: at least i8q_dq_lstm_workspace_size bytes, 256-byte aligned.
 * Errors: INVALID_ARG, CUDA. */
int i8q_dq_lstm_forward(const float* X, int64_t T, int64_t batch, int64_t input, int64_t hidden,
                        int direction, const int8_t* W, const float* W_scale, const int8_t* W_zero_point,
                        size_t n_wscale, const int8_t* R, const float* R_scale,
                        const int8_t* R_zero_point, size_t n_rscale, const float* Bias, const float* h0,
                        const float* c0, float* Y, float* Y_h, float* Y_c, void* workspace,
                        size_t ws_bytes, void* stream);

size_t i8q_dq_lstm_workspace_size(int64_t T, int64_t batch, int64_t input, int64_t hidden, int direction);

/* DynamicQuantizeLSTM [LSTM] with the schema's optional inputs and
 * attributes ("activations", "activation_alpha", "activation_beta", "clip",
 * "input_forget"; graiphic.io "DynamicQuantizeLSTM", attributes).
 *   W, R: device codes of wtype (I8Q_S8 | I8Q_U8), shapes as above.
 *   W_zero_point, R_zero_point: device codes of wtype, n_wscale / n_rscale
 *   entries (per direction or per channel, in iofc column order), or NULL.
 *   sequence_lens: device int32 [batch] or NULL.  Row b runs t = 0..L-1
 *   (forward) or L-1..0 (reverse) with L = sequence_lens[b] clamped to
 *   [0, T]; Y is 0 from t = L on; Y_h, Y_c hold the row's last state.
 *   P: device fp32 [D, 3H] peepholes (Pi, Po, Pf) or NULL.
 *   clip > 0 bounds every gate input to [-clip, clip]; clip <= 0: no clip.
 *   input_forget != 0: f = 1 - i.
 *   activations: host array of n_activations I8Q_LSTM_ACT_* values, 3 per
 *   direction (f, g, h; forward first), or NULL / 0 for Sigmoid, Tanh, Tanh.
 *   activation_alpha / activation_beta: host arrays (n_alpha, n_beta values,
 *   may be 0), consumed in the order of the activation functions: each
 *   function that takes an alpha (beta) takes the next unused value, or its
 *   ONNX operator's default when the list runs out (LeakyRelu 0.01,
 *   ThresholdedRelu 1, HardSigmoid 0.2 / 0.5, Elu 1, Affine 1 / 0,
 *   ScaledTanh 1 / 1).
 *   Gate terms are summed in the order of the ONNX LSTM equations:
 *   i = f(clip(X Wi + H Ri + Pi*C_prev + Wbi + Rbi)),
 *   f = f(clip(X Wf + H Rf + Pf*C_prev + Wbf + Rbf)),
 *   c~ = g(clip(X Wc + H Rc + Wbc + Rbc)), C = f*C_prev + i*c~,
 *   o = f(clip(X Wo + H Ro + Po*C + Wbo + Rbo)), H = o*h(C),
 *   where X W and H R are the dequantized products of the per-row uint8
 *   codes with (W - W_zero_point), (R - R_zero_point).
 * Same workspace as i8q_dq_lstm_forward.  Errors: INVALID_ARG (also for an
 * activation outside the list or a wrong count), CUDA. */
int i8q_dq_lstm_forward_ex(const float* X, int64_t T, int64_t batch, int64_t input, int64_t hidden, int direction,
                           const void* W, const void* R, int wtype, const float* W_scale, const void* W_zero_point,
                           size_t n_wscale, const float* R_scale, const void* R_zero_point, size_t n_rscale,
                           const float* Bias, const int32_t* sequence_lens, const float* h0, const float* c0,
                           const float* P, float clip, int input_forget, const int* activations,
                           size_t n_activations, const float* activation_alpha, size_t n_alpha,
                           const float* activation_beta, size_t n_beta, float* Y, float* Y_h, float* Y_c,
                           void* workspace, size_t ws_bytes, void* stream);

/* Test hook (not on the pages): where, inside the workspace of a completed
 * i8q_dq_lstm_forward / _ex call with these shape arguments, the per-row
 * uint8 quantization of a hidden state lies.  which = 0: the state the
 * last step read (h after T-1 steps; h0 when T == 1); which = 1: the final
 * state (Y_h).  *codes: device bf16 values uh - 128 (exact integers),
 * [D * batch rows][*row_stride elements], the first `hidden` of each row
 * meaningful, rows ordered direction-major; *scale, *zero: device fp32 and
 * int32 [D * batch].  Valid until the workspace is reused.  Synchronize
 * the call's stream before reading.  Errors: INVALID_ARG. */
int i8q_dq_lstm_state_codes(const void* workspace, int64_t T, int64_t batch, int64_t input, int64_t hidden,
                            int direction, int which, const void** codes, const float** scale, const int32_t** zero,
                            int64_t* row_stride);

/* ========================================================================
 * Measurement (not on the pages)
 * ====================================================================== */

/* Kernel timing.  While enabled, every kernel launch of this library is
 * bracketed by CUDA events on its launch stream.  Enabling (or disabling)
 * drops all records.  Single-threaded use. */
int i8q_profile_enable(int on);

/* Synchronize the device, fold the records into per-kernel totals and
 * return the number of distinct kernel names (or a negative error). */
int i8q_profile_collect(void);

/* Totals of kernel i (0 <= i < count): name (owned by the library, valid
 * until the next enable), number of launches, summed event time in ms. */
int i8q_profile_entry(int i, const char** name, long long* launches, double* total_ms);

/* Throughput of back-to-back mma.sync m16n8k32 u8 x s8 -> s32 on every SM
 * (the int8 tensor instruction sm_103a accepts), `iters` rounds of 8 MMAs
 * per warp.  Synchronous.  *tops receives 10^12 integer ops per second,
 * counting a multiply-add as 2 ops. */
int i8q_measure_int8_mma_peak(int64_t iters, void* stream, double* tops);

/* Synchronize `stream` and report any error recorded by a device-side
 * bounded wait since the last call (I8Q_ERR_DEVICE_TIMEOUT), or a pending
 * CUDA error (I8Q_ERR_CUDA).  Clears the recorded state. */
int i8q_sync_status(void* stream);

/* Failure-detection probe (not on the pages): launch one small kernel on
 * `stream` that runs one of the library's bounded device waits, with a
 * limit of limit_ns nanoseconds (1 us .. 1 s), on an event that never
 * comes: kind 0, an mbarrier phase nobody arrives on (the waits of the
 * tcgen05 pipelines); kind 1, a grid barrier whose other CTAs never arrive
 * (the persistent LSTM's).  The wait gives up, records the timeout in the
 * device status word and the kernel returns, so the next i8q_sync_status
 * reports I8Q_ERR_DEVICE_TIMEOUT and the context stays usable.  Nothing
 * else is in flight in the probe.  Errors: INVALID_ARG, CUDA. */
int i8q_debug_wait_timeout(int kind, int64_t limit_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* I8Q_H */
