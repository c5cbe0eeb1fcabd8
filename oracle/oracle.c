/*
 * oracle.c -- plain, slow CPU oracle for linear int8 quantization and the
 * quantized products it feeds.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may load or call
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header, table or helper with the CUDA library.
 *
 * Every function is a direct restatement of the operator text it cites, in
 * the order of operations the text gives.  Floating point is IEEE fp32 where
 * the operator is defined on fp32 (the scales, the division x / scale, the
 * dequantization products); each operation rounds once, to nearest even.
 * The build uses -O2 -ffp-contract=off and no fast-math so the compiler
 * neither fuses a multiply into an add nor reorders anything.  Integer sums
 * are carried in int64 and checked to fit the int32 the operators name.
 *
 * Sources (page title, section):
 *  [QL]  ONNX Runtime contrib schemas, "QuantizeLinear" (ver 1) doc string
 *  [DQL] ONNX Runtime contrib schemas, "DequantizeLinear" (ver 1) doc string
 *  [DQIP] Simd, "SynetDynamicQuantizedInnerProduct16b", Detailed Description
 *         (algorithm listing, typeB/avoidOverflow paragraph) and the
 *         Init()/SetParams()/Forward() member documentation
 *  [QLC] onnx-light docs, "QLinearConv" (inputs, bias rule, examples)
 *  [LSTM] ONNX Runtime contrib schemas, "DynamicQuantizeLSTM" (inputs W, R, B,
 *         initial_h/c, outputs Y, Y_h, Y_c); graiphic.io "DynamicQuantizeLSTM"
 *  [QG]  ONNX Runtime contrib schemas, "QGemm" (inputs A .. y_zero_point,
 *         attributes transA, transB, alpha)
 *  [MITF] ONNX Runtime contrib schemas, "MatMulIntegerToFloat" and
 *         "DynamicQuantizeMatMul" (inputs A, B, scales, zero points, bias)
 *  [QEW] ONNX Runtime contrib schemas, "MulInteger", "QLinearAdd",
 *         "QLinearMul" (doc formulas, Numpy-style broadcasting),
 *         "QLinearLeakyRelu", "QLinearSigmoid" (doc strings)
 *
 * Where the pages leave a step open the readings used are listed in the
 * repository's design notes; each is restated at the function below.
 */
#include <fenv.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_ERR_ROUNDING -1
#define OR_ERR_OVERFLOW -2
#define OR_ERR_ARG -3

#define OR_U8 0
#define OR_S8 1

#define OR_ACT_IDENTITY 0
#define OR_ACT_RELU 1
#define OR_ACT_GELU 2

static int rounding_is_nearest(void) { return fegetround() == FE_TONEAREST; }

/* rintf gives the nearest integer, ties to even, under FE_TONEAREST.
 * The result is held in a double so values far outside int32 saturate
 * correctly instead of overflowing a conversion. */
static int64_t sat_rint_plus(float v, int64_t zp, int64_t lo, int64_t hi) {
  double r = (double)rintf(v) + (double)zp;
  if (r < (double)lo) return lo;
  if (r > (double)hi) return hi;
  return (int64_t)r;
}

static int64_t q_lo(int t) { return t == OR_U8 ? 0 : -128; }
static int64_t q_hi(int t) { return t == OR_U8 ? 255 : 127; }

static int64_t load_q(const void* p, int t, int64_t i) {
  return t == OR_U8 ? (int64_t)((const uint8_t*)p)[i] : (int64_t)((const int8_t*)p)[i];
}

static void store_q(void* p, int t, int64_t i, int64_t v) {
  if (t == OR_U8)
    ((uint8_t*)p)[i] = (uint8_t)v;
  else
    ((int8_t*)p)[i] = (int8_t)v;
}

/* [QL]: y = saturate(round_half_even(x / y_scale) + y_zero_point), saturating
 * to [0,255] for uint8 and [-128,127] for int8.  The tensor is viewed as
 * [outer, axis_len, inner]; with per_axis the scale and zero point are picked
 * by the middle index (the 'axis' attribute), otherwise element 0 is used
 * for every element (per tensor). */
int or_quantize_linear(const float* x, int64_t outer, int64_t axis_len, int64_t inner,
                       const float* y_scale, const int32_t* y_zero_point, int per_axis,
                       int ytype, void* y) {
  if (!rounding_is_nearest()) return OR_ERR_ROUNDING;
  if (ytype != OR_U8 && ytype != OR_S8) return OR_ERR_ARG;
  int64_t lo = q_lo(ytype), hi = q_hi(ytype);
#pragma omp parallel for schedule(static)
  for (int64_t o = 0; o < outer; ++o) {
    for (int64_t a = 0; a < axis_len; ++a) {
      int64_t c = per_axis ? a : 0;
      float s = y_scale[c];
      int64_t zp = y_zero_point[c];
      for (int64_t n = 0; n < inner; ++n) {
        int64_t i = (o * axis_len + a) * inner + n;
        float q = x[i] / s;
        store_q(y, ytype, i, sat_rint_plus(q, zp, lo, hi));
      }
    }
  }
  return OR_OK;
}

/* [DQL]: y = (x - x_zero_point) * x_scale, output float.  The integer
 * difference is exact and converts to float exactly (|x - zp| <= 510). */
int or_dequantize_linear(const void* x, int xtype, int64_t outer, int64_t axis_len, int64_t inner,
                         const float* x_scale, const int32_t* x_zero_point, int per_axis, float* y) {
  if (xtype != OR_U8 && xtype != OR_S8) return OR_ERR_ARG;
#pragma omp parallel for schedule(static)
  for (int64_t o = 0; o < outer; ++o) {
    for (int64_t a = 0; a < axis_len; ++a) {
      int64_t c = per_axis ? a : 0;
      float s = x_scale[c];
      int64_t zp = x_zero_point[c];
      for (int64_t n = 0; n < inner; ++n) {
        int64_t i = (o * axis_len + a) * inner + n;
        float d = (float)(load_q(x, xtype, i) - zp);
        y[i] = d * s;
      }
    }
  }
  return OR_OK;
}

/* [DQIP] step "A[i,k] -> uA[i,k], scaleA[i], zeroA[i]".  The page names only
 * the outputs; the reading used (asymmetric uint8 per row, range widened to
 * contain 0) is:
 *   mn = min(0, min_k A[i,k]),  mx = max(0, max_k A[i,k])
 *   scaleA = (mx - mn) / 255                      (fp32 division)
 *   zeroA  = saturate_u8(round_half_even(-mn / scaleA))
 *   uA     = saturate_u8(round_half_even(A / scaleA) + zeroA)
 * The last line is [QL] applied with the row's scale and zero point.
 * Degenerate row (scaleA == 0, i.e. the row is all zeros): scaleA = 1,
 * zeroA = 0, so every uA is 0. */
int or_quantize_rows_u8(const float* A, int64_t M, int64_t K, uint8_t* uA, float* scaleA,
                        int32_t* zeroA) {
  if (!rounding_is_nearest()) return OR_ERR_ROUNDING;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < M; ++i) {
    const float* a = A + i * K;
    float mn = 0.0f, mx = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
      if (a[k] < mn) mn = a[k];
      if (a[k] > mx) mx = a[k];
    }
    float s = (mx - mn) / 255.0f;
    int64_t z;
    if (s == 0.0f) {
      s = 1.0f;
      z = 0;
    } else {
      z = sat_rint_plus(-mn / s, 0, 0, 255);
    }
    scaleA[i] = s;
    zeroA[i] = (int32_t)z;
    for (int64_t k = 0; k < K; ++k) uA[i * K + k] = (uint8_t)sat_rint_plus(a[k] / s, z, 0, 255);
  }
  return OR_OK;
}

/* [DQIP] step "B[k,j] -> iB[k,j], scaleB[j]" with the typeB/avoidOverflow
 * paragraph: int8 in [-128,127], or the narrowed [-64,63] when avoidOverflow
 * is set.  Reading: symmetric per column, zero point 0,
 *   scaleB = max_k |B[k,j]| / qmax       (qmax = 127, or 63 narrowed)
 *   iB     = saturate(round_half_even(B / scaleB))
 * Degenerate column (all zeros): scaleB = 1, iB = 0.  B is K x N row-major. */
int or_quantize_cols_s8(const float* B, int64_t K, int64_t N, int avoid_overflow, int8_t* iB,
                        float* scaleB) {
  if (!rounding_is_nearest()) return OR_ERR_ROUNDING;
  const int64_t qmax = avoid_overflow ? 63 : 127;
  const int64_t qmin = avoid_overflow ? -64 : -128;
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < N; ++j) {
    float m = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
      float v = fabsf(B[k * N + j]);
      if (v > m) m = v;
    }
    float s = m / (float)qmax;
    if (s == 0.0f) s = 1.0f;
    scaleB[j] = s;
    for (int64_t k = 0; k < K; ++k)
      iB[k * N + j] = (int8_t)sat_rint_plus(B[k * N + j] / s, 0, qmin, qmax);
  }
  return OR_OK;
}

/* GELU, x * Phi(x) = 0.5 * x * (1 + erf(x / sqrt(2))), in fp32.  Evaluated
 * as (0.5 * x) * erfc(-(x * (1/sqrt(2)))): the same function, written with
 * the complementary error function so that no 1 + erf(.) cancels for
 * negative x. */
static float gelu_f32(float x) {
  float t = x * 0.70710678118654752440f;
  float e = erfcf(-t);
  float h = 0.5f * x;
  return h * e;
}

static float activate(float v, int act) {
  switch (act) {
    case OR_ACT_RELU: return v > 0.0f ? v : 0.0f;
    case OR_ACT_GELU: return gelu_f32(v);
    default: return v;
  }
}

/* [DQIP] algorithm listing, for the rows listed in `rows` (all rows when
 * rows == NULL):
 *   sum = sum_k (uA[i,k] - zeroA[i]) * iB[k,j]        (integer)
 *   val = sum * scaleA[i] * scaleB[j]                  (left to right, fp32)
 *   C[i,j] = Activate(val + bias[j])
 * uA is M x K row-major, iB is K x N row-major.  The sum is carried in int64
 * and must fit int32; its conversion to fp32 rounds to nearest even.
 * acc_out (optional) receives the int32 sums, C_out the fp32 results,
 * both nrows x N. */
int or_qgemm_dyn_rows(const uint8_t* uA, const int32_t* zeroA, const float* scaleA,
                      const int8_t* iB, const float* scaleB, const float* bias, int act,
                      int64_t M, int64_t N, int64_t K, const int64_t* rows, int64_t nrows,
                      int32_t* acc_out, float* C_out) {
  if (!rounding_is_nearest()) return OR_ERR_ROUNDING;
  int err = OR_OK;
  if (rows == NULL) nrows = M;
#pragma omp parallel for schedule(dynamic, 1) reduction(min : err)
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t i = rows ? rows[r] : r;
    if (i < 0 || i >= M) {
      err = OR_ERR_ARG;
      continue;
    }
    for (int64_t j = 0; j < N; ++j) {
      int64_t sum = 0;
      for (int64_t k = 0; k < K; ++k)
        sum += ((int64_t)uA[i * K + k] - (int64_t)zeroA[i]) * (int64_t)iB[k * N + j];
      if (sum > INT32_MAX || sum < INT32_MIN) {
        err = OR_ERR_OVERFLOW;
        continue;
      }
      if (acc_out) acc_out[r * N + j] = (int32_t)sum;
      float val = (float)(int32_t)sum;
      val = val * scaleA[i];
      val = val * scaleB[j];
      if (bias) val = val + bias[j];
      C_out[r * N + j] = activate(val, act);
    }
  }
  return err;
}

/* Conversion of fp32 to bf16, round to nearest even on the upper 16 bits
 * (the conversion the output type bf16 implies).  NaN maps to a quiet NaN. */
void or_f32_to_bf16(const float* x, int64_t n, uint16_t* y) {
  for (int64_t i = 0; i < n; ++i) {
    uint32_t u;
    memcpy(&u, &x[i], 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) {
      y[i] = (uint16_t)((u >> 16) | 0x40u);
      continue;
    }
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    y[i] = (uint16_t)(u >> 16);
  }
}

/* [QLC] 2-D QLinearConv on NCHW tensors.
 *   acc[n,m,oh,ow] = sum over c in m's group, kh, kw of
 *                    (x[n,c,ih,iw] - x_zero_point) * (w[m,c',kh,kw] - w_zero_point[m])
 *   with ih = oh*stride_h - pad_top + kh*dil_h (likewise iw).  A position
 *   outside the input holds real 0, i.e. the quantized value x_zero_point,
 *   so it adds nothing.
 *   acc += B[m]            (bias quantized with scale x_scale*w_scale, zp 0)
 *   y = saturate(round_half_even(((float)acc * (x_scale * w_scale[m])) / y_scale)
 *                + y_zero_point)
 * The last line dequantizes the accumulator and applies QuantizeLinear with
 * (y_scale, y_zero_point); the page gives no formula of its own.
 * pads = {top, left, bottom, right}; strides, dilations = {h, w}.
 * w_scale / w_zero_point hold M entries when per_channel, else one. */
int or_qlinearconv(const void* x, int xtype, int64_t N, int64_t C, int64_t H, int64_t W,
                   float x_scale, int32_t x_zero_point, const void* w, int wtype, int64_t M,
                   int64_t kH, int64_t kW, const float* w_scale, const int32_t* w_zero_point,
                   int per_channel, float y_scale, int32_t y_zero_point, const int32_t* B,
                   const int64_t* pads, const int64_t* strides, const int64_t* dilations,
                   int64_t group, void* y, int ytype) {
  if (!rounding_is_nearest()) return OR_ERR_ROUNDING;
  if (group <= 0 || C % group != 0 || M % group != 0) return OR_ERR_ARG;
  const int64_t Cg = C / group, Mg = M / group;
  const int64_t OH = (H + pads[0] + pads[2] - ((kH - 1) * dilations[0] + 1)) / strides[0] + 1;
  const int64_t OW = (W + pads[1] + pads[3] - ((kW - 1) * dilations[1] + 1)) / strides[1] + 1;
  if (OH <= 0 || OW <= 0) return OR_ERR_ARG;
  const int64_t lo = q_lo(ytype), hi = q_hi(ytype);
  int err = OR_OK;
#pragma omp parallel for collapse(2) schedule(static) reduction(min : err)
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t m = 0; m < M; ++m) {
      const int64_t g = m / Mg;
      const int64_t wz = w_zero_point[per_channel ? m : 0];
      const float ws = w_scale[per_channel ? m : 0];
      for (int64_t oh = 0; oh < OH; ++oh) {
        for (int64_t ow = 0; ow < OW; ++ow) {
          int64_t acc = 0;
          for (int64_t cc = 0; cc < Cg; ++cc) {
            const int64_t c = g * Cg + cc;
            for (int64_t kh = 0; kh < kH; ++kh) {
              const int64_t ih = oh * strides[0] - pads[0] + kh * dilations[0];
              if (ih < 0 || ih >= H) continue;
              for (int64_t kw = 0; kw < kW; ++kw) {
                const int64_t iw = ow * strides[1] - pads[1] + kw * dilations[1];
                if (iw < 0 || iw >= W) continue;
                const int64_t xv = load_q(x, xtype, ((n * C + c) * H + ih) * W + iw);
                const int64_t wv = load_q(w, wtype, ((m * Cg + cc) * kH + kh) * kW + kw);
                acc += (xv - x_zero_point) * (wv - wz);
              }
            }
          }
          if (B) acc += B[m];
          if (acc > INT32_MAX || acc < INT32_MIN) {
            err = OR_ERR_OVERFLOW;
            continue;
          }
          float v = (float)(int32_t)acc;
          float mul = x_scale * ws;
          v = v * mul;
          v = v / y_scale;
          store_q(y, ytype, ((n * M + m) * OH + oh) * OW + ow, sat_rint_plus(v, y_zero_point, lo, hi));
        }
      }
    }
  }
  return err;
}

/* [QG] QGemm.  A is (M, K), or (K, M) when transA; B is (K, N), or (N, K)
 * when transB; both hold 8-bit codes of type atype / btype.
 *   acc[i,j] = sum_k (A[i,k] - a_zero_point) * (B[k,j] - b_zero_point[j])
 *   acc += C[i,j] when C is given; C is (c_rows, c_cols) with c_rows in
 *          {1, M} and c_cols in {1, N}, broadcast to (M, N).  Its scale is
 *          alpha * a_scale * b_scale and its zero point 0, so it adds to the
 *          integer sum (the page writes alpha / beta but defines no beta:
 *          beta = 1).
 *   y = (float)acc * ((alpha * a_scale) * b_scale[j])
 *   quantized output: y = saturate(round_half_even(y / y_scale) + y_zero_point)
 * The page gives no formula for the rescale; this is DequantizeLinear of the
 * integer sum, then QuantizeLinear with (y_scale, y_zero_point), the three
 * scale factors multiplied in the order they are listed.  b_scale and
 * b_zero_point hold N entries when n_b == N, else one.  Y is float (M, N)
 * unless quantize_y, then ytype codes. */
int or_qgemm(const void* A, int atype, int transA, int64_t M, int64_t K, float a_scale, int32_t a_zero_point,
             const void* B, int btype, int transB, int64_t N, const float* b_scale, const int32_t* b_zero_point,
             int64_t n_b, const int32_t* C, int64_t c_rows, int64_t c_cols, float alpha, int quantize_y,
             float y_scale, int32_t y_zero_point, int ytype, void* Y) {
  if (!rounding_is_nearest()) return OR_ERR_ROUNDING;
  if (n_b != 1 && n_b != N) return OR_ERR_ARG;
  if (C && !((c_rows == 1 || c_rows == M) && (c_cols == 1 || c_cols == N))) return OR_ERR_ARG;
  const int64_t lo = q_lo(ytype), hi = q_hi(ytype);
  int err = OR_OK;
#pragma omp parallel for schedule(static) reduction(min : err)
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t j = 0; j < N; ++j) {
      const int64_t bz = b_zero_point ? b_zero_point[n_b == N ? j : 0] : 0;
      int64_t acc = 0;
      for (int64_t k = 0; k < K; ++k) {
        const int64_t av = load_q(A, atype, transA ? k * M + i : i * K + k);
        const int64_t bv = load_q(B, btype, transB ? j * K + k : k * N + j);
        acc += (av - a_zero_point) * (bv - bz);
      }
      if (C) acc += C[(c_rows == 1 ? 0 : i) * c_cols + (c_cols == 1 ? 0 : j)];
      if (acc > INT32_MAX || acc < INT32_MIN) {
        err = OR_ERR_OVERFLOW;
        continue;
      }
      float mul = alpha * a_scale;
      mul = mul * b_scale[n_b == N ? j : 0];
      float v = (float)(int32_t)acc;
      v = v * mul;
      if (quantize_y) {
        v = v / y_scale;
        store_q(Y, ytype, i * N + j, sat_rint_plus(v, y_zero_point, lo, hi));
      } else {
        ((float*)Y)[i * N + j] = v;
      }
    }
  }
  return err;
}

/* [MITF] MatMulIntegerToFloat on 2-D operands (leading dimensions of an
 * N-dimensional A are rows):
 *   acc[i,j] = sum_k (A[i,k] - a_zero_point[i]) * (B[k,j] - b_zero_point[j])
 *   Y[i,j]   = (float)acc * (a_scale[i] * b_scale[j]) + bias[j]
 * b_scale / b_zero_point hold 1 or N entries (per tensor or per column of B).
 * For A the schema repeats B's sentence ("per-column", "the number of
 * columns of input 'A'"); a scale per summation index cannot be taken out
 * of the integer sum, so the reading used is 1 entry (per tensor) or M
 * entries (one per row of A, the dimension that remains in Y).  A missing
 * zero point is 0, a missing bias adds nothing.  The product of the two
 * scales is formed first, as the per-element multiplier. */
int or_matmul_integer_to_float(const void* A, int atype, int64_t M, int64_t K, const void* B, int btype,
                               int64_t N, const float* a_scale, const int32_t* a_zero_point, int64_t n_a,
                               const float* b_scale, const int32_t* b_zero_point, int64_t n_b, const float* bias,
                               float* Y) {
  if (!rounding_is_nearest()) return OR_ERR_ROUNDING;
  if ((n_a != 1 && n_a != M) || (n_b != 1 && n_b != N)) return OR_ERR_ARG;
  int err = OR_OK;
#pragma omp parallel for schedule(static) reduction(min : err)
  for (int64_t i = 0; i < M; ++i) {
    const int64_t pa = n_a == M ? i : 0;
    const int64_t az = a_zero_point ? a_zero_point[pa] : 0;
    for (int64_t j = 0; j < N; ++j) {
      const int64_t pb = n_b == N ? j : 0;
      const int64_t bz = b_zero_point ? b_zero_point[pb] : 0;
      int64_t acc = 0;
      for (int64_t k = 0; k < K; ++k)
        acc += (load_q(A, atype, i * K + k) - az) * (load_q(B, btype, k * N + j) - bz);
      if (acc > INT32_MAX || acc < INT32_MIN) {
        err = OR_ERR_OVERFLOW;
        continue;
      }
      float mul = a_scale[pa] * b_scale[pb];
      float v = (float)(int32_t)acc;
      v = v * mul;
      if (bias) v = v + bias[j];
      Y[i * N + j] = v;
    }
  }
  return err;
}

/* Numpy-style broadcasting of two shapes already padded to one rank: the
 * offset of output element `flat` in an operand with shape `sh` (its size-1
 * dimensions repeat). */
static int64_t bcast_offset(int64_t flat, const int64_t* out_shape, const int64_t* sh, int rank) {
  int64_t off = 0, stride = 1;
  for (int d = rank - 1; d >= 0; --d) {
    const int64_t idx = flat % out_shape[d];
    flat /= out_shape[d];
    if (sh[d] != 1) off += idx * stride;
    stride *= sh[d];
  }
  return off;
}

/* [QEW] MulInteger: C (int32) = (A - A_zero_point) * (B - B_zero_point),
 * broadcast.  a_shape / b_shape / out_shape share one rank (left-padded with
 * 1s by the caller). */
int or_mul_integer(const void* A, int atype, const int64_t* a_shape, int32_t a_zp, const void* B, int btype,
                   const int64_t* b_shape, int32_t b_zp, const int64_t* out_shape, int rank, int32_t* C) {
  int64_t n = 1;
  for (int d = 0; d < rank; ++d) n *= out_shape[d];
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    const int64_t a = load_q(A, atype, bcast_offset(i, out_shape, a_shape, rank)) - a_zp;
    const int64_t b = load_q(B, btype, bcast_offset(i, out_shape, b_shape, rank)) - b_zp;
    C[i] = (int32_t)(a * b);
  }
  return OR_OK;
}

/* [QEW] QLinearAdd (op 0) and QLinearMul (op 1), broadcast; A, B and C are
 * codes of one 8-bit type.  Read in the order the formulas are written:
 *   add: C = (A_scale * (A - A_zp) + B_scale * (B - B_zp)) / C_scale + C_zp
 *   mul: C = ((A - A_zp) * (B - B_zp)) * (A_scale * B_scale) / C_scale + C_zp
 * with the integer differences (and their product) exact, every fp32
 * operation rounding once, then round half to even and saturation. */
int or_qlinear_binary(int op, const void* A, const int64_t* a_shape, float a_scale, int32_t a_zp, const void* B,
                      const int64_t* b_shape, float b_scale, int32_t b_zp, float c_scale, int32_t c_zp,
                      const int64_t* out_shape, int rank, int qtype, void* C) {
  if (!rounding_is_nearest()) return OR_ERR_ROUNDING;
  int64_t n = 1;
  for (int d = 0; d < rank; ++d) n *= out_shape[d];
  const int64_t lo = q_lo(qtype), hi = q_hi(qtype);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    const int64_t a = load_q(A, qtype, bcast_offset(i, out_shape, a_shape, rank)) - a_zp;
    const int64_t b = load_q(B, qtype, bcast_offset(i, out_shape, b_shape, rank)) - b_zp;
    float v;
    if (op == 0) {
      float fa = a_scale * (float)a;
      float fb = b_scale * (float)b;
      v = fa + fb;
    } else {
      float m = a_scale * b_scale;
      v = (float)(a * b) * m;
    }
    v = v / c_scale;
    store_q(C, qtype, i, sat_rint_plus(v, c_zp, lo, hi));
  }
  return OR_OK;
}

/* ---------------------------------------------------------------------------
 * [EF] fp32 elementary functions: exp, expm1, log1p, sigmoid, tanh and
 * softplus, as used by the LSTM activations and QLinearSigmoid.
 *
 * The pages fix no evaluation of these functions.  Library versions differ
 * in the last bit between platforms, and one such bit in h can move a uint8
 * code of the next step's dynamically quantized hidden state.  So each is
 * defined here as a fixed sequence of IEEE fp32 operations (each rounds
 * once to nearest even; fmaf rounds the exact a*b+c once, and scaling by a
 * power of two is exact unless the result leaves the normal range); any
 * implementation that performs the same sequence gets the same bits.  The
 * methods are textbook ones:
 *
 *  exp   Cody and Waite's argument reduction (W. J. Cody and W. Waite,
 *        "Software Manual for the Elementary Functions", 1980):
 *        x = n ln2 + r, n = rint(x / ln2), r = (x - n LN2_HI) - n LN2_LO,
 *        where LN2_HI is ln 2 rounded to fp32 and LN2_LO the fp32 rounding
 *        of the remainder; e^r by its Taylor series to r^7/7! in Horner
 *        form (|r| <= ln2/2: the truncation is below 2^-27 relative); the
 *        result scaled by 2^n as two multiplications by powers of two, so
 *        that a subnormal result rounds once.
 *  expm1 the same reduction; e^r - 1 = r (1 + r/2! + ... + r^7/8!), and
 *        e^x - 1 = 2^n (e^r - 1) + (2^n - 1).
 *  log1p (argument in [0, 1]) 1 + u = 2^k (1 + v) with k = 0 or 1 and v in
 *        [sqrt(1/2) - 1, sqrt(2) - 1]; log(1 + v) = 2 atanh(s) with
 *        s = v / (2 + v), by the series 2 s (1 + s^2/3 + ... + s^8/9).
 *  sigmoid(x) = 1 / (1 + exp(-x));  tanh(x) = sign(x) t(|x|) with
 *        t(a) = e / (e + 2), e = expm1(2a), for a < 0.625, where the
 *        cancellation of 1 - 2 / (e^2a + 1) would cost accuracy;
 *        1 - 2 / (exp(2a) + 1) up to 9.5; and 1 above (tanh rounds to 1);
 *        softplus(x) = log(1 + e^x), as x + log1p(e^-x) for x > 0.
 * Each constant is written in hexadecimal; the comment names the number it
 * is the fp32 rounding of.
 */
static float pow2i(int k) { return ldexpf(1.0f, k); } /* exact for -149 <= k <= 127 */

static const float EF_L2E = 0x1.715476p+0f;     /* 1 / ln 2 */
static const float EF_LN2_HI = 0x1.62e430p-1f;  /* ln 2 */
static const float EF_LN2_LO = -0x1.05c610p-29f; /* ln 2 - EF_LN2_HI */

static float ef_exp(float x) {
  if (x > 89.0f) x = 89.0f;    /* e^89 is above the fp32 range: the result is +inf */
  if (x < -104.0f) x = -104.0f; /* e^-104 is below half the least subnormal: 0 */
  const float nf = rintf(x * EF_L2E);
  const int n = (int)nf;
  float r = fmaf(-nf, EF_LN2_HI, x);
  r = fmaf(-nf, EF_LN2_LO, r);
  float p = 0x1.a01a02p-13f;       /* 1/7! */
  p = fmaf(p, r, 0x1.6c16c2p-10f); /* 1/6! */
  p = fmaf(p, r, 0x1.111112p-7f);  /* 1/5! */
  p = fmaf(p, r, 0x1.555556p-5f);  /* 1/4! */
  p = fmaf(p, r, 0x1.555556p-3f);  /* 1/3! */
  p = fmaf(p, r, 0.5f);            /* 1/2! */
  p = fmaf(p, r, 1.0f);
  p = fmaf(p, r, 1.0f);
  const int n1 = n / 2, n2 = n - n1;
  return (p * pow2i(n1)) * pow2i(n2);
}

/* e^x - 1 for x <= 20 (e^x itself above, -1 below -20, where e^x is under
 * a quarter of an fp32 ulp of 1). */
static float ef_expm1(float x) {
  if (x > 20.0f) return ef_exp(x);
  if (x < -20.0f) return -1.0f;
  const float nf = rintf(x * EF_L2E);
  const int n = (int)nf;
  float r = fmaf(-nf, EF_LN2_HI, x);
  r = fmaf(-nf, EF_LN2_LO, r);
  float q = 0x1.a01a02p-16f;       /* 1/8! */
  q = fmaf(q, r, 0x1.a01a02p-13f); /* 1/7! */
  q = fmaf(q, r, 0x1.6c16c2p-10f); /* 1/6! */
  q = fmaf(q, r, 0x1.111112p-7f);  /* 1/5! */
  q = fmaf(q, r, 0x1.555556p-5f);  /* 1/4! */
  q = fmaf(q, r, 0x1.555556p-3f);  /* 1/3! */
  q = fmaf(q, r, 0.5f);            /* 1/2! */
  q = fmaf(q, r, 1.0f);
  q = q * r; /* e^r - 1 */
  if (n == 0) return q;
  const float t = pow2i(n);
  return fmaf(t, q, t - 1.0f);
}

/* log(1 + u) for 0 <= u <= 1. */
static float ef_log1p01(float u) {
  float v = u, k = 0.0f;
  if (u > 0x1.a8279ap-2f) { /* sqrt(2) - 1 */
    v = (u - 1.0f) * 0.5f;  /* exact: 1 + u = 2 (1 + v) */
    k = 1.0f;
  }
  const float s = v / (2.0f + v);
  const float z = s * s;
  float w = 0x1.c71c72p-4f;       /* 1/9 */
  w = fmaf(w, z, 0x1.24924ap-3f); /* 1/7 */
  w = fmaf(w, z, 0x1.99999ap-3f); /* 1/5 */
  w = fmaf(w, z, 0x1.555556p-2f); /* 1/3 */
  w = fmaf(w, z, 1.0f);
  const float l = (s + s) * w; /* log(1 + v) */
  return fmaf(k, EF_LN2_HI, l);
}

static float ef_sigmoid(float x) { return 1.0f / (1.0f + ef_exp(-x)); }

/* tanh(a) = e / (e + 2) = 1 - 2 / (e + 2) with e = e^(2a) - 1: the first
   form below |a| = 0.625, the second above (no cancellation in either);
   1 beyond 9.5, where tanh rounds to 1 in fp32. */
static float ef_tanh(float x) {
  const float a = fabsf(x);
  float t = 1.0f;
  if (a <= 9.5f) {
    const float e = ef_expm1(a + a);
    const float q = (a < 0.625f ? e : 2.0f) / (e + 2.0f);
    t = a < 0.625f ? q : 1.0f - q;
  }
  return copysignf(t, x);
}

static float ef_softplus(float x) {
  return x > 0.0f ? x + ef_log1p01(ef_exp(-x)) : ef_log1p01(ef_exp(x));
}

/* Single-argument entry points for the pins (n values each). */
int or_elementary(int fn, const float* x, int64_t n, float* y) {
  for (int64_t i = 0; i < n; ++i) {
    switch (fn) {
      case 0: y[i] = ef_exp(x[i]); break;
      case 1: y[i] = ef_expm1(x[i]); break;
      case 2: y[i] = ef_log1p01(x[i]); break;
      case 3: y[i] = ef_sigmoid(x[i]); break;
      case 4: y[i] = ef_tanh(x[i]); break;
      case 5: y[i] = ef_softplus(x[i]); break;
      default: return OR_ERR_ARG;
    }
  }
  return OR_OK;
}

/* [QEW] QLinearLeakyRelu (op 0) and QLinearSigmoid (op 1) on n codes:
 *   d = DequantizeLinear(x) = (x - X_zp) * X_scale
 *   leaky relu: f = alpha * d when d < 0, else d
 *   sigmoid:    f = 1 / (1 + exp(-d))   ([EF] sigmoid)
 *   y = QuantizeLinear(f) = saturate(rint(f / Y_scale) + Y_zp) */
int or_qlinear_unary(int op, const void* X, int64_t n, int qtype, float x_scale, int32_t x_zp, float y_scale,
                     int32_t y_zp, float alpha, void* Y) {
  if (!rounding_is_nearest()) return OR_ERR_ROUNDING;
  const int64_t lo = q_lo(qtype), hi = q_hi(qtype);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    const float d = (float)(load_q(X, qtype, i) - x_zp) * x_scale;
    float f;
    if (op == 0)
      f = d < 0.0f ? alpha * d : d;
    else
      f = ef_sigmoid(d);
    store_q(Y, qtype, i, sat_rint_plus(f / y_scale, y_zp, lo, hi));
  }
  return OR_OK;
}

/* [LSTM] The activation functions the "activations" attribute may name: the
 * ONNX LSTM operator's list (the schema refers to it; it is not printed on
 * the pages), in that list's order.  alpha and beta are the function's
 * attributes, resolved by the caller (defaults of the corresponding ONNX
 * operators where the attribute lists run out).  Each is its operator's
 * formula in fp32, one rounding per operation:
 *   Relu            max(0, x)
 *   Tanh, Sigmoid   [EF] tanh, sigmoid
 *   Affine          alpha x + beta
 *   LeakyRelu       x for x >= 0, alpha x otherwise
 *   ThresholdedRelu x for x > alpha, 0 otherwise
 *   ScaledTanh      alpha tanh(beta x)
 *   HardSigmoid     min(max(alpha x + beta, 0), 1)
 *   Elu             x for x >= 0, alpha (e^x - 1) otherwise ([EF] expm1)
 *   Softsign        x / (1 + |x|)
 *   Softplus        log(e^x + 1) ([EF] softplus) */
enum {
  OR_LA_RELU, OR_LA_TANH, OR_LA_SIGMOID, OR_LA_AFFINE, OR_LA_LEAKY_RELU, OR_LA_THRESHOLDED_RELU,
  OR_LA_SCALED_TANH, OR_LA_HARD_SIGMOID, OR_LA_ELU, OR_LA_SOFTSIGN, OR_LA_SOFTPLUS
};

static float lstm_activation(int kind, float alpha, float beta, float x) {
  switch (kind) {
    case OR_LA_RELU: return x > 0.0f ? x : 0.0f;
    case OR_LA_TANH: return ef_tanh(x);
    case OR_LA_SIGMOID: return ef_sigmoid(x);
    case OR_LA_AFFINE: return alpha * x + beta;
    case OR_LA_LEAKY_RELU: return x >= 0.0f ? x : alpha * x;
    case OR_LA_THRESHOLDED_RELU: return x > alpha ? x : 0.0f;
    case OR_LA_SCALED_TANH: return alpha * ef_tanh(beta * x);
    case OR_LA_HARD_SIGMOID: {
      const float v = alpha * x + beta;
      return v < 0.0f ? 0.0f : (v > 1.0f ? 1.0f : v);
    }
    case OR_LA_ELU: return x >= 0.0f ? x : alpha * ef_expm1(x);
    case OR_LA_SOFTSIGN: return x / (1.0f + fabsf(x));
    case OR_LA_SOFTPLUS: return ef_softplus(x);
  }
  return x;
}

/* [LSTM] one cell update for one direction and one time step, gate columns
 * in iofc order.  The ONNX LSTM equations the schema points to (not printed
 * on the pages) give each gate's terms in this order, summed left to right:
 *   i = f(X Wi + H Ri + Pi (.) C_prev + Wbi + Rbi)
 *   f = f(X Wf + H Rf + Pf (.) C_prev + Wbf + Rbf)     (1 - i when input_forget)
 *   c~ = g(X Wc + H Rc + Wbc + Rbc)
 *   C = f (.) C_prev + i (.) c~
 *   o = f(X Wo + H Ro + Po (.) C + Wbo + Rbo)
 *   H = o (.) h(C)
 * f, g, h are act[0..2] with their alpha/beta (NULL act: the defaults
 * Sigmoid, Tanh, Tanh).  Gx and Gh are the two dequantized products.  P
 * holds Pi, Po, Pf (3H, "P[iof]") or is NULL (no peephole terms).  clip > 0
 * bounds each gate's input to [-clip, clip] before its activation; clip <= 0
 * is no clip (the schema: "No clip if not specified"; the third-party page
 * lists a default of 0, read as the same).  A missing bias adds nothing. */
int or_lstm_cell_ex(const float* Gx, const float* Gh, const float* Wb, const float* Rb, const float* P, float clip,
                    int input_forget, const int* act, const float* act_alpha, const float* act_beta,
                    const float* c_prev, float* h_out, float* c_out, int64_t batch, int64_t H) {
  static const int default_act[3] = {OR_LA_SIGMOID, OR_LA_TANH, OR_LA_TANH};
  static const float zero3[3] = {0.0f, 0.0f, 0.0f};
  if (!act) act = default_act;
  if (!act_alpha) act_alpha = zero3;
  if (!act_beta) act_beta = zero3;
  for (int q = 0; q < 3; ++q)
    if (act[q] < OR_LA_RELU || act[q] > OR_LA_SOFTPLUS) return OR_ERR_ARG;
#define F_(v) lstm_activation(act[0], act_alpha[0], act_beta[0], (v))
#define G_(v) lstm_activation(act[1], act_alpha[1], act_beta[1], (v))
#define H_(v) lstm_activation(act[2], act_alpha[2], act_beta[2], (v))
  for (int64_t b = 0; b < batch; ++b) {
    for (int64_t u = 0; u < H; ++u) {
      const float cp = c_prev[b * H + u];
      float g[4];
      for (int q = 0; q < 4; ++q) {
        int64_t n = q * H + u;
        float v = Gx[b * 4 * H + n] + Gh[b * 4 * H + n];
        if (P && q == 0) v = v + P[u] * cp;
        if (P && q == 2) v = v + P[2 * H + u] * cp;
        if (q != 1) {
          if (Wb) v = v + Wb[n];
          if (Rb) v = v + Rb[n];
          if (clip > 0.0f) v = v < -clip ? -clip : (v > clip ? clip : v);
        }
        g[q] = v;
      }
      float ig = F_(g[0]);
      float fg = input_forget ? 1.0f - ig : F_(g[2]);
      float ct = G_(g[3]);
      float c = fg * cp + ig * ct;
      float vo = g[1];
      if (P) vo = vo + P[H + u] * c;
      if (Wb) vo = vo + Wb[H + u];
      if (Rb) vo = vo + Rb[H + u];
      if (clip > 0.0f) vo = vo < -clip ? -clip : (vo > clip ? clip : vo);
      float og = F_(vo);
      c_out[b * H + u] = c;
      h_out[b * H + u] = og * H_(c);
    }
  }
#undef F_
#undef G_
#undef H_
  return OR_OK;
}

/* The default cell: no peepholes, no clip, input_forget 0. */
int or_lstm_cell(const float* Gx, const float* Gh, const float* Wb, const float* Rb, const float* c_prev,
                 float* h_out, float* c_out, int64_t batch, int64_t H) {
  return or_lstm_cell_ex(Gx, Gh, Wb, Rb, NULL, 0.0f, 0, NULL, NULL, NULL, c_prev, h_out, c_out, batch, H);
}

/* [DQIP] / [LSTM] the dequantized product of per-row uint8 codes uA (M x K,
 * scaleA, zeroA) with 8-bit B codes (K x N, type btype) that carry a zero
 * point per column (n_zb == N) or per tensor (n_zb == 1; NULL: 0):
 *   C[i,j] = ((float)sum_k (uA[i,k] - zeroA[i]) * (B[k,j] - zeroB[j]) * scaleA[i]) * scaleB[j]
 * in the order of the inner product's epilogue; the int32 sum is exact. */
int or_dyn_product_zp(const uint8_t* uA, const int32_t* zeroA, const float* scaleA, const void* B, int btype,
                      const int32_t* zeroB, int64_t n_zb, const float* scaleB, int64_t M, int64_t N, int64_t K,
                      float* C) {
  if (!rounding_is_nearest()) return OR_ERR_ROUNDING;
  int err = OR_OK;
#pragma omp parallel for schedule(static) reduction(min : err)
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t j = 0; j < N; ++j) {
      const int64_t zb = zeroB ? zeroB[n_zb == N ? j : 0] : 0;
      int64_t acc = 0;
      for (int64_t k = 0; k < K; ++k)
        acc += ((int64_t)uA[i * K + k] - (int64_t)zeroA[i]) * (load_q(B, btype, k * N + j) - zb);
      if (acc > INT32_MAX || acc < INT32_MIN) {
        err = OR_ERR_OVERFLOW;
        continue;
      }
      float v = (float)(int32_t)acc;
      v = v * scaleA[i];
      v = v * scaleB[j];
      C[i * N + j] = v;
    }
  }
  return err;
}
