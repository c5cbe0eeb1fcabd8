// qdq.cu -- QuantizeLinear and DequantizeLinear (ONNX Runtime contrib
// schemas "QuantizeLinear" / "DequantizeLinear", ver 1).
//
//   QuantizeLinear:   y = saturate(rint(x / y_scale) + y_zero_point)
//   DequantizeLinear: y = (x - x_zero_point) * x_scale
//
// Both are pure streams over HBM (5 bytes per element), so the kernels are
// shaped for bandwidth: each thread moves 16 elements per iteration with
// 16-byte loads and stores (4 x float4 on the fp32 side, one uint4 on the
// 8-bit side), streaming cache hints, and a grid-stride loop over a grid
// sized to fill every SM.  The per-axis parameter index is the middle index
// of the [outer, axis_len, inner] view of the tensor; the common case of the
// last axis (inner == 1) keeps a running channel counter instead of dividing.
#include "common.cuh"

namespace i8q {
namespace {

enum AxisMode : int { AX_TENSOR = 0, AX_LAST = 1, AX_BLOCK = 2 };

template <typename QT>
struct QRange;
template <>
struct QRange<uint8_t> {
  static constexpr float lo = 0.0f, hi = 255.0f;
};
template <>
struct QRange<int8_t> {
  static constexpr float lo = -128.0f, hi = 127.0f;
};

template <typename QT>
__device__ __forceinline__ uint32_t quant_one(float x, float s, int zp) {
  float q = __fdiv_rn(x, s);
  int v = sat_rint(q, QRange<QT>::lo - (float)zp, QRange<QT>::hi - (float)zp) + zp;
  return (uint32_t)(v & 0xff);
}

template <typename QT>
__device__ __forceinline__ float dequant_one(uint32_t byte, float s, int zp) {
  int v = (int)(QT)(byte & 0xff);
  return __fmul_rn(__int2float_rn(v - zp), s);
}

template <typename QT>
__device__ __forceinline__ int load_zp(const QT* zp, int64_t c) {
  return (int)zp[c];
}

// Parameters of 16 consecutive elements starting at element e.
template <int MODE, typename QT>
__device__ __forceinline__ void params16(const float* __restrict__ scale, const QT* __restrict__ zp,
                                         int64_t c0, float (&s)[16], int (&z)[16]) {
  if (MODE == AX_LAST) {
    // 16 consecutive channels; c0 is a multiple of 16 (axis_len % 16 == 0)
    const float4* s4 = reinterpret_cast<const float4*>(scale + c0);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float4 v = __ldg(s4 + q);
      s[4 * q + 0] = v.x;
      s[4 * q + 1] = v.y;
      s[4 * q + 2] = v.z;
      s[4 * q + 3] = v.w;
    }
    uint4 zz = __ldg(reinterpret_cast<const uint4*>(zp + c0));
    uint32_t w[4] = {zz.x, zz.y, zz.z, zz.w};
#pragma unroll
    for (int q = 0; q < 16; ++q) z[q] = (int)(QT)((w[q >> 2] >> (8 * (q & 3))) & 0xff);
  } else {
    float sv = __ldg(scale + c0);
    int zv = (int)zp[c0];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      s[q] = sv;
      z[q] = zv;
    }
  }
}

template <int MODE, typename QT>
__global__ void __launch_bounds__(256) quantize_vec16(const float* __restrict__ x, QT* __restrict__ y,
                                                      int64_t nvec, const float* __restrict__ scale,
                                                      const QT* __restrict__ zp, int64_t axis_len,
                                                      int64_t inner) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  // running channel of element 16*v for the last-axis mode
  int64_t c_last = 0, c_step = 0;
  if (MODE == AX_LAST) {
    c_last = (16 * v) % axis_len;
    c_step = (16 * stride) % axis_len;
  }
  const float4* x4 = reinterpret_cast<const float4*>(x);
  uint4* y16 = reinterpret_cast<uint4*>(y);
  for (; v < nvec; v += stride) {
    float4 a[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) a[q] = __ldcs(x4 + 4 * v + q);
    int64_t c0 = 0;
    if (MODE == AX_LAST) c0 = c_last;
    if (MODE == AX_BLOCK) c0 = ((16 * v) / inner) % axis_len;
    float s[16];
    int z[16];
    params16<MODE, QT>(scale, zp, c0, s, z);
    const float* f = reinterpret_cast<const float*>(a);
    uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
    for (int q = 0; q < 16; ++q) w[q >> 2] |= quant_one<QT>(f[q], s[q], z[q]) << (8 * (q & 3));
    __stcs(y16 + v, make_uint4(w[0], w[1], w[2], w[3]));
    if (MODE == AX_LAST) {
      c_last += c_step;
      if (c_last >= axis_len) c_last -= axis_len;
    }
  }
}

template <int MODE, typename QT>
__global__ void __launch_bounds__(256) dequantize_vec16(const QT* __restrict__ x, float* __restrict__ y,
                                                        int64_t nvec, const float* __restrict__ scale,
                                                        const QT* __restrict__ zp, int64_t axis_len,
                                                        int64_t inner) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  int64_t c_last = 0, c_step = 0;
  if (MODE == AX_LAST) {
    c_last = (16 * v) % axis_len;
    c_step = (16 * stride) % axis_len;
  }
  const uint4* x16 = reinterpret_cast<const uint4*>(x);
  float4* y4 = reinterpret_cast<float4*>(y);
  for (; v < nvec; v += stride) {
    uint4 in = __ldcs(x16 + v);
    int64_t c0 = 0;
    if (MODE == AX_LAST) c0 = c_last;
    if (MODE == AX_BLOCK) c0 = ((16 * v) / inner) % axis_len;
    float s[16];
    int z[16];
    params16<MODE, QT>(scale, zp, c0, s, z);
    uint32_t w[4] = {in.x, in.y, in.z, in.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float4 o;
      o.x = dequant_one<QT>(w[q], s[4 * q + 0], z[4 * q + 0]);
      o.y = dequant_one<QT>(w[q] >> 8, s[4 * q + 1], z[4 * q + 1]);
      o.z = dequant_one<QT>(w[q] >> 16, s[4 * q + 2], z[4 * q + 2]);
      o.w = dequant_one<QT>(w[q] >> 24, s[4 * q + 3], z[4 * q + 3]);
      __stcs(y4 + 4 * v + q, o);
    }
    if (MODE == AX_LAST) {
      c_last += c_step;
      if (c_last >= axis_len) c_last -= axis_len;
    }
  }
}

// Element-wise kernels for the tail and for layouts the vector path does
// not take (unaligned pointers, axis length not a multiple of 16).
template <typename QT>
__global__ void quantize_scalar(const float* __restrict__ x, QT* __restrict__ y, int64_t begin, int64_t n,
                                const float* __restrict__ scale, const QT* __restrict__ zp, int per_axis,
                                int64_t axis_len, int64_t inner) {
  for (int64_t i = begin + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    int64_t c = per_axis ? (i / inner) % axis_len : 0;
    y[i] = (QT)quant_one<QT>(x[i], scale[c], (int)zp[c]);
  }
}

template <typename QT>
__global__ void dequantize_scalar(const QT* __restrict__ x, float* __restrict__ y, int64_t begin, int64_t n,
                                  const float* __restrict__ scale, const QT* __restrict__ zp, int per_axis,
                                  int64_t axis_len, int64_t inner) {
  for (int64_t i = begin + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    int64_t c = per_axis ? (i / inner) % axis_len : 0;
    y[i] = dequant_one<QT>((uint32_t)(uint8_t)x[i], scale[c], (int)zp[c]);
  }
}

struct AxisView {
  int64_t n = 1, axis_len = 1, inner = 1;
  bool per_axis = false;
};

int make_view(const int64_t* shape, int rank, int axis, size_t n_scale, AxisView* v) {
  if (rank < 0 || rank > 8) return fail(I8Q_ERR_INVALID_ARG, "rank must be in [0, 8]");
  if (rank > 0 && !shape) return fail(I8Q_ERR_INVALID_ARG, "shape is NULL");
  int64_t n = 1;
  for (int d = 0; d < rank; ++d) {
    if (shape[d] < 0) return fail(I8Q_ERR_INVALID_ARG, "negative dimension");
    n *= shape[d];
  }
  v->n = n;
  if (axis == I8Q_NO_AXIS) {
    if (n_scale != 1) return fail(I8Q_ERR_INVALID_ARG, "per-tensor scale and zero point must be scalars");
    v->per_axis = false;
    return I8Q_OK;
  }
  if (axis < -rank || axis >= rank) return fail(I8Q_ERR_INVALID_ARG, "axis out of range [-rank, rank-1]");
  int a = axis < 0 ? axis + rank : axis;
  if ((int64_t)n_scale != shape[a])
    return fail(I8Q_ERR_INVALID_ARG, "per-axis scale/zero point length must equal dim[axis]");
  int64_t inner = 1;
  for (int d = a + 1; d < rank; ++d) inner *= shape[d];
  v->axis_len = shape[a];
  v->inner = inner;
  v->per_axis = true;
  return I8Q_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <typename QT>
int run_quantize(const float* x, const AxisView& v, const float* scale, const QT* zp, QT* y, cudaStream_t s) {
  if (v.n == 0) return I8Q_OK;
  I8Q_PROF("quantize_linear", s);
  int mode = -1;
  if (!v.per_axis) mode = AX_TENSOR;
  else if (v.inner == 1 && v.axis_len % 16 == 0 && aligned16(scale) && aligned16(zp)) mode = AX_LAST;
  else if (v.inner % 16 == 0) mode = AX_BLOCK;
  int64_t nvec = (mode >= 0 && aligned16(x) && aligned16(y)) ? v.n / 16 : 0;
  const int threads = 256;
  if (nvec > 0) {
    int64_t blocks = std::min<int64_t>(ceil_div(nvec, threads), (int64_t)sm_count() * 8);
    if (mode == AX_TENSOR)
      quantize_vec16<AX_TENSOR, QT><<<blocks, threads, 0, s>>>(x, y, nvec, scale, zp, v.axis_len, v.inner);
    else if (mode == AX_LAST)
      quantize_vec16<AX_LAST, QT><<<blocks, threads, 0, s>>>(x, y, nvec, scale, zp, v.axis_len, v.inner);
    else
      quantize_vec16<AX_BLOCK, QT><<<blocks, threads, 0, s>>>(x, y, nvec, scale, zp, v.axis_len, v.inner);
    I8Q_LAUNCH_CHECK("quantize_vec16");
  }
  int64_t begin = nvec * 16;
  if (begin < v.n) {
    int64_t blocks = std::min<int64_t>(ceil_div(v.n - begin, threads), (int64_t)sm_count() * 8);
    quantize_scalar<QT><<<blocks, threads, 0, s>>>(x, y, begin, v.n, scale, zp, v.per_axis, v.axis_len, v.inner);
    I8Q_LAUNCH_CHECK("quantize_scalar");
  }
  return I8Q_OK;
}

template <typename QT>
int run_dequantize(const QT* x, const AxisView& v, const float* scale, const QT* zp, float* y, cudaStream_t s) {
  if (v.n == 0) return I8Q_OK;
  I8Q_PROF("dequantize_linear", s);
  int mode = -1;
  if (!v.per_axis) mode = AX_TENSOR;
  else if (v.inner == 1 && v.axis_len % 16 == 0 && aligned16(scale) && aligned16(zp)) mode = AX_LAST;
  else if (v.inner % 16 == 0) mode = AX_BLOCK;
  int64_t nvec = (mode >= 0 && aligned16(x) && aligned16(y)) ? v.n / 16 : 0;
  const int threads = 256;
  if (nvec > 0) {
    int64_t blocks = std::min<int64_t>(ceil_div(nvec, threads), (int64_t)sm_count() * 8);
    if (mode == AX_TENSOR)
      dequantize_vec16<AX_TENSOR, QT><<<blocks, threads, 0, s>>>(x, y, nvec, scale, zp, v.axis_len, v.inner);
    else if (mode == AX_LAST)
      dequantize_vec16<AX_LAST, QT><<<blocks, threads, 0, s>>>(x, y, nvec, scale, zp, v.axis_len, v.inner);
    else
      dequantize_vec16<AX_BLOCK, QT><<<blocks, threads, 0, s>>>(x, y, nvec, scale, zp, v.axis_len, v.inner);
    I8Q_LAUNCH_CHECK("dequantize_vec16");
  }
  int64_t begin = nvec * 16;
  if (begin < v.n) {
    int64_t blocks = std::min<int64_t>(ceil_div(v.n - begin, threads), (int64_t)sm_count() * 8);
    dequantize_scalar<QT><<<blocks, threads, 0, s>>>(x, y, begin, v.n, scale, zp, v.per_axis, v.axis_len, v.inner);
    I8Q_LAUNCH_CHECK("dequantize_scalar");
  }
  return I8Q_OK;
}

}  // namespace
}  // namespace i8q

using namespace i8q;

extern "C" int i8q_quantize_linear(const float* x, const int64_t* shape, int rank, int axis,
                                   const float* y_scale, const void* y_zero_point, size_t n_scale,
                                   int ytype, void* y, void* stream) {
  AxisView v;
  int rc = make_view(shape, rank, axis, n_scale, &v);
  if (rc) return rc;
  if (ytype != I8Q_U8 && ytype != I8Q_S8) return fail(I8Q_ERR_INVALID_ARG, "ytype must be I8Q_U8 or I8Q_S8");
  if (v.n > 0 && (!x || !y || !y_scale || !y_zero_point)) return fail(I8Q_ERR_INVALID_ARG, "NULL tensor pointer");
  cudaStream_t s = as_stream(stream);
  if (ytype == I8Q_U8)
    return run_quantize<uint8_t>(x, v, y_scale, (const uint8_t*)y_zero_point, (uint8_t*)y, s);
  return run_quantize<int8_t>(x, v, y_scale, (const int8_t*)y_zero_point, (int8_t*)y, s);
}

extern "C" int i8q_dequantize_linear(const void* x, int xtype, const int64_t* shape, int rank, int axis,
                                     const float* x_scale, const void* x_zero_point, size_t n_scale, float* y,
                                     void* stream) {
  AxisView v;
  int rc = make_view(shape, rank, axis, n_scale, &v);
  if (rc) return rc;
  if (xtype != I8Q_U8 && xtype != I8Q_S8) return fail(I8Q_ERR_INVALID_ARG, "xtype must be I8Q_U8 or I8Q_S8");
  if (v.n > 0 && (!x || !y || !x_scale || !x_zero_point)) return fail(I8Q_ERR_INVALID_ARG, "NULL tensor pointer");
  cudaStream_t s = as_stream(stream);
  if (xtype == I8Q_U8)
    return run_dequantize<uint8_t>((const uint8_t*)x, v, x_scale, (const uint8_t*)x_zero_point, y, s);
  return run_dequantize<int8_t>((const int8_t*)x, v, x_scale, (const int8_t*)x_zero_point, y, s);
}
