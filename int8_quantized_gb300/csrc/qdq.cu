// qdq.cu -- QuantizeLinear and DequantizeLinear (ONNX Runtime contrib
// schemas "QuantizeLinear" / "DequantizeLinear", ver 1).
//
//   QuantizeLinear:   y = saturate(rint(x / y_scale) + y_zero_point)
//   DequantizeLinear: y = (x - x_zero_point) * x_scale
//
// Both are pure streams over HBM (5 bytes per element), so the kernels are
// shaped for bandwidth: a warp moves 512 consecutive elements per iteration
// in four warp-wide accesses that are each one contiguous span (lane t takes
// elements 128*q + 4*t .. +3: a float4 on the fp32 side, one 32-bit word of
// codes on the 8-bit side), with streaming cache hints and a grid-stride
// loop over a grid sized to fill every SM.  The per-axis parameter index is
// the middle index of the [outer, axis_len, inner] view of the tensor; the
// common case of the last axis (inner == 1) keeps a running channel per warp
// tile instead of dividing.
#include "common.cuh"

#include <numeric>

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

// Low byte of the result: the code of x (IEEE division, then saturating
// round-half-even with the zero point).  The quotient is first bounded to
// [-2^16, 2^16] (beyond every code once the zero point is added; NaN goes
// to the lower bound), rounded to the nearest integer, ties to even, by
// adding 1.5 * 2^23, shifted by the zero point and saturated in integers:
// the same code as saturating rint(q) + zp, without a conversion.
template <typename QT>
__device__ __forceinline__ uint32_t quant_one(float x, float s, int zp) {
  const float q = fminf(fmaxf(__fdiv_rn(x, s), -65536.0f), 65536.0f);
  const int r = __float_as_int(__fadd_rn(q, 12582912.0f)) - 0x4B400000 + zp;
  return (uint32_t)min(max(r, (int)QRange<QT>::lo), (int)QRange<QT>::hi);
}

// (x - zp) * s; the difference (|x - zp| <= 255) goes to float exactly
// through the 1.5 * 2^23 bit pattern instead of a conversion instruction.
template <typename QT>
__device__ __forceinline__ float dequant_one(uint32_t byte, float s, int zp) {
  const int v = (int)(QT)(byte & 0xff) - zp;
  return __fmul_rn(__fsub_rn(__int_as_float(0x4B400000 + v), 12582912.0f), s);
}

template <typename QT>
__device__ __forceinline__ int load_zp(const QT* zp, int64_t c) {
  return (int)zp[c];
}

// Channel of element e (per-axis modes).  AX_LAST: e % axis_len, kept as a
// running value per warp tile; AX_BLOCK: (e / inner) % axis_len.
// Parameters of 4 consecutive elements starting at channel c (AX_LAST: the
// 4 channels c..c+3; otherwise one channel for all 4).
template <int MODE, typename QT>
__device__ __forceinline__ void params4(const float* __restrict__ scale, const QT* __restrict__ zp, int64_t c,
                                        float (&s)[4], int (&z)[4]) {
  if (MODE == AX_LAST) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(scale + c));
    s[0] = v.x;
    s[1] = v.y;
    s[2] = v.z;
    s[3] = v.w;
    const uint32_t w = __ldg(reinterpret_cast<const unsigned int*>(zp + c));
#pragma unroll
    for (int q = 0; q < 4; ++q) z[q] = (int)(QT)((w >> (8 * q)) & 0xffu);
  } else {
    const float sv = __ldg(scale + c);
    const int zv = (int)zp[c];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      s[q] = sv;
      z[q] = zv;
    }
  }
}

// A warp tile is 512 consecutive elements.  Lane t of the warp handles, for
// q = 0..3, the 4 elements at 128*q + 4*t: so each warp-wide access moves
// one contiguous span (512 B of fp32 or 128 B of codes).
template <int MODE>
__device__ __forceinline__ int64_t channel_of(int64_t e, int64_t c_tile, int off, int64_t axis_len, int64_t inner) {
  if (MODE == AX_TENSOR) return 0;
  if (MODE == AX_BLOCK) return (e / inner) % axis_len;
  int64_t c = c_tile + off;               // c_tile < axis_len, off < 512
  if (axis_len >= 512) return c >= axis_len ? c - axis_len : c;
  return c % axis_len;
}

// Per tensor, or the last axis with a grid stride of whole channel cycles:
// every tile of a warp sees the same parameters, so they are loaded once and
// held in registers.  On the last axis those are 16 channels' worth, which
// leaves room for 4 blocks per SM with one warp tile in flight (measured
// slightly ahead of 3 blocks with two tiles each); per tensor, one scalar
// pair leaves room for 6 blocks per SM.
template <int MODE, typename QT>
__global__ void __launch_bounds__(256, MODE == AX_TENSOR ? 6 : 4) quantize_fixed(const float* __restrict__ x, QT* __restrict__ y, int64_t ntiles,
                                                     const float* __restrict__ scale, const QT* __restrict__ zp,
                                                     int64_t axis_len) {
  static_assert(MODE == AX_TENSOR || MODE == AX_LAST, "fixed parameters: per tensor or the last axis");
  constexpr int U = 1;
  const int lane = threadIdx.x & 31;
  const int64_t wstride = ((int64_t)gridDim.x * blockDim.x) >> 5;
  int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t c_tile = MODE == AX_LAST ? (w * 512) % axis_len : 0;
  const float4* x4 = reinterpret_cast<const float4*>(x);
  uint32_t* y32 = reinterpret_cast<uint32_t*>(y);
  float s[4][4];
  int z[4][4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int off = 128 * q + 4 * lane;
    params4<MODE, QT>(scale, zp, channel_of<MODE>(w * 512 + off, c_tile, off, axis_len, 1), s[q], z[q]);
  }
  for (; w < ntiles; w += U * wstride) {
    float4 a[U][4];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t wu = w + u * wstride;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        a[u][q] = wu < ntiles ? __ldcs(x4 + wu * 128 + 32 * q + lane) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t wu = w + u * wstride;
      if (wu < ntiles) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t code =
              pack_low_bytes(quant_one<QT>(a[u][q].x, s[q][0], z[q][0]), quant_one<QT>(a[u][q].y, s[q][1], z[q][1]),
                             quant_one<QT>(a[u][q].z, s[q][2], z[q][2]), quant_one<QT>(a[u][q].w, s[q][3], z[q][3]));
          __stcs(y32 + wu * 128 + 32 * q + lane, code);
        }
      }
    }
  }
}

// Per-axis parameters that change from tile to tile (the last axis with a
// grid stride that is not whole channel cycles, or an inner axis).
template <int MODE, typename QT>
__global__ void __launch_bounds__(256) quantize_warp512(const float* __restrict__ x, QT* __restrict__ y,
                                                        int64_t ntiles, const float* __restrict__ scale,
                                                        const QT* __restrict__ zp, int64_t axis_len, int64_t inner) {
  const int lane = threadIdx.x & 31;
  const int64_t wstride = ((int64_t)gridDim.x * blockDim.x) >> 5;
  int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  int64_t c_tile = 0, c_step = 0;
  if (MODE == AX_LAST) {
    c_tile = (w * 512) % axis_len;
    c_step = (wstride * 512) % axis_len;
  }
  const float4* x4 = reinterpret_cast<const float4*>(x);
  uint32_t* y32 = reinterpret_cast<uint32_t*>(y);
  for (; w < ntiles; w += wstride) {
    const int64_t base4 = w * 128;  // tile start in units of 4 elements
    float4 a[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) a[q] = __ldcs(x4 + base4 + 32 * q + lane);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int off = 128 * q + 4 * lane;
      float s[4];
      int z[4];
      params4<MODE, QT>(scale, zp, channel_of<MODE>(w * 512 + off, c_tile, off, axis_len, inner), s, z);
      const uint32_t code = pack_low_bytes(quant_one<QT>(a[q].x, s[0], z[0]), quant_one<QT>(a[q].y, s[1], z[1]),
                                           quant_one<QT>(a[q].z, s[2], z[2]), quant_one<QT>(a[q].w, s[3], z[3]));
      __stcs(y32 + base4 + 32 * q + lane, code);
    }
    if (MODE == AX_LAST) {
      c_tile += c_step;
      if (c_tile >= axis_len) c_tile -= axis_len;
    }
  }
}

template <int MODE, typename QT>
__global__ void __launch_bounds__(256) dequantize_warp512(const QT* __restrict__ x, float* __restrict__ y,
                                                          int64_t ntiles, const float* __restrict__ scale,
                                                          const QT* __restrict__ zp, int64_t axis_len,
                                                          int64_t inner) {
  const int lane = threadIdx.x & 31;
  const int64_t wstride = ((int64_t)gridDim.x * blockDim.x) >> 5;
  int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  int64_t c_tile = 0, c_step = 0;
  if (MODE == AX_LAST) {
    c_tile = (w * 512) % axis_len;
    c_step = (wstride * 512) % axis_len;
  }
  const uint32_t* x32 = reinterpret_cast<const uint32_t*>(x);
  float4* y4 = reinterpret_cast<float4*>(y);
  // The 8-bit side moves only 4 bytes per lane per access, so four warp
  // tiles (16 loads per lane) are put in flight before any is used.
  constexpr int U = 4;
  // per tensor, or the last axis when the grid stride is a whole number of
  // channel cycles: every tile of this warp sees the same parameters
  if (MODE == AX_TENSOR || (MODE == AX_LAST && c_step == 0)) {
    float s[4][4];
    int z[4][4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int off = 128 * q + 4 * lane;
      params4<MODE, QT>(scale, zp, channel_of<MODE>(w * 512 + off, c_tile, off, axis_len, inner), s[q], z[q]);
    }
    for (; w < ntiles; w += U * wstride) {
      uint32_t in[U][4];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t wu = w + u * wstride;
#pragma unroll
        for (int q = 0; q < 4; ++q) in[u][q] = wu < ntiles ? __ldcs(x32 + wu * 128 + 32 * q + lane) : 0u;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t wu = w + u * wstride;
        if (wu < ntiles) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float4 o;
            o.x = dequant_one<QT>(in[u][q], s[q][0], z[q][0]);
            o.y = dequant_one<QT>(in[u][q] >> 8, s[q][1], z[q][1]);
            o.z = dequant_one<QT>(in[u][q] >> 16, s[q][2], z[q][2]);
            o.w = dequant_one<QT>(in[u][q] >> 24, s[q][3], z[q][3]);
            __stcs(y4 + wu * 128 + 32 * q + lane, o);
          }
        }
      }
    }
    return;
  }
  for (; w < ntiles; w += U * wstride) {
    uint32_t in[U][4];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t wu = w + u * wstride;
#pragma unroll
      for (int q = 0; q < 4; ++q) in[u][q] = wu < ntiles ? __ldcs(x32 + wu * 128 + 32 * q + lane) : 0u;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t wu = w + u * wstride;
      if (wu < ntiles) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int off = 128 * q + 4 * lane;
          float s[4];
          int z[4];
          params4<MODE, QT>(scale, zp, channel_of<MODE>(wu * 512 + off, c_tile, off, axis_len, inner), s, z);
          float4 o;
          o.x = dequant_one<QT>(in[u][q], s[0], z[0]);
          o.y = dequant_one<QT>(in[u][q] >> 8, s[1], z[1]);
          o.z = dequant_one<QT>(in[u][q] >> 16, s[2], z[2]);
          o.w = dequant_one<QT>(in[u][q] >> 24, s[3], z[3]);
          __stcs(y4 + wu * 128 + 32 * q + lane, o);
        }
      }
      if (MODE == AX_LAST) {
        c_tile += c_step;
        if (c_tile >= axis_len) c_tile -= axis_len;
      }
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

// Blocks of `threads` threads that are resident at once on the whole GPU.
int64_t wave_blocks(const void* kern, int threads) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, 0) != cudaSuccess) per_sm = 1;
  return (int64_t)sm_count() * std::max(per_sm, 1);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

template <typename QT>
int run_quantize(const float* x, const AxisView& v, const float* scale, const QT* zp, QT* y, cudaStream_t s) {
  if (v.n == 0) return I8Q_OK;
  I8Q_PROF("quantize_linear", s);
  int mode = -1;
  if (!v.per_axis) mode = AX_TENSOR;
  else if (v.inner == 1 && v.axis_len % 4 == 0 && aligned16(scale) && aligned4(zp)) mode = AX_LAST;
  else if (v.inner % 4 == 0) mode = AX_BLOCK;
  const bool ok_ptr = aligned16(x) && aligned4(y);
  const int64_t ntiles = (mode >= 0 && ok_ptr) ? v.n / 512 : 0;
  const int threads = 256;
  if (ntiles > 0) {
    // One wave of resident blocks (two for the per-tensor form): a partial
    // last wave leaves SMs with too few reads in flight.  On the last axis
    // the block count is rounded down, where that keeps at least half of
    // it, to a multiple that makes the grid stride whole channel cycles
    // (the form with parameters held in registers).
    const int64_t want = ceil_div(ntiles, threads / 32);
    if (mode == AX_TENSOR) {
      static const int64_t full = wave_blocks((const void*)quantize_fixed<AX_TENSOR, QT>, threads);
      const int64_t blocks = std::min<int64_t>(want, 2 * full);
      quantize_fixed<AX_TENSOR, QT><<<blocks, threads, 0, s>>>(x, y, ntiles, scale, zp, 1);
    } else if (mode == AX_LAST) {
      static const int64_t full = wave_blocks((const void*)quantize_fixed<AX_LAST, QT>, threads);
      const int64_t cyc = v.axis_len / std::gcd<int64_t>(v.axis_len, (int64_t)threads / 32 * 512);
      int64_t blocks = std::min<int64_t>(want, full);
      if (blocks % cyc != 0 && 2 * (blocks / cyc) * cyc >= blocks) blocks = (blocks / cyc) * cyc;
      if ((blocks * (threads / 32) * 512) % v.axis_len == 0)
        quantize_fixed<AX_LAST, QT><<<blocks, threads, 0, s>>>(x, y, ntiles, scale, zp, v.axis_len);
      else
        quantize_warp512<AX_LAST, QT><<<blocks, threads, 0, s>>>(x, y, ntiles, scale, zp, v.axis_len, v.inner);
    } else {
      static const int64_t full = wave_blocks((const void*)quantize_warp512<AX_BLOCK, QT>, threads);
      const int64_t blocks = std::min<int64_t>(want, full);
      quantize_warp512<AX_BLOCK, QT><<<blocks, threads, 0, s>>>(x, y, ntiles, scale, zp, v.axis_len, v.inner);
    }
    I8Q_LAUNCH_CHECK("quantize_warp512");
  }
  int64_t begin = ntiles * 512;
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
  else if (v.inner == 1 && v.axis_len % 4 == 0 && aligned16(scale) && aligned4(zp)) mode = AX_LAST;
  else if (v.inner % 4 == 0) mode = AX_BLOCK;
  const bool ok_ptr = aligned4(x) && aligned16(y);
  const int64_t ntiles = (mode >= 0 && ok_ptr) ? v.n / 512 : 0;
  const int threads = 256;
  if (ntiles > 0) {
    // Measured on the [32,1024,4096] round trip: per tensor, four whole
    // waves of resident blocks write fastest; per axis, 8 blocks per SM.
    int64_t blocks = std::min<int64_t>(ceil_div(ntiles, threads / 32), (int64_t)sm_count() * 8);
    if (mode == AX_TENSOR) {
      static const int64_t full = wave_blocks((const void*)dequantize_warp512<AX_TENSOR, QT>, threads);
      blocks = std::min<int64_t>(ceil_div(ntiles, threads / 32), 4 * full);
    }
    if (mode == AX_TENSOR)
      dequantize_warp512<AX_TENSOR, QT><<<blocks, threads, 0, s>>>(x, y, ntiles, scale, zp, v.axis_len, v.inner);
    else if (mode == AX_LAST)
      dequantize_warp512<AX_LAST, QT><<<blocks, threads, 0, s>>>(x, y, ntiles, scale, zp, v.axis_len, v.inner);
    else
      dequantize_warp512<AX_BLOCK, QT><<<blocks, threads, 0, s>>>(x, y, ntiles, scale, zp, v.axis_len, v.inner);
    I8Q_LAUNCH_CHECK("dequantize_warp512");
  }
  int64_t begin = ntiles * 512;
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
