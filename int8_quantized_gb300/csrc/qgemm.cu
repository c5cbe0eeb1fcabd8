// qgemm.cu -- the products of 8-bit codes on the exact-integer tensor-core
// path: QGemm, MatMulIntegerToFloat and DynamicQuantizeMatMul (ONNX Runtime
// contrib schemas).
//
// QGemm:
//   acc[i,j] = sum_k (A[i,k] - a_zero_point) * (B[k,j] - b_zero_point[j])
//   acc += C[i,j]                           (int32, broadcast from (1|M, 1|N))
//   y = (float)acc * ((alpha * a_scale) * b_scale[j])
//   quantized output: y = saturate(rint(y / y_scale) + y_zero_point)
// C carries the scale alpha * a_scale * b_scale and zero point 0 (the schema
// writes alpha / beta but defines no beta), so it adds to the integer sum;
// the rescale is DequantizeLinear of the sum followed by QuantizeLinear.
// MatMulIntegerToFloat:
//   Y[i,j] = (float)acc * (a_scale[i] * b_scale[j]) + bias[j]
// with A's scale and zero point per tensor or per row of A.
// DynamicQuantizeMatMul: fp32 A quantized to uint8 per tensor (range widened
// to contain 0, scale (max - min) / 255, zero point rint(-min / scale)),
// then MatMulIntegerToFloat.
//
// The 8-bit codes enter the tensor pipe centred, A' = A - ca and
// B' = B - cb with ca, cb = 128 for uint8 and 0 for int8, so every operand is
// in [-128, 127] (exact in bf16) and every product within 2^14, as in the
// dynamic quantized inner product.  The zero points come back in the
// epilogue from the row sums of A', the column sums of B' and K (see
// QgEpilogue).  One pass per operand writes the centred bf16 copy, K
// contiguous (transposing when the operand's K is its slow index), with the
// sums; one small pass forms the per-column epilogue parameters.
#include "common.cuh"

namespace i8q {
namespace {

constexpr int PT = 64;   // rows x K elements per tile of the operand pass
constexpr int CK = 512;  // K elements per CTA (8 tiles)

// Xc[r][k] = bf16(X(r,k) - cx) for k < K, 0 for K <= k < Kp, and
// sums[r] += sum_k (X(r,k) - cx) over the CTA's K range (sums zeroed by the
// caller).  X(r,k) = X[r*K + k] when k_fast, else X[k*R + r].  CTA (x, y)
// owns rows 64x .. 64x + 63 and K elements 512y .. 512y + 511, in 64-wide
// tiles through shared memory, reading the source along its contiguous
// index 16 bytes at a time where the layout allows (VEC), else bytewise.
template <bool SIGNED, bool VEC>
__global__ void __launch_bounds__(256)
center_operand(const uint8_t* __restrict__ X, int64_t R, int64_t K, int64_t Kp, int k_fast,
               __nv_bfloat16* __restrict__ Xc, int32_t* __restrict__ sums) {
  __shared__ __align__(16) int8_t tile[PT][PT + 4];  // [r][k], centred codes
  const int t = threadIdx.x;
  const int64_t r0 = (int64_t)blockIdx.x * PT;
  const int64_t kbeg = (int64_t)blockIdx.y * CK, kend = kbeg + CK < Kp ? kbeg + CK : Kp;
  const uint32_t flip = SIGNED ? 0u : 0x80808080u;  // u8 code - 128 == int8 of (code ^ 0x80)
  const int a = t >> 2, b = (t & 3) * 16;
  int part = 0;
  for (int64_t k0 = kbeg; k0 < kend; k0 += PT) {
    // load 64 x 64 codes: thread -> one 16-byte segment of a source line
    if (k_fast) {
      const int64_t r = r0 + a, k = k0 + b;
      if (VEC && r < R && k + 16 <= K) {
        const uint4 v = __ldcs(reinterpret_cast<const uint4*>(X + r * K + k));
        uint32_t* d = reinterpret_cast<uint32_t*>(&tile[a][b]);
        d[0] = v.x ^ flip; d[1] = v.y ^ flip; d[2] = v.z ^ flip; d[3] = v.w ^ flip;
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e)
          tile[a][b + e] = (r < R && k + e < K) ? (int8_t)(X[r * K + k + e] ^ (uint8_t)flip) : (int8_t)0;
      }
    } else {
      const int64_t k = k0 + a, r = r0 + b;
      if (VEC && k < K && r + 16 <= R) {
        const uint4 v = __ldcs(reinterpret_cast<const uint4*>(X + k * R + r));
        const uint32_t w[4] = {v.x ^ flip, v.y ^ flip, v.z ^ flip, v.w ^ flip};
#pragma unroll
        for (int e = 0; e < 16; ++e) tile[b + e][a] = (int8_t)(w[e >> 2] >> (8 * (e & 3)));
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e)
          tile[b + e][a] = (r + e < R && k < K) ? (int8_t)(X[k * R + r + e] ^ (uint8_t)flip) : (int8_t)0;
      }
    }
    __syncthreads();
    // write: thread -> row a, 16 consecutive k as bf16 (two 16-byte stores)
    const int64_t r = r0 + a;
    if (r < R) {
      // centred code c as the fp32 1.5 * 2^23 + (c + 128) by one byte
      // permute, minus 1.5 * 2^23 + 128: exactly c; its bf16 is the top half
      const uint32_t* src = reinterpret_cast<const uint32_t*>(&tile[a][b]);
      uint32_t w[8];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t cw = src[q];
        part = __dp4a((int)cw, 0x01010101, part);
        const uint32_t uw = cw ^ 0x80808080u;
        float f[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          f[e] = __fsub_rn(__uint_as_float(__byte_perm(uw, 0x4B400000u, 0x7640u + e)), 12583040.0f);
        w[2 * q] = __byte_perm(__float_as_uint(f[0]), __float_as_uint(f[1]), 0x7632);
        w[2 * q + 1] = __byte_perm(__float_as_uint(f[2]), __float_as_uint(f[3]), 0x7632);
      }
      uint4* dst = reinterpret_cast<uint4*>(Xc + r * Kp + k0 + b);
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
    __syncthreads();
  }
  // the four threads of a row are adjacent lanes
  part += __shfl_xor_sync(0xffffffffu, part, 1);
  part += __shfl_xor_sync(0xffffffffu, part, 2);
  const int64_t r = r0 + a;
  if ((t & 3) == 0 && r < R) atomicAdd(sums + r, part);
}

// The same result when K is the contiguous index (no transpose): a stream
// of 16-code groups, Xc keeping X's row order.  Thread g takes group g of
// the padded rows (Kp / 16 groups each) and three more a grid apart, all
// loaded before any is used; groups at or beyond K are written as zeros.
// A row's groups are consecutive threads, so its sum is reduced across the
// warp when all lanes share the row, else added lane by lane.  Needs
// K % 16 == 0 and a 16-byte aligned X.
template <bool SIGNED>
__global__ void __launch_bounds__(256)
center_rows(const uint8_t* __restrict__ X, int64_t R, int64_t K, int64_t Kp, __nv_bfloat16* __restrict__ Xc,
            int32_t* __restrict__ sums) {
  constexpr int U = 4;
  const uint32_t flip = SIGNED ? 0u : 0x80808080u;  // u8 code - 128 == int8 of (code ^ 0x80)
  const int64_t gpr = Kp / 16, total = R * gpr;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int lane = threadIdx.x & 31;
  // (row, group in row) of g, advanced by addition: one division per thread
  const int64_t sr = stride / gpr, sg = stride - sr * gpr;
  int64_t g0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  int64_t r_at = g0 / gpr, c_at = g0 - r_at * gpr;
  auto advance = [&](int64_t& r, int64_t& c) {
    r += sr;
    c += sg;
    if (c >= gpr) {
      c -= gpr;
      ++r;
    }
  };
  for (; g0 - lane < total; g0 += U * stride) {
    uint4 v[U];
    int64_t rr[U], kk[U];
    {
      int64_t r = r_at, c = c_at;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (u) advance(r, c);
        rr[u] = r;
        kk[u] = c * 16;
      }
      advance(r, c);
      r_at = r;
      c_at = c;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t g = g0 + u * stride;
      v[u] = (g < total && kk[u] < K) ? __ldcs(reinterpret_cast<const uint4*>(X + rr[u] * K + kk[u]))
                                      : make_uint4(flip, flip, flip, flip);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t g = g0 + u * stride;
      const uint32_t wd[4] = {v[u].x ^ flip, v[u].y ^ flip, v[u].z ^ flip, v[u].w ^ flip};
      uint32_t o[8];
      int part = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        // two centred codes (int8 bytes) as bf16: exact through fp32
        const int c0 = (int)(int8_t)(wd[e >> 1] >> (16 * (e & 1))), c1 = (int)(int8_t)(wd[e >> 1] >> (16 * (e & 1) + 8));
        part += c0 + c1;
        o[e] = (__float_as_uint((float)c0) >> 16) | (__float_as_uint((float)c1) & 0xffff0000u);
      }
      if (g < total) {
        uint4* dst = reinterpret_cast<uint4*>(Xc + rr[u] * Kp + kk[u]);
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
      }
      // row sum: one atomic per warp when the warp's groups share a row
      const int64_t r = g < total ? rr[u] : -1;
      const int64_t r_first = __shfl_sync(0xffffffffu, r, 0);
      if (__all_sync(0xffffffffu, r == r_first)) {
        part = __reduce_add_sync(0xffffffffu, part);
        if (lane == 0 && r >= 0) atomicAdd(sums + r, part);
      } else if (r >= 0 && part != 0) {
        atomicAdd(sums + r, part);
      }
    }
  }
}

// g[j] = cb - bz[j]; e[j] = colsum[j] + K g[j] (wrapping int32);
// bsc[j] = b_scale[j] (expanded when per tensor).  Thread 0 also writes the
// per-tensor row values d0 = ca - za and asc0 when asked (write_row0).
__global__ void col_params(const int32_t* __restrict__ colsum, const float* __restrict__ b_scale,
                           const uint8_t* __restrict__ b_zp, int b_signed, int64_t n_b, int64_t N, int64_t K, int cb,
                           int32_t* __restrict__ g, int32_t* __restrict__ e, float* __restrict__ bsc, int write_row0,
                           int32_t d0, float asc0, int32_t* __restrict__ d, float* __restrict__ asc) {
  const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (write_row0 && j == 0) {
    d[0] = d0;
    asc[0] = asc0;
  }
  if (j >= N) return;
  const int64_t pj = n_b == N ? j : 0;
  const int bz = b_zp ? (b_signed ? (int)(int8_t)b_zp[pj] : (int)b_zp[pj]) : 0;
  const int32_t gj = cb - bz;
  g[j] = gj;
  e[j] = (int32_t)((uint32_t)colsum[j] + (uint32_t)K * (uint32_t)gj);
  bsc[j] = __ldg(b_scale + pj);
}

// d[i] = ca - a_zero_point[i] for per-row zero points (0 when none).
__global__ void row_params(const uint8_t* __restrict__ a_zp, int a_signed, int64_t n, int ca,
                           int32_t* __restrict__ d) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int za = a_zp ? (a_signed ? (int)(int8_t)a_zp[i] : (int)a_zp[i]) : 0;
  d[i] = ca - za;
}

// Range of a whole fp32 tensor, widened to contain 0: mm[0] = -min(0, min x)
// and mm[1] = max(0, max x), both non-negative, so their bit patterns order
// like the values and atomicMax on them is exact.  mm starts at 0.
__global__ void __launch_bounds__(256) tensor_range(const float* __restrict__ x, int64_t n, uint32_t* mm) {
  float nmn = 0.0f, mx = 0.0f;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if ((reinterpret_cast<uintptr_t>(x) & 15) == 0) {
    const int64_t n4 = n / 4;
    // four 16-byte loads per thread in flight
    for (int64_t i0 = t; i0 < n4; i0 += 4 * stride) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t i = i0 + u * stride;
        v[u] = i < n4 ? __ldcs(reinterpret_cast<const float4*>(x) + i) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        mx = fmaxf(fmaxf(mx, fmaxf(v[u].x, v[u].y)), fmaxf(v[u].z, v[u].w));
        nmn = fmaxf(fmaxf(nmn, fmaxf(-v[u].x, -v[u].y)), fmaxf(-v[u].z, -v[u].w));
      }
    }
    for (int64_t i = n4 * 4 + t; i < n; i += stride) {
      mx = fmaxf(mx, x[i]);
      nmn = fmaxf(nmn, -x[i]);
    }
  } else {
    for (int64_t i = t; i < n; i += stride) {
      mx = fmaxf(mx, x[i]);
      nmn = fmaxf(nmn, -x[i]);
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    nmn = fmaxf(nmn, __shfl_xor_sync(0xffffffffu, nmn, o));
  }
  // one merge per block: atomics on a single word serialize
  __shared__ float red[2][8];
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    red[0][warp] = nmn;
    red[1][warp] = mx;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) {
      nmn = fmaxf(nmn, red[0][w]);
      mx = fmaxf(mx, red[1][w]);
    }
    atomicMax(mm, __float_as_uint(nmn));
    atomicMax(mm + 1, __float_as_uint(mx));
  }
}

// Per-tensor uint8 quantization of fp32 A (M x K) straight into the centred
// bf16 operand: code = saturate(rint(A / s) + z), A' = code - 128, with s, z
// from the tensor's range exactly as a row of the dynamic inner product;
// rowsum[i] = sum_k A'.  One warp per row.  Block 0 publishes d = 128 - z and
// s for the epilogue and, when given, the scale and zero point.
__global__ void __launch_bounds__(256)
quantize_tensor_center(const float* __restrict__ A, int64_t M, int64_t K, int64_t Kp, const uint32_t* __restrict__ mm,
                       __nv_bfloat16* __restrict__ Ac, int32_t* __restrict__ rowsum, int32_t* __restrict__ d_out,
                       float* __restrict__ asc_out, float* __restrict__ a_scale_out,
                       uint8_t* __restrict__ a_zp_out) {
  const float mn = -__uint_as_float(mm[0]), mx = __uint_as_float(mm[1]);
  float sc;
  int z;
  row_scale_zero(mn, mx, sc, z);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *d_out = 128 - z;
    *asc_out = sc;
    if (a_scale_out) *a_scale_out = sc;
    if (a_zp_out) *a_zp_out = (uint8_t)z;
  }
  const int lane = threadIdx.x & 31;
  const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (row >= M) return;
  const float lo_z = (float)(-z), hi_z = (float)(255 - z);
  const float* a = A + row * K;
  __nv_bfloat16* out = Ac + row * Kp;
  int part = 0;
  // bf16 bits of a code - 128 (exact small integer) from its fp32 image
  auto bits = [](int c) { return __float_as_uint(__fsub_rn(__int_as_float(0x4B400000 + c), 12582912.0f)); };
  auto emit = [&](int64_t k0, const float (&v)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int e2 = 0; e2 < 4; ++e2) {
      int c[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        c[h] = k0 + 2 * e2 + h < K ? (int)(row_code(v[2 * e2 + h], sc, lo_z, hi_z, z)) - 128 : 0;
        part += c[h];
      }
      w[e2] = (bits(c[0]) >> 16) | (bits(c[1]) & 0xffff0000u);
    }
    *reinterpret_cast<uint4*>(out + k0) = make_uint4(w[0], w[1], w[2], w[3]);
  };
  const bool vec = K % 8 == 0 && (reinterpret_cast<uintptr_t>(A) & 15) == 0;
  if (vec) {
    // two 8-element groups per lane in flight (four 16-byte loads)
    for (int64_t k0 = (int64_t)lane * 8; k0 < Kp; k0 += 512) {
      float v[2][8];
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        const int64_t k = k0 + 256 * g;
        float4 x0 = make_float4(0.0f, 0.0f, 0.0f, 0.0f), x1 = x0;
        if (k < K) {
          x0 = __ldcs(reinterpret_cast<const float4*>(a + k));
          x1 = __ldcs(reinterpret_cast<const float4*>(a + k + 4));
        }
        v[g][0] = x0.x; v[g][1] = x0.y; v[g][2] = x0.z; v[g][3] = x0.w;
        v[g][4] = x1.x; v[g][5] = x1.y; v[g][6] = x1.z; v[g][7] = x1.w;
      }
#pragma unroll
      for (int g = 0; g < 2; ++g)
        if (k0 + 256 * g < Kp) emit(k0 + 256 * g, v[g]);
    }
  } else {
    for (int64_t k0 = (int64_t)lane * 8; k0 < Kp; k0 += 256) {
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = k0 + e < K ? a[k0 + e] : 0.0f;
      emit(k0, v);
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  if (lane == 0) rowsum[row] = part;
}

size_t a256(size_t v) { return (v + 255) & ~size_t(255); }

struct QgLayout {
  size_t Ac, rowsum, Bc, colsum, g, e, bsc, d, asc, mm, total;
};

QgLayout qg_layout(int64_t M, int64_t N, int64_t K) {
  const int64_t Kp = round_up(K, 64);
  QgLayout L{};
  size_t o = 0;
  auto take = [&](size_t n) {
    const size_t at = o;
    o += a256(n);
    return at;
  };
  L.Ac = take((size_t)M * Kp * 2);
  L.rowsum = take((size_t)M * 4);
  L.Bc = take((size_t)N * Kp * 2);
  L.colsum = take((size_t)N * 4);
  L.g = take((size_t)N * 4);
  L.e = take((size_t)N * 4);
  L.bsc = take((size_t)N * 4);
  L.d = take((size_t)M * 4);
  L.asc = take(4);
  L.mm = take(8);
  L.total = o;
  return L;
}

int launch_center(const void* X, int type, int64_t R, int64_t K, int64_t Kp, int k_fast, __nv_bfloat16* Xc,
                  int32_t* sums, cudaStream_t s) {
  const int64_t bx = ceil_div(R, PT), by = ceil_div(Kp, CK);
  if (bx > 0x7fffffff || by > 65535) return fail(I8Q_ERR_UNSUPPORTED, "qgemm: operand too large");
  if (bx == 0) return I8Q_OK;
  I8Q_PROF("qgemm_center", s);
  I8Q_CUDA_TRY(cudaMemsetAsync(sums, 0, (size_t)R * sizeof(int32_t), s));
  if (!k_fast && repack_tiles_ok(X, K, R, R, nullptr, Xc, Kp)) {
    // transposed: 128 x 128 tiles turned by byte permutes
    launch_repack_tiles(X, type != I8Q_S8, K, R, R, nullptr, Xc, Kp, sums, 0, s);
    I8Q_LAUNCH_CHECK("repack_tiles (centre)");
    return I8Q_OK;
  }
  const bool vec = (reinterpret_cast<uintptr_t>(X) & 15) == 0 && (k_fast ? K % 16 == 0 : R % 16 == 0);
  const auto* x8 = static_cast<const uint8_t*>(X);
  if (k_fast && vec) {
    // no transpose: a stream; one wave of resident blocks
    static const int per_sm = [] {
      int a = 0, b = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&a, center_rows<true>, 256, 0) != cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, center_rows<false>, 256, 0) != cudaSuccess)
        cudaGetLastError();
      return std::max(1, std::min(a, b));
    }();
    const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>(ceil_div(R * (Kp / 16), 256 * 4),
                                                                  (int64_t)sm_count() * per_sm));
    if (type == I8Q_S8) center_rows<true><<<(unsigned)blocks, 256, 0, s>>>(x8, R, K, Kp, Xc, sums);
    else center_rows<false><<<(unsigned)blocks, 256, 0, s>>>(x8, R, K, Kp, Xc, sums);
    I8Q_LAUNCH_CHECK("center_rows");
    return I8Q_OK;
  }
  const dim3 grid((unsigned)bx, (unsigned)by);
  if (type == I8Q_S8) {
    if (vec) center_operand<true, true><<<grid, 256, 0, s>>>(x8, R, K, Kp, k_fast, Xc, sums);
    else center_operand<true, false><<<grid, 256, 0, s>>>(x8, R, K, Kp, k_fast, Xc, sums);
  } else {
    if (vec) center_operand<false, true><<<grid, 256, 0, s>>>(x8, R, K, Kp, k_fast, Xc, sums);
    else center_operand<false, false><<<grid, 256, 0, s>>>(x8, R, K, Kp, k_fast, Xc, sums);
  }
  I8Q_LAUNCH_CHECK("center_operand");
  return I8Q_OK;
}

// Where the per-row values d = ca - a_zero_point and asc (the row scale) come
// from.
enum RowMode : int {
  ROWS_HOST = 0,    // one d and asc given on the host (written by col_params)
  ROWS_DEVICE = 1,  // a_scale and a_zero_point on the device, 1 or M entries
  ROWS_READY = 2,   // d[0] and asc[0] already written on the device
};
struct RowParams {
  int mode;
  int32_t d0;             // ROWS_HOST
  float asc0;             // ROWS_HOST
  const float* asc_dev;   // ROWS_DEVICE
  const uint8_t* za_dev;  // ROWS_DEVICE, or null (zero)
  int64_t n_a;            // ROWS_DEVICE: 1 or M
  int a_signed;
};

// Everything after the A operand is centred: centre B, form the column and
// row parameters, run the product with the epilogue in qg (its C, bias and
// output fields already set).
int finish_product(const QgLayout& L, uint8_t* base, int64_t M, int64_t N, int64_t K, int64_t Kp, const void* B,
                   int btype, int transB, const float* b_scale, const void* b_zero_point, int64_t n_b, int ca,
                   const RowParams& rp, QgEpilogue qg, cudaStream_t s) {
  auto* Ac = reinterpret_cast<__nv_bfloat16*>(base + L.Ac);
  auto* Bc = reinterpret_cast<__nv_bfloat16*>(base + L.Bc);
  auto* colsum = reinterpret_cast<int32_t*>(base + L.colsum);
  auto* g = reinterpret_cast<int32_t*>(base + L.g);
  auto* e = reinterpret_cast<int32_t*>(base + L.e);
  auto* bsc = reinterpret_cast<float*>(base + L.bsc);
  auto* d = reinterpret_cast<int32_t*>(base + L.d);
  auto* asc = reinterpret_cast<float*>(base + L.asc);
  int rc = launch_center(B, btype, N, K, Kp, transB ? 1 : 0, Bc, colsum, s);
  if (rc) return rc;
  const int cb = btype == I8Q_U8 ? 128 : 0;
  {
    I8Q_PROF("qgemm_params", s);
    col_params<<<(unsigned)ceil_div(N, 256), 256, 0, s>>>(colsum, b_scale, static_cast<const uint8_t*>(b_zero_point),
                                                         btype == I8Q_S8, n_b, N, K, cb, g, e, bsc,
                                                         rp.mode == ROWS_HOST ? 1 : 0, rp.d0, rp.asc0, d, asc);
    I8Q_LAUNCH_CHECK("col_params");
    if (rp.mode == ROWS_DEVICE) {
      row_params<<<(unsigned)ceil_div(rp.n_a, 256), 256, 0, s>>>(rp.za_dev, rp.a_signed, rp.n_a, ca, d);
      I8Q_LAUNCH_CHECK("row_params");
    }
  }
  qg.rowsum = reinterpret_cast<int32_t*>(base + L.rowsum);
  qg.d = d;
  qg.g = g;
  qg.e = e;
  qg.bsc = bsc;
  if (rp.mode == ROWS_DEVICE) {
    const int64_t st = rp.n_a == M && M > 1 ? 1 : 0;
    qg.d_stride = st;
    qg.asc = rp.asc_dev;
    qg.asc_stride = st;
  } else {
    qg.d_stride = 0;
    qg.asc = asc;
    qg.asc_stride = 0;
  }
  qg.ldy = N;
  // |A'| <= 2^7 and |B'| <= 2^7
  return launch_qgemm_tc(Ac, Bc, M, N, Kp, 14, qg, s);
}

int check_common(const char* who, int64_t M, int64_t N, int64_t K, int btype, const void* B, const float* b_scale,
                 const void* Y, size_t n_b, void* workspace, size_t ws_bytes, const QgLayout& L) {
  const std::string w(who);
  if (M <= 0 || N <= 0 || K <= 0) return fail(I8Q_ERR_INVALID_ARG, w + ": M, N, K must be >= 1");
  if (K > 65536) return fail(I8Q_ERR_UNSUPPORTED, w + ": K > 65536 (int32 sums could overflow)");
  if (btype != I8Q_U8 && btype != I8Q_S8) return fail(I8Q_ERR_INVALID_ARG, w + ": B must be I8Q_U8 or I8Q_S8");
  if (!B || !b_scale || !Y) return fail(I8Q_ERR_INVALID_ARG, w + ": B, b_scale and Y are required");
  if (n_b != 1 && (int64_t)n_b != N) return fail(I8Q_ERR_INVALID_ARG, w + ": b_scale must have 1 or N entries");
  if (!workspace || ws_bytes < L.total)
    return fail(I8Q_ERR_INVALID_ARG, w + ": workspace missing or smaller than the workspace size");
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return fail(I8Q_ERR_INVALID_ARG, w + ": workspace must be 256-byte aligned");
  return I8Q_OK;
}

}  // namespace
}  // namespace i8q

using namespace i8q;

extern "C" size_t i8q_qgemm_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  return qg_layout(M, N, K).total;
}

extern "C" size_t i8q_matmul_integer_workspace_size(int64_t M, int64_t N, int64_t K) {
  return i8q_qgemm_workspace_size(M, N, K);
}

extern "C" int i8q_qgemm(const void* A, int atype, int transA, int64_t M, int64_t K, float a_scale,
                         int a_zero_point, const void* B, int btype, int transB, int64_t N, const float* b_scale,
                         const void* b_zero_point, size_t n_b, const int32_t* C, int64_t c_rows, int64_t c_cols,
                         float alpha, int quantize_y, float y_scale, int y_zero_point, int ytype, void* Y,
                         void* workspace, size_t ws_bytes, void* stream) {
  if (atype != I8Q_U8 && atype != I8Q_S8) return fail(I8Q_ERR_INVALID_ARG, "qgemm: A and B must be I8Q_U8 or I8Q_S8");
  const QgLayout L = qg_layout(M, N, K);
  int rc = check_common("qgemm", M, N, K, btype, B, b_scale, Y, n_b, workspace, ws_bytes, L);
  if (rc) return rc;
  if (!A) return fail(I8Q_ERR_INVALID_ARG, "qgemm: A is required");
  const int alo = atype == I8Q_U8 ? 0 : -128, ahi = atype == I8Q_U8 ? 255 : 127;
  if (a_zero_point < alo || a_zero_point > ahi) return fail(I8Q_ERR_INVALID_ARG, "qgemm: a_zero_point out of A's range");
  if (C && !((c_rows == 1 || c_rows == M) && (c_cols == 1 || c_cols == N)))
    return fail(I8Q_ERR_INVALID_ARG, "qgemm: C must be broadcastable to (M, N) as (1|M, 1|N)");
  if (quantize_y) {
    if (ytype != I8Q_U8 && ytype != I8Q_S8) return fail(I8Q_ERR_INVALID_ARG, "qgemm: quantized Y must be U8 or S8");
    const int ylo = ytype == I8Q_U8 ? 0 : -128, yhi = ytype == I8Q_U8 ? 255 : 127;
    if (y_zero_point < ylo || y_zero_point > yhi) return fail(I8Q_ERR_INVALID_ARG, "qgemm: y_zero_point out of range");
  }
  cudaStream_t s = as_stream(stream);
  const int64_t Kp = round_up(K, 64);
  uint8_t* base = static_cast<uint8_t*>(workspace);
  // A is (M, K), K contiguous, unless transA; B is (K, N), N contiguous,
  // unless transB
  rc = launch_center(A, atype, M, K, Kp, transA ? 0 : 1, reinterpret_cast<__nv_bfloat16*>(base + L.Ac),
                     reinterpret_cast<int32_t*>(base + L.rowsum), s);
  if (rc) return rc;
  const int ca = atype == I8Q_U8 ? 128 : 0;
  RowParams rp{};
  rp.mode = ROWS_HOST;
  rp.d0 = ca - a_zero_point;
  rp.asc0 = alpha * a_scale;  // the multiplier's first factor, rounded once
  QgEpilogue qg{};
  qg.C = C;
  qg.c_si = C ? (c_rows == 1 ? 0 : c_cols) : 0;
  qg.c_sj = C ? (c_cols == 1 ? 0 : 1) : 0;
  qg.c_col = (C && qg.c_si == 0) ? 1 : 0;  // QGemm has no bias
  qg.ytype = quantize_y ? ytype : I8Q_F32;
  qg.y_scale = y_scale;
  qg.y_rcp = quot_rcp(y_scale);
  qg.y_zero_point = y_zero_point;
  qg.Y = Y;
  return finish_product(L, base, M, N, K, Kp, B, btype, transB, b_scale, b_zero_point, (int64_t)n_b, ca, rp, qg, s);
}

extern "C" int i8q_matmul_integer_to_float(const void* A, int atype, int64_t M, int64_t K, const void* B, int btype,
                                           int64_t N, const float* a_scale, const void* a_zero_point, size_t n_a,
                                           const float* b_scale, const void* b_zero_point, size_t n_b,
                                           const float* bias, float* Y, void* workspace, size_t ws_bytes,
                                           void* stream) {
  if (atype != I8Q_U8 && atype != I8Q_S8)
    return fail(I8Q_ERR_INVALID_ARG, "matmul_integer_to_float: A must be I8Q_U8 or I8Q_S8");
  const QgLayout L = qg_layout(M, N, K);
  int rc = check_common("matmul_integer_to_float", M, N, K, btype, B, b_scale, Y, n_b, workspace, ws_bytes, L);
  if (rc) return rc;
  if (!A || !a_scale) return fail(I8Q_ERR_INVALID_ARG, "matmul_integer_to_float: A and a_scale are required");
  if (n_a != 1 && (int64_t)n_a != M)
    return fail(I8Q_ERR_INVALID_ARG, "matmul_integer_to_float: a_scale must have 1 entry or one per row of A");
  cudaStream_t s = as_stream(stream);
  const int64_t Kp = round_up(K, 64);
  uint8_t* base = static_cast<uint8_t*>(workspace);
  rc = launch_center(A, atype, M, K, Kp, 1, reinterpret_cast<__nv_bfloat16*>(base + L.Ac),
                     reinterpret_cast<int32_t*>(base + L.rowsum), s);
  if (rc) return rc;
  RowParams rp{};
  rp.mode = ROWS_DEVICE;
  rp.asc_dev = a_scale;
  rp.za_dev = static_cast<const uint8_t*>(a_zero_point);
  rp.n_a = (int64_t)n_a;
  rp.a_signed = atype == I8Q_S8;
  QgEpilogue qg{};
  qg.bias = bias;
  qg.ytype = I8Q_F32;
  qg.Y = Y;
  return finish_product(L, base, M, N, K, Kp, B, btype, 0, b_scale, b_zero_point, (int64_t)n_b,
                        atype == I8Q_U8 ? 128 : 0, rp, qg, s);
}

extern "C" int i8q_dynamic_quantize_matmul(const float* A, int64_t M, int64_t K, const void* B, int btype, int64_t N,
                                           const float* b_scale, const void* b_zero_point, size_t n_b,
                                           const float* bias, float* Y, float* a_scale_out,
                                           uint8_t* a_zero_point_out, void* workspace, size_t ws_bytes,
                                           void* stream) {
  const QgLayout L = qg_layout(M, N, K);
  int rc = check_common("dynamic_quantize_matmul", M, N, K, btype, B, b_scale, Y, n_b, workspace, ws_bytes, L);
  if (rc) return rc;
  if (!A) return fail(I8Q_ERR_INVALID_ARG, "dynamic_quantize_matmul: A is required");
  cudaStream_t s = as_stream(stream);
  const int64_t Kp = round_up(K, 64);
  uint8_t* base = static_cast<uint8_t*>(workspace);
  auto* mm = reinterpret_cast<uint32_t*>(base + L.mm);
  {
    I8Q_PROF("dqmm_quantize_a", s);
    I8Q_CUDA_TRY(cudaMemsetAsync(mm, 0, 8, s));
    const int64_t n = M * K;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(ceil_div(n, 256 * 8), (int64_t)sm_count() * 8));
    tensor_range<<<grid, 256, 0, s>>>(A, n, mm);
    I8Q_LAUNCH_CHECK("tensor_range");
    const int64_t blocks = ceil_div(M, 8);
    if (blocks > 0x7fffffff) return fail(I8Q_ERR_UNSUPPORTED, "dynamic_quantize_matmul: too many rows");
    quantize_tensor_center<<<(unsigned)blocks, 256, 0, s>>>(
        A, M, K, Kp, mm, reinterpret_cast<__nv_bfloat16*>(base + L.Ac), reinterpret_cast<int32_t*>(base + L.rowsum),
        reinterpret_cast<int32_t*>(base + L.d), reinterpret_cast<float*>(base + L.asc), a_scale_out, a_zero_point_out);
    I8Q_LAUNCH_CHECK("quantize_tensor_center");
  }
  RowParams rp{};
  rp.mode = ROWS_READY;
  QgEpilogue qg{};
  qg.bias = bias;
  qg.ytype = I8Q_F32;
  qg.Y = Y;
  return finish_product(L, base, M, N, K, Kp, B, btype, 0, b_scale, b_zero_point, (int64_t)n_b, 128, rp, qg, s);
}
