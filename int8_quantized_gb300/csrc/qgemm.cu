// qgemm.cu -- QGemm (ONNX Runtime contrib schemas, "QGemm") on the
// exact-integer tensor-core path.
//
//   acc[i,j] = sum_k (A[i,k] - a_zero_point) * (B[k,j] - b_zero_point[j])
//   acc += C[i,j]                           (int32, broadcast from (1|M, 1|N))
//   y = (float)acc * ((alpha * a_scale) * b_scale[j])
//   quantized output: y = saturate(rint(y / y_scale) + y_zero_point)
// C carries the scale alpha * a_scale * b_scale and zero point 0 (the schema
// writes alpha / beta but defines no beta), so it adds to the integer sum;
// the rescale is DequantizeLinear of the sum followed by QuantizeLinear.
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

constexpr int PT = 64;  // rows x K elements per tile of the operand pass

// Xc[r][k] = bf16(X(r,k) - cx) for k < K, 0 for K <= k < Kp, and
// sums[r] = sum_k (X(r,k) - cx).  X(r,k) = X[r*K + k] when k_fast, else
// X[k*R + r].  One CTA owns 64 rows and walks K in 64-wide tiles through
// shared memory, reading the source along its contiguous index.
template <bool SIGNED>
__global__ void __launch_bounds__(256)
center_operand(const uint8_t* __restrict__ X, int64_t R, int64_t K, int64_t Kp, int k_fast,
               __nv_bfloat16* __restrict__ Xc, int32_t* __restrict__ sums) {
  __shared__ int8_t tile[PT][PT + 4];  // [r][k], centred codes
  const int t = threadIdx.x;
  const int64_t r0 = (int64_t)blockIdx.x * PT;
  const uint8_t flip = SIGNED ? 0 : 0x80;  // u8 code - 128 == int8 of (code ^ 0x80)
  int part = 0;
  for (int64_t k0 = 0; k0 < Kp; k0 += PT) {
    // load 64 x 64 codes: thread -> one source line segment of 16 bytes
    const int a = t >> 2, b = (t & 3) * 16;
    if (k_fast) {
      const int64_t r = r0 + a;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int64_t k = k0 + b + e;
        tile[a][b + e] = (r < R && k < K) ? (int8_t)(X[r * K + k] ^ flip) : (int8_t)0;
      }
    } else {
      const int64_t k = k0 + a;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int64_t r = r0 + b + e;
        tile[b + e][a] = (r < R && k < K) ? (int8_t)(X[k * R + r] ^ flip) : (int8_t)0;
      }
    }
    __syncthreads();
    // write: thread -> row a, 16 consecutive k as bf16 (two 16-byte stores)
    const int64_t r = r0 + a;
    if (r < R) {
      uint32_t w[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int c0 = tile[a][b + 2 * e], c1 = tile[a][b + 2 * e + 1];
        part += c0 + c1;
        w[e] = (__float_as_uint((float)c0) >> 16) | (__float_as_uint((float)c1) & 0xffff0000u);
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
  const int64_t r = r0 + (t >> 2);
  if ((t & 3) == 0 && r < R) sums[r] = part;
}

// g[j] = cb - bz[j]; h[j] = (ca - za) * colsum[j] + K (ca - za) g[j] (wrapping
// int32); mult[j] = (alpha * a_scale) * b_scale[j].
__global__ void qgemm_col_params(const int32_t* __restrict__ colsum, const float* __restrict__ b_scale,
                                 const uint8_t* __restrict__ b_zp, int b_signed, int64_t n_b, int64_t N, int64_t K,
                                 int ca, int za, int cb, float alpha, float a_scale, int32_t* __restrict__ g,
                                 int32_t* __restrict__ h, float* __restrict__ mult) {
  const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= N) return;
  const int64_t pj = n_b == N ? j : 0;
  const int bz = b_zp ? (b_signed ? (int)(int8_t)b_zp[pj] : (int)b_zp[pj]) : 0;
  const int32_t gj = cb - bz;
  const uint32_t da = (uint32_t)(ca - za);
  g[j] = gj;
  h[j] = (int32_t)(da * (uint32_t)colsum[j] + (uint32_t)K * da * (uint32_t)gj);
  const float m = __fmul_rn(alpha, a_scale);
  mult[j] = __fmul_rn(m, __ldg(b_scale + pj));
}

size_t a256(size_t v) { return (v + 255) & ~size_t(255); }

struct QgLayout {
  size_t Ac, rowsum, Bc, colsum, g, h, mult, total;
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
  L.h = take((size_t)N * 4);
  L.mult = take((size_t)N * 4);
  L.total = o;
  return L;
}

int launch_center(const void* X, int type, int64_t R, int64_t K, int64_t Kp, int k_fast, __nv_bfloat16* Xc,
                  int32_t* sums, cudaStream_t s) {
  const int64_t blocks = ceil_div(R, PT);
  if (blocks > 0x7fffffff) return fail(I8Q_ERR_UNSUPPORTED, "qgemm: too many rows");
  I8Q_PROF("qgemm_center", s);
  if (type == I8Q_S8)
    center_operand<true><<<(unsigned)blocks, 256, 0, s>>>(static_cast<const uint8_t*>(X), R, K, Kp, k_fast, Xc, sums);
  else
    center_operand<false><<<(unsigned)blocks, 256, 0, s>>>(static_cast<const uint8_t*>(X), R, K, Kp, k_fast, Xc,
                                                            sums);
  I8Q_LAUNCH_CHECK("center_operand");
  return I8Q_OK;
}

}  // namespace
}  // namespace i8q

using namespace i8q;

extern "C" size_t i8q_qgemm_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  return qg_layout(M, N, K).total;
}

extern "C" int i8q_qgemm(const void* A, int atype, int transA, int64_t M, int64_t K, float a_scale,
                         int a_zero_point, const void* B, int btype, int transB, int64_t N, const float* b_scale,
                         const void* b_zero_point, size_t n_b, const int32_t* C, int64_t c_rows, int64_t c_cols,
                         float alpha, int quantize_y, float y_scale, int y_zero_point, int ytype, void* Y,
                         void* workspace, size_t ws_bytes, void* stream) {
  if (M <= 0 || N <= 0 || K <= 0) return fail(I8Q_ERR_INVALID_ARG, "qgemm: M, N, K must be >= 1");
  if (K > 65536) return fail(I8Q_ERR_UNSUPPORTED, "qgemm: K > 65536 (int32 sums could overflow)");
  if ((atype != I8Q_U8 && atype != I8Q_S8) || (btype != I8Q_U8 && btype != I8Q_S8))
    return fail(I8Q_ERR_INVALID_ARG, "qgemm: A and B must be I8Q_U8 or I8Q_S8");
  if (!A || !B || !b_scale || !Y) return fail(I8Q_ERR_INVALID_ARG, "qgemm: A, B, b_scale and Y are required");
  if (n_b != 1 && (int64_t)n_b != N) return fail(I8Q_ERR_INVALID_ARG, "qgemm: b_scale must have 1 or N entries");
  const int alo = atype == I8Q_U8 ? 0 : -128, ahi = atype == I8Q_U8 ? 255 : 127;
  if (a_zero_point < alo || a_zero_point > ahi) return fail(I8Q_ERR_INVALID_ARG, "qgemm: a_zero_point out of A's range");
  if (C && !((c_rows == 1 || c_rows == M) && (c_cols == 1 || c_cols == N)))
    return fail(I8Q_ERR_INVALID_ARG, "qgemm: C must be broadcastable to (M, N) as (1|M, 1|N)");
  if (quantize_y) {
    if (ytype != I8Q_U8 && ytype != I8Q_S8) return fail(I8Q_ERR_INVALID_ARG, "qgemm: quantized Y must be U8 or S8");
    const int ylo = ytype == I8Q_U8 ? 0 : -128, yhi = ytype == I8Q_U8 ? 255 : 127;
    if (y_zero_point < ylo || y_zero_point > yhi) return fail(I8Q_ERR_INVALID_ARG, "qgemm: y_zero_point out of range");
  }
  const QgLayout L = qg_layout(M, N, K);
  if (!workspace || ws_bytes < L.total)
    return fail(I8Q_ERR_INVALID_ARG, "qgemm: workspace missing or smaller than qgemm_workspace_size");
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return fail(I8Q_ERR_INVALID_ARG, "qgemm: workspace must be 256-byte aligned");
  cudaStream_t s = as_stream(stream);
  const int64_t Kp = round_up(K, 64);
  uint8_t* base = static_cast<uint8_t*>(workspace);
  auto* Ac = reinterpret_cast<__nv_bfloat16*>(base + L.Ac);
  auto* Bc = reinterpret_cast<__nv_bfloat16*>(base + L.Bc);
  auto* rowsum = reinterpret_cast<int32_t*>(base + L.rowsum);
  auto* colsum = reinterpret_cast<int32_t*>(base + L.colsum);
  auto* g = reinterpret_cast<int32_t*>(base + L.g);
  auto* h = reinterpret_cast<int32_t*>(base + L.h);
  auto* mult = reinterpret_cast<float*>(base + L.mult);
  // A is (M, K), K contiguous, unless transA; B is (K, N), N contiguous,
  // unless transB
  int rc = launch_center(A, atype, M, K, Kp, transA ? 0 : 1, Ac, rowsum, s);
  if (rc) return rc;
  rc = launch_center(B, btype, N, K, Kp, transB ? 1 : 0, Bc, colsum, s);
  if (rc) return rc;
  const int ca = atype == I8Q_U8 ? 128 : 0, cb = btype == I8Q_U8 ? 128 : 0;
  {
    I8Q_PROF("qgemm_col_params", s);
    qgemm_col_params<<<(unsigned)ceil_div(N, 256), 256, 0, s>>>(colsum, b_scale,
                                                               static_cast<const uint8_t*>(b_zero_point),
                                                               btype == I8Q_S8, (int64_t)n_b, N, K, ca, a_zero_point,
                                                               cb, alpha, a_scale, g, h, mult);
    I8Q_LAUNCH_CHECK("qgemm_col_params");
  }
  QgEpilogue qg;
  qg.rowsum = rowsum;
  qg.g = g;
  qg.h = h;
  qg.mult = mult;
  qg.C = C;
  qg.c_si = C ? (c_rows == 1 ? 0 : c_cols) : 0;
  qg.c_sj = C ? (c_cols == 1 ? 0 : 1) : 0;
  qg.ytype = quantize_y ? ytype : I8Q_F32;
  qg.y_scale = y_scale;
  qg.y_zero_point = y_zero_point;
  qg.Y = Y;
  qg.ldy = N;
  // |A'| <= 2^7 and |B'| <= 2^7
  return launch_qgemm_tc(Ac, Bc, M, N, Kp, 14, qg, s);
}
