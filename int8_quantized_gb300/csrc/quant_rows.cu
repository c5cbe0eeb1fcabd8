// quant_rows.cu -- operand preparation of the dynamic quantized inner
// product (Simd "SynetDynamicQuantizedInnerProduct16b", Detailed
// Description: "A[i,k] -> uA[i,k], scaleA[i], zeroA[i]" and
// "B[k,j] -> iB[k,j], scaleB[j]").
//
// Row quantization of A (uint8, per row, range widened to contain 0):
//   mn = min(0, min_k A), mx = max(0, max_k A), scale = (mx - mn) / 255,
//   zero = sat_u8(rint(-mn / scale)), uA = sat_u8(rint(A / scale) + zero)
//   (an all-zero row takes scale 1, zero 0).
// Column quantization of B (int8, symmetric, per column):
//   scale = max_k |B| / qmax (qmax 127, or 63 with avoidOverflow),
//   iB = saturate(rint(B / scale)) to [-128,127] / [-64,63]
//   (an all-zero column takes scale 1).
// Both write the operand layouts the GEMM cores read: uA as M x Kp and B
// transposed to N x Kp (K contiguous), zero padded to Kp, plus optional bf16
// copies for the tensor-core path (B's codes as they are, A's shifted to
// uA - 128 so every product stays within 2^14 in magnitude), and the column
// sums of iB used by the zero-point correction  -zeroA[i] * colsum[j].
#include "tcgen05.cuh"

namespace i8q {
namespace {

constexpr int kRowThreads = 256;

__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

// Load 8 consecutive elements as fp32 (16-byte aligned vector loads).
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
  float4 a = __ldg(reinterpret_cast<const float4*>(p));
  float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
  uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
  uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    v[2 * q] = __uint_as_float(w[q] << 16);
    v[2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
  }
}

// bf16 bit pattern of a small non-negative or negative integer code (exact).
__device__ __forceinline__ uint32_t code_bf16_bits(int c) {
  return (uint32_t)__bfloat16_as_ushort(__int2bfloat16_rn(c));
}

// One CTA per row (grid-stride over rows).  VEC: 8 elements per access.
template <typename T, bool VEC>
__global__ void __launch_bounds__(kRowThreads)
quantize_rows_kernel(const T* __restrict__ A, int64_t M, int64_t K, int64_t lda, uint8_t* __restrict__ uA,
                     __nv_bfloat16* __restrict__ uA_bf16, int64_t Kp, float* __restrict__ scaleA,
                     int32_t* __restrict__ zeroA) {
  __shared__ float red_mn[kRowThreads / 32], red_mx[kRowThreads / 32];
  __shared__ float sh_scale;
  __shared__ int sh_zero;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
    const T* a = A + row * lda;
    float mn = 0.0f, mx = 0.0f;
    if (VEC) {
      for (int64_t k = (int64_t)tid * 8; k < K; k += kRowThreads * 8) {
        float v[8];
        load8(a + k, v);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          mn = fminf(mn, v[q]);
          mx = fmaxf(mx, v[q]);
        }
      }
    } else {
      for (int64_t k = tid; k < K; k += kRowThreads) {
        float v = to_f32<T>(a[k]);
        mn = fminf(mn, v);
        mx = fmaxf(mx, v);
      }
    }
    mn = warp_min(mn);
    mx = warp_max(mx);
    if (lane == 0) {
      red_mn[warp] = mn;
      red_mx[warp] = mx;
    }
    __syncthreads();
    if (tid == 0) {
      float m0 = red_mn[0], m1 = red_mx[0];
      for (int w = 1; w < kRowThreads / 32; ++w) {
        m0 = fminf(m0, red_mn[w]);
        m1 = fmaxf(m1, red_mx[w]);
      }
      float s = __fdiv_rn(__fsub_rn(m1, m0), 255.0f);
      int z = 0;
      if (s == 0.0f) {
        s = 1.0f;
      } else {
        z = sat_rint(__fdiv_rn(-m0, s), 0.0f, 255.0f);
      }
      sh_scale = s;
      sh_zero = z;
      scaleA[row] = s;
      zeroA[row] = z;
    }
    __syncthreads();
    const float s = sh_scale;
    const int z = sh_zero;
    const float lo = (float)(-z), hi = (float)(255 - z);
    uint8_t* u = uA + row * Kp;
    __nv_bfloat16* ub = uA_bf16 ? uA_bf16 + row * Kp : nullptr;
    // Kp is a multiple of 64, so 8-wide chunks tile it exactly.
    for (int64_t k = (int64_t)tid * 8; k < Kp; k += kRowThreads * 8) {
      int code[8];
      if (VEC && k + 8 <= K) {
        float v[8];
        load8(a + k, v);
#pragma unroll
        for (int q = 0; q < 8; ++q) code[q] = sat_rint(__fdiv_rn(v[q], s), lo, hi) + z;
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          code[q] = (k + q < K) ? sat_rint(__fdiv_rn(to_f32<T>(a[k + q]), s), lo, hi) + z : 0;
      }
      uint32_t lo4 = 0, hi4 = 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        lo4 |= (uint32_t)code[q] << (8 * q);
        hi4 |= (uint32_t)code[q + 4] << (8 * q);
      }
      *reinterpret_cast<uint2*>(u + k) = make_uint2(lo4, hi4);
      if (ub) {
        // the tensor-core operand holds uA - 128 (exact in bf16), 0 in the
        // padding beyond K
        int cc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) cc[q] = (k + q < K) ? code[q] - 128 : 0;
        uint4 o;
        o.x = code_bf16_bits(cc[0]) | (code_bf16_bits(cc[1]) << 16);
        o.y = code_bf16_bits(cc[2]) | (code_bf16_bits(cc[3]) << 16);
        o.z = code_bf16_bits(cc[4]) | (code_bf16_bits(cc[5]) << 16);
        o.w = code_bf16_bits(cc[6]) | (code_bf16_bits(cc[7]) << 16);
        *reinterpret_cast<uint4*>(ub + k) = o;
      }
    }
    __syncthreads();
  }
}

// One warp per row, the whole row held in registers (one pass over HBM):
// lane l holds the 8-element vectors l, l+32, ..., NV of them, as raw 16-byte
// words (bf16: one word per vector; fp32: two).  Needs K % 8 == 0,
// K <= 256 * NV, a 16-byte aligned A and a row stride that keeps rows aligned.
template <typename T, int NV>
__global__ void __launch_bounds__(128)
quantize_rows_warp(const T* __restrict__ A, int64_t M, int64_t K, int64_t lda, uint8_t* __restrict__ uA,
                   __nv_bfloat16* __restrict__ uA_bf16, int64_t Kp, float* __restrict__ scaleA,
                   int32_t* __restrict__ zeroA) {
  constexpr int W = sizeof(T) == 4 ? 2 : 1;  // 16-byte words per 8-element vector
  const int lane = threadIdx.x & 31;
  const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (row >= M) return;
  const T* a = A + row * lda;
  uint4 raw[NV * W];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int64_t k = 8 * (int64_t)(lane + 32 * i);
#pragma unroll
    for (int w = 0; w < W; ++w)
      raw[i * W + w] = k < K ? __ldcs(reinterpret_cast<const uint4*>(a + k) + w) : make_uint4(0, 0, 0, 0);
  }
  auto elem = [&](int i, int e) -> float {
    if (W == 1) {
      const uint32_t word = (&raw[i].x)[e >> 1];
      return __uint_as_float((e & 1) ? (word & 0xffff0000u) : (word << 16));
    }
    return __uint_as_float((&raw[i * 2 + (e >> 2)].x)[e & 3]);
  };
  float mn = 0.0f, mx = 0.0f;  // zero padding beyond K leaves min(0, .) / max(0, .) unchanged
#pragma unroll
  for (int i = 0; i < NV; ++i)
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float v = elem(i, e);
      mn = fminf(mn, v);
      mx = fmaxf(mx, v);
    }
  mn = warp_min(mn);
  mx = warp_max(mx);
  float s = __fdiv_rn(__fsub_rn(mx, mn), 255.0f);
  int z = 0;
  if (s == 0.0f) {
    s = 1.0f;
  } else {
    z = sat_rint(__fdiv_rn(-mn, s), 0.0f, 255.0f);
  }
  if (lane == 0) {
    scaleA[row] = s;
    zeroA[row] = z;
  }
  const float lo_z = (float)(-z), hi_z = (float)(255 - z);
  const float shift = (float)(z - 128) - 12582912.0f;  // takes rint + 1.5*2^23 to uA - 128
  uint8_t* u = uA + row * Kp;
  __nv_bfloat16* ub = uA_bf16 ? uA_bf16 + row * Kp : nullptr;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int64_t k = 8 * (int64_t)(lane + 32 * i);
    if (k >= Kp) break;
    uint32_t code[8], cb[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      // IEEE quotient, clamp, round half to even by the 1.5*2^23 add
      const float t = fminf(fmaxf(__fdiv_rn(elem(i, e), s), lo_z), hi_z);
      const float r = __fadd_rn(t, 12582912.0f);
      const bool valid = k + e < K;
      code[e] = valid ? (uint32_t)(__float_as_int(r) + z) : 0u;
      cb[e] = valid ? (__float_as_uint(__fadd_rn(r, shift)) >> 16) : 0u;
    }
    *reinterpret_cast<uint2*>(u + k) =
        make_uint2(pack_low_bytes(code[0], code[1], code[2], code[3]), pack_low_bytes(code[4], code[5], code[6], code[7]));
    if (ub) {
      uint4 o;
      o.x = cb[0] | (cb[1] << 16);
      o.y = cb[2] | (cb[3] << 16);
      o.z = cb[4] | (cb[5] << 16);
      o.w = cb[6] | (cb[7] << 16);
      *reinterpret_cast<uint4*>(ub + k) = o;
    }
  }
}

// Rows staged in shared memory: a persistent CTA of 16 warps takes groups of
// 4 rows; one thread copies each group into shared memory with bulk copies
// (one per row, double-buffered, the next group in flight while this one is
// processed), then 4 warps share each row: a min/max pass (combined through
// shared memory) and a quantization pass over shared memory, 8 elements per
// lane and step, with coalesced stores of the codes and of their bf16 copy
// (uA - 128).  The
// arithmetic is that of quantize_rows_warp.  Needs K % 8 == 0, 16-byte
// aligned rows, and 2 * 4 rows in shared memory.  Groups of 4 rows rather
// than 8 (measured on bf16 rows of 4096): 3 % faster on 8192 or 32768 rows,
// 2.4x on 1024 rows, and fp32 rows of 4096 fit.
constexpr int kStageRows = 4;
constexpr int kWarpsPerRow = 4;

// Four codes saturated to [0, 255] and packed, byte 0 from a.
__device__ __forceinline__ uint32_t pack_sat_u8x4(int a, int b, int c, int d) {
  uint32_t hi, r;
  asm("cvt.pack.sat.u8.s32.b32 %0, %1, %2, %3;" : "=r"(hi) : "r"(d), "r"(c), "r"(0u));
  asm("cvt.pack.sat.u8.s32.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(b), "r"(a), "r"(hi));
  return r;
}

// z + rint(fl(v / s)), saturated to [0, 255], from the quotient itself: the
// fallback of the bracketed codes below.  Out of line: rare.
__device__ __noinline__ int row_code_exact(float v, float s, float lo_z, float hi_z, int z) {
  return (int)(rint_code_bits(__fdiv_rn(v, s), lo_z, hi_z, z) - 0x4B400000u);
}
constexpr int kStageThreads = 32 * kStageRows * kWarpsPerRow;
constexpr uint32_t ST_TIMEOUT_ROWS = 1u << 12;

template <typename T>
__global__ void __launch_bounds__(kStageThreads, 1)
quantize_rows_staged(const T* __restrict__ A, int64_t M, int64_t K, int64_t lda, uint8_t* __restrict__ uA,
                     __nv_bfloat16* __restrict__ uA_bf16, int64_t Kp, float* __restrict__ scaleA,
                     int32_t* __restrict__ zeroA, uint32_t* status) {
  extern __shared__ __align__(128) uint8_t sm[];
  const uint32_t row_bytes = (uint32_t)(K * sizeof(T));
  const uint32_t group_bytes = kStageRows * row_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + 2 * (size_t)group_bytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2);
  __shared__ float red[kStageRows][kWarpsPerRow][2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rw = warp / kWarpsPerRow, part = warp % kWarpsPerRow;  // row of the group, quarter of the work
  const int64_t groups = (M + kStageRows - 1) / kStageRows;
  if (threadIdx.x == 0) {
    tc::mbar_init(tc::smem_u32(bars), 1);
    tc::mbar_init(tc::smem_u32(bars + 1), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  auto issue = [&](int64_t g, int b) {
    const int64_t r0 = g * kStageRows;
    const int rows = (int)(M - r0 < kStageRows ? M - r0 : kStageRows);
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    tc::mbar_arrive_expect_tx(tc::smem_u32(bars + b), (uint32_t)rows * row_bytes);
    for (int r = 0; r < rows; ++r)
      tc::bulk_load(tc::smem_u32(sm + (size_t)b * group_bytes + (size_t)r * row_bytes), A + (r0 + r) * lda, row_bytes,
                    tc::smem_u32(bars + b));
  };
  int64_t g = blockIdx.x;
  int issued = 0, waited = 0;  // groups copied / consumed (thread 0 issues)
  if (threadIdx.x == 0 && g < groups) {
    issue(g, 0);
    issued = 1;
  }
  const int nunits = (int)(K / 8);  // 8-element units of a row
  for (int it = 0; g < groups; g += gridDim.x, ++it) {
    const int b = it & 1;
    const int64_t gn = g + gridDim.x;
    if (threadIdx.x == 0 && gn < groups) {
      issue(gn, b ^ 1);
      ++issued;
    }
    if (!tc::wait_bar(tc::smem_u32(bars + b), (uint32_t)(it >> 1) & 1u, abort_flag, status, ST_TIMEOUT_ROWS)) break;
    ++waited;
    const int64_t row = g * kStageRows + rw;
    const bool live = row < M;
    {
      const uint8_t* base = sm + (size_t)b * group_bytes + (size_t)rw * row_bytes;
      auto unit = [&](int c, float (&v)[8]) {
        if (sizeof(T) == 2) {
          const uint4 w = *reinterpret_cast<const uint4*>(base + (size_t)c * 16);
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            v[2 * q] = __uint_as_float(ws[q] << 16);
            v[2 * q + 1] = __uint_as_float(ws[q] & 0xffff0000u);
          }
        } else {
          const float4 x0 = *reinterpret_cast<const float4*>(base + (size_t)c * 32);
          const float4 x1 = *reinterpret_cast<const float4*>(base + (size_t)c * 32 + 16);
          v[0] = x0.x; v[1] = x0.y; v[2] = x0.z; v[3] = x0.w;
          v[4] = x1.x; v[5] = x1.y; v[6] = x1.z; v[7] = x1.w;
        }
      };
      float mn = 0.0f, mx = 0.0f;
      if (live) {
#pragma unroll 4
        for (int c = part * 32 + lane; c < nunits; c += 32 * kWarpsPerRow) {
          float v[8];
          unit(c, v);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            mn = fminf(mn, v[e]);
            mx = fmaxf(mx, v[e]);
          }
        }
      }
      mn = warp_min(mn);
      mx = warp_max(mx);
      if (lane == 0) {
        red[rw][part][0] = mn;
        red[rw][part][1] = mx;
      }
      __syncthreads();
#pragma unroll
      for (int w2 = 0; w2 < kWarpsPerRow; ++w2) {
        mn = fminf(mn, red[rw][w2][0]);
        mx = fmaxf(mx, red[rw][w2][1]);
      }
      float sc = __fdiv_rn(__fsub_rn(mx, mn), 255.0f);
      int z = 0;
      if (sc == 0.0f) {
        sc = 1.0f;
      } else {
        z = sat_rint(__fdiv_rn(-mn, sc), 0.0f, 255.0f);
      }
      if (live && part == 0 && lane == 0) {
        scaleA[row] = sc;
        zeroA[row] = z;
      }
      const float lo_z = (float)(-z), hi_z = (float)(255 - z);
      const float shift = (float)(z - 128) - 12582912.0f;  // takes rint + 1.5*2^23 to uA - 128
      uint8_t* u = uA + (live ? row : 0) * Kp;
      __nv_bfloat16* ub = uA_bf16 ? uA_bf16 + (live ? row : 0) * Kp : nullptr;
      // Bracketed codes: with r = fl(1 / sc) scaled by 1 -+ 2^-20 (rl < 1 / sc
      // < rh), the exact products v * rl and v * rh enclose v / sc with a margin
      // above 2^-21 |v / sc|, so they strictly enclose the IEEE quotient too;
      // an fma adds mz = 1.5 * 2^23 + z and rounds once to an integer (|v / sc|
      // <= 256 here), a non-decreasing function of the product, so equal ends
      // give z + rint(quotient) (a half-integer quotient would have both
      // neighbours inside).  Unequal ends (near a tie) take the quotient.
      const float rcp = quot_rcp(sc);
      const bool brk = rcp == rcp;
      const float rh = __fmul_rn(rcp, 1.0f + 0x1p-20f), rl = __fmul_rn(rcp, 1.0f - 0x1p-20f);
      const float mz = 12582912.0f + (float)z;
#pragma unroll 2
      for (int c = part * 32 + lane; live && c < nunits; c += 32 * kWarpsPerRow) {
        float v[8];
        unit(c, v);
        uint32_t w0, w1;
        if (brk) {
          int n[8];
          uint32_t diff = 0;
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const float2 h = fma2_rn(make_float2(v[e], v[e + 1]), make_float2(rh, rh), make_float2(mz, mz));
            const float2 l = fma2_rn(make_float2(v[e], v[e + 1]), make_float2(rl, rl), make_float2(mz, mz));
            diff |= (__float_as_uint(h.x) ^ __float_as_uint(l.x)) | (__float_as_uint(h.y) ^ __float_as_uint(l.y));
            n[e] = __float_as_int(h.x) - 0x4B400000;
            n[e + 1] = __float_as_int(h.y) - 0x4B400000;
          }
          if (diff) {
#pragma unroll
            for (int e = 0; e < 8; ++e) n[e] = row_code_exact(v[e], sc, lo_z, hi_z, z);
          }
          w0 = pack_sat_u8x4(n[0], n[1], n[2], n[3]);
          w1 = pack_sat_u8x4(n[4], n[5], n[6], n[7]);
          *reinterpret_cast<uint2*>(u + (size_t)c * 8) = make_uint2(w0, w1);
          if (ub) {
            // code c as the fp32 1.5 * 2^23 + c by one byte permute, minus
            // 1.5 * 2^23 + 128: exactly c - 128, whose bf16 is the top half
            uint32_t cb[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint32_t w = q < 2 ? w0 : w1, sel = 0x7640u + 2 * (q & 1);
              const float2 f = fma2_rn(make_float2(__uint_as_float(__byte_perm(w, 0x4B400000u, sel)),
                                                   __uint_as_float(__byte_perm(w, 0x4B400000u, sel + 1))),
                                       make_float2(1.0f, 1.0f), make_float2(-12583040.0f, -12583040.0f));
              cb[q] = __byte_perm(__float_as_uint(f.x), __float_as_uint(f.y), 0x7632);
            }
            *reinterpret_cast<uint4*>(ub + (size_t)c * 8) = make_uint4(cb[0], cb[1], cb[2], cb[3]);
          }
          continue;
        }
        uint32_t code[8], cb[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float t = fminf(fmaxf(__fdiv_rn(v[e], sc), lo_z), hi_z);
          const float r = __fadd_rn(t, 12582912.0f);
          code[e] = (uint32_t)(__float_as_int(r) + z);
          cb[e] = __float_as_uint(__fadd_rn(r, shift)) >> 16;
        }
        *reinterpret_cast<uint2*>(u + (size_t)c * 8) = make_uint2(pack_low_bytes(code[0], code[1], code[2], code[3]),
                                                                   pack_low_bytes(code[4], code[5], code[6], code[7]));
        if (ub)
          *reinterpret_cast<uint4*>(ub + (size_t)c * 8) = make_uint4(cb[0] | (cb[1] << 16), cb[2] | (cb[3] << 16),
                                                                     cb[4] | (cb[5] << 16), cb[6] | (cb[7] << 16));
      }
      // zero padding K .. Kp
      for (int c = nunits + part * 32 + lane; live && c < (int)(Kp / 8); c += 32 * kWarpsPerRow) {
        *reinterpret_cast<uint2*>(u + (size_t)c * 8) = make_uint2(0u, 0u);
        if (ub) *reinterpret_cast<uint4*>(ub + (size_t)c * 8) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    __syncthreads();  // the buffer is free for the group after next
  }
  // after a timeout: let the copies this CTA still has in flight land
  // (bounded) before it exits
  if (threadIdx.x == 0)
    for (int j = waited; j < issued; ++j) {
      const unsigned long long t0 = tc::global_ns();
      while (!tc::mbar_try_wait(tc::smem_u32(bars + (j & 1)), (uint32_t)(j >> 1) & 1u))
        if (tc::global_ns() - t0 > tc::WAIT_LIMIT_NS) break;
    }
}

// ---- columns -------------------------------------------------------------
// A CTA owns 32 columns [j0, j0+32) and walks all of K twice: once for the
// max-abs per column, once to quantize, transposing 64 x 32 tiles through
// shared memory so the N x Kp output is written with contiguous K.
constexpr int kColW = 32;
constexpr int kColKT = 64;

// Destination row of column j: j itself, or, with gates_H > 0, the gate
// interleaving 4 * (j % gates_H) + j / gates_H (column q*H + u of an
// iofc-ordered 4H-wide matrix lands at 4u + q).
__device__ __forceinline__ int64_t dest_row(int64_t j, int64_t gates_H) {
  return gates_H > 0 ? 4 * (j % gates_H) + j / gates_H : j;
}

template <typename T, int MODE>  // MODE 0: quantize fp32/bf16 B; 1: repack int8 B
__global__ void __launch_bounds__(256)
cols_kernel(const T* __restrict__ B, int64_t K, int64_t N, int64_t ldb, int qmin, int qmax,
            int8_t* __restrict__ iBt, __nv_bfloat16* __restrict__ iBt_bf16, int64_t Kp,
            float* __restrict__ scaleB, int32_t* __restrict__ colsum, int64_t gates_H) {
  __shared__ float red[8][kColW];
  __shared__ float sh_scale[kColW];
  __shared__ int sh_sum[8][kColW];
  __shared__ int8_t tile[kColW][kColKT + 16];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t j0 = (int64_t)blockIdx.x * kColW;
  const int64_t j = j0 + lane;
  const bool jok = j < N;
  if constexpr (MODE == 0) {
    float m = 0.0f;
    if (jok)
      for (int64_t k = warp; k < K; k += 8) m = fmaxf(m, fabsf(to_f32<T>(B[k * ldb + j])));
    red[warp][lane] = m;
    __syncthreads();
    if (warp == 0) {
      float mm = red[0][lane];
      for (int w = 1; w < 8; ++w) mm = fmaxf(mm, red[w][lane]);
      float s = __fdiv_rn(mm, (float)qmax);
      if (s == 0.0f) s = 1.0f;
      sh_scale[lane] = s;
      if (jok) scaleB[j] = s;
    }
    __syncthreads();
  }
  const float s = MODE == 0 ? sh_scale[lane] : 1.0f;
  int sum = 0;
  for (int64_t k0 = 0; k0 < Kp; k0 += kColKT) {
    // each warp quantizes rows k0 + warp + 8*r of the 32 columns
#pragma unroll
    for (int r = 0; r < kColKT / 8; ++r) {
      const int kk = warp + 8 * r;
      const int64_t k = k0 + kk;
      int code = 0;
      if (jok && k < K) {
        if constexpr (MODE == 0)
          code = sat_rint(__fdiv_rn(to_f32<T>(B[k * ldb + j]), s), (float)qmin, (float)qmax);
        else
          code = (int)(int8_t)B[k * ldb + j];
      }
      sum += code;
      tile[lane][kk] = (int8_t)code;
    }
    __syncthreads();
    // write the 32 x 64 tile: thread -> (column c, 8-byte segment)
    const int c = tid >> 3, seg = tid & 7;
    const int64_t jj = j0 + c;
    if (jj < N) {
      const int8_t* src = &tile[c][seg * 8];
      const int64_t jd = dest_row(jj, gates_H);
      uint32_t w0 = 0, w1 = 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        w0 |= (uint32_t)(uint8_t)src[q] << (8 * q);
        w1 |= (uint32_t)(uint8_t)src[q + 4] << (8 * q);
      }
      if (iBt) *reinterpret_cast<uint2*>(iBt + jd * Kp + k0 + seg * 8) = make_uint2(w0, w1);
      if (iBt_bf16) {
        uint4 o;
        o.x = code_bf16_bits(src[0]) | (code_bf16_bits(src[1]) << 16);
        o.y = code_bf16_bits(src[2]) | (code_bf16_bits(src[3]) << 16);
        o.z = code_bf16_bits(src[4]) | (code_bf16_bits(src[5]) << 16);
        o.w = code_bf16_bits(src[6]) | (code_bf16_bits(src[7]) << 16);
        *reinterpret_cast<uint4*>(iBt_bf16 + jd * Kp + k0 + seg * 8) = o;
      }
    }
    __syncthreads();
  }
  sh_sum[warp][lane] = sum;
  __syncthreads();
  if (warp == 0 && jok) {
    int t = 0;
    for (int w = 0; w < 8; ++w) t += sh_sum[w][lane];
    colsum[dest_row(j, gates_H)] = t;
  }
}

// ---- 8-bit repack in 128 x 128 tiles -------------------------------------------
// The repack of a given 8-bit B (no quantization) over a grid of K x N tiles,
// codes centred on the way for uint8 (FLIP: code - 128, the int8 of code ^
// 0x80); the int8 and bf16 copies are each optional:
// a thread loads a 4-row x 16-column block (four 16-byte loads, two lanes
// per 32-byte sector of a row), turns it into 16 words of 4 rows each of one
// column by byte permutes, and stores them to a column-major shared tile
// (column stride 33 words: the lanes of a warp store to 32 distinct banks).
// Eight consecutive lanes then write one column's 128 bytes (and its 256
// bf16 bytes) contiguously, and merge their column-sum partials by shuffles
// into one atomicAdd per column and tile.  Rows k >= K load as zeros, so the
// tiles up to Kp write the padding.
constexpr int kRtCols = 128, kRtK = 128, kRtStride = kRtK / 4 + 1;

template <bool FLIP>
__global__ void __launch_bounds__(256)
repack_tiles_s8(const int8_t* __restrict__ B, int64_t K, int64_t N, int64_t ldb, int8_t* __restrict__ iBt,
                __nv_bfloat16* __restrict__ iBt_bf16, int64_t Kp, int32_t* __restrict__ colsum, int64_t gates_H) {
  constexpr uint32_t flip = FLIP ? 0x80808080u : 0u;
  __shared__ uint32_t tile[kRtCols * kRtStride];
  const int t = (int)threadIdx.x, lane = t & 31, warp = t >> 5;
  const int64_t j0 = (int64_t)blockIdx.x * kRtCols, k0 = (int64_t)blockIdx.y * kRtK;
  {
    const int cq = 2 * (warp & 3) + (lane & 1), rq = 16 * (warp >> 2) + (lane >> 1);
    const int64_t j = j0 + 16 * cq;
    uint4 v[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int64_t k = k0 + 4 * rq + r;
      v[r] = (k < K && j < N) ? __ldg(reinterpret_cast<const uint4*>(B + k * ldb + j))
                              : make_uint4(flip, flip, flip, flip);
    }
    // padding rows stay 0 after the flip too
    const uint32_t a[4][4] = {{v[0].x ^ flip, v[0].y ^ flip, v[0].z ^ flip, v[0].w ^ flip},
                              {v[1].x ^ flip, v[1].y ^ flip, v[1].z ^ flip, v[1].w ^ flip},
                              {v[2].x ^ flip, v[2].y ^ flip, v[2].z ^ flip, v[2].w ^ flip},
                              {v[3].x ^ flip, v[3].y ^ flip, v[3].z ^ flip, v[3].w ^ flip}};
    uint32_t* dst = tile + (16 * cq) * kRtStride + rq;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      // 4 x 4 byte transpose: word b = byte b of rows 0..3
      const uint32_t t0 = __byte_perm(a[0][g], a[1][g], 0x5140), t1 = __byte_perm(a[0][g], a[1][g], 0x7362);
      const uint32_t t2 = __byte_perm(a[2][g], a[3][g], 0x5140), t3 = __byte_perm(a[2][g], a[3][g], 0x7362);
      dst[(4 * g + 0) * kRtStride] = __byte_perm(t0, t2, 0x5410);
      dst[(4 * g + 1) * kRtStride] = __byte_perm(t0, t2, 0x7632);
      dst[(4 * g + 2) * kRtStride] = __byte_perm(t1, t3, 0x5410);
      dst[(4 * g + 3) * kRtStride] = __byte_perm(t1, t3, 0x7632);
    }
  }
  __syncthreads();
  // code c as fp32: byte c ^ 0x80 in 1.5 * 2^23 + (c + 128), minus 1.5 * 2^23 + 128
  const float off = 12583040.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int task = t + 256 * i, c = task >> 3, q = task & 7;
    const int64_t j = j0 + c, k = k0 + 16 * q;
    const uint32_t* src = tile + c * kRtStride + 4 * q;
    const uint32_t w[4] = {src[0], src[1], src[2], src[3]};
    int sum = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) sum = __dp4a((int)w[e], 0x01010101, sum);
    const bool live = j < N && k < Kp;
    if (live) {
      const int64_t jd = dest_row(j, gates_H);
      if (iBt) *reinterpret_cast<uint4*>(iBt + jd * Kp + k) = make_uint4(w[0], w[1], w[2], w[3]);
      if (iBt_bf16) {
        uint32_t o[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t u = w[e] ^ 0x80808080u;
          float f[4];
#pragma unroll
          for (int b = 0; b < 4; ++b) f[b] = __fsub_rn(__uint_as_float(__byte_perm(u, 0x4B400000u, 0x7640 + b)), off);
          o[2 * e] = __byte_perm(__float_as_uint(f[0]), __float_as_uint(f[1]), 0x7632);
          o[2 * e + 1] = __byte_perm(__float_as_uint(f[2]), __float_as_uint(f[3]), 0x7632);
        }
        uint4* ob = reinterpret_cast<uint4*>(iBt_bf16 + jd * Kp + k);
        ob[0] = make_uint4(o[0], o[1], o[2], o[3]);
        ob[1] = make_uint4(o[4], o[5], o[6], o[7]);
      }
    }
    // the column's 8 lanes (consecutive, aligned) hold its 128 rows
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    sum += __shfl_xor_sync(0xffffffffu, sum, 4);
    if (q == 0 && j < N) atomicAdd(colsum + dest_row(j, gates_H), sum);
  }
}

// ---- columns, two wide passes ---------------------------------------------
// Each lane owns 4 consecutive columns, so a warp reads 128 columns of one
// row per access (512 B of fp32, 256 B of bf16).  Pass 1 folds max|B| per
// column over a K range and merges it with atomicMax on the bit pattern
// (non-negative floats order like their bits).  Pass 2 quantizes 64-row
// tiles, transposes them through shared memory into the K-contiguous
// outputs and merges partial column sums with atomicAdd.
constexpr int kWideCols = 128, kWideKT = 64, kWideKSplit = 512;

__device__ __forceinline__ void load4(const float* p, float (&v)[4]) {
  const float4 a = __ldcs(reinterpret_cast<const float4*>(p));
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16* p, float (&v)[4]) {
  const uint2 a = __ldcs(reinterpret_cast<const uint2*>(p));
  v[0] = __uint_as_float(a.x << 16);
  v[1] = __uint_as_float(a.x & 0xffff0000u);
  v[2] = __uint_as_float(a.y << 16);
  v[3] = __uint_as_float(a.y & 0xffff0000u);
}

template <typename T>
__global__ void __launch_bounds__(256)
col_absmax_wide(const T* __restrict__ B, int64_t K, int64_t N, uint32_t* __restrict__ colmax) {
  __shared__ float red[8][kWideCols];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t j = (int64_t)blockIdx.x * kWideCols + 4 * lane;
  const int64_t k_end = std::min<int64_t>(K, (int64_t)(blockIdx.y + 1) * kWideKSplit);
  float m[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  if (j < N)
#pragma unroll 8
    for (int64_t k = (int64_t)blockIdx.y * kWideKSplit + warp; k < k_end; k += 8) {
      float v[4];
      load4(B + k * N + j, v);
#pragma unroll
      for (int u = 0; u < 4; ++u) m[u] = fmaxf(m[u], fabsf(v[u]));
    }
#pragma unroll
  for (int u = 0; u < 4; ++u) red[warp][4 * lane + u] = m[u];
  __syncthreads();
  if (threadIdx.x < kWideCols) {
    float r = red[0][threadIdx.x];
    for (int w = 1; w < 8; ++w) r = fmaxf(r, red[w][threadIdx.x]);
    const int64_t jj = (int64_t)blockIdx.x * kWideCols + threadIdx.x;
    if (jj < N) atomicMax(colmax + jj, __float_as_uint(r));
  }
}

template <typename T>
__global__ void __launch_bounds__(256)
col_quant_wide(const T* __restrict__ B, int64_t K, int64_t N, int64_t Kp, const uint32_t* __restrict__ colmax,
               int qmin, int qmax, int8_t* __restrict__ iBt, __nv_bfloat16* __restrict__ iBt_bf16,
               float* __restrict__ scaleB, int32_t* __restrict__ colsum) {
  __shared__ int8_t tile[kWideCols][kWideKT + 16];
  __shared__ int sums[8][kWideCols];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t j0 = (int64_t)blockIdx.x * kWideCols;
  const int64_t j = j0 + 4 * lane;
  const bool jok = j < N;
  float s[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    float sv = jok ? __fdiv_rn(__uint_as_float(colmax[j + u]), (float)qmax) : 1.0f;
    s[u] = sv == 0.0f ? 1.0f : sv;
  }
  if (blockIdx.y == 0 && warp == 0 && jok) {
#pragma unroll
    for (int u = 0; u < 4; ++u) scaleB[j + u] = s[u];
  }
  int sum[4] = {0, 0, 0, 0};
  const int64_t kbeg = (int64_t)blockIdx.y * kWideKSplit;
  const int64_t kend = std::min<int64_t>(Kp, kbeg + kWideKSplit);
  for (int64_t k0 = kbeg; k0 < kend; k0 += kWideKT) {
#pragma unroll
    for (int r = 0; r < kWideKT / 8; ++r) {
      const int kk = warp + 8 * r;
      const int64_t k = k0 + kk;
      int code[4] = {0, 0, 0, 0};
      if (jok && k < K) {
        float v[4];
        load4(B + k * N + j, v);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          code[u] = sat_rint(__fdiv_rn(v[u], s[u]), (float)qmin, (float)qmax);
          sum[u] += code[u];
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) tile[4 * lane + u][kk] = (int8_t)code[u];
    }
    __syncthreads();
    // each thread writes half of one column's 64 codes (32 B) and their bf16 copies (64 B)
    const int c = threadIdx.x >> 1, h = threadIdx.x & 1;
    const int64_t jj = j0 + c;
    if (jj < N) {
      const int8_t* src = &tile[c][h * 32];
      uint32_t wds[8];
#pragma unroll
      for (int q = 0; q < 8; ++q)
        wds[q] = (uint32_t)(uint8_t)src[4 * q] | ((uint32_t)(uint8_t)src[4 * q + 1] << 8) |
                 ((uint32_t)(uint8_t)src[4 * q + 2] << 16) | ((uint32_t)(uint8_t)src[4 * q + 3] << 24);
      if (iBt) {
        uint4* dst = reinterpret_cast<uint4*>(iBt + jj * Kp + k0 + h * 32);
        dst[0] = make_uint4(wds[0], wds[1], wds[2], wds[3]);
        dst[1] = make_uint4(wds[4], wds[5], wds[6], wds[7]);
      }
      if (iBt_bf16) {
        uint4* db = reinterpret_cast<uint4*>(iBt_bf16 + jj * Kp + k0 + h * 32);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            pk[e] = code_bf16_bits(src[8 * q + 2 * e]) | (code_bf16_bits(src[8 * q + 2 * e + 1]) << 16);
          db[q] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) sums[warp][4 * lane + u] = sum[u];
  __syncthreads();
  if (threadIdx.x < kWideCols) {
    int t = 0;
    for (int w = 0; w < 8; ++w) t += sums[w][threadIdx.x];
    const int64_t jj = j0 + threadIdx.x;
    if (jj < N) atomicAdd(colsum + jj, t);
  }
}

// ---- columns, one strip per CTA -------------------------------------------
// A persistent CTA owns a strip of 64 bytes of every row of B (16 fp32 or
// 32 bf16 columns).  One thread streams the strip through an 8-stage ring of
// 256-row TMA boxes twice: first for max|B| per column, then -- from L2: a
// strip per SM is 0.25 MB at K = 4096 -- for the codes; the second pass of
// a strip runs box by box alongside the first pass of the CTA's next strip.  Each consumer
// thread owns one column and a run of R adjacent rows of every box (8 for
// fp32, 16 for bf16), reads it down the column in shared memory and writes
// its R codes, contiguous along K, straight to the transposed outputs.  Rows
// past K read as zero from the tensor map, which gives the zero padding up
// to Kp.  The rounding avoids the conversion units: q is clamped to
// [qmin, qmax] (integer bounds, so clamping commutes with rounding) and
// 1.5 * 2^23 is added, which rounds to nearest even; taking it off again
// gives the code as an exact float, whose bf16 bits are its top 16 bits and
// whose column sum is exact in fp32 (|sum| <= 2^23).
constexpr int kCqConsumers = 512, kCqThreads = kCqConsumers + 32;
constexpr int kCqRowBytes = 64;  // strip width in bytes (128: 4 % slower; 32: 6 % slower)
constexpr int kCqBoxRows = 256, kCqStages = 8, kCqStageBytes = kCqBoxRows * kCqRowBytes;
constexpr size_t kCqSmem = 1024 + (size_t)kCqStages * kCqStageBytes + 2 * kCqStages * 8 + 16;
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23
constexpr uint32_t ST_TIMEOUT_COLS = 1u << 13;

__device__ __forceinline__ float elem_f32(const uint8_t* p, float) { return *reinterpret_cast<const float*>(p); }
__device__ __forceinline__ float elem_f32(const uint8_t* p, __nv_bfloat16) {
  return __uint_as_float((uint32_t)*reinterpret_cast<const uint16_t*>(p) << 16);
}

template <typename T>
__global__ void __launch_bounds__(kCqThreads, 1)
col_quant_tma(const __grid_constant__ CUtensorMap tmB, int64_t K, int64_t N, int64_t Kp, int qmin, int qmax,
              int8_t* __restrict__ iBt, __nv_bfloat16* __restrict__ iBt_bf16, float* __restrict__ scaleB,
              int32_t* __restrict__ colsum, uint32_t* status) {
  constexpr int W = kCqRowBytes / (int)sizeof(T);  // strip width in columns
  constexpr int RG = kCqConsumers / W;      // row groups of a box
  constexpr int R = kCqBoxRows / RG;        // rows per consumer thread per box
  extern __shared__ uint8_t cq_raw[];
  // 1024-byte aligned, indexed from the shared array itself so that accesses stay shared-space
  uint8_t* ring = cq_raw + ((1024u - (tc::smem_u32(cq_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)kCqStages * kCqStageBytes);
  uint64_t* empty = full + kCqStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kCqStages);
  __shared__ float red[RG][W];
  __shared__ float sscale[W];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int b = 0; b < kCqStages; ++b) {
      tc::mbar_init(tc::smem_u32(full + b), 1);
      tc::mbar_init(tc::smem_u32(empty + b), kCqConsumers / 32);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  const int64_t nstrips = (N + W - 1) / W;
  const int nb1 = (int)((K + kCqBoxRows - 1) / kCqBoxRows);   // boxes of the max pass
  const int nb2 = (int)((Kp + kCqBoxRows - 1) / kCqBoxRows);  // boxes of the code pass
  if (warp == kCqConsumers / 32) {
    // ---------------- producer ----------------
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      // a strip's second pass reads its lines for the last time
      const uint64_t drop = tc::policy_evict_first();
      auto load = [&](int64_t strip, int b, bool first_pass) {
        const uint32_t st = it % kCqStages;
        if (it >= (uint32_t)kCqStages &&
            !tc::wait_bar(tc::smem_u32(empty + st), ((it / kCqStages) - 1) & 1u, abort_flag, status, ST_TIMEOUT_COLS)) {
          ok = false;
          return;
        }
        tc::mbar_arrive_expect_tx(tc::smem_u32(full + st), (uint32_t)kCqStageBytes);
        if (first_pass)
          tc::tma_load_2d(tc::smem_u32(ring + (size_t)st * kCqStageBytes), &tmB, tc::smem_u32(full + st),
                          (int)(strip * W), b * kCqBoxRows);
        else
          tc::tma_load_2d_hint(tc::smem_u32(ring + (size_t)st * kCqStageBytes), &tmB, tc::smem_u32(full + st),
                               (int)(strip * W), b * kCqBoxRows, drop);
        ++it;
      };
      // the boxes in the consumers' order: the first strip's max pass, then
      // each strip's code pass interleaved box by box with the next strip's
      // max pass
      for (int b = 0; ok && b < nb1 && (int64_t)blockIdx.x < nstrips; ++b) load(blockIdx.x, b, true);
      for (int64_t strip = blockIdx.x; ok && strip < nstrips; strip += gridDim.x) {
        const int64_t nxt = strip + gridDim.x;
        const int nbm = nxt < nstrips ? nb1 : 0;
        for (int b = 0; ok && b < (nb2 > nbm ? nb2 : nbm); ++b) {
          if (b < nb2) load(strip, b, false);
          if (ok && b < nbm) load(nxt, b, true);
        }
      }
      // the copies in flight land before the CTA leaves (bounded)
      const uint32_t first = it > (uint32_t)kCqStages ? it - kCqStages : 0u;
      for (uint32_t i = first; i < it; ++i) {
        const uint64_t t0 = tc::global_ns();
        while (!tc::mbar_try_wait(tc::smem_u32(full + i % kCqStages), (i / kCqStages) & 1u))
          if (tc::global_ns() - t0 > tc::WAIT_LIMIT_NS) {
            atomicOr(status, ST_TIMEOUT_COLS);
            break;
          }
      }
    }
    return;
  }
  // ---------------- consumers ----------------
  const int c = tid % W, rg = tid / W;
  const float lo = (float)qmin, hi = (float)qmax;
  uint32_t it = 0;
  bool ok = true;
  auto consumers_sync = [] { asm volatile("bar.sync 1, %0;\n" ::"n"(kCqConsumers) : "memory"); };
  // max |B| of this thread's column over its rows of the next box
  auto max_box = [&](float& m) {
    const uint32_t st = it % kCqStages;
    if (ok) ok = tc::wait_bar(tc::smem_u32(full + st), (it / kCqStages) & 1u, abort_flag, status, ST_TIMEOUT_COLS);
    if (ok) {
      const uint8_t* src = ring + (size_t)st * kCqStageBytes + (size_t)(rg * R) * kCqRowBytes + (size_t)c * sizeof(T);
#pragma unroll
      for (int r = 0; r < R; ++r) m = fmaxf(m, fabsf(elem_f32(src + r * kCqRowBytes, T())));
    }
    __syncwarp();
    if (ok && lane == 0) tc::mbar_arrive(tc::smem_u32(empty + st));
    ++it;
  };
  // the codes of this thread's R rows of the next box (box b of column j)
  // from q = fl(B * rs), rs = fl(1 / s): q and the quotient fl(B / s) differ
  // by less than 2^-22 |q|, so they round alike unless q lies within
  // 2^-21 |q| of a half-integer (checked for the R values at once), where
  // the quotient itself is formed; a scale whose reciprocal is not a normal
  // number always takes the quotient
  auto code_box = [&](int64_t j, int b, float s, float rs, bool rs_ok, float& fsum) {
    const uint32_t st = it % kCqStages;
    if (ok) ok = tc::wait_bar(tc::smem_u32(full + st), (it / kCqStages) & 1u, abort_flag, status, ST_TIMEOUT_COLS);
    uint32_t w[R / 2], o[R / 4];
    if (ok) {
      const uint8_t* src = ring + (size_t)st * kCqStageBytes + (size_t)(rg * R) * kCqRowBytes + (size_t)c * sizeof(T);
      // rr = code + 1.5 * 2^23 (the code in its low byte, two's complement),
      // ff = the code as an exact float; pairs on the paired fp32 pipe (an
      // fma by 1 rounds once, as the addition does)
      float2 rr[R / 2], ff[R / 2];
      bool slow = !rs_ok;
#pragma unroll
      for (int r = 0; r < R; r += 2) {
        float2 q = mul2_rn(make_float2(elem_f32(src + r * kCqRowBytes, T()), elem_f32(src + (r + 1) * kCqRowBytes, T())),
                           make_float2(rs, rs));
        q = make_float2(fminf(fmaxf(q.x, lo), hi), fminf(fmaxf(q.y, lo), hi));
        rr[r / 2] = fma2_rn(q, make_float2(1.0f, 1.0f), make_float2(kRoundMagic, kRoundMagic));
        ff[r / 2] = fma2_rn(rr[r / 2], make_float2(1.0f, 1.0f), make_float2(-kRoundMagic, -kRoundMagic));
        const float2 d = fma2_rn(ff[r / 2], make_float2(-1.0f, -1.0f), q);  // q - code, exact
        // |q| <= 128, so 0.5 - 2^-21 |q| >= 0.5 - 2^-14: a constant bound
        // that flags every near tie (and a few more)
        slow |= fabsf(d.x) > 0.5f - 0x1p-14f || fabsf(d.y) > 0.5f - 0x1p-14f;
      }
      if (slow) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float q = fminf(fmaxf(__fdiv_rn(elem_f32(src + r * kCqRowBytes, T()), s), lo), hi);
          const float r1 = __fadd_rn(q, kRoundMagic);
          if (r & 1) {
            rr[r / 2].y = r1;
            ff[r / 2].y = __fsub_rn(r1, kRoundMagic);
          } else {
            rr[r / 2].x = r1;
            ff[r / 2].x = __fsub_rn(r1, kRoundMagic);
          }
        }
      }
      float2 fs2 = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int r = 0; r < R; r += 2) {
        fs2 = fma2_rn(ff[r / 2], make_float2(1.0f, 1.0f), fs2);  // exact integer sums
        w[r / 2] = __byte_perm(__float_as_uint(ff[r / 2].x), __float_as_uint(ff[r / 2].y), 0x7632);
      }
      fsum = __fadd_rn(fsum, __fadd_rn(fs2.x, fs2.y));
#pragma unroll
      for (int e = 0; e < R / 4; ++e)
        o[e] = pack_low_bytes(__float_as_uint(rr[2 * e].x), __float_as_uint(rr[2 * e].y),
                              __float_as_uint(rr[2 * e + 1].x), __float_as_uint(rr[2 * e + 1].y));
    }
    __syncwarp();
    if (ok && lane == 0) tc::mbar_arrive(tc::smem_u32(empty + st));
    ++it;
    const int64_t k = (int64_t)b * kCqBoxRows + rg * R;
    if (ok && j < N && k < Kp) {
      if (iBt_bf16) {
        uint4* d = reinterpret_cast<uint4*>(iBt_bf16 + j * Kp + k);
#pragma unroll
        for (int q = 0; q < R / 8; ++q) d[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
      }
      if (iBt) {  // streaming stores: the product reads the bf16 copy, not these
        if constexpr (R % 16 == 0) {
          uint4* d = reinterpret_cast<uint4*>(iBt + j * Kp + k);
#pragma unroll
          for (int q = 0; q < R / 16; ++q) __stcs(d + q, make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]));
        } else {
          uint2* d = reinterpret_cast<uint2*>(iBt + j * Kp + k);
#pragma unroll
          for (int q = 0; q < R / 8; ++q) __stcs(d + q, make_uint2(o[2 * q], o[2 * q + 1]));
        }
      }
    }
  };
  // pass 1 of the first strip, then each strip's pass 2 interleaved box by
  // box with the next strip's pass 1, so that every CTA keeps reading new
  // rows from DRAM while it codes the strip it has in L2
  float m = 0.0f;
  for (int b = 0; b < nb1 && (int64_t)blockIdx.x < nstrips; ++b) max_box(m);
  for (int64_t strip = blockIdx.x; strip < nstrips; strip += gridDim.x) {
    const int64_t j = strip * W + c;
    red[rg][c] = m;
    consumers_sync();
    if (tid < W) {
      float r = red[0][tid];
#pragma unroll
      for (int g = 1; g < RG; ++g) r = fmaxf(r, red[g][tid]);
      float sv = __fdiv_rn(r, hi);
      sv = sv == 0.0f ? 1.0f : sv;
      sscale[tid] = sv;
      if (ok && strip * W + tid < N) scaleB[strip * W + tid] = sv;
    }
    consumers_sync();
    const float sc = sscale[c];
    const float rs = quot_rcp(sc);
    const bool rs_ok = rs == rs;
    float fsum = 0.0f;
    const int64_t nxt = strip + gridDim.x;
    const int nbm = nxt < nstrips ? nb1 : 0;
    m = 0.0f;
    for (int b = 0; b < (nb2 > nbm ? nb2 : nbm); ++b) {
      if (b < nb2) code_box(j, b, sc, rs, rs_ok, fsum);
      if (b < nbm) max_box(m);
    }
    // column sums (exact integers in fp32)
    red[rg][c] = fsum;
    consumers_sync();
    if (tid < W && ok && strip * W + tid < N) {
      float t = red[0][tid];
#pragma unroll
      for (int g = 1; g < RG; ++g) t = __fadd_rn(t, red[g][tid]);
      colsum[strip * W + tid] = __float2int_rn(t);
    }
    consumers_sync();
  }
}

template <typename T>
int launch_col_quant_tma(const T* B, int64_t K, int64_t N, int64_t Kp, int qmin, int qmax, int8_t* iBt,
                         __nv_bfloat16* iBt_bf16, float* scaleB, int32_t* colsum, uint32_t* status, cudaStream_t s) {
  const int ar = smem_attr((const void*)col_quant_tma<T>, (int)kCqSmem);
  if (ar) return ar;
  constexpr int W = kCqRowBytes / (int)sizeof(T);
  CUtensorMap map;
  const int rc = tc::make_map_plain_2d(&map, B,
                                       sizeof(T) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                       N, K, N * (int64_t)sizeof(T), W, kCqBoxRows, "quantize_cols");
  if (rc) return rc;
  const int grid = (int)std::min<int64_t>(ceil_div(N, (int64_t)W), (int64_t)sm_count());
  col_quant_tma<T><<<grid, kCqThreads, kCqSmem, s>>>(map, K, N, Kp, qmin, qmax, iBt, iBt_bf16, scaleB, colsum, status);
  I8Q_LAUNCH_CHECK("col_quant_tma");
  return I8Q_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int launch_quantize_rows(const void* A, int typeA, int64_t M, int64_t K, int64_t lda, uint8_t* uA,
                         __nv_bfloat16* uA_bf16, int64_t Kp, float* scaleA, int32_t* zeroA, cudaStream_t s) {
  if (M <= 0) return I8Q_OK;
  int64_t blocks = std::min<int64_t>(M, (int64_t)sm_count() * 8);
  I8Q_PROF("quantize_rows", s);
  // rows staged in shared memory, when they fit and a row is too long for
  // 8 vectors a lane in registers (measured on 32768 rows: registers win up
  // to 2048 elements of either type, 1.1-1.7x; staging wins for bf16 rows of
  // 4096, 1.4x, where 16 vectors a lane crowd the registers)
  {
    const bool bf = typeA == I8Q_BF16;
    const int64_t esz = bf ? 2 : 4;
    const size_t smem = 2 * (size_t)kStageRows * (size_t)(K * esz) + 64;
    const bool aligned = aligned16(A) && K % 8 == 0 && (lda * esz) % 16 == 0;
    uint32_t* status = device_status_word();
    const int64_t groups = ceil_div(M, (int64_t)kStageRows);
    // worth it once the row groups fill the GPU; fewer rows keep the
    // register form (lower latency per launch)
    if (aligned && status && K > 2048 && smem <= 200 * 1024 && groups >= sm_count() && !getenv("I8Q_ROWS_REGISTER")) {
      int ar = smem_attr((const void*)quantize_rows_staged<float>, 200 * 1024 + 64);
      if (!ar) ar = smem_attr((const void*)quantize_rows_staged<__nv_bfloat16>, 200 * 1024 + 64);
      if (ar) return ar;
      const void* kern = bf ? (const void*)quantize_rows_staged<__nv_bfloat16> : (const void*)quantize_rows_staged<float>;
      // one wave of the blocks that fit at once (shared memory and threads)
      int per_sm = 0;
      I8Q_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kStageThreads, smem));
      const int grid = (int)std::min<int64_t>(groups, (int64_t)sm_count() * std::max(per_sm, 1));
      if (bf)
        quantize_rows_staged<__nv_bfloat16><<<grid, kStageThreads, smem, s>>>(static_cast<const __nv_bfloat16*>(A), M, K, lda,
                                                                    uA, uA_bf16, Kp, scaleA, zeroA, status);
      else
        quantize_rows_staged<float><<<grid, kStageThreads, smem, s>>>(static_cast<const float*>(A), M, K, lda, uA, uA_bf16, Kp,
                                                            scaleA, zeroA, status);
      I8Q_LAUNCH_CHECK("quantize_rows_staged");
      return I8Q_OK;
    }
  }
  // warp per row with the row in registers, when it fits
  {
    const bool bf = typeA == I8Q_BF16;
    const int64_t esz = bf ? 2 : 4;
    const bool aligned = aligned16(A) && K % 8 == 0 && (lda * esz) % 16 == 0;
    const int nv_max = bf ? 16 : 8;
    int nv = 1;
    while (nv < nv_max && 256 * nv < K) nv *= 2;
    if (aligned && 256 * nv >= K) {
      const int64_t wblocks = ceil_div(M, 4);  // 4 rows (warps) per 128-thread block
      if (bf) {
        const __nv_bfloat16* a = static_cast<const __nv_bfloat16*>(A);
        switch (nv) {
          case 1: quantize_rows_warp<__nv_bfloat16, 1><<<(unsigned)wblocks, 128, 0, s>>>(a, M, K, lda, uA, uA_bf16, Kp, scaleA, zeroA); break;
          case 2: quantize_rows_warp<__nv_bfloat16, 2><<<(unsigned)wblocks, 128, 0, s>>>(a, M, K, lda, uA, uA_bf16, Kp, scaleA, zeroA); break;
          case 4: quantize_rows_warp<__nv_bfloat16, 4><<<(unsigned)wblocks, 128, 0, s>>>(a, M, K, lda, uA, uA_bf16, Kp, scaleA, zeroA); break;
          case 8: quantize_rows_warp<__nv_bfloat16, 8><<<(unsigned)wblocks, 128, 0, s>>>(a, M, K, lda, uA, uA_bf16, Kp, scaleA, zeroA); break;
          default: quantize_rows_warp<__nv_bfloat16, 16><<<(unsigned)wblocks, 128, 0, s>>>(a, M, K, lda, uA, uA_bf16, Kp, scaleA, zeroA); break;
        }
      } else {
        const float* a = static_cast<const float*>(A);
        switch (nv) {
          case 1: quantize_rows_warp<float, 1><<<(unsigned)wblocks, 128, 0, s>>>(a, M, K, lda, uA, uA_bf16, Kp, scaleA, zeroA); break;
          case 2: quantize_rows_warp<float, 2><<<(unsigned)wblocks, 128, 0, s>>>(a, M, K, lda, uA, uA_bf16, Kp, scaleA, zeroA); break;
          case 4: quantize_rows_warp<float, 4><<<(unsigned)wblocks, 128, 0, s>>>(a, M, K, lda, uA, uA_bf16, Kp, scaleA, zeroA); break;
          default: quantize_rows_warp<float, 8><<<(unsigned)wblocks, 128, 0, s>>>(a, M, K, lda, uA, uA_bf16, Kp, scaleA, zeroA); break;
        }
      }
      I8Q_LAUNCH_CHECK("quantize_rows_warp");
      return I8Q_OK;
    }
  }
  if (typeA == I8Q_F32) {
    const float* a = static_cast<const float*>(A);
    bool vec = aligned16(a) && K % 8 == 0 && lda % 4 == 0;
    if (vec)
      quantize_rows_kernel<float, true><<<blocks, kRowThreads, 0, s>>>(a, M, K, lda, uA, uA_bf16, Kp, scaleA, zeroA);
    else
      quantize_rows_kernel<float, false><<<blocks, kRowThreads, 0, s>>>(a, M, K, lda, uA, uA_bf16, Kp, scaleA, zeroA);
  } else {
    const __nv_bfloat16* a = static_cast<const __nv_bfloat16*>(A);
    bool vec = aligned16(a) && K % 8 == 0 && lda % 8 == 0;
    if (vec)
      quantize_rows_kernel<__nv_bfloat16, true><<<blocks, kRowThreads, 0, s>>>(a, M, K, lda, uA, uA_bf16, Kp, scaleA, zeroA);
    else
      quantize_rows_kernel<__nv_bfloat16, false><<<blocks, kRowThreads, 0, s>>>(a, M, K, lda, uA, uA_bf16, Kp, scaleA, zeroA);
  }
  I8Q_LAUNCH_CHECK("quantize_rows_kernel");
  return I8Q_OK;
}

int launch_quantize_cols(const void* B, int typeB, int64_t K, int64_t N, int avoid_overflow, int8_t* iBt,
                         __nv_bfloat16* iBt_bf16, int64_t Kp, float* scaleB, int32_t* colsum,
                         uint32_t* colmax_scratch, cudaStream_t s) {
  if (N <= 0) return I8Q_OK;
  const int qmax = avoid_overflow ? 63 : 127, qmin = avoid_overflow ? -64 : -128;
  I8Q_PROF("quantize_cols", s);
  const bool bf = typeB == I8Q_BF16;
  uint32_t* status = device_status_word();
  if (status && N % (bf ? 8 : 4) == 0 && Kp % 64 == 0 && K < ((int64_t)1 << 31) && N < ((int64_t)1 << 31) &&
      aligned16(B) && aligned16(iBt) && aligned16(iBt_bf16) && !getenv("I8Q_COLS_TWO_PASS")) {
    if (bf)
      return launch_col_quant_tma(static_cast<const __nv_bfloat16*>(B), K, N, Kp, qmin, qmax, iBt, iBt_bf16, scaleB,
                                  colsum, status, s);
    return launch_col_quant_tma(static_cast<const float*>(B), K, N, Kp, qmin, qmax, iBt, iBt_bf16, scaleB, colsum,
                                status, s);
  }
  if (colmax_scratch && N % 4 == 0 && aligned16(B)) {
    I8Q_CUDA_TRY(cudaMemsetAsync(colmax_scratch, 0, (size_t)N * 4, s));
    I8Q_CUDA_TRY(cudaMemsetAsync(colsum, 0, (size_t)N * 4, s));
    dim3 g1((unsigned)ceil_div(N, kWideCols), (unsigned)ceil_div(K, kWideKSplit));
    dim3 g2((unsigned)ceil_div(N, kWideCols), (unsigned)ceil_div(Kp, kWideKSplit));
    if (typeB == I8Q_F32) {
      const float* b = static_cast<const float*>(B);
      col_absmax_wide<float><<<g1, 256, 0, s>>>(b, K, N, colmax_scratch);
      col_quant_wide<float><<<g2, 256, 0, s>>>(b, K, N, Kp, colmax_scratch, qmin, qmax, iBt, iBt_bf16, scaleB, colsum);
    } else {
      const __nv_bfloat16* b = static_cast<const __nv_bfloat16*>(B);
      col_absmax_wide<__nv_bfloat16><<<g1, 256, 0, s>>>(b, K, N, colmax_scratch);
      col_quant_wide<__nv_bfloat16><<<g2, 256, 0, s>>>(b, K, N, Kp, colmax_scratch, qmin, qmax, iBt, iBt_bf16, scaleB,
                                                       colsum);
    }
    I8Q_LAUNCH_CHECK("col_quant_wide");
    return I8Q_OK;
  }
  dim3 grid((unsigned)ceil_div(N, kColW));
  if (typeB == I8Q_F32)
    cols_kernel<float, 0><<<grid, 256, 0, s>>>(static_cast<const float*>(B), K, N, N, qmin, qmax, iBt, iBt_bf16, Kp,
                                               scaleB, colsum, 0);
  else
    cols_kernel<__nv_bfloat16, 0><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(B), K, N, N, qmin, qmax,
                                                       iBt, iBt_bf16, Kp, scaleB, colsum, 0);
  I8Q_LAUNCH_CHECK("cols_kernel(quantize)");
  return I8Q_OK;
}

bool repack_tiles_ok(const void* B, int64_t K, int64_t N, int64_t ldb, const void* iBt, const void* iBt_bf16,
                     int64_t Kp) {
  const auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  return N > 0 && N % 16 == 0 && ldb % 16 == 0 && Kp % 16 == 0 && Kp >= K && al16(B) && (!iBt || al16(iBt)) &&
         (!iBt_bf16 || al16(iBt_bf16)) && (iBt || iBt_bf16) && ceil_div(Kp, kRtK) <= 65535 &&
         ceil_div(N, kRtCols) <= 0x7fffffff;
}

void launch_repack_tiles(const void* B, bool flip, int64_t K, int64_t N, int64_t ldb, int8_t* iBt,
                         __nv_bfloat16* iBt_bf16, int64_t Kp, int32_t* colsum, int64_t gates_H, cudaStream_t s) {
  const dim3 grid((unsigned)ceil_div(N, kRtCols), (unsigned)ceil_div(Kp, kRtK));
  const auto* b8 = static_cast<const int8_t*>(B);
  if (flip) repack_tiles_s8<true><<<grid, 256, 0, s>>>(b8, K, N, ldb, iBt, iBt_bf16, Kp, colsum, gates_H);
  else repack_tiles_s8<false><<<grid, 256, 0, s>>>(b8, K, N, ldb, iBt, iBt_bf16, Kp, colsum, gates_H);
}

int launch_repack_cols_s8(const int8_t* B, int64_t K, int64_t N, int64_t ldb, int8_t* iBt, __nv_bfloat16* iBt_bf16,
                          int64_t Kp, int32_t* colsum, cudaStream_t s) {
  return launch_repack_cols_s8_gates(B, K, N, ldb, iBt, iBt_bf16, Kp, colsum, 0, s);
}

int launch_repack_cols_s8_gates(const int8_t* B, int64_t K, int64_t N, int64_t ldb, int8_t* iBt,
                                __nv_bfloat16* iBt_bf16, int64_t Kp, int32_t* colsum, int64_t gates_H, cudaStream_t s) {
  if (N <= 0) return I8Q_OK;
  if (gates_H > 0 && N != 4 * gates_H) return fail(I8Q_ERR_INVALID_ARG, "repack: gate interleave needs N == 4H");
  I8Q_PROF("repack_cols", s);
  if (repack_tiles_ok(B, K, N, ldb, iBt, iBt_bf16, Kp)) {
    I8Q_CUDA_TRY(cudaMemsetAsync(colsum, 0, (size_t)N * sizeof(int32_t), s));
    launch_repack_tiles(B, false, K, N, ldb, iBt, iBt_bf16, Kp, colsum, gates_H, s);
    I8Q_LAUNCH_CHECK("repack_tiles_s8");
    return I8Q_OK;
  }
  dim3 grid((unsigned)ceil_div(N, kColW));
  cols_kernel<int8_t, 1><<<grid, 256, 0, s>>>(B, K, N, ldb, -128, 127, iBt, iBt_bf16, Kp, nullptr, colsum, gates_H);
  I8Q_LAUNCH_CHECK("cols_kernel(repack)");
  return I8Q_OK;
}

}  // namespace i8q
