// conv.cu -- QLinearConv (onnx-light docs, "QLinearConv", since version 10),
// 2-D NCHW.
//
//   acc = sum_{c in group, kh, kw} (x - x_zero_point) * (w - w_zero_point[m])
//   acc += B[m]                       (int32 bias: scale x_scale*w_scale, zp 0)
//   y   = saturate(rint(((float)acc * (x_scale * w_scale[m])) / y_scale) + y_zero_point)
// A position outside the input holds real 0 (the code x_zero_point), so it
// adds nothing.  The requantization is DequantizeLinear of the accumulator
// followed by QuantizeLinear with (y_scale, y_zero_point).
//
// This file holds the direct form used for every group count: one thread
// per output pixel, the centered filter of the CTA's output channel staged
// in shared memory, exact int32 accumulation.
#include "common.cuh"

namespace i8q {
namespace {

template <typename XT, typename WT, typename YT>
__global__ void __launch_bounds__(256)
qlinearconv_direct(const XT* __restrict__ x, const WT* __restrict__ w, const float* __restrict__ w_scale,
                   const WT* __restrict__ w_zp, int per_channel, const int32_t* __restrict__ B, int C, int H,
                   int W, int M, int Cg, int Mg, int kH, int kW, int OH, int OW, int pt, int pl, int sh, int sw,
                   int dh, int dw, float x_scale, int x_zp, float y_scale, int y_zp, float qlo, float qhi,
                   YT* __restrict__ y) {
  extern __shared__ int wc[];  // centered filter of channel m: Cg * kH * kW
  const int m = blockIdx.y, n = blockIdx.z;
  const int taps = Cg * kH * kW;
  const int wz = (int)w_zp[per_channel ? m : 0];
  for (int i = threadIdx.x; i < taps; i += blockDim.x) wc[i] = (int)w[(int64_t)m * taps + i] - wz;
  __syncthreads();
  const int g = m / Mg;
  const int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= (int64_t)OH * OW) return;
  const int oh = (int)(p / OW), ow = (int)(p % OW);
  const XT* xb = x + ((int64_t)n * C + (int64_t)g * Cg) * H * W;
  int32_t acc = 0;
  for (int cc = 0; cc < Cg; ++cc) {
    const XT* xc = xb + (int64_t)cc * H * W;
    const int* wcc = wc + cc * kH * kW;
    for (int kh = 0; kh < kH; ++kh) {
      const int ih = oh * sh - pt + kh * dh;
      if (ih < 0 || ih >= H) continue;
      for (int kw = 0; kw < kW; ++kw) {
        const int iw = ow * sw - pl + kw * dw;
        if (iw < 0 || iw >= W) continue;
        acc += ((int)xc[(int64_t)ih * W + iw] - x_zp) * wcc[kh * kW + kw];
      }
    }
  }
  if (B) acc += B[m];
  float v = __int2float_rn(acc);
  const float mul = __fmul_rn(x_scale, w_scale[per_channel ? m : 0]);
  v = __fmul_rn(v, mul);
  v = __fdiv_rn(v, y_scale);
  y[(((int64_t)n * M + m) * OH + oh) * OW + ow] = (YT)(sat_rint(v, qlo - (float)y_zp, qhi - (float)y_zp) + y_zp);
}

// Depthwise form (group == C == M): one CTA per (image, channel) plane.  The
// input plane is staged in shared memory as centred int16 (x - x_zp, with the
// padding never read: out-of-range taps are skipped, i.e. real 0), the
// plane's filter in registers, and every output of the plane computed from
// shared memory, requantized and stored with consecutive threads on
// consecutive outputs.
template <typename XT, typename WT, typename YT>
__global__ void __launch_bounds__(256)
qlinearconv_depthwise_plane(const XT* __restrict__ x, const WT* __restrict__ w, const float* __restrict__ w_scale,
                            const WT* __restrict__ w_zp, int per_channel, const int32_t* __restrict__ B, int C, int H,
                            int W, int kH, int kW, int OH, int OW, int pt, int pl, int sh, int sw, int dh, int dw,
                            float x_scale, int x_zp, float y_scale, int y_zp, float qlo, float qhi,
                            YT* __restrict__ y) {
  extern __shared__ int16_t plane[];  // H * W centred inputs
  const int c = blockIdx.x % C, n = blockIdx.x / C;
  const XT* xp = x + ((int64_t)n * C + c) * H * W;
  const int HW = H * W;
  // 16-byte loads where the plane is aligned (planes of a multiple of 16 bytes)
  if ((reinterpret_cast<uintptr_t>(xp) & 15) == 0) {
    const int nv = HW / 16;
    for (int v = threadIdx.x; v < nv; v += blockDim.x) {
      const uint4 q = __ldg(reinterpret_cast<const uint4*>(xp) + v);
      const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int e = 0; e < 16; ++e) plane[16 * v + e] = (int16_t)((int)(XT)((wd[e >> 2] >> (8 * (e & 3))) & 0xff) - x_zp);
    }
    for (int i = nv * 16 + threadIdx.x; i < HW; i += blockDim.x) plane[i] = (int16_t)((int)xp[i] - x_zp);
  } else {
    for (int i = threadIdx.x; i < HW; i += blockDim.x) plane[i] = (int16_t)((int)xp[i] - x_zp);
  }
  const int taps = kH * kW;
  const int wz = (int)w_zp[per_channel ? c : 0];
  __shared__ int wc[25];
  if (threadIdx.x < taps) wc[threadIdx.x] = (int)w[(int64_t)c * taps + threadIdx.x] - wz;
  const int32_t bc = B ? B[c] : 0;
  const float mul = __fmul_rn(x_scale, w_scale[per_channel ? c : 0]);
  const float lo_z = qlo - (float)y_zp, hi_z = qhi - (float)y_zp;
  __syncthreads();
  YT* yp = y + ((int64_t)n * C + c) * OH * OW;
  const int OHW = OH * OW;
  for (int o = threadIdx.x; o < OHW; o += blockDim.x) {
    const int oh = o / OW, ow = o - oh * OW;
    int32_t acc = 0;
    for (int kh = 0; kh < kH; ++kh) {
      const int ih = oh * sh - pt + kh * dh;
      if (ih < 0 || ih >= H) continue;
      for (int kw = 0; kw < kW; ++kw) {
        const int iw = ow * sw - pl + kw * dw;
        if (iw >= 0 && iw < W) acc += (int)plane[ih * W + iw] * wc[kh * kW + kw];
      }
    }
    float v = __fmul_rn(__int2float_rn(acc + bc), mul);
    v = __fdiv_rn(v, y_scale);
    yp[o] = (YT)rint_code_bits(v, lo_z, hi_z, y_zp);
  }
}

// Depthwise with a KxK filter, stride 1, dilation 1: the plane is staged with
// a halo of zeros (centred zero = the padding value) so every tap reads
// shared memory without a bounds check.  Shared layout: (H + 2P) rows of
// (W + 2P) int16, P = the larger pad.
template <typename XT, typename WT, typename YT, int KS>
__global__ void __launch_bounds__(256)
qlinearconv_depthwise_halo(const XT* __restrict__ x, const WT* __restrict__ w, const float* __restrict__ w_scale,
                           const WT* __restrict__ w_zp, int per_channel, const int32_t* __restrict__ B, int C, int H,
                           int W, int OH, int OW, int pt, int pl, int P, float x_scale, int x_zp, float y_scale,
                           int y_zp, float qlo, float qhi, YT* __restrict__ y) {
  extern __shared__ int16_t hp[];
  const int c = blockIdx.x % C, n = blockIdx.x / C;
  const int HP = H + 2 * P, WP = W + 2 * P;
  const XT* xp = x + ((int64_t)n * C + c) * H * W;
  for (int i = threadIdx.x; i < HP * WP; i += blockDim.x) hp[i] = 0;
  __syncthreads();
  const int HW = H * W;
  if ((reinterpret_cast<uintptr_t>(xp) & 15) == 0 && (W & 15) == 0) {
    for (int v = threadIdx.x; v < HW / 16; v += blockDim.x) {
      const uint4 q = __ldg(reinterpret_cast<const uint4*>(xp) + v);
      const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
      const int e0 = 16 * v, r = e0 / W, col = e0 - r * W;
      int16_t* dst = hp + (r + P) * WP + col + P;
#pragma unroll
      for (int e = 0; e < 16; ++e) dst[e] = (int16_t)((int)(XT)((wd[e >> 2] >> (8 * (e & 3))) & 0xff) - x_zp);
    }
  } else {
    for (int i = threadIdx.x; i < HW; i += blockDim.x) {
      const int r = i / W, col = i - r * W;
      hp[(r + P) * WP + col + P] = (int16_t)((int)xp[i] - x_zp);
    }
  }
  const int wz = (int)w_zp[per_channel ? c : 0];
  int wc[KS * KS];
#pragma unroll
  for (int t = 0; t < KS * KS; ++t) wc[t] = (int)w[(int64_t)c * KS * KS + t] - wz;
  const int32_t bc = B ? B[c] : 0;
  const float mul = __fmul_rn(x_scale, w_scale[per_channel ? c : 0]);
  const float lo_z = qlo - (float)y_zp, hi_z = qhi - (float)y_zp;
  __syncthreads();
  YT* yp = y + ((int64_t)n * C + c) * OH * OW;
  // output (oh, ow) reads hp rows oh - pt + P + kh, columns ow - pl + P + kw
  const int ro = P - pt, co = P - pl;
  for (int oh = threadIdx.x / 32; oh < OH; oh += blockDim.x / 32)
    for (int ow = threadIdx.x & 31; ow < OW; ow += 32) {
      const int16_t* base = hp + (oh + ro) * WP + ow + co;
      int32_t acc = 0;
#pragma unroll
      for (int kh = 0; kh < KS; ++kh)
#pragma unroll
        for (int kw = 0; kw < KS; ++kw) acc += (int)base[kh * WP + kw] * wc[kh * KS + kw];
      float v = __fmul_rn(__int2float_rn(acc + bc), mul);
      v = __fdiv_rn(v, y_scale);
      yp[oh * OW + ow] = (YT)rint_code_bits(v, lo_z, hi_z, y_zp);
    }
}

// Depthwise KS x KS, stride 1, dilation 1, on the two-way dot product of
// 16-bit and 8-bit integers (dp2a) over the raw input codes.  A CTA takes
// `ppc` consecutive (image, channel) planes; each sits in shared memory as
// its codes, row r of the plane at byte kX0 of shared row r + pt (rows of
// RW words), the halo filled with the x zero point's code.  With the
// centred filter w' = w - w_zp (|w'| <= 255, exact in 16 bits),
//   sum (x - x_zp)(w - w_zp) = sum x w' - x_zp sum w'
// over all KS^2 taps: a padded tap holds x = x_zp and so adds nothing, and
// x_zp sum w' is a constant of the channel.  dp2a multiplies the two 16-bit
// halves of one operand with two bytes of the other (bytes 0, 1 or 2, 3),
// so a 4-byte window of an input row starting at output e serves outputs e
// and e + 1: e takes (w'0, w'1) on bytes 0, 1 and (w'2, 0) on bytes 2, 3;
// e + 1 takes (0, w'0) and (w'1, w'2) (for KS = 5 a second window adds the
// taps past the fourth byte).  Every sum is exact in int32.
//
// A thread owns an item: R output rows x 8 consecutive outputs.  It reads
// each of the R + KS - 1 input rows the item needs once (NWD words, shifted
// once to the item's first byte), forms the windows of the even outputs by
// byte permutes with constant selectors, and feeds every output row that
// row reaches (up to KS of them); an output row is requantized and stored
// (one 8-byte store) as soon as its last input row is in.  A plane whose
// sums all stay below 2^22 in magnitude and whose quotients stay below 2^20
// (bounded from its filter, bias and scales when its constants are staged)
// takes the bracketed form of dw_requant_fast: its sums carry 1.5 * 2^23
// from the start, so each int32 pattern is already an exact float, and two
// rounded ends of an interval around the quotient give the code when they
// agree.  Other planes take each code from the reciprocal product
// (quot_code_bits), with the quotient itself near a half-integer or when
// 1 / y_scale is not a normal number.  (Tap sums on the fp32 pipe, exact
// for these magnitudes, were measured slower: the byte-to-float conversions
// outweigh the faster multiply-adds.)
constexpr int kStrip = 8, kX0 = 8;  // outputs per item row; byte of x column 0 in a shared row

// Words of a shared row: the slack before column 0, the items' outputs, the
// filter's reach past them; a multiple of 4 so rows are 16-byte aligned.
__host__ __device__ constexpr int dw_row_words(int nstrips, int ks) {
  return ((kX0 + nstrips * kStrip + 4 * ((ks + 3) / 4) + 8 + 15) / 16) * 4;
}

// Output rows per item: KS = 3 keeps three rows of sums in flight, KS = 5 five.
template <int KS>
constexpr int dw_rows() { return KS == 3 ? 7 : 4; }

// Per-plane constants staged in shared memory after the planes.
template <int KS>
struct DwPlane {
  // per filter row, the 16-bit pairs of w' = w - w_zp the dp2a steps take:
  // KS = 3: (w'0, w'1), (w'2, 0) for an even output, (0, w'0), (w'1, w'2)
  // for the odd one; KS = 5 adds (w'4, 0) and (w'3, w'4) on the window four
  // bytes on
  uint32_t wp[KS][KS == 3 ? 4 : 6];
  int k0;     // B - x_zp sum w', plus 0x4B400000 when fast
  float mul;  // x_scale * w_scale
  int fast;   // the plane's sums and quotients fit the bracketed requantization
};

// d = c + a.lo16 * b.byte(0|2) + a.hi16 * b.byte(1|3): a holds two signed
// 16-bit values, b four codes (signed when BS).
template <bool HI, bool BS>
__device__ __forceinline__ int dp2a(uint32_t a, uint32_t b, int c) {
  int d;
  if (HI && BS) asm("dp2a.hi.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  else if (HI) asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  else if (BS) asm("dp2a.lo.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  else asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ uint32_t pair16(int lo, int hi) {
  return (uint32_t)(lo & 0xffff) | ((uint32_t)hi << 16);
}

__device__ __forceinline__ void dw_cp_async(uint32_t dst, const void* src, int bytes) {
  if (bytes == 8) asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(dst), "l"(src) : "memory");
  else asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void dw_cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void dw_cp_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// The code of one sum from the quotient itself: the fallback of
// dw_requant_fast (accb carries 1.5 * 2^23 + acc).
__device__ __forceinline__ int dw_code_exact(int accb, float mul, float y_scale, float lo_z, float hi_z, int y_zp) {
  const float v = __fmul_rn(__fsub_rn(__int_as_float(accb), 12582912.0f), mul);
  return (int)(rint_code_bits(__fdiv_rn(v, y_scale), lo_z, hi_z, y_zp) - 0x4B400000u);
}

// Four codes saturated to the range of YT, packed with byte 0 from a.
template <typename YT>
__device__ __forceinline__ uint32_t pack_sat4(int a, int b, int c, int d) {
  uint32_t hi, r;
  if (std::is_same<YT, uint8_t>::value) {
    asm("cvt.pack.sat.u8.s32.b32 %0, %1, %2, %3;" : "=r"(hi) : "r"(d), "r"(c), "r"(0u));
    asm("cvt.pack.sat.u8.s32.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(b), "r"(a), "r"(hi));
  } else {
    asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, %3;" : "=r"(hi) : "r"(d), "r"(c), "r"(0u));
    asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(b), "r"(a), "r"(hi));
  }
  return r;
}

// The rare ends of a bracketed row, out of line so that the row loop's code
// stays small: the codes from the quotient itself when the bracket's ends
// differed, and the bytewise stores of a row that is not one whole aligned
// 8-byte piece.
template <typename YT>
__device__ __noinline__ void dw_row_rare(int b0, int b1, int b2, int b3, int b4, int b5, int b6, int b7, int c0, int c1,
                                         int c2, int c3, int c4, int c5, int c6, int c7, bool exact, float mul,
                                         float y_scale, float lo_z, float hi_z, int y_zp, YT* out, bool vec, int n) {
  const int accb[kStrip] = {b0, b1, b2, b3, b4, b5, b6, b7};
  int code[kStrip] = {c0, c1, c2, c3, c4, c5, c6, c7};
  if (exact) {
#pragma unroll
    for (int e = 0; e < kStrip; ++e) code[e] = dw_code_exact(accb[e], mul, y_scale, lo_z, hi_z, y_zp);
  }
  if (vec) {
    *reinterpret_cast<uint2*>(out) = make_uint2(pack_sat4<YT>(code[0], code[1], code[2], code[3]),
                                                pack_sat4<YT>(code[4], code[5], code[6], code[7]));
  } else {
    constexpr int lo = std::is_same<YT, uint8_t>::value ? 0 : -128, hi = lo + 255;
#pragma unroll
    for (int e = 0; e < kStrip; ++e)
      if (e < n) out[e] = (YT)min(max(code[e], lo), hi);
  }
}

// Requantize the 8 sums of an output row of a fast plane and store the
// codes.  Each sum arrives as the bit pattern of 1.5 * 2^23 + acc (the
// plane's constant carries the offset; |acc| < 2^22, so the pattern is the
// exact float and subtracting the offset gives fl(acc) exactly).  With
// v = fl(acc * mul) and yrl < 1 / y_scale < yrh (yr scaled by 1 -+ 2^-20,
// each rounded once), the exact products v * yrl and v * yrh enclose v /
// y_scale with a margin of more than 2^-21 |v / y_scale|, so they strictly
// enclose the quotient fl(v / y_scale) too.  Each fma adds mz = 1.5 * 2^23 +
// y_zp to one product and rounds once to an integer (|q| < 2^21 keeps the
// sum in the binade of unit spacing), a non-decreasing function of the
// product: when both ends give the same integer, so does the quotient,
// which is then no half-integer (both neighbours would lie inside), so the
// integer is y_zp + rint(quotient), saturated by the pack.  Ends that differ
// send the row to the quotient itself.
template <typename YT>
__device__ __forceinline__ void dw_requant_fast(const int (&accb)[kStrip], float mul, float yrh, float yrl, float mz,
                                                float y_scale, float lo_z, float hi_z, int y_zp, YT* out, bool vec,
                                                int n) {
  int code[kStrip];
  uint32_t diff = 0;
#pragma unroll
  for (int e = 0; e < kStrip; e += 2) {
    const float2 a = fma2_rn(make_float2(__int_as_float(accb[e]), __int_as_float(accb[e + 1])),
                             make_float2(1.0f, 1.0f), make_float2(-12582912.0f, -12582912.0f));
    const float2 v = mul2_rn(a, make_float2(mul, mul));
    const float2 rh = fma2_rn(v, make_float2(yrh, yrh), make_float2(mz, mz));
    const float2 rl = fma2_rn(v, make_float2(yrl, yrl), make_float2(mz, mz));
    diff |= (__float_as_uint(rh.x) ^ __float_as_uint(rl.x)) | (__float_as_uint(rh.y) ^ __float_as_uint(rl.y));
    code[e] = __float_as_int(rh.x) - 0x4B400000;
    code[e + 1] = __float_as_int(rh.y) - 0x4B400000;
  }
  if (vec && !diff) {
    *reinterpret_cast<uint2*>(out) = make_uint2(pack_sat4<YT>(code[0], code[1], code[2], code[3]),
                                                pack_sat4<YT>(code[4], code[5], code[6], code[7]));
  } else {
    dw_row_rare<YT>(accb[0], accb[1], accb[2], accb[3], accb[4], accb[5], accb[6], accb[7], code[0], code[1],
                    code[2], code[3], code[4], code[5], code[6], code[7], diff != 0, mul, y_scale, lo_z, hi_z, y_zp,
                    out, vec, n);
  }
}

// The planes outside the bracketed form: each code from the reciprocal
// product, or from the quotient near a half-integer.  Out of line, so the
// row loop's code stays small.
template <typename YT>
__device__ __noinline__ void dw_requant_general(int a0, int a1, int a2, int a3, int a4, int a5, int a6, int a7,
                                                float mul, float y_scale, float yr, float lo_z, float hi_z, int y_zp,
                                                YT* out, bool vec, int n) {
  const int a[kStrip] = {a0, a1, a2, a3, a4, a5, a6, a7};
  uint32_t code[kStrip];
#pragma unroll
  for (int e = 0; e < kStrip; ++e)
    code[e] = quot_code_bits(__fmul_rn(__int2float_rn(a[e]), mul), y_scale, yr, lo_z, hi_z, y_zp);
  if (vec) {
    *reinterpret_cast<uint2*>(out) = make_uint2(pack_low_bytes(code[0], code[1], code[2], code[3]),
                                                pack_low_bytes(code[4], code[5], code[6], code[7]));
  } else {
#pragma unroll
    for (int e = 0; e < kStrip; ++e)
      if (e < n) out[e] = (YT)code[e];
  }
}

// Persistent: CTA b takes the groups of `ppc` consecutive planes b, b +
// gridDim.x, ...; two shared buffers, the next group's planes copied in
// (cp.async, 8- or 4-byte pieces) while the current one is computed.  The
// halo of both buffers is written once: copies touch only the interior.
template <typename XT, typename WT, typename YT, int KS>
__global__ void __launch_bounds__(224, 3)  // 3 CTAs of 7 warps per SM: at most 80 registers
qlinearconv_depthwise_rows(const XT* __restrict__ x, const WT* __restrict__ w, const float* __restrict__ w_scale,
                           const WT* __restrict__ w_zp, int per_channel, const int32_t* __restrict__ B, int C, int H,
                           int W, int OH, int OW, int pt, int pl, int planes, int ppc, float x_scale, int x_zp,
                           float y_scale, int y_zp, float qlo, float qhi, YT* __restrict__ y) {
  constexpr bool XS = std::is_signed<XT>::value;  // the weights enter centred, as 16-bit values
  constexpr int NWD = KS == 3 ? 4 : 5;  // words read per input row of an item (8 outputs + KS - 1)
  constexpr int R = dw_rows<KS>();
  extern __shared__ __align__(16) uint32_t smw[];
  const int nstrips = (OW + kStrip - 1) / kStrip, nblocks = (OH + R - 1) / R;
  const int HP = OH + KS - 1, RW = dw_row_words(nstrips, KS), PW = HP * RW;
  const int buf_words = ppc * PW;
  DwPlane<KS>* prm_base = reinterpret_cast<DwPlane<KS>*>(smw + 2 * buf_words);
  const int nthr = (int)blockDim.x, tid = (int)threadIdx.x;
  const uint32_t fill = (uint32_t)(uint8_t)x_zp * 0x01010101u;
  const int rows_in = min(H, HP - pt);  // input rows that reach an output
  const int ngroups = (planes + ppc - 1) / ppc;
  const float yr = quot_rcp(y_scale);
  const bool rcp_ok = yr == yr;
  const float yrh = __fmul_rn(yr, 1.0f + 0x1p-20f), yrl = __fmul_rn(yr, 1.0f - 0x1p-20f);
  const float mz = 12582912.0f + (float)y_zp;

  // both buffers: every word the zero point's code, once
  for (int i = tid; i < 2 * buf_words / 4; i += nthr)
    reinterpret_cast<uint4*>(smw)[i] = make_uint4(fill, fill, fill, fill);
  __syncthreads();

  // copies: a thread takes whole input rows, in pieces of 8 or 4 bytes
  // (single bytes when the rows are not word aligned)
  const int pb = ((W & 7) == 0 && (reinterpret_cast<uintptr_t>(x) & 7) == 0) ? 8
                 : ((W & 3) == 0 && (reinterpret_cast<uintptr_t>(x) & 3) == 0) ? 4 : 1;

  // issue the copies of group grp into buffer bi and its plane constants
  auto stage = [&](int grp, int bi) {
    const int p0 = grp * ppc, np = min(ppc, planes - p0);
    const uint8_t* xs = reinterpret_cast<const uint8_t*>(x + (int64_t)p0 * H * W);
    const uint32_t dsts = (uint32_t)__cvta_generic_to_shared(smw + bi * buf_words) + kX0;
    for (int g = tid; g < np * H; g += nthr) {
      const int p = g / H, r = g - p * H;
      if (r >= rows_in) continue;
      const uint8_t* src = xs + (int64_t)g * W;
      const uint32_t dst = dsts + (uint32_t)((p * HP + pt + r) * RW) * 4u;
      if (pb > 1) {
        for (int j = 0; j < W; j += pb) dw_cp_async(dst + j, src + j, pb);
      } else {
        uint8_t* db = reinterpret_cast<uint8_t*>(smw + bi * buf_words) + (size_t)((p * HP + pt + r) * RW) * 4 + kX0;
        for (int j = 0; j < W; ++j) db[j] = src[j];
      }
    }
    for (int i = tid; i < np * (KS + 1); i += nthr) {
      if (i < np * KS) {
        // (plane, filter row): the row's 16-bit weight pairs
        const int pi = i / KS, kh = i - pi * KS;
        const int c = (p0 + pi) % C;
        DwPlane<KS>& P = prm_base[bi * ppc + pi];
        const int wz = (int)w_zp[per_channel ? c : 0];
        int v[KS];
#pragma unroll
        for (int kw = 0; kw < KS; ++kw) v[kw] = (int)w[(int64_t)c * KS * KS + kh * KS + kw] - wz;
        P.wp[kh][0] = pair16(v[0], v[1]);
        P.wp[kh][2] = pair16(0, v[0]);
        P.wp[kh][3] = pair16(v[1], v[2]);
        if constexpr (KS == 3) {
          P.wp[kh][1] = pair16(v[2], 0);
        } else {
          P.wp[kh][1] = pair16(v[2], v[3]);
          P.wp[kh][4] = pair16(v[4], 0);
          P.wp[kh][5] = pair16(v[3], v[4]);
        }
      } else {
        // (plane): the constant term and the scale
        const int pi = i - np * KS;
        const int c = (p0 + pi) % C;
        DwPlane<KS>& P = prm_base[bi * ppc + pi];
        const int wz = (int)w_zp[per_channel ? c : 0];
        int wsum = 0, wabs = 0;
        for (int t = 0; t < KS * KS; ++t) {
          const int d = (int)w[(int64_t)c * KS * KS + t] - wz;
          wsum += d;
          wabs += abs(d);
        }
        const long long k0 = (long long)(B ? B[c] : 0) - (long long)x_zp * wsum;
        const float mul = __fmul_rn(x_scale, w_scale[per_channel ? c : 0]);
        // every sum of the plane is within amax of 0: below 2^22 it rides on
        // 1.5 * 2^23 as an exact float; and |q| <= 2^20 keeps the rounded
        // codes in the binade of unit spacing
        const long long amax = (k0 < 0 ? -k0 : k0) + (long long)(XS ? 128 : 255) * wabs;
        const bool fast =
            rcp_ok && amax < (1ll << 22) && fabsf(__fmul_rn(__fmul_rn((float)amax, mul), yrh)) <= 0x1p20f;
        P.k0 = (int)k0 + (fast ? 0x4B400000 : 0);
        P.mul = mul;
        P.fast = fast;
      }
    }
    dw_cp_commit();
  };

  const float lo_z = qlo - (float)y_zp, hi_z = qhi - (float)y_zp;
  const int ipp = nstrips * nblocks;

  int grp = blockIdx.x;
  if (grp < ngroups) stage(grp, 0);
  for (int k = 0; grp < ngroups; ++k, grp += gridDim.x) {
    const int bi = k & 1;
    const int nxt = grp + (int)gridDim.x;
    dw_cp_wait<0>();  // this group's copies, the only ones in flight
    // this group's planes and constants are in, and every thread is done
    // with the previous group, whose buffer the next group's copies take
    __syncthreads();
    if (nxt < ngroups) stage(nxt, bi ^ 1);
    const int p0 = grp * ppc, np = min(ppc, planes - p0);
    const uint32_t* buf = smw + bi * buf_words;
    const DwPlane<KS>* prm = prm_base + bi * ppc;
    for (int it = tid; it < np * ipp; it += nthr) {
      const int p = it / ipp, rem = it - p * ipp;
      const int blk = rem / nstrips, st = rem - blk * nstrips;
      const DwPlane<KS>& P = prm[p];
      constexpr int NP = KS == 3 ? 4 : 6;
      uint32_t wp[KS][NP];
#pragma unroll
      for (int kh = 0; kh < KS; ++kh)
#pragma unroll
        for (int t = 0; t < NP; ++t) wp[kh][t] = P.wp[kh][t];
      const int k0 = P.k0;
      const float mul = P.mul;
      const bool fast = P.fast != 0;
      const int oh0 = blk * R, ow0 = st * kStrip;
      const int s0 = kX0 - pl + ow0;  // first byte of the item's windows in a shared row
      const uint32_t shift = 0x3210u + (uint32_t)(s0 & 3) * 0x1111u;
      const uint32_t* rows = buf + (size_t)p * PW + oh0 * RW + (s0 >> 2);
      YT* yp = y + (int64_t)(p0 + p) * OH * OW + ow0;
      // whole 8-byte stores when the item's rows are complete and aligned
      const bool vec = ow0 + kStrip <= OW && (OW & 7) == 0 && (reinterpret_cast<uintptr_t>(yp) & 7) == 0;
      int acc[R][kStrip];
#pragma unroll
      for (int ir = 0; ir < R + KS - 1; ++ir) {
        // input row oh0 + ir of the shared plane (rows past the plane feed
        // only rows past OH, which are not stored)
        uint32_t wd[NWD];
        const bool rin = oh0 + ir < HP;
#pragma unroll
        for (int i = 0; i < NWD; ++i) wd[i] = rin ? rows[ir * RW + i] : fill;
        uint32_t a[NWD - 1];
#pragma unroll
        for (int i = 0; i < NWD - 1; ++i) a[i] = __byte_perm(wd[i], wd[i + 1], shift);  // bytes from s0 on
        // win[m]: the 4 bytes from output 2m's first tap; KS = 5 also reads win[m + 2]
        constexpr int NWIN = kStrip / 2 + (KS == 5 ? 2 : 0);
        uint32_t win[NWIN];
#pragma unroll
        for (int m = 0; m < NWIN; ++m) win[m] = (m & 1) ? __byte_perm(a[m >> 1], a[(m >> 1) + 1], 0x5432u) : a[m >> 1];
#pragma unroll
        for (int kh = 0; kh < KS; ++kh) {
          const int o = ir - kh;  // the item's output row this input row feeds through filter row kh
          if (o < 0 || o >= R) continue;
#pragma unroll
          for (int m = 0; m < kStrip / 2; ++m) {
            int ve = kh == 0 ? k0 : acc[o][2 * m];
            int vo = kh == 0 ? k0 : acc[o][2 * m + 1];
            ve = dp2a<false, XS>(wp[kh][0], win[m], ve);
            ve = dp2a<true, XS>(wp[kh][1], win[m], ve);
            vo = dp2a<false, XS>(wp[kh][2], win[m], vo);
            vo = dp2a<true, XS>(wp[kh][3], win[m], vo);
            if constexpr (KS == 5) {
              ve = dp2a<false, XS>(wp[kh][4], win[m + 2], ve);
              vo = dp2a<false, XS>(wp[kh][5], win[m + 2], vo);
            }
            acc[o][2 * m] = ve;
            acc[o][2 * m + 1] = vo;
          }
          if (kh == KS - 1 && oh0 + o < OH) {
            // output row oh0 + o is complete: requantize and store its 8 codes
            if (fast) {
              dw_requant_fast<YT>(acc[o], mul, yrh, yrl, mz, y_scale, lo_z, hi_z, y_zp,
                                  yp + (int64_t)(oh0 + o) * OW, vec, OW - ow0);
            } else {
              dw_requant_general<YT>(acc[o][0], acc[o][1], acc[o][2], acc[o][3], acc[o][4], acc[o][5], acc[o][6],
                                     acc[o][7], mul, y_scale, yr, lo_z, hi_z, y_zp, yp + (int64_t)(oh0 + o) * OW, vec,
                                     OW - ow0);
            }
          }
        }
      }
    }
  }
}

struct ConvShape {
  int64_t N, C, H, W, M, Cg, kH, kW, OH, OW;
  int64_t pt, pl, pb, pr, sh, sw, dh, dw, group;
};

int conv_shape(const int64_t* xs, const int64_t* ws, const int64_t* pads, const int64_t* strides,
               const int64_t* dil, int64_t group, ConvShape* s) {
  if (!xs || !ws) return fail(I8Q_ERR_INVALID_ARG, "qlinearconv: NULL shape");
  s->N = xs[0]; s->C = xs[1]; s->H = xs[2]; s->W = xs[3];
  s->M = ws[0]; s->Cg = ws[1]; s->kH = ws[2]; s->kW = ws[3];
  s->pt = pads ? pads[0] : 0; s->pl = pads ? pads[1] : 0;
  s->pb = pads ? pads[2] : 0; s->pr = pads ? pads[3] : 0;
  s->sh = strides ? strides[0] : 1; s->sw = strides ? strides[1] : 1;
  s->dh = dil ? dil[0] : 1; s->dw = dil ? dil[1] : 1;
  s->group = group;
  for (int i = 0; i < 4; ++i)
    if (xs[i] <= 0 || ws[i] <= 0) return fail(I8Q_ERR_INVALID_ARG, "qlinearconv: dimensions must be positive");
  if (s->pt < 0 || s->pl < 0 || s->pb < 0 || s->pr < 0) return fail(I8Q_ERR_INVALID_ARG, "qlinearconv: negative pad");
  if (s->sh < 1 || s->sw < 1 || s->dh < 1 || s->dw < 1)
    return fail(I8Q_ERR_INVALID_ARG, "qlinearconv: strides and dilations must be >= 1");
  if (group < 1 || s->C != s->Cg * group || s->M % group != 0)
    return fail(I8Q_ERR_INVALID_ARG, "qlinearconv: need x.shape[1] == w.shape[1] * group and M % group == 0");
  s->OH = (s->H + s->pt + s->pb - ((s->kH - 1) * s->dh + 1)) / s->sh + 1;
  s->OW = (s->W + s->pl + s->pr - ((s->kW - 1) * s->dw + 1)) / s->sw + 1;
  if (s->OH <= 0 || s->OW <= 0) return fail(I8Q_ERR_INVALID_ARG, "qlinearconv: empty output");
  // every |(x - xz)(w - wz)| <= 255*255; keep the int32 sum exact
  if (s->Cg * s->kH * s->kW > 33025) return fail(I8Q_ERR_UNSUPPORTED, "qlinearconv: C/group*kH*kW > 33025");
  if (s->M > 65535 || s->N > 65535) return fail(I8Q_ERR_UNSUPPORTED, "qlinearconv: M or N > 65535");
  if (s->OH * s->OW > (int64_t)1 << 31) return fail(I8Q_ERR_UNSUPPORTED, "qlinearconv: output plane too large");
  return I8Q_OK;
}

template <typename XT, typename WT, typename YT>
int run_direct(const ConvShape& s, const void* x, float x_scale, int x_zp, const void* w, const float* w_scale,
               const void* w_zp, int per_ch, float y_scale, int y_zp, const int32_t* B, void* y, cudaStream_t st) {
  const float dq_lo = std::is_same<YT, uint8_t>::value ? 0.0f : -128.0f;
  const float dq_hi = std::is_same<YT, uint8_t>::value ? 255.0f : 127.0f;
  const int64_t P = std::max(std::max(s.pt, s.pb), std::max(s.pl, s.pr));
  {
    // dp4a row kernel: depthwise 3x3 / 5x5, stride 1, dilation 1; planes
    // per CTA so that the items (rows x 8 outputs) of a CTA fill 224 threads
    const int64_t nstrips = (s.OW + kStrip - 1) / kStrip;
    const int64_t R = s.kH == 3 ? dw_rows<3>() : dw_rows<5>();
    const int64_t ipp = nstrips * ((s.OH + R - 1) / R);
    const size_t pbytes = nstrips <= (1 << 20)
                              ? (size_t)(s.OH + s.kH - 1) * dw_row_words((int)nstrips, (int)s.kW) * 4
                              : (size_t)-1 / 2;
    const size_t prm = s.kH == 3 ? sizeof(DwPlane<3>) : sizeof(DwPlane<5>);
    int64_t ppc = std::max<int64_t>(1, std::min<int64_t>(224 / std::max<int64_t>(ipp, 1), 8));
    while (ppc > 1 && 2 * ppc * (pbytes + prm) > 160 * 1024) --ppc;
    const size_t ssmem = 2 * (size_t)ppc * (pbytes + prm);
    if (s.group == s.C && s.M == s.C && s.Cg == 1 && s.sh == 1 && s.sw == 1 && s.dh == 1 && s.dw == 1 &&
        s.kH == s.kW && (s.kH == 3 || s.kH == 5) && s.pl <= kX0 && ssmem <= 160 * 1024 &&
        s.N * s.C < ((int64_t)1 << 31) && !getenv("I8Q_FORCE_CONV_HALO")) {
      auto kern = s.kH == 3 ? qlinearconv_depthwise_rows<XT, WT, YT, 3> : qlinearconv_depthwise_rows<XT, WT, YT, 5>;
      const int ar = smem_attr((const void*)kern, 160 * 1024);
      if (ar) return ar;
      const int threads = (int)std::min<int64_t>(224, round_up(ppc * ipp, 32));
      const int64_t planes = s.N * s.C, groups = ceil_div(planes, ppc);
      // persistent: as many CTAs as fit at once, at most one per group
      int per_sm = 0;
      I8Q_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, ssmem));
      const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(groups, (int64_t)std::max(per_sm, 1) * sm_count()));
      I8Q_PROF("qlinearconv_depthwise", st);
      kern<<<(unsigned)grid, threads, ssmem, st>>>(
          (const XT*)x, (const WT*)w, w_scale, (const WT*)w_zp, per_ch, B, (int)s.C, (int)s.H, (int)s.W, (int)s.OH,
          (int)s.OW, (int)s.pt, (int)s.pl, (int)planes, (int)ppc, x_scale, x_zp, y_scale, y_zp, dq_lo, dq_hi, (YT*)y);
      I8Q_LAUNCH_CHECK("qlinearconv_depthwise_rows");
      return I8Q_OK;
    }
  }
  if (s.group == s.C && s.M == s.C && s.Cg == 1 && s.sh == 1 && s.sw == 1 && s.dh == 1 && s.dw == 1 &&
      s.kH == s.kW && (s.kH == 3 || s.kH == 5) && (s.H + 2 * P) * (s.W + 2 * P) * 2 <= 160 * 1024) {
    const size_t hsmem = (size_t)(s.H + 2 * P) * (s.W + 2 * P) * 2;
    auto kern = s.kH == 3 ? qlinearconv_depthwise_halo<XT, WT, YT, 3> : qlinearconv_depthwise_halo<XT, WT, YT, 5>;
    if (hsmem > 48 * 1024)
      I8Q_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)hsmem));
    I8Q_PROF("qlinearconv_depthwise", st);
    kern<<<(unsigned)(s.N * s.C), 256, hsmem, st>>>((const XT*)x, (const WT*)w, w_scale, (const WT*)w_zp, per_ch, B,
                                                    (int)s.C, (int)s.H, (int)s.W, (int)s.OH, (int)s.OW, (int)s.pt,
                                                    (int)s.pl, (int)P, x_scale, x_zp, y_scale, y_zp, dq_lo, dq_hi,
                                                    (YT*)y);
    I8Q_LAUNCH_CHECK("qlinearconv_depthwise_halo");
    return I8Q_OK;
  }
  if (s.group == s.C && s.M == s.C && s.Cg == 1 && s.kH * s.kW <= 25 && s.H * s.W * 2 <= 160 * 1024) {
    auto kern = qlinearconv_depthwise_plane<XT, WT, YT>;
    const size_t psmem = (size_t)s.H * s.W * 2;
    if (psmem > 48 * 1024)
      I8Q_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)psmem));
    I8Q_PROF("qlinearconv_depthwise", st);
    kern<<<(unsigned)(s.N * s.C), 256, psmem, st>>>((const XT*)x, (const WT*)w, w_scale, (const WT*)w_zp, per_ch, B,
                                                    (int)s.C, (int)s.H, (int)s.W, (int)s.kH, (int)s.kW, (int)s.OH,
                                                    (int)s.OW, (int)s.pt, (int)s.pl, (int)s.sh, (int)s.sw, (int)s.dh,
                                                    (int)s.dw, x_scale, x_zp, y_scale, y_zp, dq_lo, dq_hi, (YT*)y);
    I8Q_LAUNCH_CHECK("qlinearconv_depthwise_plane");
    return I8Q_OK;
  }
  const int64_t taps = s.Cg * s.kH * s.kW;
  const size_t smem = (size_t)taps * sizeof(int);
  if (smem > 200 * 1024) return fail(I8Q_ERR_UNSUPPORTED, "qlinearconv: filter too large for shared memory");
  auto kern = qlinearconv_direct<XT, WT, YT>;
  if (smem > 48 * 1024) I8Q_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  const float qlo = std::is_same<YT, uint8_t>::value ? 0.0f : -128.0f;
  const float qhi = std::is_same<YT, uint8_t>::value ? 255.0f : 127.0f;
  dim3 grid((unsigned)ceil_div(s.OH * s.OW, 256), (unsigned)s.M, (unsigned)s.N);
  I8Q_PROF("qlinearconv_direct", st);
  kern<<<grid, 256, smem, st>>>((const XT*)x, (const WT*)w, w_scale, (const WT*)w_zp, per_ch, B, (int)s.C, (int)s.H,
                                (int)s.W, (int)s.M, (int)s.Cg, (int)(s.M / s.group), (int)s.kH, (int)s.kW, (int)s.OH,
                                (int)s.OW, (int)s.pt, (int)s.pl, (int)s.sh, (int)s.sw, (int)s.dh, (int)s.dw, x_scale,
                                x_zp, y_scale, y_zp, qlo, qhi, (YT*)y);
  I8Q_LAUNCH_CHECK("qlinearconv_direct");
  return I8Q_OK;
}

template <typename XT, typename WT>
int dispatch_y(int ytype, const ConvShape& s, const void* x, float xs, int xz, const void* w, const float* ws,
               const void* wz, int pc, float ys, int yz, const int32_t* B, void* y, cudaStream_t st) {
  if (ytype == I8Q_U8) return run_direct<XT, WT, uint8_t>(s, x, xs, xz, w, ws, wz, pc, ys, yz, B, y, st);
  return run_direct<XT, WT, int8_t>(s, x, xs, xz, w, ws, wz, pc, ys, yz, B, y, st);
}

}  // namespace
}  // namespace i8q

using namespace i8q;

extern "C" size_t i8q_qlinearconv_workspace_size(const int64_t* xshape, const int64_t* wshape, const int64_t* pads,
                                                 const int64_t* strides, const int64_t* dilations, int64_t group) {
  ConvShape s;
  if (conv_shape(xshape, wshape, pads, strides, dilations, group, &s) != I8Q_OK) return 0;
  return conv_tc_workspace(s.N, s.C, s.H, s.W, s.M, s.Cg, s.kH, s.kW, s.OH, s.OW, s.group, s.sh, s.sw, s.dh, s.dw);
}

extern "C" int i8q_qlinearconv(const void* x, int xtype, const int64_t* xshape, float x_scale, int x_zero_point,
                               const void* w, int wtype, const int64_t* wshape, const float* w_scale,
                               const void* w_zero_point, size_t n_w, float y_scale, int y_zero_point,
                               const int32_t* B, const int64_t* pads, const int64_t* strides,
                               const int64_t* dilations, int64_t group, void* y, int ytype, void* workspace,
                               size_t ws_bytes, void* stream) {
  ConvShape s;
  int rc = conv_shape(xshape, wshape, pads, strides, dilations, group, &s);
  if (rc) return rc;
  const size_t ws_need =
      conv_tc_workspace(s.N, s.C, s.H, s.W, s.M, s.Cg, s.kH, s.kW, s.OH, s.OW, s.group, s.sh, s.sw, s.dh, s.dw);
  if (ws_need) {
    if (!workspace || ws_bytes < ws_need)
      return fail(I8Q_ERR_INVALID_ARG, "qlinearconv: workspace missing or smaller than qlinearconv_workspace_size");
    if (reinterpret_cast<uintptr_t>(workspace) & 255)
      return fail(I8Q_ERR_INVALID_ARG, "qlinearconv: workspace must be 256-byte aligned");
  }
  auto is8 = [](int t) { return t == I8Q_U8 || t == I8Q_S8; };
  if (!is8(xtype) || !is8(wtype) || !is8(ytype)) return fail(I8Q_ERR_INVALID_ARG, "qlinearconv: types must be U8 or S8");
  if (!x || !w || !y || !w_scale || !w_zero_point) return fail(I8Q_ERR_INVALID_ARG, "qlinearconv: NULL tensor pointer");
  if (n_w != 1 && (int64_t)n_w != s.M)
    return fail(I8Q_ERR_INVALID_ARG, "qlinearconv: w_scale / w_zero_point must have 1 or M entries");
  const int xlo = xtype == I8Q_U8 ? 0 : -128, xhi = xtype == I8Q_U8 ? 255 : 127;
  const int ylo = ytype == I8Q_U8 ? 0 : -128, yhi = ytype == I8Q_U8 ? 255 : 127;
  if (x_zero_point < xlo || x_zero_point > xhi || y_zero_point < ylo || y_zero_point > yhi)
    return fail(I8Q_ERR_INVALID_ARG, "qlinearconv: zero point outside its type's range");
  if (!(x_scale > 0.0f) || !(y_scale > 0.0f)) return fail(I8Q_ERR_INVALID_ARG, "qlinearconv: scales must be > 0");
  const int pc = n_w != 1;
  cudaStream_t st = as_stream(stream);
  if (ws_need)
    return launch_conv_tc(x, xtype, s.N, s.C, s.H, s.W, x_scale, x_zero_point, w, wtype, s.M, s.kH, s.kW, w_scale,
                          w_zero_point, pc, y_scale, y_zero_point, ytype, B, s.pt, s.pl, s.OH, s.OW, y, workspace, st);
  if (xtype == I8Q_U8 && wtype == I8Q_U8)
    return dispatch_y<uint8_t, uint8_t>(ytype, s, x, x_scale, x_zero_point, w, w_scale, w_zero_point, pc, y_scale,
                                        y_zero_point, B, y, st);
  if (xtype == I8Q_U8)
    return dispatch_y<uint8_t, int8_t>(ytype, s, x, x_scale, x_zero_point, w, w_scale, w_zero_point, pc, y_scale,
                                       y_zero_point, B, y, st);
  if (wtype == I8Q_U8)
    return dispatch_y<int8_t, uint8_t>(ytype, s, x, x_scale, x_zero_point, w, w_scale, w_zero_point, pc, y_scale,
                                       y_zero_point, B, y, st);
  return dispatch_y<int8_t, int8_t>(ytype, s, x, x_scale, x_zero_point, w, w_scale, w_zero_point, pc, y_scale,
                                    y_zero_point, B, y, st);
}
