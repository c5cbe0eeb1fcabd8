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

// Depthwise KS x KS, stride 1, dilation 1: one CTA of 128 threads per
// (image, channel) plane, integer tap sums on the byte dot product (dp4a)
// over the raw codes.  The plane sits in shared memory as its codes, each
// row at byte kX0 of a row of RW words, the halo filled with the x zero
// point's code (so that a padded tap contributes x - x_zp = 0).  For the KS
// taps of a filter row, with w packed four codes a word (zeros beyond KS),
//   sum (x - x_zp)(w - w_zp) = sum x w - w_zp sum x - x_zp sum w + KS x_zp w_zp
// per row, all exact in int32: sum x w and sum x come from dp4a of a 4-byte
// window of the row with the packed weights and with ones.  Each thread
// computes strips of 8 consecutive outputs of a row: it loads the strip's
// words of each input row, shifts them once to the strip's first byte and
// takes the eight windows with byte permutes whose selectors are constants.
// The codes are requantized (quot_code_bits) and written as one 8-byte store.
constexpr int kStrip = 8, kX0 = 8;  // outputs per strip; byte of x column 0 in a shared row

template <bool AS, bool BS>
__device__ __forceinline__ int dp4a(uint32_t a, uint32_t b, int c) {
  int d;
  if (AS && BS) asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  else if (AS) asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  else if (BS) asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  else asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__host__ __device__ constexpr int dw_row_words(int nstrips, int ks) {
  return (kX0 + nstrips * kStrip + 4 * ((ks + 3) / 4) + 8 + 3) / 4;
}

template <typename XT, typename WT, typename YT, int KS>
__global__ void __launch_bounds__(128)
qlinearconv_depthwise_strip(const XT* __restrict__ x, const WT* __restrict__ w, const float* __restrict__ w_scale,
                            const WT* __restrict__ w_zp, int per_channel, const int32_t* __restrict__ B, int C, int H,
                            int W, int OH, int OW, int pt, int pl, float x_scale, int x_zp, float y_scale, int y_zp,
                            float qlo, float qhi, YT* __restrict__ y) {
  constexpr bool XS = std::is_signed<XT>::value, WS = std::is_signed<WT>::value;
  constexpr int TW = (KS + 3) / 4;  // words of a filter row
  constexpr int NWD = 3 + TW;       // words loaded per input row of a strip
  extern __shared__ __align__(16) uint32_t plw[];
  const int c = blockIdx.x % C, n = blockIdx.x / C;
  const int nstrips = (OW + kStrip - 1) / kStrip;
  const int HP = OH + KS - 1, RW = dw_row_words(nstrips, KS);
  const uint32_t fill = (uint32_t)(uint8_t)x_zp * 0x01010101u;
  for (int i = threadIdx.x; i < HP * RW; i += blockDim.x) plw[i] = fill;
  __syncthreads();
  const XT* xp = x + ((int64_t)n * C + c) * H * W;
  uint8_t* plb = reinterpret_cast<uint8_t*>(plw);
  const int rows = min(H, HP - pt);  // input rows that reach an output
  if ((W & 3) == 0 && (reinterpret_cast<uintptr_t>(xp) & 3) == 0) {
    // the plane is contiguous: 32-bit words, consecutive threads on
    // consecutive words, each landing at a word of its shared row
    const int wpr = W / 4;
    const int dr = (int)blockDim.x / wpr, dj = (int)blockDim.x - dr * wpr;  // the stride as (rows, words)
    int r = (int)threadIdx.x / wpr, j = (int)threadIdx.x - r * wpr;
    for (int i = threadIdx.x; i < rows * wpr; i += blockDim.x) {
      plw[(r + pt) * RW + kX0 / 4 + j] = __ldg(reinterpret_cast<const uint32_t*>(xp) + i);
      r += dr;
      j += dj;
      if (j >= wpr) {
        j -= wpr;
        ++r;
      }
    }
  } else {
    for (int i = threadIdx.x; i < rows * W; i += blockDim.x) {
      const int r = i / W, col = i - r * W;
      plb[(r + pt) * RW * 4 + kX0 + col] = (uint8_t)xp[i];
    }
  }
  // the filter rows packed four codes a word, their code sum, the constant terms
  uint32_t wr[KS][TW];
  int wsum = 0;
#pragma unroll
  for (int kh = 0; kh < KS; ++kh)
#pragma unroll
    for (int t = 0; t < TW; ++t) {
      uint32_t v = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (4 * t + e < KS) {
          const WT q = w[(int64_t)c * KS * KS + kh * KS + 4 * t + e];
          wsum += (int)q;
          v |= (uint32_t)(uint8_t)q << (8 * e);
        }
      wr[kh][t] = v;
    }
  // ones over the taps a filter-row word holds (all four but in the last word)
  constexpr uint32_t ones0 = 0x01010101u >> (8 * (4 - (KS - 4 * (TW - 1))));
  const int wz = (int)w_zp[per_channel ? c : 0];
  const int32_t k0 = (B ? B[c] : 0) - x_zp * wsum + KS * KS * x_zp * wz;
  const float mul = __fmul_rn(x_scale, w_scale[per_channel ? c : 0]);
  const float yr = quot_rcp(y_scale);
  const float lo_z = qlo - (float)y_zp, hi_z = qhi - (float)y_zp;
  __syncthreads();
  YT* yp = y + ((int64_t)n * C + c) * OH * OW;
  const bool vec_rows = (OW % kStrip) == 0 && (reinterpret_cast<uintptr_t>(y) & 7) == 0;
  const int doh = (int)blockDim.x / nstrips, dst = (int)blockDim.x - doh * nstrips;  // the stride as (rows, strips)
  int oh = (int)threadIdx.x / nstrips, st = (int)threadIdx.x - oh * nstrips;
  for (int sidx = threadIdx.x; sidx < OH * nstrips; sidx += blockDim.x) {
    const int ow0 = st * kStrip;
    const int s0 = kX0 - pl + ow0;  // first byte of the strip's windows in a shared row
    const uint32_t shift = 0x3210u + (uint32_t)(s0 & 3) * 0x1111u;
    int sxw[kStrip], sx[kStrip];
#pragma unroll
    for (int e = 0; e < kStrip; ++e) sxw[e] = sx[e] = 0;
#pragma unroll
    for (int kh = 0; kh < KS; ++kh) {
      const uint32_t* row = plw + (oh + kh) * RW + (s0 >> 2);
      uint32_t wd[NWD], a[NWD - 1];
#pragma unroll
      for (int i = 0; i < NWD; ++i) wd[i] = row[i];
#pragma unroll
      for (int i = 0; i < NWD - 1; ++i) a[i] = __byte_perm(wd[i], wd[i + 1], shift);  // bytes from s0 on
#pragma unroll
      for (int e = 0; e < kStrip; ++e)
#pragma unroll
        for (int t = 0; t < TW; ++t) {
          const int k = (e >> 2) + t;
          const uint32_t win = (e & 3) ? __byte_perm(a[k], a[k + 1], 0x3210u + (uint32_t)(e & 3) * 0x1111u) : a[k];
          sxw[e] = dp4a<XS, WS>(win, wr[kh][t], sxw[e]);
          sx[e] = dp4a<XS, false>(win, t == TW - 1 ? ones0 : 0x01010101u, sx[e]);
        }
    }
    uint32_t code[kStrip];
#pragma unroll
    for (int e = 0; e < kStrip; ++e) {
      const int32_t acc = sxw[e] - wz * sx[e] + k0;
      code[e] = quot_code_bits(__fmul_rn(__int2float_rn(acc), mul), y_scale, yr, lo_z, hi_z, y_zp);
    }
    YT* out = yp + oh * OW + ow0;
    if (vec_rows && ((reinterpret_cast<uintptr_t>(out) & 7) == 0)) {
      *reinterpret_cast<uint2*>(out) =
          make_uint2(pack_low_bytes(code[0], code[1], code[2], code[3]), pack_low_bytes(code[4], code[5], code[6], code[7]));
    } else {
#pragma unroll
      for (int e = 0; e < kStrip; ++e)
        if (ow0 + e < OW) out[e] = (YT)code[e];
    }
    oh += doh;
    st += dst;
    if (st >= nstrips) {
      st -= nstrips;
      ++oh;
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
    // strip kernel: depthwise 3x3 / 5x5, stride 1, dilation 1
    const int64_t nstrips = (s.OW + kStrip - 1) / kStrip;
    const size_t ssmem = (size_t)(s.OH + s.kH - 1) * dw_row_words((int)std::min<int64_t>(nstrips, 1 << 20), (int)s.kW) * 4;
    if (s.group == s.C && s.M == s.C && s.Cg == 1 && s.sh == 1 && s.sw == 1 && s.dh == 1 && s.dw == 1 &&
        s.kH == s.kW && (s.kH == 3 || s.kH == 5) && s.pl <= kX0 && ssmem <= 160 * 1024 &&
        !getenv("I8Q_FORCE_CONV_HALO")) {
      auto kern = s.kH == 3 ? qlinearconv_depthwise_strip<XT, WT, YT, 3> : qlinearconv_depthwise_strip<XT, WT, YT, 5>;
      if (ssmem > 48 * 1024)
        I8Q_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ssmem));
      I8Q_PROF("qlinearconv_depthwise", st);
      kern<<<(unsigned)(s.N * s.C), 128, ssmem, st>>>((const XT*)x, (const WT*)w, w_scale, (const WT*)w_zp, per_ch, B,
                                                      (int)s.C, (int)s.H, (int)s.W, (int)s.OH, (int)s.OW, (int)s.pt,
                                                      (int)s.pl, x_scale, x_zp, y_scale, y_zp, dq_lo, dq_hi, (YT*)y);
      I8Q_LAUNCH_CHECK("qlinearconv_depthwise_strip");
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
