// common.cuh -- shared helpers of libi8q (CUDA side only).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>
#include <string>
#include <type_traits>

#include "../../include/i8q.h"

namespace i8q {

// ---- error reporting (thread-local text, see i8q_last_error) -------------
void set_error(const std::string& msg);
int fail(int code, const std::string& msg);
int cuda_fail(cudaError_t e, const char* what);

#define I8Q_CUDA_TRY(expr)                                   \
  do {                                                       \
    cudaError_t e_ = (expr);                                 \
    if (e_ != cudaSuccess) return ::i8q::cuda_fail(e_, #expr); \
  } while (0)

#define I8Q_LAUNCH_CHECK(what)                               \
  do {                                                       \
    cudaError_t e_ = cudaGetLastError();                     \
    if (e_ != cudaSuccess) return ::i8q::cuda_fail(e_, what); \
  } while (0)

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// Streaming-multiprocessor count of the current device (cached per device).
int sm_count();

// Run init once per (key, current device), thread-safely, and return its
// status; later calls on that device return the first status.  Kernel
// attributes and occupancy figures belong to a device, so each device sets
// them up the first time a launch meets it.
int once_per_device(const void* key, int (*init)(void*), void* arg);

// cudaFuncSetAttribute(func, MaxDynamicSharedMemorySize, bytes) once per
// device.
int smem_attr(const void* func, int bytes);

// Device-side status word for bounded waits (see i8q_sync_status).
uint32_t* device_status_word();

// Kernel timing (i8q_profile_*): while enabled, a ProfScope brackets the
// launches made in its lifetime with CUDA events on the launch stream.
bool profiling_enabled();
void profile_record(const char* name, cudaStream_t s, bool begin);
struct ProfScope {
  const char* name;
  cudaStream_t s;
  bool on;
  ProfScope(const char* n, cudaStream_t st) : name(n), s(st), on(profiling_enabled()) {
    if (on) profile_record(name, s, true);
  }
  ~ProfScope() {
    if (on) profile_record(name, s, false);
  }
};
#define I8Q_PROF(name, stream) ::i8q::ProfScope i8q_prof_scope_(name, stream)

// ---- exact fp32 helpers (no contraction into FMA) ------------------------
// rint(v) saturated to [lo, hi] then cast; lo/hi already include the zero
// point shift so the comparison happens on exactly representable values.
__device__ __forceinline__ int sat_rint(float v, float lo, float hi) {
  float r = rintf(v);
  r = fminf(fmaxf(r, lo), hi);
  return __float2int_rz(r);
}

// saturate(rint(q) + zp) as the low byte of the result, for lo_z = lo - zp
// and hi_z = hi - zp (small integers, exact in fp32).  Clamping to integer
// bounds commutes with rounding, so q is clamped first; adding 1.5 * 2^23
// then rounds it to the nearest integer, ties to even (the constant is an
// even integer, so the parity of the rounded part is unchanged), and the
// integer sits in the low mantissa bits: bits(q' + 1.5*2^23) = 0x4B400000 +
// rint(q') for |q'| < 2^22.  Adding zp to that pattern leaves the code in
// the low byte (two's complement for int8).
__device__ __forceinline__ uint32_t rint_code_bits(float q, float lo_z, float hi_z, int zp) {
  const float c = fminf(fmaxf(q, lo_z), hi_z);
  const float r = __fadd_rn(c, 12582912.0f);
  return (uint32_t)(__float_as_int(r) + zp);
}

// fl(1 / s) when s and its reciprocal are normal numbers (quot_code_bits
// may then use it), else NaN (quot_code_bits then always divides).
__host__ __device__ inline float quot_rcp(float s) {
  const float a = s < 0.0f ? -s : s;
  return (a >= 0x1p-125f && a <= 0x1p125f) ? 1.0f / s : __builtin_nanf("");
}

// rint_code_bits of the IEEE quotient fl(v / s), usually without forming
// it: with r = quot_rcp(s), q = fl(v * r) is within (2^-23 + 2^-48) |v / s|
// of v / s (r carries one rounding, the product another) and fl(v / s)
// within 2^-24 |v / s|, so the two differ by less than 2^-22 |q|.  Where q
// is farther than 2^-21 |q| from every half-integer, both round to the same
// integer, and the saturation bounds are integers, so the codes agree;
// beyond 1024 in magnitude both saturate alike (the bounds are within
// +-255).  Any other q (close to a half-integer, NaN, or r NaN) is replaced
// by the quotient itself.
__device__ __forceinline__ uint32_t quot_code_bits(float v, float s, float r, float lo_z, float hi_z, int zp) {
  float q = __fmul_rn(v, r);
  const float a = fabsf(q);
  if (!(a > 1024.0f)) {
    const float dist = fabsf(__fsub_rn(__fsub_rn(q, floorf(q)), 0.5f));
    if (!(dist > a * 0x1p-21f)) q = __fdiv_rn(v, s);
  }
  return rint_code_bits(q, lo_z, hi_z, zp);
}

// Row quantization of A (uint8, per row, range widened to contain 0) from
// the row's mn = min(0, min A) and mx = max(0, max A):
//   scale = (mx - mn) / 255, zero = sat_u8(rint(-mn / scale)),
// and an all-zero row (scale 0) takes scale 1, zero 0.
__device__ __forceinline__ void row_scale_zero(float mn, float mx, float& s, int& z) {
  s = __fdiv_rn(__fsub_rn(mx, mn), 255.0f);
  z = 0;
  if (s == 0.0f) {
    s = 1.0f;
  } else {
    z = sat_rint(__fdiv_rn(-mn, s), 0.0f, 255.0f);
  }
}

// uA = sat_u8(rint(v / scale) + zero) as the low byte of the result, for
// lo_z = -zero and hi_z = 255 - zero.
__device__ __forceinline__ uint32_t row_code(float v, float s, float lo_z, float hi_z, int z) {
  return rint_code_bits(__fdiv_rn(v, s), lo_z, hi_z, z) & 0xffu;
}

// Pack the low bytes of four words into one word (byte 0 from a).
__device__ __forceinline__ uint32_t pack_low_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(c, d, 0x0040), 0x5410);
}

// GELU = x * Phi(x) = 0.5 * x * (1 + erf(x / sqrt 2)), evaluated as
// (0.5 * x) * erfc(-(x / sqrt 2)) so nothing cancels for negative x.
__device__ __forceinline__ float gelu_erf(float x) {
  float t = __fmul_rn(x, 0.70710678118654752440f);
  float e = erfcf(-t);
  float h = __fmul_rn(0.5f, x);
  return __fmul_rn(h, e);
}

// GELU for outputs stored as bf16, where a relative error far below half a
// bf16 ulp (2^-9) is all the rounding can see.  erfc takes the form of
// Numerical Recipes' erfcc (Press, Teukolsky, Vetterling, Flannery, section
// 6.2): erfc(z) = t * exp(-z^2 + P(t)), t = 1 / (1 + z / 2), z >= 0, here
// with P in base 2 and of degree 5: a minimax fit, made for this library, of
// log2(erfc(z) e^(z^2) / t) over t in [0.147, 1] (z up to 11.6, beyond which
// every GELU(-x) is below the smallest bf16), maximum error 1.1e-5 (a
// relative 7.8e-6 in erfc).  With z = |x| / sqrt 2,
//   GELU(x) = x Phi(x) = max(x, 0) - |x| erfc(z) / 2,
// for either sign of x.  2^(P - z^2 log2 e) is formed as 2^64 * 2^(...) so
// that ex2 stays in the normal range down to z = 11.6; the 2^-64 (and the
// -1/2) go into t, where an underflow costs at most 2^-150 * |x|.  Measured
// against erfc in double precision over the fp32 line (with the approximate
// reciprocal and exponential off by up to 2^-23 and 2^-22), the result is
// within a relative 1.6e-5 of GELU, or 1.5e-42 where GELU is below 1e-37.
namespace gelu_fit {
constexpr float kD = 0.35355339059327376f;    // 1 + z / 2 = 1 + kD |x|
constexpr float kX2 = -0.72134752044448170f;  // -z^2 log2 e = kX2 x^2
constexpr float kC5 = 0.32952117f, kC4 = -1.02156514f, kC3 = 0.68284217f, kC2 = 0.36794539f,
                kC1 = 1.46848227f;
constexpr float kC0 = 62.17278356f;           // -1.82721644 + 64
constexpr float kT = -2.710505431213761e-20f; // -2^-65
}  // namespace gelu_fit

// Paired fp32 multiply and fused multiply-add, round to nearest, lane by
// lane as __fmul_rn / fmaf.  The compiler may fuse a paired multiply with a
// following paired add (not with an fma), so there is no paired add here.
__device__ __forceinline__ float2 mul2_rn(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "mul.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

__device__ __forceinline__ float2 fma2_rn(float2 a, float2 b, float2 c) {
  float2 r;
  asm("{\n\t.reg .b64 a, b, c, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "mov.b64 c, {%6, %7};\n\tfma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}

__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ float gelu_bf16out(float x) {
  using namespace gelu_fit;
  const float ax = fabsf(x);
  const float t = rcp_approx(fmaf(ax, kD, 1.0f));
  float p = fmaf(kC5, t, kC4);
  p = fmaf(p, t, kC3);
  p = fmaf(p, t, kC2);
  p = fmaf(p, t, kC1);
  p = fmaf(p, t, kC0);
  const float a = fmaf(__fmul_rn(x, kX2), x, p);
  const float te = __fmul_rn(__fmul_rn(t, kT), ex2_approx(a));
  return fmaf(ax, te, fmaxf(x, 0.0f));
}

// The same on two values with the paired fp32 instructions: each lane
// rounds exactly as the scalar form does (every product here is an operand
// of a fused multiply-add or of another product, never of an add).
__device__ __forceinline__ float2 gelu_bf16out2(float2 x) {
  using namespace gelu_fit;
  const float2 ax = make_float2(fabsf(x.x), fabsf(x.y));
  const float2 d = fma2_rn(ax, make_float2(kD, kD), make_float2(1.0f, 1.0f));
  const float2 t = make_float2(rcp_approx(d.x), rcp_approx(d.y));
  float2 p = fma2_rn(make_float2(kC5, kC5), t, make_float2(kC4, kC4));
  p = fma2_rn(p, t, make_float2(kC3, kC3));
  p = fma2_rn(p, t, make_float2(kC2, kC2));
  p = fma2_rn(p, t, make_float2(kC1, kC1));
  p = fma2_rn(p, t, make_float2(kC0, kC0));
  const float2 a = fma2_rn(mul2_rn(x, make_float2(kX2, kX2)), x, p);
  const float2 e = make_float2(ex2_approx(a.x), ex2_approx(a.y));
  const float2 te = mul2_rn(mul2_rn(t, make_float2(kT, kT)), e);
  return fma2_rn(ax, te, make_float2(fmaxf(x.x, 0.0f), fmaxf(x.y, 0.0f)));
}

// ---- fp32 elementary functions with a fixed operation sequence ----------
// exp, expm1, log1p, sigmoid, tanh and softplus as used by the LSTM gates
// and QLinearSigmoid.  Library versions of these differ in the last bit
// between platforms, and one bit of an LSTM hidden state can move a uint8
// code of the next step's dynamic quantization.  Each is therefore one fixed
// sequence of IEEE fp32 operations (every add, multiply, divide and fused
// multiply-add rounds once to nearest even; scaling by a power of two is
// exact in the normal range), so any IEEE implementation of the same
// sequence gives the same bits.
//  exp   Cody and Waite's argument reduction (Software Manual for the
//        Elementary Functions, 1980): n = rint(x / ln2), r = (x - n LN2_HI)
//        - n LN2_LO with LN2_HI = fl(ln 2), LN2_LO = fl(ln 2 - LN2_HI);
//        e^r = sum_{k<=7} r^k / k! in Horner form (truncation below 2^-27
//        for |r| <= ln2 / 2); times 2^n as two exact power-of-two factors,
//        so that a subnormal result rounds once.  Within 1 ulp.
//  expm1 the same reduction, e^r - 1 = r (1 + r/2! + ... + r^7/8!), and
//        e^x - 1 = 2^n (e^r - 1) + (2^n - 1); e^x above 20, -1 below -20.
//  log1p on [0, 1]: 1 + u = 2^k (1 + v), k in {0, 1}, v in [sqrt(1/2) - 1,
//        sqrt(2) - 1]; log(1 + v) = 2 atanh(s), s = v / (2 + v), by the
//        series 2 s (1 + s^2/3 + s^4/5 + s^6/7 + s^8/9).
//  sigmoid(x) = 1 / (1 + e^-x).  tanh(a) for a = |x|: with e = expm1(2a),
//        e / (e + 2) below 0.625 and 1 - 2 / (e + 2) up to 9.5, 1 above
//        (where tanh rounds to 1); the sign of x copied on.
//  softplus(x) = x + log1p(e^-x) for x > 0, log1p(e^x) otherwise.
// The constants are the fp32 roundings of the numbers named beside them.
namespace ef {
constexpr float kL2E = 0x1.715476p+0f;      // 1 / ln 2
constexpr float kLn2Hi = 0x1.62e430p-1f;    // ln 2
constexpr float kLn2Lo = -0x1.05c610p-29f;  // ln 2 - kLn2Hi

// 2^k for -126 <= k <= 127, exactly.
__device__ __forceinline__ float pow2i(int k) { return __int_as_float((k + 127) << 23); }

__device__ __forceinline__ float exp32(float x) {
  x = fminf(fmaxf(x, -104.0f), 89.0f);  // e^89 overflows to inf; e^-104 rounds to 0
  const float nf = rintf(__fmul_rn(x, kL2E));
  const int n = (int)nf;
  float r = __fmaf_rn(-nf, kLn2Hi, x);
  r = __fmaf_rn(-nf, kLn2Lo, r);
  float p = 0x1.a01a02p-13f;            // 1/7!
  p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);  // 1/6!
  p = __fmaf_rn(p, r, 0x1.111112p-7f);   // 1/5!
  p = __fmaf_rn(p, r, 0x1.555556p-5f);   // 1/4!
  p = __fmaf_rn(p, r, 0x1.555556p-3f);   // 1/3!
  p = __fmaf_rn(p, r, 0.5f);             // 1/2!
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  const int n1 = n / 2, n2 = n - n1;     // both within [-75, 65]
  return __fmul_rn(__fmul_rn(p, pow2i(n1)), pow2i(n2));
}

__device__ __forceinline__ float expm1_32(float x) {
  if (x > 20.0f) return exp32(x);
  if (x < -20.0f) return -1.0f;
  const float nf = rintf(__fmul_rn(x, kL2E));
  const int n = (int)nf;                 // |n| <= 29
  float r = __fmaf_rn(-nf, kLn2Hi, x);
  r = __fmaf_rn(-nf, kLn2Lo, r);
  float q = 0x1.a01a02p-16f;             // 1/8!
  q = __fmaf_rn(q, r, 0x1.a01a02p-13f);  // 1/7!
  q = __fmaf_rn(q, r, 0x1.6c16c2p-10f);  // 1/6!
  q = __fmaf_rn(q, r, 0x1.111112p-7f);   // 1/5!
  q = __fmaf_rn(q, r, 0x1.555556p-5f);   // 1/4!
  q = __fmaf_rn(q, r, 0x1.555556p-3f);   // 1/3!
  q = __fmaf_rn(q, r, 0.5f);             // 1/2!
  q = __fmaf_rn(q, r, 1.0f);
  q = __fmul_rn(q, r);                   // e^r - 1
  if (n == 0) return q;
  const float t = pow2i(n);
  return __fmaf_rn(t, q, __fsub_rn(t, 1.0f));
}

// log(1 + u), 0 <= u <= 1.
__device__ __forceinline__ float log1p01(float u) {
  float v = u, k = 0.0f;
  if (u > 0x1.a8279ap-2f) {  // sqrt(2) - 1
    v = __fmul_rn(__fsub_rn(u, 1.0f), 0.5f);  // exact: 1 + u = 2 (1 + v)
    k = 1.0f;
  }
  const float s = __fdiv_rn(v, __fadd_rn(2.0f, v));
  const float z = __fmul_rn(s, s);
  float w = 0x1.c71c72p-4f;              // 1/9
  w = __fmaf_rn(w, z, 0x1.24924ap-3f);   // 1/7
  w = __fmaf_rn(w, z, 0x1.99999ap-3f);   // 1/5
  w = __fmaf_rn(w, z, 0x1.555556p-2f);   // 1/3
  w = __fmaf_rn(w, z, 1.0f);
  return __fmaf_rn(k, kLn2Hi, __fmul_rn(__fadd_rn(s, s), w));
}

__device__ __forceinline__ float sigmoid32(float x) { return __fdiv_rn(1.0f, __fadd_rn(1.0f, exp32(-x))); }

// tanh(a) = e / (e + 2) = 1 - 2 / (e + 2), e = e^(2a) - 1: the first form
// below |a| = 0.625, the second up to 9.5, 1 beyond (and for NaN).  One
// expm1 and one division for every lane, so a warp does not run two forms.
__device__ __forceinline__ float tanh32(float x) {
  const float a = fabsf(x);
  const float ac = fminf(a, 9.5f);
  const float e = expm1_32(__fadd_rn(ac, ac));
  const bool small = a < 0.625f;
  const float q = __fdiv_rn(small ? e : 2.0f, __fadd_rn(e, 2.0f));
  const float t = a <= 9.5f ? (small ? q : __fsub_rn(1.0f, q)) : 1.0f;
  return copysignf(t, x);
}

// Two lanes at once: the same operations as exp32, expm1_32 (for |x| <=
// 20), sigmoid32 and tanh32 on x.x and x.y, with the multiplies and fused
// multiply-adds paired (each rounds per lane as its scalar form); sums
// of two terms are written as fused multiply-adds by 1, which round once as
// the scalar additions do, and the divisions stay scalar.
__device__ __forceinline__ float2 exp32x2(float2 x) {
  x = make_float2(fminf(fmaxf(x.x, -104.0f), 89.0f), fminf(fmaxf(x.y, -104.0f), 89.0f));
  const float2 t = mul2_rn(x, make_float2(kL2E, kL2E));
  const float2 nf = make_float2(rintf(t.x), rintf(t.y));
  const int nx = (int)nf.x, ny = (int)nf.y;
  const float2 mn = make_float2(-nf.x, -nf.y);
  float2 r = fma2_rn(mn, make_float2(kLn2Hi, kLn2Hi), x);
  r = fma2_rn(mn, make_float2(kLn2Lo, kLn2Lo), r);
  float2 p = fma2_rn(make_float2(0x1.a01a02p-13f, 0x1.a01a02p-13f), r, make_float2(0x1.6c16c2p-10f, 0x1.6c16c2p-10f));
  p = fma2_rn(p, r, make_float2(0x1.111112p-7f, 0x1.111112p-7f));
  p = fma2_rn(p, r, make_float2(0x1.555556p-5f, 0x1.555556p-5f));
  p = fma2_rn(p, r, make_float2(0x1.555556p-3f, 0x1.555556p-3f));
  p = fma2_rn(p, r, make_float2(0.5f, 0.5f));
  p = fma2_rn(p, r, make_float2(1.0f, 1.0f));
  p = fma2_rn(p, r, make_float2(1.0f, 1.0f));
  const int n1x = nx / 2, n2x = nx - n1x, n1y = ny / 2, n2y = ny - n1y;
  return mul2_rn(mul2_rn(p, make_float2(pow2i(n1x), pow2i(n1y))), make_float2(pow2i(n2x), pow2i(n2y)));
}

__device__ __forceinline__ float2 expm1_32x2(float2 x) {  // |x.x|, |x.y| <= 20
  const float2 t = mul2_rn(x, make_float2(kL2E, kL2E));
  const float2 nf = make_float2(rintf(t.x), rintf(t.y));
  const int nx = (int)nf.x, ny = (int)nf.y;
  const float2 mn = make_float2(-nf.x, -nf.y);
  float2 r = fma2_rn(mn, make_float2(kLn2Hi, kLn2Hi), x);
  r = fma2_rn(mn, make_float2(kLn2Lo, kLn2Lo), r);
  float2 q = fma2_rn(make_float2(0x1.a01a02p-16f, 0x1.a01a02p-16f), r, make_float2(0x1.a01a02p-13f, 0x1.a01a02p-13f));
  q = fma2_rn(q, r, make_float2(0x1.6c16c2p-10f, 0x1.6c16c2p-10f));
  q = fma2_rn(q, r, make_float2(0x1.111112p-7f, 0x1.111112p-7f));
  q = fma2_rn(q, r, make_float2(0x1.555556p-5f, 0x1.555556p-5f));
  q = fma2_rn(q, r, make_float2(0x1.555556p-3f, 0x1.555556p-3f));
  q = fma2_rn(q, r, make_float2(0.5f, 0.5f));
  q = fma2_rn(q, r, make_float2(1.0f, 1.0f));
  q = mul2_rn(q, r);
  const float2 s = make_float2(pow2i(nx), pow2i(ny));
  const float2 v = fma2_rn(s, q, make_float2(__fsub_rn(s.x, 1.0f), __fsub_rn(s.y, 1.0f)));
  return make_float2(nx == 0 ? q.x : v.x, ny == 0 ? q.y : v.y);
}

__device__ __forceinline__ float2 sigmoid32x2(float2 x) {
  const float2 d = fma2_rn(exp32x2(make_float2(-x.x, -x.y)), make_float2(1.0f, 1.0f), make_float2(1.0f, 1.0f));
  return make_float2(__fdiv_rn(1.0f, d.x), __fdiv_rn(1.0f, d.y));
}

__device__ __forceinline__ float2 tanh32x2(float2 x) {
  const float2 a = make_float2(fabsf(x.x), fabsf(x.y));
  const float2 ac = make_float2(fminf(a.x, 9.5f), fminf(a.y, 9.5f));
  const float2 e = expm1_32x2(mul2_rn(ac, make_float2(2.0f, 2.0f)));  // ac + ac, exactly
  const float2 d = fma2_rn(e, make_float2(1.0f, 1.0f), make_float2(2.0f, 2.0f));
  const bool sx = a.x < 0.625f, sy = a.y < 0.625f;
  const float qx = __fdiv_rn(sx ? e.x : 2.0f, d.x), qy = __fdiv_rn(sy ? e.y : 2.0f, d.y);
  const float tx = a.x <= 9.5f ? (sx ? qx : __fsub_rn(1.0f, qx)) : 1.0f;
  const float ty = a.y <= 9.5f ? (sy ? qy : __fsub_rn(1.0f, qy)) : 1.0f;
  return make_float2(copysignf(tx, x.x), copysignf(ty, x.y));
}

__device__ __forceinline__ float softplus32(float x) {
  return x > 0.0f ? __fadd_rn(x, log1p01(exp32(-x))) : log1p01(exp32(x));
}

// The LSTM activation functions (I8Q_LSTM_ACT_*, the ONNX LSTM list) with
// their alpha / beta, each its operator's formula, one rounding per step.
__device__ __forceinline__ float lstm_act(int kind, float alpha, float beta, float x) {
  switch (kind) {
    case I8Q_LSTM_ACT_RELU: return x > 0.0f ? x : 0.0f;
    case I8Q_LSTM_ACT_TANH: return tanh32(x);
    case I8Q_LSTM_ACT_SIGMOID: return sigmoid32(x);
    case I8Q_LSTM_ACT_AFFINE: return __fadd_rn(__fmul_rn(alpha, x), beta);
    case I8Q_LSTM_ACT_LEAKY_RELU: return x >= 0.0f ? x : __fmul_rn(alpha, x);
    case I8Q_LSTM_ACT_THRESHOLDED_RELU: return x > alpha ? x : 0.0f;
    case I8Q_LSTM_ACT_SCALED_TANH: return __fmul_rn(alpha, tanh32(__fmul_rn(beta, x)));
    case I8Q_LSTM_ACT_HARD_SIGMOID: {
      const float v = __fadd_rn(__fmul_rn(alpha, x), beta);
      return v < 0.0f ? 0.0f : (v > 1.0f ? 1.0f : v);
    }
    case I8Q_LSTM_ACT_ELU: return x >= 0.0f ? x : __fmul_rn(alpha, expm1_32(x));
    case I8Q_LSTM_ACT_SOFTSIGN: return __fdiv_rn(x, __fadd_rn(1.0f, fabsf(x)));
    case I8Q_LSTM_ACT_SOFTPLUS: return softplus32(x);
  }
  return x;
}
}  // namespace ef

__device__ __forceinline__ float activate(float v, int act) {
  if (act == I8Q_ACT_RELU) return v > 0.0f ? v : 0.0f;
  if (act == I8Q_ACT_GELU) return gelu_erf(v);
  return v;
}

// Epilogue of the dynamic quantized inner product for one element:
//   ((float)sum * scaleA) * scaleB + bias, activation.
__device__ __forceinline__ float dequant_epilogue(int32_t sum, float sA, float sB, float b, int act) {
  float v = __int2float_rn(sum);
  v = __fmul_rn(v, sA);
  v = __fmul_rn(v, sB);
  v = __fadd_rn(v, b);
  return activate(v, act);
}

// Same, for an output stored as bf16: GELU may use the cheaper erfc.
__device__ __forceinline__ float dequant_epilogue_bf16out(int32_t sum, float sA, float sB, float b, int act) {
  float v = __int2float_rn(sum);
  v = __fmul_rn(v, sA);
  v = __fmul_rn(v, sB);
  v = __fadd_rn(v, b);
  if (act == I8Q_ACT_GELU) return gelu_bf16out(v);
  return activate(v, act);
}

// ---- internal kernel launchers (implemented in the .cu files) ------------

// Row quantization of A (M x K, fp32 or bf16, row stride lda elements) into
// uA (M x Kp uint8, zero padded), optional uA_bf16 (M x Kp bf16 holding
// uA - 128, zero padded), scaleA[M], zeroA[M].
int launch_quantize_rows(const void* A, int typeA, int64_t M, int64_t K, int64_t lda, uint8_t* uA,
                         __nv_bfloat16* uA_bf16, int64_t Kp, float* scaleA, int32_t* zeroA,
                         cudaStream_t s);

// Column quantization of B (K x N fp32/bf16 row-major) into iBt (N x Kp
// int8, transposed, zero padded) and iBt_bf16 (the same codes as bf16),
// either of which may be null, scaleB[N], colsum[N].
// colmax_scratch: N words of device scratch for the two-pass form, or null.
int launch_quantize_cols(const void* B, int typeB, int64_t K, int64_t N, int avoid_overflow,
                         int8_t* iBt, __nv_bfloat16* iBt_bf16, int64_t Kp, float* scaleB,
                         int32_t* colsum, uint32_t* colmax_scratch, cudaStream_t s);

// Repack a given int8 B (K x N row-major, row stride ldb) into iBt
// (N x Kp), optional iBt_bf16, and colsum[N].
int launch_repack_cols_s8(const int8_t* B, int64_t K, int64_t N, int64_t ldb, int8_t* iBt,
                          __nv_bfloat16* iBt_bf16, int64_t Kp, int32_t* colsum, cudaStream_t s);

// The tiled form of those repacks: whether it takes the operands (16-byte
// aligned rows and pieces, N % 16 == 0, Kp % 16 == 0), and its launch, the
// codes centred on the way when flip (uint8: code - 128); iBt or iBt_bf16
// may be null; colsum (N entries) must be zeroed before.
bool repack_tiles_ok(const void* B, int64_t K, int64_t N, int64_t ldb, const void* iBt, const void* iBt_bf16,
                     int64_t Kp);
void launch_repack_tiles(const void* B, bool flip, int64_t K, int64_t N, int64_t ldb, int8_t* iBt,
                         __nv_bfloat16* iBt_bf16, int64_t Kp, int32_t* colsum, int64_t gates_H, cudaStream_t s);

// Same, with the columns of an iofc-ordered 4H-wide matrix (N == 4 * gates_H)
// interleaved per hidden unit: column q*H + u becomes row 4u + q of iBt.
int launch_repack_cols_s8_gates(const int8_t* B, int64_t K, int64_t N, int64_t ldb, int8_t* iBt,
                                __nv_bfloat16* iBt_bf16, int64_t Kp, int32_t* colsum, int64_t gates_H,
                                cudaStream_t s);

// Output modes of the GEMM epilogue.
enum OutMode : int {
  OUT_F32 = 0,   // dequantized fp32
  OUT_BF16 = 1,  // dequantized bf16
  OUT_S32 = 2,   // raw corrected int32 sums
};

struct GemmEpilogue {
  const int32_t* zeroA;   // [M]
  const float* scaleA;    // [M]
  const int32_t* colsum;  // [N]
  const float* scaleB;    // [N]
  const float* bias;      // [N] or null
  int act;
  int out_mode;
  void* C;
  int64_t ldc;            // elements
};

// Epilogue of the 8-bit-code products on the tensor-core path (QGemm,
// MatMulIntegerToFloat, DynamicQuantizeMatMul).  The operands enter
// centred, A' = A - ca and B' = B - cb (ca, cb = 128 for uint8 codes, 0 for
// int8), so with run = sum_k A'[i,k] B'[k,j]:
//   acc = run + rowsum[i] * g[j] + d[i] * e[j] + C[i,j]
//   rowsum[i] = sum_k A'[i,k],  d[i] = ca - a_zero_point[i],
//   g[j] = cb - b_zero_point[j],  e[j] = sum_k B'[k,j] + K g[j]
// (int32, wrapping: the true sum fits int32, so the modular result is it),
// then y = (float)acc * (asc[i] * bsc[j]) (+ bias[j]), stored as fp32 or
// requantized: saturate(rint(y / y_scale) + y_zero_point).  Per-row values
// are read at i * stride (stride 0: one value for the tensor).
struct QgEpilogue {
  const int32_t* rowsum;  // [M]
  const int32_t* d;       // d[i * d_stride]
  int64_t d_stride;
  const float* asc;       // asc[i * asc_stride]
  int64_t asc_stride;
  const int32_t* g;       // [N]
  const int32_t* e;       // [N]
  const float* bsc;       // [N]
  const float* bias;      // [N] or null
  const int32_t* C;       // element (i, j) at C[i * c_si + j * c_sj], or null
  int64_t c_si, c_sj;
  int c_col;              // C is the same for every row (c_si == 0) and bias is null: C is staged per column
  int ytype;              // I8Q_F32, I8Q_U8 or I8Q_S8
  float y_scale;
  float y_rcp;            // quot_rcp(y_scale)
  int y_zero_point;
  void* Y;
  int64_t ldy;
};

// Integer GEMM core: sum_k uA[i,k] * iBt[j,k] (uint8 x int8), corrected by
// -zeroA[i]*colsum[j], then the epilogue.  uA is M x Kp (row stride Kp),
// iBt is N x Kp, Kp a multiple of 64 with zero padding beyond K.
int launch_gemm_imma(const uint8_t* uA, const int8_t* iBt, int64_t M, int64_t N, int64_t Kp,
                     const GemmEpilogue& ep, cudaStream_t s);

// Exact-integer GEMM on the bf16 tensor pipe (tcgen05), same result as
// launch_gemm_imma but reading the bf16 operand copies: uA - 128 and iBt.
// max_abs_product_log2 bounds |(uA - 128) * iB| <= 2^max_abs_product_log2.
// Returns I8Q_ERR_UNSUPPORTED when the shape is outside what it handles.
int launch_gemm_tc(const __nv_bfloat16* uA, const __nv_bfloat16* iBt, int64_t M, int64_t N,
                   int64_t Kp, int max_abs_product_log2, const GemmEpilogue& ep, cudaStream_t s);

// The same product of centred operands A' (M x Kp) and B' (N x Kp) with the
// QGemm epilogue.
int launch_qgemm_tc(const __nv_bfloat16* Ac, const __nv_bfloat16* Bc, int64_t M, int64_t N, int64_t Kp,
                    int max_abs_product_log2, const QgEpilogue& qg, cudaStream_t s);

// Small products in one launch: row quantization of A (fp32/bf16, row
// stride K) into uA / scaleA / zeroA, then the integer sums against iBt
// (N x Kp int8) with dp4a and the epilogue.  Kp <= small_max_kp().
int64_t small_max_kp();
int launch_gemm_small(const void* A, int typeA, int64_t M, int64_t K, int64_t Kp, const int8_t* iBt, int64_t N,
                      uint8_t* uA, float* scaleA, int32_t* zeroA, const GemmEpilogue& ep, cudaStream_t s);

// QLinearConv on the tensor pipe (group 1, stride 1, dilation 1, tile shapes
// it instantiates).  conv_tc_workspace: scratch bytes, 0 when the shape does
// not take this path.
size_t conv_tc_workspace(int64_t N, int64_t C, int64_t H, int64_t W, int64_t M, int64_t Cg, int64_t kH, int64_t kW,
                         int64_t OH, int64_t OW, int64_t group, int64_t sh, int64_t sw, int64_t dh, int64_t dw);
int launch_conv_tc(const void* x, int xtype, int64_t N, int64_t C, int64_t H, int64_t W, float x_scale, int x_zp,
                   const void* w, int wtype, int64_t M, int64_t kH, int64_t kW, const float* w_scale,
                   const void* w_zp, int per_channel, float y_scale, int y_zp, int ytype, const int32_t* B,
                   int64_t pt, int64_t pl, int64_t OH, int64_t OW, void* y, void* workspace, cudaStream_t s);

}  // namespace i8q
