// lstm.cu -- DynamicQuantizeLSTM (ONNX Runtime contrib schema
// "DynamicQuantizeLSTM"; graiphic.io "DynamicQuantizeLSTM") on the dynamic
// quantized GEMM engine.
//
// int8 W [D, input, 4H] and R [D, H, 4H] with per-channel (or per-direction)
// scales and zero point 0; fp32 X; default activations (sigmoid for the
// i, o, f gates, tanh for the cell candidate and the output; the general
// form takes any of the ONNX LSTM activation functions); gate column
// order i, o, f, c.  sigmoid and tanh are the fixed-sequence fp32
// functions of common.cuh (ef::), so a step's result does not depend on
// the platform's math library.  X and each step's hidden state are quantized per row to
// uint8 exactly like A of the dynamic quantized inner product.
//   input projection (all steps at once): Gx = X W[d]
//   per step t: Gh = h_{t-1} R[d]; g = ((Gx_t + Gh) + Wb) + Rb
//               i, o, f = sigmoid(g); ct = tanh(g_c)
//               c = f*c_{t-1} + i*ct;  h = o*tanh(c)
// The reverse direction walks t = T-1 .. 0.
//
// Layout: the 4H gate columns of W, R, their scales and the biases are
// interleaved per hidden unit (column q*H + u stored at 4u + q), so any
// 64-column tile holds all four gates of 16 hidden units.  The projection
// runs once over all T * batch rows on the tensor-core GEMM; X is quantized
// once for both directions.  The recurrence runs, where the layer fits, as
// one persistent cooperative kernel (prs:: below: R resident in shared
// memory, the new h quantized per row inside the kernel).  Otherwise one
// kernel per step does, for both directions at once, the recurrent integer
// product and the whole cell update in its epilogue: on the tensor pipe
// (tcgen05, 128 gate columns x 64 batch rows per CTA, h codes centred to
// uh - 128 in bf16, fp32 chunks drained exactly to int32, the step's
// x-projection and previous cell state loaded while the MMAs run) for wide
// layers, or on the int8 mma.sync form (64 x 64 tiles) otherwise.  Each
// step's new h is then quantized per row (both directions in one launch) for
// the next step, and the whole sequence of steps is replayed as one CUDA
// graph, cached per argument set.
#include <cstring>
#include <functional>
#include <mutex>

#include "tcgen05.cuh"

namespace i8q {
namespace {

struct LstmLayout {
  int64_t D, TB, Ip, Hp, H4;
  size_t off_Wt, off_Wtb, off_Wcs, off_Rt, off_Rtb, off_Rcs, off_Wsc, off_Rsc, off_Wbi, off_Rbi, off_uX, off_uXc,
      off_sX, off_zX, off_Gx, off_uh, off_uhc, off_sh, off_zh, off_mm, off_gbar, off_h, off_c, total;
};

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

LstmLayout lstm_layout(int64_t T, int64_t batch, int64_t input, int64_t hidden, int direction) {
  LstmLayout L;
  L.D = direction == I8Q_LSTM_BIDIRECTIONAL ? 2 : 1;
  L.TB = T * batch;
  L.Ip = round_up(input, 64);
  L.Hp = round_up(hidden, 64);
  L.H4 = 4 * hidden;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  L.off_Wt = take((size_t)L.D * L.H4 * L.Ip);
  L.off_Wtb = take((size_t)L.D * L.H4 * L.Ip * 2);
  L.off_Wcs = take((size_t)L.D * L.H4 * 4);
  L.off_Rt = take((size_t)L.D * L.H4 * L.Hp);
  L.off_Rtb = take((size_t)L.D * L.H4 * L.Hp * 2);
  L.off_Rcs = take((size_t)L.D * L.H4 * 4);
  L.off_Wsc = take((size_t)L.D * L.H4 * 4);
  L.off_Rsc = take((size_t)L.D * L.H4 * 4);
  L.off_Wbi = take((size_t)L.D * L.H4 * 4);
  L.off_Rbi = take((size_t)L.D * L.H4 * 4);
  L.off_uX = take((size_t)L.TB * L.Ip);
  L.off_uXc = take((size_t)L.TB * L.Ip * 2);
  L.off_sX = take((size_t)L.TB * 4);
  L.off_zX = take((size_t)L.TB * 4);
  L.off_Gx = take((size_t)L.D * L.TB * L.H4 * 4);
  // h codes (uint8 for the mma.sync step, bf16 uh - 128 for the tensor
  // pipe), scales and zero points, in two step parities: step s reads
  // parity (s + 1) & 1 and the codes of its new h go to parity s & 1 (h0's
  // to parity 1); then per-row min/max pairs and a barrier counter for the
  // persistent recurrence
  L.off_uh = take((size_t)2 * L.D * batch * L.Hp);
  L.off_uhc = take((size_t)2 * L.D * batch * L.Hp * 2);
  L.off_sh = take((size_t)2 * L.D * batch * 4);
  L.off_zh = take((size_t)2 * L.D * batch * 4);
  L.off_mm = take((size_t)2 * L.D * batch * 2 * 4);
  L.off_gbar = take(2 * 4);
  L.off_h = take((size_t)2 * L.D * batch * hidden * 4);
  L.off_c = take((size_t)L.D * batch * hidden * 4);
  L.total = o;
  return L;
}

// Per-direction (n == D) or per-channel (n == D*4H) scales, interleaved.
__global__ void interleave_scales(const float* __restrict__ src, int64_t n, int64_t D, int64_t H,
                                  float* __restrict__ dst) {
  const int64_t H4 = 4 * H;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < D * H4; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t d = i / H4, jp = i % H4, u = jp / 4, q = jp % 4;
    dst[i] = n == D ? src[d] : src[d * H4 + q * H + u];
  }
}

// Wb, Rb halves of B [D, 8H], interleaved (zeros when B is absent).
__global__ void interleave_bias(const float* __restrict__ B, int64_t D, int64_t H, float* __restrict__ Wbi,
                                float* __restrict__ Rbi) {
  const int64_t H4 = 4 * H;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < D * H4; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t d = i / H4, jp = i % H4, u = jp / 4, q = jp % 4;
    Wbi[i] = B ? B[d * 2 * H4 + q * H + u] : 0.0f;
    Rbi[i] = B ? B[d * 2 * H4 + H4 + q * H + u] : 0.0f;
  }
}

__global__ void init_state(const float* __restrict__ h0, const float* __restrict__ c0, int64_t n, float* __restrict__ h,
                           float* __restrict__ c) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    h[i] = h0 ? h0[i] : 0.0f;
    c[i] = c0 ? c0[i] : 0.0f;
  }
}

__global__ void copy_f32(const float* __restrict__ src, float* __restrict__ dst, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

__global__ void any_nonzero_s8(const int8_t* __restrict__ p, int64_t n, int* __restrict__ flag) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    if (p[i] != 0) atomicOr(flag, 1);
}

// W or R of one direction (K x 4H, 8-bit codes, columns in iofc order) with
// its zero point subtracted, as bf16 rows of the gate-interleaved K-major
// operand: column q*H + u lands at row 4u + q, K contiguous, zeros beyond K;
// colsum[row] = sum_k (W - zp).  zp: typed codes, one per direction
// (n_zp == 1) or per column (n_zp == 4H), or null (0).  |W - zp| <= 255 is
// exact in bf16.  One CTA per 32 columns; 64 K-rows per step through shared
// memory.
template <bool SIGNED>
__global__ void __launch_bounds__(256)
repack_gates_zp(const uint8_t* __restrict__ W, int64_t K, int64_t H, const uint8_t* __restrict__ zp, int64_t n_zp,
                int64_t Kp, __nv_bfloat16* __restrict__ out, int32_t* __restrict__ colsum) {
  __shared__ int16_t tile[32][64 + 2];
  __shared__ int32_t sums[8][32];
  const int64_t H4 = 4 * H;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int64_t j0 = (int64_t)blockIdx.x * 32;
  const int64_t j = j0 + lane;  // loading: lane -> column
  const bool jok = j < H4;
  auto code = [&](uint8_t v) { return SIGNED ? (int)(int8_t)v : (int)v; };
  const int z = (jok && zp) ? code(zp[n_zp == 1 ? 0 : j]) : 0;
  int part = 0;
  for (int64_t k0 = 0; k0 < Kp; k0 += 64) {
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int kk = warp + 8 * r;
      const int64_t k = k0 + kk;
      const int v = (jok && k < K) ? code(W[k * H4 + j]) - z : 0;
      part += v;
      tile[lane][kk] = (int16_t)v;
    }
    __syncthreads();
    // write: thread -> column c (of 32), 16-byte chunk ch (of 8)
    const int c = t >> 3, ch = t & 7;
    const int64_t jj = j0 + c;
    if (jj < H4) {
      const int64_t row = 4 * (jj % H) + jj / H;
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float f0 = (float)tile[c][ch * 8 + 2 * e], f1 = (float)tile[c][ch * 8 + 2 * e + 1];
        w[e] = (__float_as_uint(f0) >> 16) | (__float_as_uint(f1) & 0xffff0000u);
      }
      *reinterpret_cast<uint4*>(out + row * Kp + k0 + ch * 8) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    __syncthreads();
  }
  sums[warp][lane] = part;
  __syncthreads();
  if (warp == 0 && jok) {
    int total = 0;
    for (int w8 = 0; w8 < 8; ++w8) total += sums[w8][lane];
    colsum[4 * (j % H) + j / H] = total;
  }
}

using ef::sigmoid32;
using ef::tanh32;

// The three activation functions (f, g, h) of each direction with their
// alpha / beta (the general form only).
struct LstmActs {
  int kind[2][3];
  float alpha[2][3], beta[2][3];
};

// ---- the fused step ------------------------------------------------------------
constexpr int SB = 64, SN = 64, SK = 64, SSTAGES = 3, STHREADS = 128;
constexpr int S_STAGE = (SB + SN) * SK;

__device__ __forceinline__ uint32_t s_smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void s_cp_async16(uint32_t dst, const void* src, int bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(bytes));
}
__device__ __forceinline__ void s_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void s_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}
__device__ __forceinline__ void s_ldsm4(uint32_t a, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(a));
}
__device__ __forceinline__ void s_mma(int32_t (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.u8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ int s_swz(int r, int c) { return r * SK + ((c ^ ((r >> 1) & 3)) << 4); }

struct StepParams {
  const uint8_t* uh;   // [D*B, Hp] quantized h of the previous step
  const float* sh;     // [D*B]
  const int32_t* zh;   // [D*B]
  const int8_t* Rt;    // [D, 4H, Hp] interleaved rows
  const int32_t* Rcs;  // [D, 4H]
  const float* Rsc;    // [D, 4H]
  const float* Gx;     // [D, T*B, 4H] interleaved columns
  const float* Wbi;    // [D, 4H]
  const float* Rbi;    // [D, 4H]
  float* c;            // [D, B, H] in place
  float* h_next;       // [D, B, H]
  float* Y;            // [T, D, B, H] or null
  int step, T, B, H, Hp, D, direction;
};

// grid (4H/64, D, ceil(B/64)), 128 threads.
__global__ void __launch_bounds__(STHREADS) lstm_step_kernel(StepParams p) {
  __shared__ __align__(128) uint8_t smem[SSTAGES * S_STAGE];
  __shared__ float gs[SB][SN + 1];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wm = warp >> 1, wn = warp & 1;
  const int d = blockIdx.y, m0 = blockIdx.z * SB, n0 = blockIdx.x * SN;
  const int H4 = 4 * p.H;
  const int KT = p.Hp / SK;
  const uint8_t* A = p.uh + (int64_t)d * p.B * p.Hp;
  const int8_t* Bm = p.Rt + (int64_t)d * H4 * p.Hp;

  auto load_stage = [&](int stage, int kt) {
    uint8_t* sA = smem + stage * S_STAGE;
    uint8_t* sB = sA + SB * SK;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int idx = tid + i * STHREADS;  // 0..255: row = idx/4, chunk = idx%4
      const int r = idx >> 2, ch = idx & 3;
      const int ga = m0 + r, gb = n0 + r;
      const uint8_t* pa = A + (int64_t)(ga < p.B ? ga : p.B - 1) * p.Hp + kt * SK + ch * 16;
      const int8_t* pb = Bm + (int64_t)(gb < H4 ? gb : H4 - 1) * p.Hp + kt * SK + ch * 16;
      s_cp_async16(s_smem_u32(sA + s_swz(r, ch)), pa, ga < p.B ? 16 : 0);
      s_cp_async16(s_smem_u32(sB + s_swz(r, ch)), pb, gb < H4 ? 16 : 0);
    }
  };

  int32_t acc[2][4][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[i][j][q] = 0;

#pragma unroll
  for (int s = 0; s < SSTAGES - 1; ++s) {
    if (s < KT) load_stage(s, s);
    s_commit();
  }
  for (int kt = 0; kt < KT; ++kt) {
    s_wait<SSTAGES - 2>();
    __syncthreads();
    {
      const int nk = kt + SSTAGES - 1;
      if (nk < KT) load_stage(nk % SSTAGES, nk);
      s_commit();
    }
    const uint8_t* sA = smem + (kt % SSTAGES) * S_STAGE;
    const uint8_t* sB = sA + SB * SK;
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      uint32_t af[2][4], bf[4][2];
#pragma unroll
      for (int mi = 0; mi < 2; ++mi) {
        const int r = wm * 32 + mi * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        s_ldsm4(s_smem_u32(sA + s_swz(r, kk * 2 + (lane >> 4))), af[mi][0], af[mi][1], af[mi][2], af[mi][3]);
      }
#pragma unroll
      for (int nj = 0; nj < 2; ++nj) {
        const int r = wn * 32 + nj * 16 + (lane & 7) + (lane >> 4) * 8;
        s_ldsm4(s_smem_u32(sB + s_swz(r, kk * 2 + ((lane >> 3) & 1))), bf[2 * nj][0], bf[2 * nj][1], bf[2 * nj + 1][0],
                bf[2 * nj + 1][1]);
      }
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) s_mma(acc[mi][ni], af[mi], bf[ni][0], bf[ni][1]);
    }
  }
  s_wait<0>();

  // gate pre-activations of the tile: ((Gx + Gh) + Wb) + Rb
  const bool rev = p.direction == I8Q_LSTM_REVERSE || (p.direction == I8Q_LSTM_BIDIRECTIONAL && d == 1);
  const int t = rev ? p.T - 1 - p.step : p.step;
  const int64_t TB = (int64_t)p.T * p.B;
  const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int r = wm * 32 + mi * 16 + g + 8 * hh;
      const int b = m0 + r;
      if (b >= p.B) continue;
      const float sH = __ldg(p.sh + d * p.B + b);
      const int32_t zH = __ldg(p.zh + d * p.B + b);
      const float* gx = p.Gx + ((int64_t)d * TB + (int64_t)t * p.B + b) * H4;
#pragma unroll
      for (int ni = 0; ni < 4; ++ni)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int cc = wn * 32 + ni * 8 + 2 * t4 + e;
          const int n = n0 + cc;
          if (n >= H4) continue;
          const int64_t dn = (int64_t)d * H4 + n;
          const int32_t v = acc[mi][ni][2 * hh + e] - zH * __ldg(p.Rcs + dn);
          float gh = __fmul_rn(__int2float_rn(v), sH);
          gh = __fmul_rn(gh, __ldg(p.Rsc + dn));
          float gg = __fadd_rn(__ldg(gx + n), gh);
          gg = __fadd_rn(gg, __ldg(p.Wbi + dn));
          gg = __fadd_rn(gg, __ldg(p.Rbi + dn));
          gs[r][cc] = gg;
        }
    }
  __syncthreads();

  // cell update: 64 rows x 16 hidden units per tile
  for (int pi = tid; pi < SB * (SN / 4); pi += STHREADS) {
    const int r = pi >> 4, uu = pi & 15;
    const int b = m0 + r, u = n0 / 4 + uu;
    if (b >= p.B || u >= p.H) continue;
    const float ig = sigmoid32(gs[r][4 * uu + 0]);
    const float og = sigmoid32(gs[r][4 * uu + 1]);
    const float fg = sigmoid32(gs[r][4 * uu + 2]);
    const float ct = tanh32(gs[r][4 * uu + 3]);
    const int64_t e = ((int64_t)d * p.B + b) * p.H + u;
    const float cn = __fadd_rn(__fmul_rn(fg, p.c[e]), __fmul_rn(ig, ct));
    const float hn = __fmul_rn(og, tanh32(cn));
    p.c[e] = cn;
    p.h_next[e] = hn;
    if (p.Y) p.Y[(((int64_t)t * p.D + d) * p.B + b) * p.H + u] = hn;
  }
}

// ---- the fused step on the tensor pipe ----------------------------------------
// The same step with the recurrent product on tcgen05 (bf16 operands holding
// exact integer codes, fp32 accumulation exact within chunks of 2^24 / 2^14
// = 1024 K-elements, drained into int32 registers).  Orientation: M = 128
// gate rows of R (rows 4u + q), N = 64 batch rows of h, so TMEM lane r holds
// gate row r for 64 batch columns; the four gates of unit u sit in four
// consecutive lanes of one warp and meet through warp shuffles.
// Warps: 0 = TMA producer, 1 = TMEM owner and MMA issuer, 2..5 = drain and
// cell update (warp w reads TMEM lanes 32 * (w % 4) ..).
namespace tcs {
using namespace tc;
constexpr int BM = 128, BN = 64, BK = 64, STAGES = 4, EPI_WARPS = 8, THREADS = 64 + 32 * EPI_WARPS, TMEM_COLS = 64;
constexpr int HALF = BN / 2;  // batch columns per epilogue warp
constexpr int A_STAGE = BM * BK * 2, B_STAGE = BN * BK * 2, STAGE_BYTES = A_STAGE + B_STAGE;
constexpr int NUM_BARS = 2 * STAGES + 2;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + NUM_BARS * 8 + 16;
constexpr uint32_t ST_TIMEOUT = 1u << 8;

struct TcStepParams {
  const float* sh;     // [D*B] of the parity this step reads
  const int32_t* zh;   // [D*B]
  int hrow0;           // first row of that parity in the h-code tensor map
  const int32_t* Rcs;  // [D, 4H]
  const float* Rsc;    // [D, 4H]
  const float* Gx;     // [D, T*B, 4H]
  const float* Wbi;    // [D, 4H]
  const float* Rbi;    // [D, 4H]
  float* c;            // [D, B, H]
  float* h_next;       // [D, B, H]
  float* Y;            // [T, D, B, H] or null
  int step, T, B, H, Hp, D, direction, CS;
  uint32_t* status;
  // variants (the VAR instantiation)
  const float* h_prev;       // [D, B, H]: carried when a row's sequence has ended
  const int32_t* seq_lens;   // [B] or null (every row has length T)
  const float* P;            // [D, 3H] peepholes (i, o, f) or null
  float clip;                // > 0: gate inputs bounded to [-clip, clip]
  int input_forget;          // f = 1 - i
  LstmActs acts;
};

__device__ __forceinline__ float clip_gate(float v, float clip) {
  return clip > 0.0f ? fminf(fmaxf(v, -clip), clip) : v;
}

// grid (ceil(4H/128), D, ceil(B/64)).  VAR adds sequence lengths,
// peepholes, clip and coupled gates: the output gate is then formed after
// the new cell state (its peephole reads it).
template <bool VAR>
__global__ void __launch_bounds__(THREADS, 1)
lstm_step_tc_kernel(const __grid_constant__ CUtensorMap tmR, const __grid_constant__ CUtensorMap tmH, TcStepParams p) {
  constexpr uint32_t IDESC = idesc_bf16(BM, BN);
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned, indexed from the shared array itself so that accesses stay shared-space
  uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t smem0 = smem_u32(smem);
  auto sA = [&](int s) { return smem0 + (uint32_t)(s * STAGE_BYTES); };
  auto sB = [&](int s) { return smem0 + (uint32_t)(s * STAGE_BYTES + A_STAGE); };
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto empty = [&](int s) { return smem_u32(bars + STAGES + s); };
  const uint32_t accf = smem_u32(bars + 2 * STAGES), acce = smem_u32(bars + 2 * STAGES + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = blockIdx.y, mt = blockIdx.x, nb = blockIdx.z;
  const int H4 = 4 * p.H;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(accf, 1);
    mbar_init(acce, EPI_WARPS);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int KT = p.Hp / BK, CS = p.CS;
  const int nchunks = (KT + CS - 1) / CS;
  if (warp == 0) {
    if (lane == 0) {
      int kt = 0;
      for (; kt < KT; ++kt) {
        const int s = kt % STAGES;
        if (!wait_bar(empty(s), ((uint32_t)(kt / STAGES) & 1u) ^ 1u, abort_flag, p.status, ST_TIMEOUT)) break;
        mbar_arrive_expect_tx(full(s), STAGE_BYTES);
        tma_load_2d(sA(s), &tmR, full(s), kt * BK, d * H4 + mt * BM);
        tma_load_2d(sB(s), &tmH, full(s), kt * BK, p.hrow0 + d * p.B + nb * BN);
      }
      if (kt < KT)
        for (int j = max(0, kt - STAGES); j < kt; ++j) {
          unsigned long long t0 = global_ns();
          while (!mbar_try_wait(full(j % STAGES), (uint32_t)(j / STAGES) & 1u))
            if (global_ns() - t0 > WAIT_LIMIT_NS) break;
        }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int chunk = 0;
      for (int kt = 0; kt < KT; ++kt) {
        const int kc = kt % CS;
        if (kc == 0) {
          if (!wait_bar(acce, ((uint32_t)chunk & 1u) ^ 1u, abort_flag, p.status, ST_TIMEOUT)) break;
          tc_fence_after();
        }
        const int s = kt % STAGES;
        if (!wait_bar(full(s), (uint32_t)(kt / STAGES) & 1u, abort_flag, p.status, ST_TIMEOUT)) break;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)
          tc_mma(tmem, desc_sw128(sA(s) + (uint32_t)(k * 32)), desc_sw128(sB(s) + (uint32_t)(k * 32)), IDESC,
                 (kc == 0 && k == 0) ? 0u : 1u);
        tc_commit(empty(s));
        if (kc == CS - 1 || kt == KT - 1) {
          tc_commit(accf);
          ++chunk;
        }
      }
    }
  } else {
    const int q4 = warp & 3;                     // TMEM lane quadrant
    const int half = (warp - 2) >> 2;            // which 32 of the 64 batch columns
    const int r = q4 * 32 + lane;                // gate row within the tile
    const int n = mt * BM + r;                   // interleaved gate column 4u + q
    const bool rev = p.direction == I8Q_LSTM_REVERSE || (p.direction == I8Q_LSTM_BIDIRECTIONAL && d == 1);
    const int t = rev ? p.T - 1 - p.step : p.step;
    const int64_t TB = (int64_t)p.T * p.B;
    const bool nvalid = n < H4;
    const int q = n & 3, u = n >> 2;
    const int b0 = nb * BN + half * HALF;
    // operands of the epilogue that do not depend on the product: fetched
    // while the tensor core works.  A row whose sequence has ended (VAR,
    // step >= its length) is inactive; the reverse direction of a row of
    // length L walks t = L-1 .. 0.
    float gx[HALF], cprev[HALF];
    uint32_t active = 0;
#pragma unroll
    for (int j = 0; j < HALF; ++j) {
      const int b = b0 + j;
      const bool ok_b = b < p.B && nvalid;
      int tb = t;
      bool act_b = ok_b;
      if (VAR && ok_b && p.seq_lens) {
        const int L = min(max(__ldg(p.seq_lens + b), 0), p.T);  // lengths outside [0, T] are clamped
        act_b = p.step < L;
        tb = rev ? L - 1 - p.step : p.step;
      }
      active |= (act_b ? 1u : 0u) << j;
      gx[j] = act_b ? __ldg(p.Gx + ((int64_t)d * TB + (int64_t)tb * p.B + b) * H4 + n) : 0.0f;
      cprev[j] = (ok_b && (VAR || q == 0) && u < p.H) ? p.c[((int64_t)d * p.B + b) * p.H + u] : 0.0f;
    }
    int32_t run[HALF];
#pragma unroll
    for (int j = 0; j < HALF; ++j) run[j] = 0;
    bool ok = true;
    for (int c = 0; c < nchunks; ++c) {
      const bool got = wait_bar(accf, (uint32_t)c & 1u, abort_flag, p.status, ST_TIMEOUT);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t v0[16], v1[16];
      tmem_ld16(tmem + ((uint32_t)(q4 * 32) << 16) + (uint32_t)(half * HALF), v0);
      tmem_ld16(tmem + ((uint32_t)(q4 * 32) << 16) + (uint32_t)(half * HALF + 16), v1);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        run[i] += __float2int_rn(__uint_as_float(v0[i]));
        run[16 + i] += __float2int_rn(__uint_as_float(v1[i]));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce);
    }
    if (ok && VAR) {
      const int64_t dn = (int64_t)d * H4 + (nvalid ? n : 0);
      const int32_t cs = nvalid ? __ldg(p.Rcs + dn) : 0;
      const float rsc = nvalid ? __ldg(p.Rsc + dn) : 0.0f;
      const float wb = nvalid ? __ldg(p.Wbi + dn) : 0.0f;
      const float rb = nvalid ? __ldg(p.Rbi + dn) : 0.0f;
      // this lane's peephole weight: P[d] holds Pi, Po, Pf (H each)
      const int pq = q == 0 ? 0 : (q == 1 ? 1 : 2);
      const float pw = (p.P && nvalid && q < 3 && u < p.H) ? __ldg(p.P + (int64_t)d * 3 * p.H + pq * p.H + u) : 0.0f;
      const int base_lane = lane & ~3;
#pragma unroll
      for (int j = 0; j < HALF; ++j) {
        const int b = b0 + j;
        const bool live = (active >> j) & 1u;
        // phase 1: i, f, c~ (the o lane keeps its partial sum)
        float sum = 0.0f, act = 0.0f;
        if (live) {
          const float sH = __ldg(p.sh + d * p.B + b);
          const int32_t v = run[j] - (__ldg(p.zh + d * p.B + b) - 128) * cs;
          float gh = __fmul_rn(__int2float_rn(v), sH);
          gh = __fmul_rn(gh, rsc);
          sum = __fadd_rn(gx[j], gh);
          if (p.P && (q == 0 || q == 2)) sum = __fadd_rn(sum, __fmul_rn(pw, cprev[j]));
          if (q != 1) {
            float gg = __fadd_rn(__fadd_rn(sum, wb), rb);
            gg = clip_gate(gg, p.clip);
            act = q == 3 ? ef::lstm_act(p.acts.kind[d][1], p.acts.alpha[d][1], p.acts.beta[d][1], gg)
                         : ef::lstm_act(p.acts.kind[d][0], p.acts.alpha[d][0], p.acts.beta[d][0], gg);
          }
        }
        const float ig = __shfl_sync(0xffffffffu, act, base_lane + 0);
        const float fg0 = __shfl_sync(0xffffffffu, act, base_lane + 2);
        const float ct = __shfl_sync(0xffffffffu, act, base_lane + 3);
        const float fg = p.input_forget ? __fsub_rn(1.0f, ig) : fg0;
        const float cn = __fadd_rn(__fmul_rn(fg, cprev[j]), __fmul_rn(ig, ct));  // meaningful on live rows
        // phase 2: o from the new cell state
        float og = 0.0f;
        if (live && q == 1) {
          float so = sum;
          if (p.P) so = __fadd_rn(so, __fmul_rn(pw, cn));
          so = __fadd_rn(__fadd_rn(so, wb), rb);
          og = ef::lstm_act(p.acts.kind[d][0], p.acts.alpha[d][0], p.acts.beta[d][0], clip_gate(so, p.clip));
        }
        og = __shfl_sync(0xffffffffu, og, base_lane + 1);
        if (q == 0 && b < p.B && nvalid && u < p.H) {
          const int64_t e = ((int64_t)d * p.B + b) * p.H + u;
          if (live) {
            const float hn = __fmul_rn(og, ef::lstm_act(p.acts.kind[d][2], p.acts.alpha[d][2], p.acts.beta[d][2], cn));
            p.c[e] = cn;
            p.h_next[e] = hn;
            if (p.Y) {
              const int tb = p.seq_lens ? (rev ? min(max(__ldg(p.seq_lens + b), 0), p.T) - 1 - p.step : p.step) : t;
              p.Y[(((int64_t)tb * p.D + d) * p.B + b) * p.H + u] = hn;
            }
          } else {
            p.h_next[e] = p.h_prev[e];  // the row's state is carried
          }
        }
      }
    }
    if (ok && !VAR) {
      const int64_t dn = (int64_t)d * H4 + (nvalid ? n : 0);
      const int32_t cs = nvalid ? __ldg(p.Rcs + dn) : 0;
      const float rsc = nvalid ? __ldg(p.Rsc + dn) : 0.0f;
      const float wb = nvalid ? __ldg(p.Wbi + dn) : 0.0f;
      const float rb = nvalid ? __ldg(p.Rbi + dn) : 0.0f;
      const int base_lane = lane & ~3;
#pragma unroll
      for (int j = 0; j < HALF; ++j) {
        const int b = b0 + j;
        const bool bvalid = b < p.B;
        float act = 0.0f;
        if (bvalid && nvalid) {
          const float sH = __ldg(p.sh + d * p.B + b);
          // h entered as uh - 128: sum_k (uh - zh) R = run - (zh - 128) colsum
          const int32_t v = run[j] - (__ldg(p.zh + d * p.B + b) - 128) * cs;
          float gh = __fmul_rn(__int2float_rn(v), sH);
          gh = __fmul_rn(gh, rsc);
          float gg = __fadd_rn(gx[j], gh);
          gg = __fadd_rn(gg, wb);
          gg = __fadd_rn(gg, rb);
          act = q < 3 ? sigmoid32(gg) : tanh32(gg);
        }
        const float ig = __shfl_sync(0xffffffffu, act, base_lane + 0);
        const float og = __shfl_sync(0xffffffffu, act, base_lane + 1);
        const float fg = __shfl_sync(0xffffffffu, act, base_lane + 2);
        const float ct = __shfl_sync(0xffffffffu, act, base_lane + 3);
        if (q == 0 && bvalid && nvalid && u < p.H) {
          const int64_t e = ((int64_t)d * p.B + b) * p.H + u;
          const float cn = __fadd_rn(__fmul_rn(fg, cprev[j]), __fmul_rn(ig, ct));
          const float hn = __fmul_rn(og, tanh32(cn));
          p.c[e] = cn;
          p.h_next[e] = hn;
          if (p.Y) p.Y[(((int64_t)t * p.D + d) * p.B + b) * p.H + u] = hn;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}
}  // namespace tcs

// ---- the persistent recurrence ------------------------------------------------
// One cooperative launch runs every step.  CTA (d, g) owns the 16 hidden
// units 16g .. 16g + 15 of direction d, i.e. the 64 interleaved gate rows
// 64g .. 64g + 63 of R[d], which it loads into shared memory once (bf16
// R - zp, K-major, 128-byte swizzle) and keeps for the whole sequence.  Per
// step the TMA producer streams the previous step's h codes (uh - 128,
// bf16, 64 batch rows x Hp) through an 8-stage ring and one thread issues
// the product as M = 64 batch rows x N = 64 gate rows on tcgen05, fp32
// chunks of 2^24 / 2^log2 K-elements drained exactly to int32 as in the
// per-step kernels.  Products this small are bound by the issuing thread
// (an MMA of this size takes about 79 SM clocks to issue back to back, and
// more with any other instruction between) and by the latency of MMAs that
// accumulate into the same tile: the issue loop is unrolled over the ring
// (K a multiple of 512).  At this issue rate one accumulator (TMEM columns
// 0..63) is fastest: two or four independent ones, which hide the MMAs'
// accumulation latency, cost more in the drain than they save.  With M = 64 the accumulator rows 16w .. 16w + 15 sit in
// TMEM lanes 32w .. 32w + 15, so the epilogue warps of all four
// sub-partitions read them; a row's 16 columns (four units, gates i, o, f, c
// interleaved) are split between a lane and the lane 16 above it, two units
// each, and each thread updates its cells without further exchange.  The
// new h is quantized per row right away: each CTA folds min/max of its units
// per row, merges them into a global per-row pair (order-preserving integer
// images, atomicMax), and after a barrier over the direction's CTAs every
// CTA derives the same scale and zero point and writes the codes of its
// units; a second barrier publishes them to the direction's next TMA reads
// (the two directions never wait on each other).  Codes, scales/zero
// points and the min/max pairs are double buffered by step parity.  Every
// wait is bounded: on expiry the kernel sets ST_TIMEOUT in the status word,
// which every other wait also polls, and all CTAs leave after their copies
// and products in flight have landed.
namespace prs {

using namespace tc;
using tcs::clip_gate;

constexpr int BM = 64, BN = 64, BK = 64, STAGES = 8;
constexpr int EPI_WARPS = 16, THREADS = 32 * (2 + EPI_WARPS);  // warps 2..17: TMEM sub-partition warp % 4
constexpr int NACC = 1;                // accumulators the 16-K sub-steps of a slab rotate over
constexpr int TMEM_COLS = NACC * 64;
constexpr int A_STAGE = BM * BK * 2;   // 8 KB
constexpr int R_SLAB = BN * BK * 2;    // 8 KB per 64 K-elements of the resident R tile
constexpr uint32_t ST_TIMEOUT = 1u << 9;
constexpr int NUM_BARS = 2 * STAGES + 5;  // full, empty, accf, acce, rbar, hready, mdone

struct Params {
  const int32_t* Rcs;  // [D, 4H]
  const float* Rsc;    // [D, 4H]
  const float* Gx;     // [D, T*B, 4H]
  const float* Wbi;    // [D, 4H]
  const float* Rbi;    // [D, 4H]
  float* c;            // [D, B, H]
  float* hbuf;         // 2 x [D, B, H] (step s reads parity s & 1, writes (s + 1) & 1)
  float* Y;            // [T, D, B, H] or null
  __nv_bfloat16* uhc;  // 2 x [D * B, Hp] h codes - 128 (step s reads parity (s + 1) & 1, writes s & 1)
  float* sh;           // 2 x [D * B]
  int32_t* zh;         // 2 x [D * B]
  uint32_t* mm;        // 2 x [D * B][2]: max image of -h, of h
  uint32_t* gbar;      // [D] barrier counters of each direction's CTAs (0 at launch)
  int T, B, H, Hp, D, direction, CS, tiles;  // tiles = H / 16 per direction
  uint32_t* status;
  const int32_t* seq_lens;
  const float* P;
  float clip;
  int input_forget;
  LstmActs acts;
};

size_t smem_bytes(int64_t Hp) { return 1024 + (size_t)STAGES * A_STAGE + (size_t)(Hp / BK) * R_SLAB + NUM_BARS * 8 + 16; }

// Order-preserving image of a float as an unsigned integer (0 is below the
// image of every float, so 0 is the empty value of an atomicMax).
__device__ __forceinline__ uint32_t ord_image(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float ord_value(uint32_t v) {
  return __uint_as_float((v & 0x80000000u) ? (v & 0x7fffffffu) : ~v);
}

// Grid barrier number k (1, 2, ...), called by one thread per CTA after a
// CTA-wide barrier: the fence makes the CTA's writes visible before the
// arrival (cumulatively); true when every CTA has arrived, false on
// timeout or when another CTA gave up.
__device__ __forceinline__ bool grid_barrier(uint32_t* gbar, uint32_t target, uint32_t* status,
                                             unsigned long long limit_ns = WAIT_LIMIT_NS) {
  __threadfence();
  asm volatile("red.release.gpu.global.add.u32 [%0], 1;\n" ::"l"(gbar) : "memory");
  const unsigned long long t0 = global_ns();
  for (uint32_t i = 0;; ++i) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(gbar) : "memory");
    if (v >= target) return true;
    if ((i & 63u) == 63u) {
      if (*(volatile uint32_t*)status & ST_TIMEOUT) return false;
      if (global_ns() - t0 > limit_ns) {
        atomicOr(status, ST_TIMEOUT);
        return false;
      }
    }
  }
}

// Failure-detection probe: one CTA runs one of the bounded waits above with
// a short limit on an event that never comes -- an mbarrier phase nobody
// arrives on (kind 0, the waits of the tcgen05 pipelines) or a grid
// barrier whose other CTAs never arrive (kind 1, the persistent
// recurrence's) -- so that the wait gives up, records its code in the
// status word and the kernel returns.  Nothing is in flight while it waits.
__device__ uint32_t g_probe_counter;

__global__ void wait_probe_kernel(int kind, unsigned long long limit_ns, uint32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  if (kind == 0) {
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    wait_bar(b, 0, &abort_flag, status, ST_TIMEOUT, limit_ns);
  } else {
    g_probe_counter = 0;
    __threadfence();
    grid_barrier(&g_probe_counter, 2, status, limit_ns);   // a second CTA that does not exist
  }
}

// bf16 bit pattern of an integer code in [-128, 127] (exact): the top half
// of its fp32 image, formed without a conversion instruction.
__device__ __forceinline__ uint32_t code_bits(int c) {
  return __float_as_uint(__fsub_rn(__int_as_float(0x4B400000 + c), 12582912.0f)) >> 16;
}

// A wait expected to last microseconds: as wait_bar, but the thread sleeps
// between polls, so that the producer and MMA threads sharing its
// sub-partition keep their issue slots.
__device__ __forceinline__ bool wait_bar_idle(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                              uint32_t* status) {
  unsigned long long t0 = 0;
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    __nanosleep(32);
    if ((i & 15u) == 15u) {
      if (*abort_flag) return false;
      const unsigned long long now = global_ns();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > WAIT_LIMIT_NS) {
        atomicOr(status, ST_TIMEOUT);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, %0;\n" ::"n"(EPI_WARPS * 32) : "memory"); }

template <bool VAR>
__global__ void __launch_bounds__(THREADS, 1)
lstm_persist_kernel(const __grid_constant__ CUtensorMap tmR, const __grid_constant__ CUtensorMap tmH, Params p) {
  constexpr uint32_t IDESC = idesc_bf16(BM, BN);
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned, indexed from the shared array itself so that accesses stay shared-space
  uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  const int KT = p.Hp / BK;
  uint8_t* rtile = smem + STAGES * A_STAGE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(rtile + (size_t)KT * R_SLAB);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  __shared__ float cst[4][BN];           // Rcs (as int), Rsc, Wbi, Rbi of the tile's 64 gate rows
  __shared__ float pw[3][16];            // peepholes i, o, f of the tile's units
  __shared__ float red[4][2][64];        // per column group: min, max of h per batch row
  __shared__ int gok;
  const uint32_t smem0 = smem_u32(smem);
  auto sA = [&](int st) { return smem0 + (uint32_t)(st * A_STAGE); };
  const uint32_t sR = smem_u32(rtile);
  auto full = [&](int st) { return smem_u32(bars + st); };
  auto empty = [&](int st) { return smem_u32(bars + STAGES + st); };
  const uint32_t accf = smem_u32(bars + 2 * STAGES), acce = smem_u32(bars + 2 * STAGES + 1);
  const uint32_t rbar = smem_u32(bars + 2 * STAGES + 2), hready = smem_u32(bars + 2 * STAGES + 3);
  const uint32_t mdone = smem_u32(bars + 2 * STAGES + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = blockIdx.x / p.tiles, g = blockIdx.x % p.tiles;
  const int H4 = 4 * p.H;
  const int nchunks = (KT + p.CS - 1) / p.CS;
  const int64_t DB = (int64_t)p.D * p.B;
  const uint32_t nctas = (uint32_t)p.tiles;  // CTAs of this direction
  uint32_t* dbar = p.gbar + d;

  if (threadIdx.x == 0) {
    for (int st = 0; st < STAGES; ++st) {
      mbar_init(full(st), 1);
      mbar_init(empty(st), 1);
    }
    mbar_init(accf, 1);
    mbar_init(acce, EPI_WARPS);
    mbar_init(rbar, 1);
    mbar_init(hready, 1);
    mbar_init(mdone, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  for (int i = threadIdx.x; i < BN; i += THREADS) {
    const int64_t dn = (int64_t)d * H4 + g * BN + i;
    cst[0][i] = __int_as_float(__ldg(p.Rcs + dn));
    cst[1][i] = __ldg(p.Rsc + dn);
    cst[2][i] = __ldg(p.Wbi + dn);
    cst[3][i] = __ldg(p.Rbi + dn);
  }
  if (VAR && threadIdx.x < 48) {
    const int k = threadIdx.x / 16, ul = threadIdx.x % 16;
    pw[k][ul] = p.P ? __ldg(p.P + (int64_t)d * 3 * p.H + k * p.H + g * 16 + ul) : 0.0f;
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      bool ok = true;
      mbar_arrive_expect_tx(rbar, (uint32_t)(KT * R_SLAB));
      for (int kt = 0; kt < KT; ++kt) tma_load_2d(sR + (uint32_t)(kt * R_SLAB), &tmR, rbar, kt * BK, d * H4 + g * BN);
      // stage st, round parity ph (counters, no division in the loop)
      uint32_t st = 0, ph = 0, it = 0;
      for (int s = 0; ok && s < p.T; ++s) {
        if (s > 0) {
          if (!wait_bar_idle(hready, (uint32_t)(s - 1) & 1u, abort_flag, p.status)) break;
          // the codes were written by other CTAs' generic stores
          asm volatile("fence.proxy.async.global;\n" ::: "memory");
        }
        const int y = (int)((((s + 1) & 1) * DB) + (int64_t)d * p.B);
        for (int kt = 0; kt < KT; ++kt, ++it) {
          if (!wait_bar(empty(st), ph ^ 1u, abort_flag, p.status, ST_TIMEOUT)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full(st), (uint32_t)A_STAGE);
          tma_load_2d(sA(st), &tmH, full(st), kt * BK, y);
          if (++st == (uint32_t)STAGES) {
            st = 0;
            ph ^= 1u;
          }
        }
      }
      // the copies in flight land before the CTA leaves (bounded)
      const uint32_t first = it > (uint32_t)STAGES ? it - STAGES : 0u;
      for (uint32_t i = first; i < it; ++i) {
        const unsigned long long t0 = global_ns();
        while (!mbar_try_wait(full(i % STAGES), (i / STAGES) & 1u))
          if (global_ns() - t0 > WAIT_LIMIT_NS) break;
      }
      {
        const unsigned long long t0 = global_ns();
        while (!mbar_try_wait(rbar, 0))
          if (global_ns() - t0 > WAIT_LIMIT_NS) break;
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      bool ok = wait_bar(rbar, 0, abort_flag, p.status, ST_TIMEOUT);
      tc_fence_after();
      // counters instead of division: stage st, round parity ph, chunk
      // step kc; descriptors advanced by addition (start address >> 4)
      const uint64_t adesc0 = desc_sw128(sA(0)), bdesc0 = desc_sw128(sR);
      uint32_t st = 0, ph = 0, chunk = 0;
      if (KT % STAGES == 0 && p.CS >= KT) {
        // K a multiple of 512 with one exact chunk per step (K = 1024 at the
        // full size): every step starts at stage 0 and slab r * 8 + j sits in
        // stage j, so the issue loop is unrolled over the ring with constant
        // stage offsets and a phase that turns once per round
        uint32_t ph = 0;
        for (int s = 0; ok && s < p.T; ++s) {
          if (!wait_bar(acce, ((uint32_t)s & 1u) ^ 1u, abort_flag, p.status, ST_TIMEOUT)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int r = 0; ok && r < KT / STAGES; ++r) {
            const uint64_t bround = bdesc0 + (uint64_t)(((uint32_t)r * STAGES * R_SLAB) >> 4);
#pragma unroll
            for (int j = 0; j < STAGES; ++j) {
              if (!wait_bar(full(j), ph, abort_flag, p.status, ST_TIMEOUT)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t ad = adesc0 + (uint64_t)((j * A_STAGE) >> 4);
              const uint64_t bd = bround + (uint64_t)((j * R_SLAB) >> 4);
              const uint32_t acc = (r > 0 || j > 0) ? 1u : 0u;
#pragma unroll
              for (int k = 0; k < BK / 16; ++k)
                tc_mma(tmem + (uint32_t)((k % NACC) * BN), ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), IDESC,
                       (acc || k >= NACC) ? 1u : 0u);
              tc_commit(empty(j));
            }
            ph ^= 1u;
          }
          if (ok) tc_commit(accf);
        }
      }
      for (int s = 0; ok && s < p.T && !(KT % STAGES == 0 && p.CS >= KT); ++s) {
        int kc = 0;
        for (int kt = 0; kt < KT; ++kt) {
          if (kc == 0) {
            if (!wait_bar(acce, (chunk & 1u) ^ 1u, abort_flag, p.status, ST_TIMEOUT)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          if (!wait_bar(full(st), ph, abort_flag, p.status, ST_TIMEOUT)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = adesc0 + (uint64_t)((st * (uint32_t)A_STAGE) >> 4);
          const uint64_t bd = bdesc0 + (uint64_t)(((uint32_t)kt * (uint32_t)R_SLAB) >> 4);
          const uint32_t acc = kc == 0 ? 0u : 1u;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            tc_mma(tmem + (uint32_t)((k % NACC) * BN), ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), IDESC,
                   (acc || k >= NACC) ? 1u : 0u);
          tc_commit(empty(st));
          if (++kc == p.CS || kt == KT - 1) {
            tc_commit(accf);
            ++chunk;
            kc = 0;
          }
          if (++st == (uint32_t)STAGES) {
            st = 0;
            ph ^= 1u;
          }
        }
      }
      // every product issued has completed before TMEM is freed (bounded)
      tc_commit(mdone);
      const unsigned long long t0 = global_ns();
      while (!mbar_try_wait(mdone, 0))
        if (global_ns() - t0 > WAIT_LIMIT_NS) break;
    }
  } else {
    // ---------------- epilogue ----------------
    // sub-partition qd holds batch rows 16 qd .. 16 qd + 15 in its lanes
    // 0..15; lane t and lane t + 16 take row 16 qd + (t mod 16), units
    // 2 hi, 2 hi + 1 of the column group cg (hi = t >= 16)
    const int qd = warp & 3, cg = (warp - 2) >> 2, hi = lane >> 4;
    const int b = qd * 16 + (lane & 15);
    const bool bvalid = b < p.B;
    const int u0 = g * 16 + 4 * cg + 2 * hi;  // first of this thread's 2 units
    const int col0 = 16 * cg + 8 * hi;        // its first gate column in the tile
    const bool rev = p.direction == I8Q_LSTM_REVERSE || (p.direction == I8Q_LSTM_BIDIRECTIONAL && d == 1);
    const int64_t TB = (int64_t)p.T * p.B;
    const int64_t row = (int64_t)d * p.B + b;  // state row
    int L = p.T;
    if (VAR && bvalid && p.seq_lens) L = min(max(__ldg(p.seq_lens + b), 0), p.T);  // lengths outside [0, T] clamp
    uint32_t chunk = 0;
    bool ok = true;
    for (int s = 0; s < p.T; ++s) {
      const bool live = bvalid && s < L;
      const int tb = rev ? L - 1 - s : s;  // for VAR rows, within the row's own length
      const int t = VAR ? tb : (rev ? p.T - 1 - s : s);
      const float* hprev = p.hbuf + (int64_t)(s & 1) * DB * p.H;
      float* hnext = p.hbuf + (int64_t)((s + 1) & 1) * DB * p.H;
      const int prv = (s + 1) & 1, cur = s & 1;
      // operands that do not depend on the product
      float gx[8], cp[2], hp[2];
#pragma unroll
      for (int i = 0; i < 8; ++i) gx[i] = 0.0f;
      cp[0] = cp[1] = hp[0] = hp[1] = 0.0f;
      float shb = 0.0f;
      int zhb = 0;
      if (live) {
        const float4* gsrc = reinterpret_cast<const float4*>(p.Gx + ((int64_t)d * TB + (int64_t)t * p.B + b) * H4 +
                                                             g * BN + col0);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const float4 v = __ldg(gsrc + k);
          gx[4 * k] = v.x; gx[4 * k + 1] = v.y; gx[4 * k + 2] = v.z; gx[4 * k + 3] = v.w;
        }
        const float2 c2 = *reinterpret_cast<const float2*>(p.c + row * p.H + u0);
        cp[0] = c2.x; cp[1] = c2.y;
        shb = __ldcg(p.sh + prv * DB + row);  // written by another CTA in the previous step
        zhb = __ldcg(p.zh + prv * DB + row);
      } else if (bvalid) {
        const float2 h2 = *reinterpret_cast<const float2*>(hprev + row * p.H + u0);
        hp[0] = h2.x; hp[1] = h2.y;
      }
      // the exact sums of this step
      int32_t run[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) run[i] = 0;
      for (int c = 0; c < nchunks; ++c, ++chunk) {
        const bool got = ok && wait_bar_idle(accf, chunk & 1u, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int a = 0; a < NACC; ++a) {
          uint32_t v[16];
          tmem_ld16(tmem + ((uint32_t)(qd * 32) << 16) + (uint32_t)(a * BN + 16 * cg), v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t up = __shfl_sync(0xffffffffu, v[8 + i], lane & 15);
            run[i] += __float2int_rn(__uint_as_float(hi ? up : v[i]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce);
      }
      // cell update of the 2 units (the operation order of the per-step kernels)
      float hn[2] = {hp[0], hp[1]};
      if (ok && live) {
        float pre[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          // h entered as uh - 128: sum_k (uh - zh) R = run - (zh - 128) colsum
          const int32_t v = run[i] - (zhb - 128) * __float_as_int(cst[0][col0 + i]);
          float gh = __fmul_rn(__int2float_rn(v), shb);
          gh = __fmul_rn(gh, cst[1][col0 + i]);
          pre[i] = __fadd_rn(gx[i], gh);
        }
#pragma unroll
        if (!VAR) {
          // the two units' gates in pairs (the per-lane operations of sigmoid32 and tanh32)
          float gi[2], go[2], gf[2], gc[2];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int c0 = col0 + 4 * k;  // gate columns of unit k: i, o, f, c
            gi[k] = __fadd_rn(__fadd_rn(pre[4 * k], cst[2][c0]), cst[3][c0]);
            go[k] = __fadd_rn(__fadd_rn(pre[4 * k + 1], cst[2][c0 + 1]), cst[3][c0 + 1]);
            gf[k] = __fadd_rn(__fadd_rn(pre[4 * k + 2], cst[2][c0 + 2]), cst[3][c0 + 2]);
            gc[k] = __fadd_rn(__fadd_rn(pre[4 * k + 3], cst[2][c0 + 3]), cst[3][c0 + 3]);
          }
          const float2 ig = ef::sigmoid32x2(make_float2(gi[0], gi[1]));
          const float2 og = ef::sigmoid32x2(make_float2(go[0], go[1]));
          const float2 fg = ef::sigmoid32x2(make_float2(gf[0], gf[1]));
          const float2 ct = ef::tanh32x2(make_float2(gc[0], gc[1]));
          const float cn0 = __fadd_rn(__fmul_rn(fg.x, cp[0]), __fmul_rn(ig.x, ct.x));
          const float cn1 = __fadd_rn(__fmul_rn(fg.y, cp[1]), __fmul_rn(ig.y, ct.y));
          const float2 th = ef::tanh32x2(make_float2(cn0, cn1));
          hn[0] = __fmul_rn(og.x, th.x);
          hn[1] = __fmul_rn(og.y, th.y);
          cp[0] = cn0;
          cp[1] = cn1;
        }
#pragma unroll
        for (int k = 0; k < 2 && VAR; ++k) {
          // the general form: peepholes, clip, coupled gates, the activation list
          const int c0 = col0 + 4 * k;  // gate columns of unit k: i, o, f, c
          float si = pre[4 * k], so = pre[4 * k + 1], sf = pre[4 * k + 2], sc = pre[4 * k + 3];
          float cn, og;
          {
            const int ul = 4 * cg + 2 * hi + k;
            if (p.P) {
              si = __fadd_rn(si, __fmul_rn(pw[0][ul], cp[k]));
              sf = __fadd_rn(sf, __fmul_rn(pw[2][ul], cp[k]));
            }
            const int fk = p.acts.kind[d][0], gk = p.acts.kind[d][1];
            const float fa = p.acts.alpha[d][0], fb = p.acts.beta[d][0];
            const float ig = ef::lstm_act(fk, fa, fb, clip_gate(__fadd_rn(__fadd_rn(si, cst[2][c0]), cst[3][c0]), p.clip));
            const float fg =
                p.input_forget
                    ? __fsub_rn(1.0f, ig)
                    : ef::lstm_act(fk, fa, fb, clip_gate(__fadd_rn(__fadd_rn(sf, cst[2][c0 + 2]), cst[3][c0 + 2]), p.clip));
            const float ct = ef::lstm_act(gk, p.acts.alpha[d][1], p.acts.beta[d][1],
                                          clip_gate(__fadd_rn(__fadd_rn(sc, cst[2][c0 + 3]), cst[3][c0 + 3]), p.clip));
            cn = __fadd_rn(__fmul_rn(fg, cp[k]), __fmul_rn(ig, ct));
            if (p.P) so = __fadd_rn(so, __fmul_rn(pw[1][ul], cn));
            og = ef::lstm_act(fk, fa, fb, clip_gate(__fadd_rn(__fadd_rn(so, cst[2][c0 + 1]), cst[3][c0 + 1]), p.clip));
            hn[k] = __fmul_rn(og, ef::lstm_act(p.acts.kind[d][2], p.acts.alpha[d][2], p.acts.beta[d][2], cn));
          }
          cp[k] = cn;
        }
        *reinterpret_cast<float2*>(p.c + row * p.H + u0) = make_float2(cp[0], cp[1]);
        if (p.Y)
          *reinterpret_cast<float2*>(p.Y + (((int64_t)t * p.D + d) * p.B + b) * p.H + u0) = make_float2(hn[0], hn[1]);
      }
      if (ok && bvalid) *reinterpret_cast<float2*>(hnext + row * p.H + u0) = make_float2(hn[0], hn[1]);
      // per-row min / max of the new h over this CTA's 16 units
      float mn = fminf(hn[0], hn[1]), mx = fmaxf(hn[0], hn[1]);
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, 16));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      if (!hi) {
        red[cg][0][b] = mn;
        red[cg][1][b] = mx;
      }
      epi_sync();
      if (cg == 0 && !hi && ok && bvalid) {
        mn = fminf(fminf(red[0][0][b], red[1][0][b]), fminf(red[2][0][b], red[3][0][b]));
        mx = fmaxf(fmaxf(red[0][1][b], red[1][1][b]), fmaxf(red[2][1][b], red[3][1][b]));
        atomicMax(p.mm + (cur * DB + row) * 2, ord_image(-mn));
        atomicMax(p.mm + (cur * DB + row) * 2 + 1, ord_image(mx));
      }
      epi_sync();
      if (warp == 2 && lane == 0) gok = ok && grid_barrier(dbar, nctas * (uint32_t)(2 * s + 1), p.status);
      epi_sync();
      ok = ok && gok;
      // the row's scale and zero point (the same in every CTA), this CTA's codes
      if (ok && bvalid) {
        const uint32_t* m2 = p.mm + (cur * DB + row) * 2;
        const float rmn = fminf(-ord_value(__ldcg(m2)), 0.0f), rmx = fmaxf(ord_value(__ldcg(m2 + 1)), 0.0f);
        float sc;
        int z;
        row_scale_zero(rmn, rmx, sc, z);
        const float lo_z = (float)(-z), hi_z = (float)(255 - z);
        const int c0 = (int)(row_code(hn[0], sc, lo_z, hi_z, z)) - 128;
        const int c1 = (int)(row_code(hn[1], sc, lo_z, hi_z, z)) - 128;
        *reinterpret_cast<uint32_t*>(p.uhc + (cur * DB + row) * p.Hp + u0) = code_bits(c0) | (code_bits(c1) << 16);
        if (g == 0 && cg == 0 && !hi) {
          p.sh[cur * DB + row] = sc;
          p.zh[cur * DB + row] = z;
        }
      }
      // the next step's min/max pairs of this direction start empty
      if (ok && g == 0) {
        const int e = threadIdx.x - 64;  // 0 .. 511 over the epilogue warps
        for (int64_t i = e; i < 2 * p.B; i += EPI_WARPS * 32) p.mm[((int64_t)prv * DB + (int64_t)d * p.B) * 2 + i] = 0u;
      }
      epi_sync();
      if (warp == 2 && lane == 0) {
        gok = ok && grid_barrier(dbar, nctas * (uint32_t)(2 * s + 2), p.status);
        if (gok) mbar_arrive(hready);
        else *abort_flag = 1;
      }
      epi_sync();
      ok = ok && gok;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace prs

int grid_for(int64_t n, int threads = 256) {
  return (int)std::max<int64_t>(1, std::min<int64_t>(ceil_div(n, threads), (int64_t)sm_count() * 8));
}

bool lstm_use_tc(int64_t rows, int64_t cols) {
  const char* f = getenv("I8Q_FORCE_CORE");
  if (f && std::string(f) == "imma") return false;
  if (f && std::string(f) == "tc") return true;
  return rows >= 128 && cols >= 256 && ((rows + 127) / 128) * ((cols + 255) / 256) >= 64;
}

}  // namespace

// The arguments that fix a captured recurrence (every field 8 bytes wide,
// so the struct has no padding and compares with memcmp).
struct LstmGraphKey {
  const void *X, *W, *R, *W_scale, *R_scale, *Bias, *h0, *c0, *Y, *Y_h, *Y_c, *workspace;
  const void *W_zero_point, *R_zero_point, *seq_lens, *P;
  int64_t T, batch, input, hidden, direction, n_wscale, n_rscale, wtype, input_forget, clip_bits;
  int64_t act_kinds;      // the six activation kinds, 4 bits each
  int64_t act_params[6];  // alpha, beta bit patterns of each
};

// Launch the recurrence as a CUDA graph on s: the cached one when key
// matches, else capture `issue` on s and instantiate (or update) it.
int run_cached_graph(const LstmGraphKey& key, cudaStream_t s, const std::function<int()>& issue);

}  // namespace i8q

using namespace i8q;

extern "C" size_t i8q_dq_lstm_workspace_size(int64_t T, int64_t batch, int64_t input, int64_t hidden, int direction) {
  if (T <= 0 || batch <= 0 || input <= 0 || hidden <= 0) return 0;
  if (direction < I8Q_LSTM_FORWARD || direction > I8Q_LSTM_BIDIRECTIONAL) return 0;
  return lstm_layout(T, batch, input, hidden, direction).total;
}

namespace {

// The activations attribute (3 per direction: f, g, h; or none, for
// Sigmoid, Tanh, Tanh) with the activation_alpha / activation_beta lists,
// which are consumed in the order of the functions: each function that
// takes an alpha (beta) takes the next unused value, or its operator's
// default once the list runs out.  Sets nondefault when any function
// differs from the defaults.
int resolve_activations(const int* kinds, size_t n_kinds, const float* alpha, size_t n_alpha, const float* beta,
                        size_t n_beta, int64_t D, LstmActs& out, bool& nondefault) {
  struct Def {
    bool has_a;
    float a;
    bool has_b;
    float b;
  };
  // indexed by I8Q_LSTM_ACT_*: the ONNX operators' defaults (LeakyRelu
  // 0.01 as the DynamicQuantizeLSTM pages state); ScaledTanh's operator
  // names none, and 1, 1 make it Tanh
  static const Def defs[11] = {{false, 0, false, 0}, {false, 0, false, 0}, {false, 0, false, 0},
                               {true, 1.0f, true, 0.0f},  {true, 0.01f, false, 0}, {true, 1.0f, false, 0},
                               {true, 1.0f, true, 1.0f},  {true, 0.2f, true, 0.5f}, {true, 1.0f, false, 0},
                               {false, 0, false, 0},      {false, 0, false, 0}};
  static const int dflt[3] = {I8Q_LSTM_ACT_SIGMOID, I8Q_LSTM_ACT_TANH, I8Q_LSTM_ACT_TANH};
  nondefault = false;
  if (n_kinds != 0 && (int64_t)n_kinds != 3 * D)
    return fail(I8Q_ERR_INVALID_ARG, "dq_lstm: activations needs 3 entries per direction (or none)");
  if (n_kinds && !kinds) return fail(I8Q_ERR_INVALID_ARG, "dq_lstm: activations is NULL");
  if ((n_alpha && !alpha) || (n_beta && !beta)) return fail(I8Q_ERR_INVALID_ARG, "dq_lstm: alpha / beta list is NULL");
  size_t ia = 0, ib = 0;
  for (int d = 0; d < 2; ++d)
    for (int k = 0; k < 3; ++k) {
      out.kind[d][k] = dflt[k];
      out.alpha[d][k] = out.beta[d][k] = 0.0f;
    }
  for (int64_t d = 0; d < D; ++d)
    for (int k = 0; k < 3; ++k) {
      const int kind = n_kinds ? kinds[3 * d + k] : dflt[k];
      if (kind < I8Q_LSTM_ACT_RELU || kind > I8Q_LSTM_ACT_SOFTPLUS)
        return fail(I8Q_ERR_INVALID_ARG, "dq_lstm: unknown activation " + std::to_string(kind));
      const Def& df = defs[kind];
      out.kind[d][k] = kind;
      if (df.has_a) out.alpha[d][k] = ia < n_alpha ? alpha[ia++] : df.a;
      if (df.has_b) out.beta[d][k] = ib < n_beta ? beta[ib++] : df.b;
      if (!(out.alpha[d][k] == out.alpha[d][k]) || !(out.beta[d][k] == out.beta[d][k]))
        return fail(I8Q_ERR_INVALID_ARG, "dq_lstm: activation alpha / beta is NaN");
      if (kind != dflt[k]) nondefault = true;
    }
  return I8Q_OK;
}

int lstm_forward_impl(const float* X, int64_t T, int64_t batch, int64_t input, int64_t hidden, int direction,
                      const void* W_, const void* R_, int wtype, const float* W_scale, const void* W_zero_point_,
                      size_t n_wscale, const float* R_scale, const void* R_zero_point_, size_t n_rscale,
                      const float* Bias, const int32_t* seq_lens, const float* h0, const float* c0, const float* P,
                      float clip, int input_forget, const LstmActs& acts, bool acts_nondefault, float* Y, float* Y_h,
                      float* Y_c, void* workspace, size_t ws_bytes, void* stream) {
  const int8_t* W = static_cast<const int8_t*>(W_);
  const int8_t* R = static_cast<const int8_t*>(R_);
  const int8_t* W_zero_point = static_cast<const int8_t*>(W_zero_point_);
  const int8_t* R_zero_point = static_cast<const int8_t*>(R_zero_point_);
  if (wtype != I8Q_S8 && wtype != I8Q_U8) return fail(I8Q_ERR_INVALID_ARG, "dq_lstm: W and R must be I8Q_S8 or I8Q_U8");
  if (!(clip == clip)) return fail(I8Q_ERR_INVALID_ARG, "dq_lstm: clip is NaN");
  if (T <= 0 || batch <= 0 || input <= 0 || hidden <= 0)
    return fail(I8Q_ERR_INVALID_ARG, "dq_lstm: T, batch, input, hidden must be positive");
  if (direction < I8Q_LSTM_FORWARD || direction > I8Q_LSTM_BIDIRECTIONAL)
    return fail(I8Q_ERR_INVALID_ARG, "dq_lstm: bad direction");
  if (!X || !W || !R || !W_scale || !R_scale) return fail(I8Q_ERR_INVALID_ARG, "dq_lstm: NULL tensor pointer");
  if (input > 65536 || hidden > 65536) return fail(I8Q_ERR_UNSUPPORTED, "dq_lstm: input/hidden > 65536");
  if (T * batch > ((int64_t)1 << 31) - 1) return fail(I8Q_ERR_UNSUPPORTED, "dq_lstm: T * batch too large");
  const LstmLayout L = lstm_layout(T, batch, input, hidden, direction);
  if ((int64_t)n_wscale != L.D && (int64_t)n_wscale != L.D * L.H4)
    return fail(I8Q_ERR_INVALID_ARG, "dq_lstm: W_scale must have D or D*4H entries");
  if ((int64_t)n_rscale != L.D && (int64_t)n_rscale != L.D * L.H4)
    return fail(I8Q_ERR_INVALID_ARG, "dq_lstm: R_scale must have D or D*4H entries");
  if (!workspace || ws_bytes < L.total) return fail(I8Q_ERR_INVALID_ARG, "dq_lstm: workspace missing or too small");
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return fail(I8Q_ERR_INVALID_ARG, "dq_lstm: workspace not 256-byte aligned");
  cudaStream_t s = as_stream(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int8_t* Wt = (int8_t*)(ws + L.off_Wt);
  __nv_bfloat16* Wtb = (__nv_bfloat16*)(ws + L.off_Wtb);
  int32_t* Wcs = (int32_t*)(ws + L.off_Wcs);
  int8_t* Rt = (int8_t*)(ws + L.off_Rt);
  __nv_bfloat16* Rtb = (__nv_bfloat16*)(ws + L.off_Rtb);
  int32_t* Rcs = (int32_t*)(ws + L.off_Rcs);
  float* Wsc = (float*)(ws + L.off_Wsc);
  float* Rsc = (float*)(ws + L.off_Rsc);
  float* Wbi = (float*)(ws + L.off_Wbi);
  float* Rbi = (float*)(ws + L.off_Rbi);
  uint8_t* uX = ws + L.off_uX;
  __nv_bfloat16* uXc = (__nv_bfloat16*)(ws + L.off_uXc);
  float* sX = (float*)(ws + L.off_sX);
  int32_t* zX = (int32_t*)(ws + L.off_zX);
  float* Gx = (float*)(ws + L.off_Gx);
  uint8_t* uh = ws + L.off_uh;
  __nv_bfloat16* uhc = (__nv_bfloat16*)(ws + L.off_uhc);
  float* sh = (float*)(ws + L.off_sh);
  int32_t* zh = (int32_t*)(ws + L.off_zh);
  uint32_t* mmb = (uint32_t*)(ws + L.off_mm);
  uint32_t* gbar = (uint32_t*)(ws + L.off_gbar);
  float* hbuf = (float*)(ws + L.off_h);
  float* cbuf = (float*)(ws + L.off_c);
  const int64_t H = hidden, BH = batch * hidden, DBH = L.D * BH, DB = L.D * batch;

  // The general form (uint8 weights, zero points, sequence lengths,
  // peepholes, clip, coupled gates) runs on the tensor-core kernels: the
  // weights enter as bf16 W - zp (|W - zp| <= 255), so products stay within
  // 2^15 and the exact fp32 chunks hold 512 K-elements.  int8 weights whose
  // given zero points are all 0 (checked on the device, reported
  // synchronously) keep the plain form.
  bool var = wtype != I8Q_S8 || seq_lens || P || clip > 0.0f || input_forget || acts_nondefault;
  if (!var && (W_zero_point || R_zero_point)) {
    int* flag = reinterpret_cast<int*>(sh);  // scratch word, overwritten later
    I8Q_CUDA_TRY(cudaMemsetAsync(flag, 0, sizeof(int), s));
    if (W_zero_point) any_nonzero_s8<<<grid_for((int64_t)n_wscale), 256, 0, s>>>(W_zero_point, (int64_t)n_wscale, flag);
    if (R_zero_point) any_nonzero_s8<<<grid_for((int64_t)n_rscale), 256, 0, s>>>(R_zero_point, (int64_t)n_rscale, flag);
    int hflag = 0;
    I8Q_CUDA_TRY(cudaMemcpyAsync(&hflag, flag, sizeof(int), cudaMemcpyDeviceToHost, s));
    I8Q_CUDA_TRY(cudaStreamSynchronize(s));
    var = hflag != 0;
  }

  // weights: gate-interleaved K-major copies, column sums, scales, biases
  const bool tc = var || lstm_use_tc(L.TB, L.H4);
  // recurrent product on the tensor pipe when the step has enough gate
  // rows to spread (or when forced); exact chunks need |uh - 128| * |R| <= 2^14
  const char* force = getenv("I8Q_FORCE_CORE");
  const bool step_tc = var || (force ? std::string(force) == "tc" : (L.H4 >= 1024));
  const int prod_log2 = var ? 15 : 14;
  int rc;
  for (int64_t d = 0; d < L.D; ++d) {
    if (var) {
      const auto* zw = reinterpret_cast<const uint8_t*>(W_zero_point);
      const auto* zr = reinterpret_cast<const uint8_t*>(R_zero_point);
      const int64_t nzw = (int64_t)n_wscale == L.D ? 1 : L.H4, nzr = (int64_t)n_rscale == L.D ? 1 : L.H4;
      const auto* Wd = reinterpret_cast<const uint8_t*>(W) + d * input * L.H4;
      const auto* Rd = reinterpret_cast<const uint8_t*>(R) + d * H * L.H4;
      const unsigned blocks = (unsigned)ceil_div(L.H4, 32);
      I8Q_PROF("repack_cols", s);
      if (wtype == I8Q_S8) {
        repack_gates_zp<true><<<blocks, 256, 0, s>>>(Wd, input, H, zw ? zw + d * nzw : nullptr, nzw, L.Ip,
                                                     Wtb + d * L.H4 * L.Ip, Wcs + d * L.H4);
        repack_gates_zp<true><<<blocks, 256, 0, s>>>(Rd, H, H, zr ? zr + d * nzr : nullptr, nzr, L.Hp,
                                                     Rtb + d * L.H4 * L.Hp, Rcs + d * L.H4);
      } else {
        repack_gates_zp<false><<<blocks, 256, 0, s>>>(Wd, input, H, zw ? zw + d * nzw : nullptr, nzw, L.Ip,
                                                      Wtb + d * L.H4 * L.Ip, Wcs + d * L.H4);
        repack_gates_zp<false><<<blocks, 256, 0, s>>>(Rd, H, H, zr ? zr + d * nzr : nullptr, nzr, L.Hp,
                                                      Rtb + d * L.H4 * L.Hp, Rcs + d * L.H4);
      }
      I8Q_LAUNCH_CHECK("repack_gates_zp");
      continue;
    }
    rc = launch_repack_cols_s8_gates(W + d * input * L.H4, input, L.H4, L.H4, Wt + d * L.H4 * L.Ip,
                                     tc ? Wtb + d * L.H4 * L.Ip : nullptr, L.Ip, Wcs + d * L.H4, H, s);
    if (rc) return rc;
    rc = launch_repack_cols_s8_gates(R + d * H * L.H4, H, L.H4, L.H4, Rt + d * L.H4 * L.Hp,
                                     step_tc ? Rtb + d * L.H4 * L.Hp : nullptr, L.Hp, Rcs + d * L.H4, H, s);
    if (rc) return rc;
  }
  interleave_scales<<<grid_for(L.D * L.H4), 256, 0, s>>>(W_scale, (int64_t)n_wscale, L.D, H, Wsc);
  interleave_scales<<<grid_for(L.D * L.H4), 256, 0, s>>>(R_scale, (int64_t)n_rscale, L.D, H, Rsc);
  interleave_bias<<<grid_for(L.D * L.H4), 256, 0, s>>>(Bias, L.D, H, Wbi, Rbi);
  I8Q_LAUNCH_CHECK("lstm parameter layout");

  // input projection: X quantized once, one GEMM per direction
  rc = launch_quantize_rows(X, I8Q_F32, L.TB, input, input, uX, tc ? uXc : nullptr, L.Ip, sX, zX, s);
  if (rc) return rc;
  for (int64_t d = 0; d < L.D; ++d) {
    GemmEpilogue ep{zX, sX, Wcs + d * L.H4, Wsc + d * L.H4, nullptr, I8Q_ACT_IDENTITY, OUT_F32,
                    Gx + d * L.TB * L.H4, L.H4};
    rc = I8Q_ERR_UNSUPPORTED;
    if (tc) rc = launch_gemm_tc(uXc, Wtb + d * L.H4 * L.Ip, L.TB, L.H4, L.Ip, prod_log2, ep, s);
    if (rc == I8Q_ERR_UNSUPPORTED && !var)
      rc = launch_gemm_imma(uX, Wt + d * L.H4 * L.Ip, L.TB, L.H4, L.Ip, ep, s);
    if (rc) return rc;
  }

  // tensor maps of the step on the tensor pipe
  CUtensorMap mR, mH;
  if (step_tc) {
    rc = tc::make_map_2d(&mR, Rtb, L.D * L.H4, L.Hp, tcs::BM, "dq_lstm");
    if (rc) return rc;
    rc = tc::make_map_2d(&mH, uhc, 2 * L.D * batch, L.Hp, tcs::BN, "dq_lstm");
    if (rc) return rc;
    rc = smem_attr((const void*)tcs::lstm_step_tc_kernel<false>, tcs::SMEM_BYTES);
    if (!rc) rc = smem_attr((const void*)tcs::lstm_step_tc_kernel<true>, tcs::SMEM_BYTES);
    if (rc) return rc;
  }

  // the persistent recurrence: every CTA resident at once (one per SM),
  // at most 64 batch rows, whole 16-unit tiles
  bool persist = false;
  CUtensorMap mR64, mH2;
  const int ptiles = (int)(H / 16);
  const size_t psmem = prs::smem_bytes(L.Hp);
  if (step_tc && batch <= 64 && H % 16 == 0 && (reinterpret_cast<uintptr_t>(Y) & 15) == 0 &&
      !getenv("I8Q_LSTM_STEPS")) {
    int dev = 0, coop = 0;
    I8Q_CUDA_TRY(cudaGetDevice(&dev));
    I8Q_CUDA_TRY(cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev));
    const int most = 227 * 1024 - 4096;
    rc = smem_attr((const void*)prs::lstm_persist_kernel<false>, most);
    if (!rc) rc = smem_attr((const void*)prs::lstm_persist_kernel<true>, most);
    if (rc) return rc;
    int per_sm = 0;
    if (coop && psmem <= (size_t)(227 * 1024 - 4096)) {
      I8Q_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &per_sm, var ? prs::lstm_persist_kernel<true> : prs::lstm_persist_kernel<false>, prs::THREADS, psmem));
    }
    persist = per_sm >= 1 && L.D * ptiles <= (int64_t)per_sm * sm_count();
    if (persist) {
      rc = tc::make_map_2d(&mR64, Rtb, L.D * L.H4, L.Hp, prs::BN, "dq_lstm");
      if (rc) return rc;
      rc = tc::make_map_2d(&mH2, uhc, 2 * L.D * batch, L.Hp, prs::BN, "dq_lstm");
      if (rc) return rc;
    }
  }

  // recurrence: both directions per launch, 2 launches per step
  auto recurrence = [&]() -> int {
    init_state<<<grid_for(DBH), 256, 0, s>>>(h0, c0, DBH, hbuf, cbuf);
    I8Q_LAUNCH_CHECK("init_state");
    // rows whose sequence ends early leave the rest of Y zero
    if (Y && seq_lens) I8Q_CUDA_TRY(cudaMemsetAsync(Y, 0, (size_t)T * DBH * sizeof(float), s));
    if (persist) {
      // h0's codes go to parity 1, which step 0 reads; the padding columns
      // of both parities stay zero
      I8Q_CUDA_TRY(cudaMemsetAsync(uhc, 0, (size_t)2 * L.D * batch * L.Hp * 2, s));
      I8Q_CUDA_TRY(cudaMemsetAsync(mmb, 0, (size_t)2 * L.D * batch * 2 * 4, s));
      I8Q_CUDA_TRY(cudaMemsetAsync(gbar, 0, 2 * 4, s));
      int rcp = launch_quantize_rows(hbuf, I8Q_F32, DB, H, H, uh + DB * L.Hp, uhc + DB * L.Hp, L.Hp, sh + DB,
                                     zh + DB, s);
      if (rcp) return rcp;
      prs::Params pp;
      pp.Rcs = Rcs;
      pp.Rsc = Rsc;
      pp.Gx = Gx;
      pp.Wbi = Wbi;
      pp.Rbi = Rbi;
      pp.c = cbuf;
      pp.hbuf = hbuf;
      pp.Y = Y;
      pp.uhc = uhc;
      pp.sh = sh;
      pp.zh = zh;
      pp.mm = mmb;
      pp.gbar = gbar;
      pp.T = (int)T;
      pp.B = (int)batch;
      pp.H = (int)H;
      pp.Hp = (int)L.Hp;
      pp.D = (int)L.D;
      pp.direction = direction;
      pp.CS = (int)((((int64_t)1 << 24) >> prod_log2) / prs::BK);
      pp.tiles = ptiles;
      pp.status = device_status_word();
      pp.seq_lens = seq_lens;
      pp.P = P;
      pp.clip = clip;
      pp.input_forget = input_forget ? 1 : 0;
      pp.acts = acts;
      if (!pp.status) return fail(I8Q_ERR_CUDA, "dq_lstm: no device status word");
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)(L.D * ptiles));
      cfg.blockDim = dim3(prs::THREADS);
      cfg.dynamicSmemBytes = psmem;
      cfg.stream = s;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeCooperative;
      attr[0].val.cooperative = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      I8Q_PROF("lstm_persist", s);
      if (var)
        I8Q_CUDA_TRY(cudaLaunchKernelEx(&cfg, prs::lstm_persist_kernel<true>, mR64, mH2, pp));
      else
        I8Q_CUDA_TRY(cudaLaunchKernelEx(&cfg, prs::lstm_persist_kernel<false>, mR64, mH2, pp));
      I8Q_LAUNCH_CHECK("lstm_persist_kernel");
      const float* h_last = hbuf + (T & 1) * DBH;
      if (Y_h) copy_f32<<<grid_for(DBH), 256, 0, s>>>(h_last, Y_h, DBH);
      if (Y_c) copy_f32<<<grid_for(DBH), 256, 0, s>>>(cbuf, Y_c, DBH);
      I8Q_LAUNCH_CHECK("copy_f32");
      return I8Q_OK;
    }
    // step s reads the codes of parity (s + 1) & 1 and writes those of its
    // new h to parity s & 1 (every step, the last included, so that the
    // workspace ends with the codes of the final state); h0's go to parity 1
    int rc2 = launch_quantize_rows(hbuf, I8Q_F32, DB, H, H, uh + DB * L.Hp, uhc + DB * L.Hp, L.Hp, sh + DB, zh + DB, s);
    if (rc2) return rc2;
    StepParams sp;
    sp.uh = uh;
    sp.sh = sh;
    sp.zh = zh;
    sp.Rt = Rt;
    sp.Rcs = Rcs;
    sp.Rsc = Rsc;
    sp.Gx = Gx;
    sp.Wbi = Wbi;
    sp.Rbi = Rbi;
    sp.c = cbuf;
    sp.Y = Y;
    sp.T = (int)T;
    sp.B = (int)batch;
    sp.H = (int)H;
    sp.Hp = (int)L.Hp;
    sp.D = (int)L.D;
    sp.direction = direction;
    const dim3 sgrid((unsigned)ceil_div(L.H4, SN), (unsigned)L.D, (unsigned)ceil_div(batch, SB));
    const dim3 tgrid((unsigned)ceil_div(L.H4, tcs::BM), (unsigned)L.D, (unsigned)ceil_div(batch, tcs::BN));
    tcs::TcStepParams tp;
    tp.sh = sh;
    tp.zh = zh;
    tp.Rcs = Rcs;
    tp.Rsc = Rsc;
    tp.Gx = Gx;
    tp.Wbi = Wbi;
    tp.Rbi = Rbi;
    tp.c = cbuf;
    tp.Y = Y;
    tp.T = (int)T;
    tp.B = (int)batch;
    tp.H = (int)H;
    tp.Hp = (int)L.Hp;
    tp.D = (int)L.D;
    tp.direction = direction;
    tp.CS = (int)((((int64_t)1 << 24) >> prod_log2) / tcs::BK);  // exact fp32 chunk: 1024 (512) K-elements
    tp.seq_lens = seq_lens;
    tp.P = P;
    tp.clip = clip;
    tp.input_forget = input_forget ? 1 : 0;
    tp.acts = acts;
    tp.status = device_status_word();
    if (step_tc && !tp.status) return fail(I8Q_ERR_CUDA, "dq_lstm: no device status word");
    for (int64_t step = 0; step < T; ++step) {
      float* h_next = hbuf + ((step + 1) & 1) * DBH;
      const int64_t pin = (step + 1) & 1, pout = step & 1;
      sp.step = (int)step;
      sp.h_next = h_next;
      sp.uh = uh + pin * DB * L.Hp;
      sp.sh = sh + pin * DB;
      sp.zh = zh + pin * DB;
      if (step_tc) {
        I8Q_PROF("lstm_step_tc", s);
        tp.step = (int)step;
        tp.sh = sh + pin * DB;
        tp.zh = zh + pin * DB;
        tp.hrow0 = (int)(pin * DB);
        tp.h_next = h_next;
        tp.h_prev = hbuf + (step & 1) * DBH;
        if (var)
          tcs::lstm_step_tc_kernel<true><<<tgrid, tcs::THREADS, tcs::SMEM_BYTES, s>>>(mR, mH, tp);
        else
          tcs::lstm_step_tc_kernel<false><<<tgrid, tcs::THREADS, tcs::SMEM_BYTES, s>>>(mR, mH, tp);
        I8Q_LAUNCH_CHECK("lstm_step_tc_kernel");
      } else {
        I8Q_PROF("lstm_step", s);
        lstm_step_kernel<<<sgrid, STHREADS, 0, s>>>(sp);
        I8Q_LAUNCH_CHECK("lstm_step_kernel");
      }
      rc2 = launch_quantize_rows(h_next, I8Q_F32, DB, H, H, uh + pout * DB * L.Hp, uhc + pout * DB * L.Hp, L.Hp,
                                 sh + pout * DB, zh + pout * DB, s);
      if (rc2) return rc2;
    }
    const float* h_last = hbuf + (T & 1) * DBH;
    if (Y_h) copy_f32<<<grid_for(DBH), 256, 0, s>>>(h_last, Y_h, DBH);
    if (Y_c) copy_f32<<<grid_for(DBH), 256, 0, s>>>(cbuf, Y_c, DBH);
    I8Q_LAUNCH_CHECK("copy_f32");
    return I8Q_OK;
  };

  // The recurrence is thousands of short launches: issue it as one CUDA
  // graph, captured once per distinct argument set and relaunched (or
  // updated in place) afterwards.  Direct launches when the caller is
  // itself capturing, on the legacy default stream, or while kernel timing
  // is on (which brackets each launch).
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  I8Q_CUDA_TRY(cudaStreamIsCapturing(s, &cap));
  if (persist || s == nullptr || cap != cudaStreamCaptureStatusNone || profiling_enabled() || T < 4)
    return recurrence();
  int64_t clip_bits = 0;
  std::memcpy(&clip_bits, &clip, sizeof(float));
  LstmGraphKey key{X, W, R, W_scale, R_scale, Bias, h0, c0, Y, Y_h, Y_c, workspace, W_zero_point, R_zero_point,
                   seq_lens, P, T, batch, input, hidden, direction, (int64_t)n_wscale, (int64_t)n_rscale,
                   (int64_t)wtype, (int64_t)(input_forget ? 1 : 0), clip_bits, 0, {0, 0, 0, 0, 0, 0}};
  for (int d = 0; d < 2; ++d)
    for (int k = 0; k < 3; ++k) {
      uint32_t a = 0, b = 0;
      std::memcpy(&a, &acts.alpha[d][k], 4);
      std::memcpy(&b, &acts.beta[d][k], 4);
      key.act_kinds |= (int64_t)acts.kind[d][k] << (4 * (3 * d + k));
      key.act_params[3 * d + k] = (int64_t)(((uint64_t)a << 32) | b);
    }
  return run_cached_graph(key, s, recurrence);
}

}  // namespace

extern "C" int i8q_dq_lstm_forward(const float* X, int64_t T, int64_t batch, int64_t input, int64_t hidden,
                                   int direction, const int8_t* W, const float* W_scale, const int8_t* W_zero_point,
                                   size_t n_wscale, const int8_t* R, const float* R_scale,
                                   const int8_t* R_zero_point, size_t n_rscale, const float* Bias, const float* h0,
                                   const float* c0, float* Y, float* Y_h, float* Y_c, void* workspace,
                                   size_t ws_bytes, void* stream) {
  LstmActs acts;
  bool nondefault = false;
  const int64_t D = direction == I8Q_LSTM_BIDIRECTIONAL ? 2 : 1;
  int rc = resolve_activations(nullptr, 0, nullptr, 0, nullptr, 0, D, acts, nondefault);
  if (rc) return rc;
  return lstm_forward_impl(X, T, batch, input, hidden, direction, W, R, I8Q_S8, W_scale, W_zero_point, n_wscale,
                           R_scale, R_zero_point, n_rscale, Bias, nullptr, h0, c0, nullptr, 0.0f, 0, acts, false, Y,
                           Y_h, Y_c, workspace, ws_bytes, stream);
}

extern "C" int i8q_dq_lstm_forward_ex(const float* X, int64_t T, int64_t batch, int64_t input, int64_t hidden,
                                      int direction, const void* W, const void* R, int wtype, const float* W_scale,
                                      const void* W_zero_point, size_t n_wscale, const float* R_scale,
                                      const void* R_zero_point, size_t n_rscale, const float* Bias,
                                      const int32_t* sequence_lens, const float* h0, const float* c0, const float* P,
                                      float clip, int input_forget, const int* activations, size_t n_activations,
                                      const float* activation_alpha, size_t n_alpha, const float* activation_beta,
                                      size_t n_beta, float* Y, float* Y_h, float* Y_c, void* workspace,
                                      size_t ws_bytes, void* stream) {
  if (direction < I8Q_LSTM_FORWARD || direction > I8Q_LSTM_BIDIRECTIONAL)
    return fail(I8Q_ERR_INVALID_ARG, "dq_lstm: bad direction");
  LstmActs acts;
  bool nondefault = false;
  const int64_t D = direction == I8Q_LSTM_BIDIRECTIONAL ? 2 : 1;
  int rc = resolve_activations(activations, n_activations, activation_alpha, n_alpha, activation_beta, n_beta, D,
                               acts, nondefault);
  if (rc) return rc;
  return lstm_forward_impl(X, T, batch, input, hidden, direction, W, R, wtype, W_scale, W_zero_point, n_wscale,
                           R_scale, R_zero_point, n_rscale, Bias, sequence_lens, h0, c0, P, clip, input_forget, acts,
                           nondefault, Y, Y_h, Y_c, workspace, ws_bytes, stream);
}

extern "C" int i8q_debug_wait_timeout(int kind, int64_t limit_ns, void* stream) {
  if (kind != 0 && kind != 1) return fail(I8Q_ERR_INVALID_ARG, "debug_wait_timeout: kind must be 0 or 1");
  if (limit_ns < 1000 || limit_ns > 1000000000)
    return fail(I8Q_ERR_INVALID_ARG, "debug_wait_timeout: limit must be within [1 us, 1 s]");
  uint32_t* status = device_status_word();
  if (!status) return fail(I8Q_ERR_CUDA, "debug_wait_timeout: no device status word");
  prs::wait_probe_kernel<<<1, 32, 0, as_stream(stream)>>>(kind, (unsigned long long)limit_ns, status);
  I8Q_LAUNCH_CHECK("wait_probe_kernel");
  return I8Q_OK;
}

extern "C" int i8q_dq_lstm_state_codes(const void* workspace, int64_t T, int64_t batch, int64_t input,
                                       int64_t hidden, int direction, int which, const void** codes,
                                       const float** scale, const int32_t** zero, int64_t* row_stride) {
  if (!workspace || !codes || !scale || !zero || !row_stride)
    return fail(I8Q_ERR_INVALID_ARG, "dq_lstm_state_codes: NULL argument");
  if (T <= 0 || batch <= 0 || input <= 0 || hidden <= 0 || direction < I8Q_LSTM_FORWARD ||
      direction > I8Q_LSTM_BIDIRECTIONAL)
    return fail(I8Q_ERR_INVALID_ARG, "dq_lstm_state_codes: bad shape or direction");
  if (which != 0 && which != 1) return fail(I8Q_ERR_INVALID_ARG, "dq_lstm_state_codes: which must be 0 or 1");
  const LstmLayout L = lstm_layout(T, batch, input, hidden, direction);
  const int64_t DB = L.D * batch;
  const int64_t par = which == 0 ? (T & 1) : ((T - 1) & 1);
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  *codes = ws + L.off_uhc + (size_t)par * DB * L.Hp * 2;
  *scale = reinterpret_cast<const float*>(ws + L.off_sh) + par * DB;
  *zero = reinterpret_cast<const int32_t*>(ws + L.off_zh) + par * DB;
  *row_stride = L.Hp;
  return I8Q_OK;
}

namespace i8q {
namespace {

std::mutex g_graph_mu;
struct {
  bool valid = false;
  int device = -1;
  LstmGraphKey key{};
  cudaGraphExec_t exec = nullptr;
} g_graph;

}  // namespace

int run_cached_graph(const LstmGraphKey& key, cudaStream_t s, const std::function<int()>& issue) {
  std::lock_guard<std::mutex> lk(g_graph_mu);
  int dev = 0;
  I8Q_CUDA_TRY(cudaGetDevice(&dev));
  if (g_graph.valid && g_graph.device == dev && std::memcmp(&g_graph.key, &key, sizeof(key)) == 0) {
    I8Q_CUDA_TRY(cudaGraphLaunch(g_graph.exec, s));
    return I8Q_OK;
  }
  I8Q_CUDA_TRY(cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal));
  const int rc = issue();
  cudaGraph_t graph = nullptr;
  const cudaError_t ec = cudaStreamEndCapture(s, &graph);
  if (rc) {
    if (graph) cudaGraphDestroy(graph);
    return rc;
  }
  if (ec != cudaSuccess) return cuda_fail(ec, "cudaStreamEndCapture(lstm recurrence)");
  bool updated = false;
  if (g_graph.valid && g_graph.device == dev) {
    cudaGraphExecUpdateResultInfo info;
    if (cudaGraphExecUpdate(g_graph.exec, graph, &info) == cudaSuccess) {
      updated = true;
    } else {
      cudaGetLastError();
      cudaGraphExecDestroy(g_graph.exec);
      g_graph.valid = false;
    }
  } else if (g_graph.valid) {
    cudaGraphExecDestroy(g_graph.exec);  // made on another device
    g_graph.valid = false;
  }
  if (!updated) {
    const cudaError_t ei = cudaGraphInstantiate(&g_graph.exec, graph, 0);
    if (ei != cudaSuccess) {
      cudaGraphDestroy(graph);
      return cuda_fail(ei, "cudaGraphInstantiate(lstm recurrence)");
    }
  }
  cudaGraphDestroy(graph);
  g_graph.valid = true;
  g_graph.device = dev;
  g_graph.key = key;
  I8Q_CUDA_TRY(cudaGraphLaunch(g_graph.exec, s));
  return I8Q_OK;
}

}  // namespace i8q
