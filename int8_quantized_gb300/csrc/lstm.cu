// lstm.cu -- DynamicQuantizeLSTM (ONNX Runtime contrib schema
// "DynamicQuantizeLSTM"; graiphic.io "DynamicQuantizeLSTM") on the dynamic
// quantized GEMM engine.
//
// int8 W [D, input, 4H] and R [D, H, 4H] with per-channel (or per-direction)
// scales and zero point 0; fp32 X; default activations (sigmoid for the
// i, o, f gates, tanh for the cell candidate and the output); gate column
// order i, o, f, c.  X and each step's hidden state are quantized per row to
// uint8 exactly like A of the dynamic quantized inner product.
//   input projection (all steps at once): Gx = X W[d]
//   per step t: Gh = h_{t-1} R[d]; g = ((Gx_t + Gh) + Wb) + Rb
//               i, o, f = sigmoid(g); ct = tanh(g_c)
//               c = f*c_{t-1} + i*ct;  h = o*tanh(c)
// The reverse direction walks t = T-1 .. 0.
//
// Layout: the 4H gate columns of W, R, their scales and the biases are
// interleaved per hidden unit (column q*H + u stored at 4u + q), so any
// 64-column tile holds all four gates of 16 hidden units.  Then one kernel
// per step does, for both directions at once, the recurrent integer product
// and the whole cell update in its epilogue: on the tensor pipe
// (tcgen05, 128 gate columns x 64 batch rows per CTA, h codes centred to
// uh - 128 in bf16, fp32 chunks drained exactly to int32, the step's
// x-projection and previous cell state loaded while the MMAs run) for wide
// layers, or on the int8 mma.sync form (64 x 64 tiles) otherwise.  The
// projection runs once over all T * batch rows on the tensor-core GEMM; X is
// quantized once for both directions.  Each step's new h is quantized per
// row (both directions in one launch) for the next step, and the whole
// sequence of steps is replayed as one CUDA graph, cached per argument set.
#include <cstring>
#include <functional>
#include <mutex>

#include "tcgen05.cuh"

namespace i8q {
namespace {

struct LstmLayout {
  int64_t D, TB, Ip, Hp, H4;
  size_t off_Wt, off_Wtb, off_Wcs, off_Rt, off_Rtb, off_Rcs, off_Wsc, off_Rsc, off_Wbi, off_Rbi, off_uX, off_uXc,
      off_sX, off_zX, off_Gx, off_uh, off_uhc, off_sh, off_zh, off_h, off_c, total;
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
  L.off_uh = take((size_t)L.D * batch * L.Hp);
  L.off_uhc = take((size_t)L.D * batch * L.Hp * 2);
  L.off_sh = take((size_t)L.D * batch * 4);
  L.off_zh = take((size_t)L.D * batch * 4);
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

__device__ __forceinline__ float sigmoid_f32(float x) { return __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-x))); }

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
    const float ig = sigmoid_f32(gs[r][4 * uu + 0]);
    const float og = sigmoid_f32(gs[r][4 * uu + 1]);
    const float fg = sigmoid_f32(gs[r][4 * uu + 2]);
    const float ct = tanhf(gs[r][4 * uu + 3]);
    const int64_t e = ((int64_t)d * p.B + b) * p.H + u;
    const float cn = __fadd_rn(__fmul_rn(fg, p.c[e]), __fmul_rn(ig, ct));
    const float hn = __fmul_rn(og, tanhf(cn));
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
  const float* sh;     // [D*B]
  const int32_t* zh;   // [D*B]
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
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
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
        tma_load_2d(sB(s), &tmH, full(s), kt * BK, d * p.B + nb * BN);
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
            act = q == 3 ? tanhf(gg) : sigmoid_f32(gg);
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
          og = sigmoid_f32(clip_gate(so, p.clip));
        }
        og = __shfl_sync(0xffffffffu, og, base_lane + 1);
        if (q == 0 && b < p.B && nvalid && u < p.H) {
          const int64_t e = ((int64_t)d * p.B + b) * p.H + u;
          if (live) {
            const float hn = __fmul_rn(og, tanhf(cn));
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
          act = q < 3 ? sigmoid_f32(gg) : tanhf(gg);
        }
        const float ig = __shfl_sync(0xffffffffu, act, base_lane + 0);
        const float og = __shfl_sync(0xffffffffu, act, base_lane + 1);
        const float fg = __shfl_sync(0xffffffffu, act, base_lane + 2);
        const float ct = __shfl_sync(0xffffffffu, act, base_lane + 3);
        if (q == 0 && bvalid && nvalid && u < p.H) {
          const int64_t e = ((int64_t)d * p.B + b) * p.H + u;
          const float cn = __fadd_rn(__fmul_rn(fg, cprev[j]), __fmul_rn(ig, ct));
          const float hn = __fmul_rn(og, tanhf(cn));
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

int lstm_forward_impl(const float* X, int64_t T, int64_t batch, int64_t input, int64_t hidden, int direction,
                      const void* W_, const void* R_, int wtype, const float* W_scale, const void* W_zero_point_,
                      size_t n_wscale, const float* R_scale, const void* R_zero_point_, size_t n_rscale,
                      const float* Bias, const int32_t* seq_lens, const float* h0, const float* c0, const float* P,
                      float clip, int input_forget, float* Y, float* Y_h, float* Y_c, void* workspace,
                      size_t ws_bytes, void* stream) {
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
  float* hbuf = (float*)(ws + L.off_h);
  float* cbuf = (float*)(ws + L.off_c);
  const int64_t H = hidden, BH = batch * hidden, DBH = L.D * BH;

  // The general form (uint8 weights, zero points, sequence lengths,
  // peepholes, clip, coupled gates) runs on the tensor-core kernels: the
  // weights enter as bf16 W - zp (|W - zp| <= 255), so products stay within
  // 2^15 and the exact fp32 chunks hold 512 K-elements.  int8 weights whose
  // given zero points are all 0 (checked on the device, reported
  // synchronously) keep the plain form.
  bool var = wtype != I8Q_S8 || seq_lens || P || clip > 0.0f || input_forget;
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
    rc = tc::make_map_2d(&mH, uhc, L.D * batch, L.Hp, tcs::BN, "dq_lstm");
    if (rc) return rc;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
      attr_err = cudaFuncSetAttribute(tcs::lstm_step_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      tcs::SMEM_BYTES);
      if (attr_err == cudaSuccess)
        attr_err = cudaFuncSetAttribute(tcs::lstm_step_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        tcs::SMEM_BYTES);
    });
    if (attr_err != cudaSuccess) return cuda_fail(attr_err, "cudaFuncSetAttribute(lstm_step_tc_kernel)");
  }

  // recurrence: both directions per launch, 2 launches per step
  auto recurrence = [&]() -> int {
    init_state<<<grid_for(DBH), 256, 0, s>>>(h0, c0, DBH, hbuf, cbuf);
    I8Q_LAUNCH_CHECK("init_state");
    // rows whose sequence ends early leave the rest of Y zero
    if (Y && seq_lens) I8Q_CUDA_TRY(cudaMemsetAsync(Y, 0, (size_t)T * DBH * sizeof(float), s));
    int rc2 = launch_quantize_rows(hbuf, I8Q_F32, L.D * batch, H, H, uh, step_tc ? uhc : nullptr, L.Hp, sh, zh, s);
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
    tp.status = device_status_word();
    if (step_tc && !tp.status) return fail(I8Q_ERR_CUDA, "dq_lstm: no device status word");
    for (int64_t step = 0; step < T; ++step) {
      float* h_next = hbuf + ((step + 1) & 1) * DBH;
      sp.step = (int)step;
      sp.h_next = h_next;
      if (step_tc) {
        I8Q_PROF("lstm_step_tc", s);
        tp.step = (int)step;
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
      if (step + 1 < T) {
        rc2 = launch_quantize_rows(h_next, I8Q_F32, L.D * batch, H, H, uh, step_tc ? uhc : nullptr, L.Hp, sh, zh, s);
        if (rc2) return rc2;
      }
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
  if (s == nullptr || cap != cudaStreamCaptureStatusNone || profiling_enabled() || T < 4) return recurrence();
  int64_t clip_bits = 0;
  std::memcpy(&clip_bits, &clip, sizeof(float));
  const LstmGraphKey key{X, W, R, W_scale, R_scale, Bias, h0, c0, Y, Y_h, Y_c, workspace, W_zero_point, R_zero_point,
                         seq_lens, P, T, batch, input, hidden, direction, (int64_t)n_wscale, (int64_t)n_rscale,
                         (int64_t)wtype, (int64_t)(input_forget ? 1 : 0), clip_bits};
  return run_cached_graph(key, s, recurrence);
}

}  // namespace

extern "C" int i8q_dq_lstm_forward(const float* X, int64_t T, int64_t batch, int64_t input, int64_t hidden,
                                   int direction, const int8_t* W, const float* W_scale, const int8_t* W_zero_point,
                                   size_t n_wscale, const int8_t* R, const float* R_scale,
                                   const int8_t* R_zero_point, size_t n_rscale, const float* Bias, const float* h0,
                                   const float* c0, float* Y, float* Y_h, float* Y_c, void* workspace,
                                   size_t ws_bytes, void* stream) {
  return lstm_forward_impl(X, T, batch, input, hidden, direction, W, R, I8Q_S8, W_scale, W_zero_point, n_wscale,
                           R_scale, R_zero_point, n_rscale, Bias, nullptr, h0, c0, nullptr, 0.0f, 0, Y, Y_h, Y_c,
                           workspace, ws_bytes, stream);
}

extern "C" int i8q_dq_lstm_forward_ex(const float* X, int64_t T, int64_t batch, int64_t input, int64_t hidden,
                                      int direction, const void* W, const void* R, int wtype, const float* W_scale,
                                      const void* W_zero_point, size_t n_wscale, const float* R_scale,
                                      const void* R_zero_point, size_t n_rscale, const float* Bias,
                                      const int32_t* sequence_lens, const float* h0, const float* c0, const float* P,
                                      float clip, int input_forget, float* Y, float* Y_h, float* Y_c,
                                      void* workspace, size_t ws_bytes, void* stream) {
  return lstm_forward_impl(X, T, batch, input, hidden, direction, W, R, wtype, W_scale, W_zero_point, n_wscale,
                           R_scale, R_zero_point, n_rscale, Bias, sequence_lens, h0, c0, P, clip, input_forget, Y,
                           Y_h, Y_c, workspace, ws_bytes, stream);
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
