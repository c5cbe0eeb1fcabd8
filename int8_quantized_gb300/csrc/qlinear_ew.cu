// qlinear_ew.cu -- the quantized elementwise operators of the ONNX Runtime
// contrib schemas: MulInteger, QLinearAdd, QLinearMul (Numpy-style
// broadcasting), QLinearLeakyRelu and QLinearSigmoid.
//
//   MulInteger: C (int32) = (A - A_zp) * (B - B_zp)
//   QLinearAdd: C = (A_scale * (A - A_zp) + B_scale * (B - B_zp)) / C_scale + C_zp
//   QLinearMul: C = ((A - A_zp) * (B - B_zp)) * (A_scale * B_scale) / C_scale + C_zp
//   QLinearLeakyRelu / QLinearSigmoid: y = QuantizeLinear(f(DequantizeLinear(x)))
// The binary formulas are evaluated in the order they are written, each fp32
// operation rounding once; the integer differences and their product are
// exact.  Quantized outputs round half to even and saturate.
//
// All of them stream HBM.  The binary kernels move 16 codes per thread and
// step (16-byte loads and stores) when the operands have the output's shape,
// when one is a single value, or when one repeats along leading dimensions;
// other broadcasts take a general path over collapsed strides.  A unary
// operator's 256 possible outputs are computed once per block, with the same
// arithmetic, into a table replicated per lane in shared memory (entry e of
// lane l at word e * 32 + l, so every lookup of a warp is conflict-free).
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace i8q {
namespace {

constexpr int kMaxRank = 8;

struct BinParams {
  int op;  // 0 add, 1 mul, 2 mul-integer
  float a_scale, b_scale, c_scale;
  int a_zp, b_zp, c_zp;
  float lo_z, hi_z;  // output range minus c_zp
};

template <bool AS, bool BS>
__device__ __forceinline__ uint32_t binary_one(uint32_t araw, uint32_t braw, const BinParams& p, int32_t* wide) {
  const int a = (AS ? (int)(int8_t)araw : (int)(uint8_t)araw) - p.a_zp;
  const int b = (BS ? (int)(int8_t)braw : (int)(uint8_t)braw) - p.b_zp;
  if (p.op == 2) {
    *wide = a * b;
    return 0;
  }
  float v;
  if (p.op == 0) {
    const float fa = __fmul_rn(p.a_scale, __int2float_rn(a));
    const float fb = __fmul_rn(p.b_scale, __int2float_rn(b));
    v = __fadd_rn(fa, fb);
  } else {
    v = __fmul_rn(__int2float_rn(a * b), __fmul_rn(p.a_scale, p.b_scale));
  }
  return rint_code_bits(__fdiv_rn(v, p.c_scale), p.lo_z, p.hi_z, p.c_zp);
}

// Output flat index -> operand offsets for the fast layouts:
//   mode 0: same shape; 1: the operand is one value; 2: the operand repeats
//   every `period` elements (its shape is a suffix of the output's).
__device__ __forceinline__ int64_t fast_offset(int mode, int64_t i, int64_t period) {
  return mode == 0 ? i : (mode == 1 ? 0 : i % period);
}

// 16 outputs per thread and step.  amode/bmode as in fast_offset; a
// period-2 operand needs period % 16 == 0 (checked on the host) so a group
// of 16 stays contiguous in it.
template <bool AS, bool BS>
__global__ void __launch_bounds__(256)
binary_fast(const uint8_t* __restrict__ A, int amode, int64_t aper, const uint8_t* __restrict__ B, int bmode,
            int64_t bper, int64_t n, BinParams p, void* __restrict__ C) {
  const int64_t groups = n / 16;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t gi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; gi < groups; gi += stride) {
    const int64_t i = gi * 16;
    uint32_t aw[4], bw[4];
    if (amode == 1) {
      const uint32_t v = A[0] * 0x01010101u;
      aw[0] = aw[1] = aw[2] = aw[3] = v;
    } else {
      const uint4 v = __ldcs(reinterpret_cast<const uint4*>(A + fast_offset(amode, i, aper)));
      aw[0] = v.x, aw[1] = v.y, aw[2] = v.z, aw[3] = v.w;
    }
    if (bmode == 1) {
      const uint32_t v = B[0] * 0x01010101u;
      bw[0] = bw[1] = bw[2] = bw[3] = v;
    } else {
      const uint4 v = __ldcs(reinterpret_cast<const uint4*>(B + fast_offset(bmode, i, bper)));
      bw[0] = v.x, bw[1] = v.y, bw[2] = v.z, bw[3] = v.w;
    }
    if (p.op == 2) {
      int32_t* out = static_cast<int32_t*>(C) + i;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        int32_t r[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) binary_one<AS, BS>(aw[w] >> (8 * e), bw[w] >> (8 * e), p, &r[e]);
        __stcs(reinterpret_cast<int4*>(out + 4 * w), make_int4(r[0], r[1], r[2], r[3]));
      }
    } else {
      uint32_t ow[4];
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t c[4];
        int32_t unused;
#pragma unroll
        for (int e = 0; e < 4; ++e) c[e] = binary_one<AS, BS>(aw[w] >> (8 * e), bw[w] >> (8 * e), p, &unused);
        ow[w] = pack_low_bytes(c[0], c[1], c[2], c[3]);
      }
      __stcs(reinterpret_cast<uint4*>(static_cast<uint8_t*>(C) + i), make_uint4(ow[0], ow[1], ow[2], ow[3]));
    }
  }
}

// QLinearAdd / QLinearMul on large tensors: the output code depends only
// on the two input codes, so each block first fills a 256 x 256 table of
// codes (byte a * 256 + b, computed by binary_one, so bit for bit the
// per-element result) in shared memory, then streams 16 codes per thread
// and group, four groups in flight, each output one table lookup.  Modes as
// in binary_fast.
constexpr int kTabThreads = 1024, kTabBytes = 65536;

// Word wi of the table: the codes of (a, 4w' .. 4w' + 3), wi = a * 64 + w'.
template <bool AS, bool BS>
__device__ __forceinline__ uint32_t table_word(int wi, const BinParams& p) {
  const uint32_t a = (uint32_t)wi >> 6, b0 = ((uint32_t)wi & 63u) * 4u;
  int32_t unused;
  return pack_low_bytes(binary_one<AS, BS>(a, b0, p, &unused), binary_one<AS, BS>(a, b0 + 1, p, &unused),
                        binary_one<AS, BS>(a, b0 + 2, p, &unused), binary_one<AS, BS>(a, b0 + 3, p, &unused));
}

// The table in global memory, one word per thread (kept for later calls
// with the same parameters, see table_slot).
template <bool AS, bool BS>
__global__ void __launch_bounds__(256) build_binary_table(BinParams p, uint32_t* __restrict__ table) {
  const int wi = blockIdx.x * blockDim.x + threadIdx.x;
  if (wi < kTabBytes / 4) table[wi] = table_word<AS, BS>(wi, p);
}

// SAME: both operands have the output's shape (modes 0), the common case,
// compiled without the broadcast branches.  The shared table is copied from
// a prebuilt global one when given (64 KB from L2), else computed here.
template <bool AS, bool BS, bool SAME>
__global__ void __launch_bounds__(kTabThreads, 1)
binary_table(const uint8_t* __restrict__ A, int amode, int64_t aper, const uint8_t* __restrict__ B, int bmode,
             int64_t bper, int64_t n, BinParams p, const uint32_t* __restrict__ gtab, uint8_t* __restrict__ C) {
  extern __shared__ uint32_t tab[];  // 16384 words, codes (a, 4w' .. 4w' + 3) in word a * 64 + w'
  if (gtab) {
    for (int q = threadIdx.x; q < kTabBytes / 16; q += kTabThreads)
      reinterpret_cast<uint4*>(tab)[q] = __ldg(reinterpret_cast<const uint4*>(gtab) + q);
  } else {
    for (int wi = threadIdx.x; wi < kTabBytes / 4; wi += kTabThreads) tab[wi] = table_word<AS, BS>(wi, p);
  }
  __syncthreads();
  const uint8_t* t8 = reinterpret_cast<const uint8_t*>(tab);
  // a warp moves U * 512 consecutive codes per step (lane t: the 16-code
  // groups t, t + 32, ...), so each operand stream is read in 1 KB runs
  constexpr int U = 2;
  const int lane = threadIdx.x & 31;
  const int64_t groups = n / 16;
  const int64_t chunks = (groups + 32 * U - 1) / (32 * U);
  const int64_t wstride = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t ch = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; ch < chunks; ch += wstride) {
    uint32_t aw[U][4], bw[U][4];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t gi = ch * 32 * U + 32 * u + lane;
      const int64_t i = gi * 16;
      const bool in = gi < groups;
      if (!SAME && amode == 1) {
        const uint32_t v = A[0] * 0x01010101u;
        aw[u][0] = aw[u][1] = aw[u][2] = aw[u][3] = v;
      } else {
        const int64_t off = SAME ? i : fast_offset(amode, i, aper);
        const uint4 v = in ? __ldcs(reinterpret_cast<const uint4*>(A + off)) : make_uint4(0, 0, 0, 0);
        aw[u][0] = v.x, aw[u][1] = v.y, aw[u][2] = v.z, aw[u][3] = v.w;
      }
      if (!SAME && bmode == 1) {
        const uint32_t v = B[0] * 0x01010101u;
        bw[u][0] = bw[u][1] = bw[u][2] = bw[u][3] = v;
      } else {
        const int64_t off = SAME ? i : fast_offset(bmode, i, bper);
        const uint4 v = in ? __ldcs(reinterpret_cast<const uint4*>(B + off)) : make_uint4(0, 0, 0, 0);
        bw[u][0] = v.x, bw[u][1] = v.y, bw[u][2] = v.z, bw[u][3] = v.w;
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t gi = ch * 32 * U + 32 * u + lane;
      if (gi >= groups) break;
      uint32_t ow[4];
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint32_t c[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          c[e] = t8[(((aw[u][w] >> (8 * e)) & 0xffu) << 8) | ((bw[u][w] >> (8 * e)) & 0xffu)];
        ow[w] = c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24);
      }
      __stcs(reinterpret_cast<uint4*>(C + gi * 16), make_uint4(ow[0], ow[1], ow[2], ow[3]));
    }
  }
}

struct Strides {
  int rank;
  int64_t out[kMaxRank];
  int64_t sa[kMaxRank], sb[kMaxRank];  // element strides, 0 on broadcast dimensions
};

// Any broadcast, one output per thread and step; also the tail of the fast
// path (start = first index not covered there).
template <bool AS, bool BS>
__global__ void __launch_bounds__(256)
binary_general(const uint8_t* __restrict__ A, const uint8_t* __restrict__ B, int64_t start, int64_t n, Strides st,
               BinParams p, void* __restrict__ C) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = start + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    int64_t rem = i, oa = 0, ob = 0;
    for (int d = st.rank - 1; d >= 0; --d) {
      const int64_t idx = rem % st.out[d];
      rem /= st.out[d];
      oa += idx * st.sa[d];
      ob += idx * st.sb[d];
    }
    int32_t wide = 0;
    const uint32_t c = binary_one<AS, BS>(A[oa], B[ob], p, &wide);
    if (p.op == 2)
      static_cast<int32_t*>(C)[i] = wide;
    else
      static_cast<uint8_t*>(C)[i] = (uint8_t)c;
  }
}

// The 256 outputs of a unary operator, one per input code, with the
// DequantizeLinear -> f -> QuantizeLinear arithmetic.
template <bool SIGNED>
__device__ __forceinline__ uint32_t unary_code(int code_index, int op, float x_scale, int x_zp, float y_scale, int y_zp,
                                               float alpha, float lo_z, float hi_z) {
  const int x = SIGNED ? (int)(int8_t)(uint8_t)code_index : code_index;
  const float d = __fmul_rn(__int2float_rn(x - x_zp), x_scale);
  float f;
  if (op == 0)
    f = d < 0.0f ? __fmul_rn(alpha, d) : d;
  else
    f = ef::sigmoid32(d);
  return rint_code_bits(__fdiv_rn(f, y_scale), lo_z, hi_z, y_zp) & 0xffu;
}

template <bool SIGNED>
__global__ void __launch_bounds__(256)
unary_lut(const uint8_t* __restrict__ X, int64_t n, int op, float x_scale, int x_zp, float y_scale, int y_zp,
          float alpha, float lo_z, float hi_z, uint8_t* __restrict__ Y) {
  __shared__ uint32_t lut[256 * 32];  // entry e of lane l at e * 32 + l
  const int lane = threadIdx.x & 31;
  {
    const int e = threadIdx.x;  // 256 threads, one entry each
    const uint32_t v = unary_code<SIGNED>(e, op, x_scale, x_zp, y_scale, y_zp, alpha, lo_z, hi_z);
#pragma unroll 8
    for (int l = 0; l < 32; ++l) lut[e * 32 + l] = v;
  }
  __syncthreads();
  const int64_t groups = n / 16;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const bool aligned = ((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(Y)) & 15) == 0;
  if (aligned) {
    // a warp moves U * 512 consecutive codes per step (lane t: the 16-code
    // groups t, t + 32, ...): 4 KB runs of the input, all loaded before any
    // is used
    constexpr int U = 8;
    const int64_t chunks = (groups + 32 * U - 1) / (32 * U);
    const int64_t wstride = stride >> 5;
    for (int64_t ch = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; ch < chunks; ch += wstride) {
      uint4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t gi = ch * 32 * U + 32 * u + lane;
        v[u] = gi < groups ? __ldcs(reinterpret_cast<const uint4*>(X) + gi) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t gi = ch * 32 * U + 32 * u + lane;
        if (gi >= groups) break;
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t c0 = lut[((w[q] >> 0) & 0xff) * 32 + lane], c1 = lut[((w[q] >> 8) & 0xff) * 32 + lane];
          const uint32_t c2 = lut[((w[q] >> 16) & 0xff) * 32 + lane], c3 = lut[(w[q] >> 24) * 32 + lane];
          o[q] = pack_low_bytes(c0, c1, c2, c3);
        }
        __stcs(reinterpret_cast<uint4*>(Y) + gi, make_uint4(o[0], o[1], o[2], o[3]));
      }
    }
  }
  for (int64_t i = (aligned ? groups * 16 : 0) + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    Y[i] = (uint8_t)lut[X[i] * 32 + lane];
}

int grid_for(int64_t work) {
  return (int)std::max<int64_t>(1, std::min<int64_t>(ceil_div(work, 256), (int64_t)sm_count() * 8));
}

// Broadcast shapes (left-padded to one rank), collapse runs of dimensions
// with the same broadcast pattern, and fill element strides.
int broadcast(const int64_t* as, int ar, const int64_t* bs, int br, Strides* st, int64_t* n_out, int64_t* an,
              int64_t* bn) {
  if (ar < 0 || br < 0 || ar > kMaxRank || br > kMaxRank)
    return fail(I8Q_ERR_INVALID_ARG, "qlinear: rank must be 0.." + std::to_string(kMaxRank));
  const int r = std::max(std::max(ar, br), 1);
  int64_t a[kMaxRank], b[kMaxRank], o[kMaxRank];
  *an = *bn = *n_out = 1;
  for (int d = 0; d < r; ++d) {
    const int ia = d - (r - ar), ib = d - (r - br);
    a[d] = ia >= 0 ? as[ia] : 1;
    b[d] = ib >= 0 ? bs[ib] : 1;
    if (a[d] < 1 || b[d] < 1) return fail(I8Q_ERR_INVALID_ARG, "qlinear: dimensions must be >= 1");
    if (a[d] != b[d] && a[d] != 1 && b[d] != 1)
      return fail(I8Q_ERR_INVALID_ARG, "qlinear: shapes are not broadcastable");
    o[d] = std::max(a[d], b[d]);
    *an *= a[d];
    *bn *= b[d];
    *n_out *= o[d];
  }
  // collapse dimensions d-1, d when both operands treat them alike
  int64_t ca[kMaxRank], cb[kMaxRank], co[kMaxRank];
  int k = 0;
  for (int d = 0; d < r; ++d) {
    if (o[d] == 1) continue;
    const bool fa = a[d] == o[d], fb = b[d] == o[d];
    if (k > 0 && ((ca[k - 1] == co[k - 1]) == fa) && ((cb[k - 1] == co[k - 1]) == fb)) {
      co[k - 1] *= o[d];
      ca[k - 1] *= a[d];
      cb[k - 1] *= b[d];
    } else {
      co[k] = o[d];
      ca[k] = a[d];
      cb[k] = b[d];
      ++k;
    }
  }
  if (k == 0) {
    co[0] = ca[0] = cb[0] = 1;
    k = 1;
  }
  st->rank = k;
  int64_t sa = 1, sb = 1;
  for (int d = k - 1; d >= 0; --d) {
    st->out[d] = co[d];
    st->sa[d] = ca[d] == 1 ? 0 : sa;
    st->sb[d] = cb[d] == 1 ? 0 : sb;
    sa *= ca[d];
    sb *= cb[d];
  }
  return I8Q_OK;
}

// mode of an operand for binary_fast (-1: none applies)
int fast_mode(const Strides& st, bool is_a, int64_t numel, int64_t* period) {
  const int64_t* s = is_a ? st.sa : st.sb;
  if (numel == 1) return 1;
  bool full = true;
  for (int d = 0; d < st.rank; ++d) full = full && s[d] != 0;
  if (full) return 0;
  // a suffix of the output: dims [j, rank) present, [0, j) broadcast
  int j = st.rank;
  while (j > 0 && s[j - 1] != 0) --j;
  for (int d = 0; d < j; ++d)
    if (s[d] != 0) return -1;
  *period = numel;
  return numel % 16 == 0 ? 2 : -1;
}

// Tables kept in file-scope device memory (no allocation), up to kTabSlots
// per device, each written once for one (signedness, parameters) key and
// never again, so any stream may read it after waiting on the event that
// follows its build.  When the slots are taken, the table is computed inside
// the product kernel.
constexpr int kTabSlots = 16, kTabMaxDev = 64;
static __device__ __align__(16) uint32_t g_tables[kTabSlots][kTabBytes / 4];

struct TabSlot {
  bool used = false;
  int as = 0, bs = 0;
  BinParams p{};
  cudaEvent_t ready = nullptr;
};
std::mutex g_tab_mu;
TabSlot g_tab[kTabMaxDev][kTabSlots];
uint32_t* g_tab_base[kTabMaxDev] = {nullptr};

bool same_params(const BinParams& a, const BinParams& b) { return std::memcmp(&a, &b, sizeof(BinParams)) == 0; }

// The prebuilt table for p on this device, built on s the first time (s
// waits for it after), or null when no slot is free.
template <bool AS, bool BS>
int table_slot(const BinParams& p, cudaStream_t s, const uint32_t** out) {
  *out = nullptr;
  int dev = 0;
  I8Q_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kTabMaxDev) return I8Q_OK;
  std::lock_guard<std::mutex> lk(g_tab_mu);
  if (!g_tab_base[dev]) {
    void* base = nullptr;
    I8Q_CUDA_TRY(cudaGetSymbolAddress(&base, g_tables));
    g_tab_base[dev] = static_cast<uint32_t*>(base);
  }
  for (int i = 0; i < kTabSlots; ++i) {
    TabSlot& t = g_tab[dev][i];
    if (t.used && t.as == AS && t.bs == BS && same_params(t.p, p)) {
      I8Q_CUDA_TRY(cudaStreamWaitEvent(s, t.ready, 0));
      *out = g_tab_base[dev] + (size_t)i * (kTabBytes / 4);
      return I8Q_OK;
    }
  }
  for (int i = 0; i < kTabSlots; ++i) {
    TabSlot& t = g_tab[dev][i];
    if (t.used) continue;
    if (!t.ready) I8Q_CUDA_TRY(cudaEventCreateWithFlags(&t.ready, cudaEventDisableTiming));
    uint32_t* tab = g_tab_base[dev] + (size_t)i * (kTabBytes / 4);
    build_binary_table<AS, BS><<<kTabBytes / 4 / 256, 256, 0, s>>>(p, tab);
    I8Q_LAUNCH_CHECK("build_binary_table");
    I8Q_CUDA_TRY(cudaEventRecord(t.ready, s));
    t.used = true;
    t.as = AS;
    t.bs = BS;
    t.p = p;
    *out = tab;
    return I8Q_OK;
  }
  return I8Q_OK;
}

template <bool AS, bool BS>
int run_binary(const uint8_t* A, const uint8_t* B, const Strides& st, int64_t n, int64_t an, int64_t bn,
               const BinParams& p, void* C, cudaStream_t s) {
  int64_t aper = 0, bper = 0;
  const int am = fast_mode(st, true, an, &aper), bm = fast_mode(st, false, bn, &bper);
  const bool aligned =
      ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(C)) & 15) == 0;
  int64_t done = 0;
  if (am >= 0 && bm >= 0 && aligned && p.op != 2 && n >= ((int64_t)1 << 20) && !getenv("I8Q_QEW_NO_TABLE")) {
    int ar = smem_attr((const void*)binary_table<AS, BS, true>, kTabBytes);
    if (!ar) ar = smem_attr((const void*)binary_table<AS, BS, false>, kTabBytes);
    if (ar) return ar;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(sm_count(), ceil_div(n / 16, (int64_t)kTabThreads)));
    const uint32_t* gtab = nullptr;
    if (!getenv("I8Q_QEW_NO_TABLE_CACHE")) {
      const int rc = table_slot<AS, BS>(p, s, &gtab);
      if (rc) return rc;
    }
    if (am == 0 && bm == 0)
      binary_table<AS, BS, true><<<grid, kTabThreads, kTabBytes, s>>>(A, am, aper, B, bm, bper, n, p, gtab,
                                                                       static_cast<uint8_t*>(C));
    else
      binary_table<AS, BS, false><<<grid, kTabThreads, kTabBytes, s>>>(A, am, aper, B, bm, bper, n, p, gtab,
                                                                        static_cast<uint8_t*>(C));
    I8Q_LAUNCH_CHECK("binary_table");
    done = (n / 16) * 16;
  } else if (am >= 0 && bm >= 0 && aligned && n >= 16) {
    binary_fast<AS, BS><<<grid_for(n / 16), 256, 0, s>>>(A, am, aper, B, bm, bper, n, p, C);
    I8Q_LAUNCH_CHECK("binary_fast");
    done = (n / 16) * 16;
  }
  if (done < n) {
    binary_general<AS, BS><<<grid_for(n - done), 256, 0, s>>>(A, B, done, n, st, p, C);
    I8Q_LAUNCH_CHECK("binary_general");
  }
  return I8Q_OK;
}

int binary_dispatch(const void* A, int atype, const int64_t* a_shape, int a_rank, const void* B, int btype,
                    const int64_t* b_shape, int b_rank, BinParams p, void* C, cudaStream_t s) {
  Strides st{};
  int64_t n, an, bn;
  int rc = broadcast(a_shape, a_rank, b_shape, b_rank, &st, &n, &an, &bn);
  if (rc) return rc;
  if (n == 0) return I8Q_OK;
  const auto* a8 = static_cast<const uint8_t*>(A);
  const auto* b8 = static_cast<const uint8_t*>(B);
  const bool as = atype == I8Q_S8, bs = btype == I8Q_S8;
  if (as && bs) return run_binary<true, true>(a8, b8, st, n, an, bn, p, C, s);
  if (as) return run_binary<true, false>(a8, b8, st, n, an, bn, p, C, s);
  if (bs) return run_binary<false, true>(a8, b8, st, n, an, bn, p, C, s);
  return run_binary<false, false>(a8, b8, st, n, an, bn, p, C, s);
}

bool in_range(int v, int type) { return type == I8Q_U8 ? (v >= 0 && v <= 255) : (v >= -128 && v <= 127); }

}  // namespace
}  // namespace i8q

using namespace i8q;

extern "C" int i8q_qlinear_binary(int op, const void* A, const int64_t* a_shape, int a_rank, float a_scale,
                                  int a_zero_point, const void* B, const int64_t* b_shape, int b_rank, float b_scale,
                                  int b_zero_point, float c_scale, int c_zero_point, int qtype, void* C,
                                  void* stream) {
  if (op != I8Q_QLINEAR_ADD && op != I8Q_QLINEAR_MUL) return fail(I8Q_ERR_INVALID_ARG, "qlinear_binary: unknown op");
  if (qtype != I8Q_U8 && qtype != I8Q_S8) return fail(I8Q_ERR_INVALID_ARG, "qlinear_binary: qtype must be U8 or S8");
  if (!A || !B || !C || (a_rank > 0 && !a_shape) || (b_rank > 0 && !b_shape))
    return fail(I8Q_ERR_INVALID_ARG, "qlinear_binary: A, B, C and the shapes are required");
  if (!in_range(a_zero_point, qtype) || !in_range(b_zero_point, qtype) || !in_range(c_zero_point, qtype))
    return fail(I8Q_ERR_INVALID_ARG, "qlinear_binary: a zero point is outside the type's range");
  BinParams p{};
  p.op = op == I8Q_QLINEAR_ADD ? 0 : 1;
  p.a_scale = a_scale;
  p.b_scale = b_scale;
  p.c_scale = c_scale;
  p.a_zp = a_zero_point;
  p.b_zp = b_zero_point;
  p.c_zp = c_zero_point;
  p.lo_z = (qtype == I8Q_U8 ? 0.0f : -128.0f) - (float)c_zero_point;
  p.hi_z = (qtype == I8Q_U8 ? 255.0f : 127.0f) - (float)c_zero_point;
  I8Q_PROF(op == I8Q_QLINEAR_ADD ? "qlinear_add" : "qlinear_mul", as_stream(stream));
  return binary_dispatch(A, qtype, a_shape, a_rank, B, qtype, b_shape, b_rank, p, C, as_stream(stream));
}

extern "C" int i8q_mul_integer(const void* A, int atype, const int64_t* a_shape, int a_rank, int a_zero_point,
                               const void* B, int btype, const int64_t* b_shape, int b_rank, int b_zero_point,
                               int32_t* C, void* stream) {
  if ((atype != I8Q_U8 && atype != I8Q_S8) || (btype != I8Q_U8 && btype != I8Q_S8))
    return fail(I8Q_ERR_INVALID_ARG, "mul_integer: A and B must be U8 or S8");
  if (!A || !B || !C || (a_rank > 0 && !a_shape) || (b_rank > 0 && !b_shape))
    return fail(I8Q_ERR_INVALID_ARG, "mul_integer: A, B, C and the shapes are required");
  if (!in_range(a_zero_point, atype) || !in_range(b_zero_point, btype))
    return fail(I8Q_ERR_INVALID_ARG, "mul_integer: a zero point is outside its type's range");
  BinParams p{};
  p.op = 2;
  p.a_zp = a_zero_point;
  p.b_zp = b_zero_point;
  I8Q_PROF("mul_integer", as_stream(stream));
  return binary_dispatch(A, atype, a_shape, a_rank, B, btype, b_shape, b_rank, p, C, as_stream(stream));
}

extern "C" int i8q_qlinear_unary(int op, const void* X, int64_t n, int qtype, float x_scale, int x_zero_point,
                                 float y_scale, int y_zero_point, float alpha, void* Y, void* stream) {
  if (op != I8Q_QLINEAR_LEAKY_RELU && op != I8Q_QLINEAR_SIGMOID)
    return fail(I8Q_ERR_INVALID_ARG, "qlinear_unary: unknown op");
  if (qtype != I8Q_U8 && qtype != I8Q_S8) return fail(I8Q_ERR_INVALID_ARG, "qlinear_unary: qtype must be U8 or S8");
  if (n < 0 || (n > 0 && (!X || !Y))) return fail(I8Q_ERR_INVALID_ARG, "qlinear_unary: X and Y are required");
  if (!in_range(x_zero_point, qtype) || !in_range(y_zero_point, qtype))
    return fail(I8Q_ERR_INVALID_ARG, "qlinear_unary: a zero point is outside the type's range");
  if (n == 0) return I8Q_OK;
  cudaStream_t s = as_stream(stream);
  const int o = op == I8Q_QLINEAR_LEAKY_RELU ? 0 : 1;
  const float lo_z = (qtype == I8Q_U8 ? 0.0f : -128.0f) - (float)y_zero_point;
  const float hi_z = (qtype == I8Q_U8 ? 255.0f : 127.0f) - (float)y_zero_point;
  // no more blocks than fit at once (each holds a 32 KB table): a second
  // wave of blocks would double the time of the SMs that run it
  int per_sm = 0;
  I8Q_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &per_sm, (qtype == I8Q_S8) ? unary_lut<true> : unary_lut<false>, 256, 0));
  const int grid = (int)std::max<int64_t>(
      1, std::min<int64_t>(ceil_div(n / 16, 256 * 8), (int64_t)sm_count() * std::max(per_sm, 1)));
  I8Q_PROF(o == 0 ? "qlinear_leaky_relu" : "qlinear_sigmoid", s);
  if (qtype == I8Q_S8)
    unary_lut<true><<<grid, 256, 0, s>>>(static_cast<const uint8_t*>(X), n, o, x_scale, x_zero_point, y_scale,
                                         y_zero_point, alpha, lo_z, hi_z, static_cast<uint8_t*>(Y));
  else
    unary_lut<false><<<grid, 256, 0, s>>>(static_cast<const uint8_t*>(X), n, o, x_scale, x_zero_point, y_scale,
                                          y_zero_point, alpha, lo_z, hi_z, static_cast<uint8_t*>(Y));
  I8Q_LAUNCH_CHECK("unary_lut");
  return I8Q_OK;
}
