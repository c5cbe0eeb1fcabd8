// gemm_tc.cu -- exact integer GEMM of the dynamic quantized inner product on
// the bf16 tensor pipe of sm_103a (tcgen05.mma kind::f16, TMEM accumulators,
// TMA-fed 128-byte-swizzled shared memory).
//
// sm_103a has no 8-bit integer tcgen05 form, but A's codes shifted to
// uA - 128 (-128..127) and B's int8 codes are exact in bf16, every product
// of two is exact in fp32 (|p| <= 2^14), and an fp32 sum of such products is
// exact while every partial sum is an integer of magnitude at most 2^24.  So
// the K loop is cut into chunks of CK = 2^24 / 2^max_abs_product_log2
// elements (1024 for int8 B, 2048 in the narrowed [-64,63] range): each
// chunk accumulates in fp32 in TMEM, then the epilogue warps drain it
// (tcgen05.ld), convert it exactly to int32 and add it to an int32 running
// sum held in registers.  Two TMEM chunk buffers let the tensor core fill
// one while the other drains.  The result is the exact int32
// sum_k (uA - 128) * iB; the fused epilogue adds back the shift with the
// zero point, -(zeroA - 128) * colsum, then applies the scales, bias,
// activation and the store, exactly as the IMMA core does.
//
// CTA tile 128 x 256, K step 64 (one 128-byte swizzle row of bf16), 4-stage
// smem ring (48 KB per stage), one CTA per SM, persistent over output tiles
// in a grouped order so the A and B panels in flight stay in L2.
// Warp roles: warp 0 issues TMA, warp 1 owns TMEM and issues the MMAs (one
// thread), warps 2..17 drain and run the epilogue: warp w reads TMEM lanes
// 32*(w%4).. (its rows) and the 64-column slice (w-2)/4 of the tile.  The
// final epilogue of a tile must finish within the two chunks the MMA can run
// ahead, so it is kept short: the slice's column parameters are staged once
// per tile in shared memory and full tiles store without bounds checks.
// Every mbarrier wait is bounded: on expiry the kernel records an error in
// the device status word (read by i8q_sync_status), waits (bounded) for its
// own copies and MMAs in flight, frees TMEM and returns.
#include "tcgen05.cuh"

namespace i8q {
namespace {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int STAGES = 4;
constexpr int A_STAGE = BM * BK * 2;  // 16 KB
constexpr int B_STAGE = BN * BK * 2;  // 32 KB
constexpr int STAGE_BYTES = A_STAGE + B_STAGE;
constexpr int NUM_EPI_WARPS = 16;
constexpr int SLICE = BN / (NUM_EPI_WARPS / 4);  // 64 columns per epilogue warp
constexpr int THREADS = 64 + NUM_EPI_WARPS * 32;
constexpr int TMEM_COLS = 512;
constexpr int NUM_BARS = 2 * STAGES + 4 + 1;
constexpr int PARAM_BYTES = NUM_EPI_WARPS * SLICE * 4 * 4;  // up to four column parameters per warp slice
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + PARAM_BYTES + NUM_BARS * 8 + 16;
constexpr int GROUP_M = 16;

// status codes written to the device status word
constexpr uint32_t ST_TIMEOUT_PRODUCER = 1u << 0;
constexpr uint32_t ST_TIMEOUT_MMA = 1u << 1;
constexpr uint32_t ST_TIMEOUT_EPILOGUE = 1u << 2;
constexpr uint32_t ST_TIMEOUT_DRAIN = 1u << 3;

struct TcParams {
  int64_t M, N;
  int KT;        // K steps of 64
  int CS;        // K steps per exact fp32 chunk
  int tiles_m, tiles_n;
  int num_tiles;
  GemmEpilogue ep;  // the dynamic quantized inner product (EPI_DYN)
  QgEpilogue qg;    // QGemm (EPI_QG)
  uint32_t* status;
};

// Epilogue kinds the kernels are instantiated for.
constexpr int EPI_DYN = 0, EPI_QG = 1;

using namespace tc;

constexpr uint32_t IDESC = idesc_bf16(BM, BN);

__device__ __forceinline__ void tile_coords(int tile, int tiles_m, int tiles_n, int& mt, int& nt) {
  const int per_group = GROUP_M * tiles_n;
  const int g = tile / per_group;
  const int first = g * GROUP_M;
  const int gsize = min(tiles_m - first, GROUP_M);
  const int r = tile - g * per_group;
  mt = first + r % gsize;
  nt = r / gsize;
}

// Eight dequantized and activated values of a row, columns j .. j + 7 of
// the slice.
template <int ACT, bool BF16>
__device__ __forceinline__ void epi8(const int32_t (&run)[SLICE], int j, int32_t zA, float sA, const int32_t* pc,
                                     const float* ps, const float* pb, float2 (&o)[4]) {
  const int4 c0 = *reinterpret_cast<const int4*>(pc + j), c1 = *reinterpret_cast<const int4*>(pc + j + 4);
  const float4 s0 = *reinterpret_cast<const float4*>(ps + j), s1 = *reinterpret_cast<const float4*>(ps + j + 4);
  const float4 b0 = *reinterpret_cast<const float4*>(pb + j), b1 = *reinterpret_cast<const float4*>(pb + j + 4);
  const int32_t cc[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const float2 sb[4] = {make_float2(s0.x, s0.y), make_float2(s0.z, s0.w), make_float2(s1.x, s1.y),
                        make_float2(s1.z, s1.w)};
  const float2 bb[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w), make_float2(b1.x, b1.y),
                        make_float2(b1.z, b1.w)};
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    // zA arrives shifted by 128.  Scalar operations: the compiler may
    // fuse a paired multiply and a following paired add.
    float2 v = make_float2(__int2float_rn(run[j + 2 * u] - zA * cc[2 * u]),
                           __int2float_rn(run[j + 2 * u + 1] - zA * cc[2 * u + 1]));
    v.x = __fadd_rn(__fmul_rn(__fmul_rn(v.x, sA), sb[u].x), bb[u].x);
    v.y = __fadd_rn(__fmul_rn(__fmul_rn(v.y, sA), sb[u].y), bb[u].y);
    if constexpr (ACT == I8Q_ACT_RELU) {
      v = make_float2(v.x > 0.0f ? v.x : 0.0f, v.y > 0.0f ? v.y : 0.0f);
    } else if constexpr (ACT == I8Q_ACT_GELU) {
      if constexpr (BF16)
        v = gelu_bf16out2(v);
      else
        v = make_float2(gelu_erf(v.x), gelu_erf(v.y));
    }
    o[u] = v;
  }
}

// Dequantized values of one row's 64-column slice, eight at a time, as
// ((float)sum * scaleA) * scaleB + bias (the roundings of dequant_epilogue),
// then the activation ACT (GELU on pairs for bf16 outputs), then stored as
// bf16 or fp32.  Column parameters come from shared
// memory: pc (colsum), ps (scaleB), pb (bias), SLICE entries each (zero
// beyond N), 16-byte aligned.
template <int ACT, bool BF16>
__device__ __forceinline__ void store_slice_float(const GemmEpilogue& ep, int64_t row, int64_t col0, int64_t N,
                                                  const int32_t (&run)[SLICE], int32_t zA, float sA,
                                                  const int32_t* pc, const float* ps, const float* pb, bool vec) {
#pragma unroll
  for (int j = 0; j < SLICE; j += 8) {
    float2 o[4];
    epi8<ACT, BF16>(run, j, zA, sA, pc, ps, pb, o);
    if constexpr (BF16) {
      __nv_bfloat16* C = static_cast<__nv_bfloat16*>(ep.C) + row * ep.ldc + col0 + j;
      __nv_bfloat162 h[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) h[u] = __float22bfloat162_rn(o[u]);
      if (vec) {
        uint4 pk;
        pk.x = *reinterpret_cast<uint32_t*>(&h[0]);
        pk.y = *reinterpret_cast<uint32_t*>(&h[1]);
        pk.z = *reinterpret_cast<uint32_t*>(&h[2]);
        pk.w = *reinterpret_cast<uint32_t*>(&h[3]);
        *reinterpret_cast<uint4*>(C) = pk;
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (col0 + j + u < N) C[u] = (u & 1) ? h[u >> 1].y : h[u >> 1].x;
      }
    } else {
      float* C = static_cast<float*>(ep.C) + row * ep.ldc + col0 + j;
      if (vec) {
        *reinterpret_cast<float4*>(C) = make_float4(o[0].x, o[0].y, o[1].x, o[1].y);
        *reinterpret_cast<float4*>(C + 4) = make_float4(o[2].x, o[2].y, o[3].x, o[3].y);
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (col0 + j + u < N) C[u] = (u & 1) ? o[u >> 1].y : o[u >> 1].x;
      }
    }
  }
}

// The epilogue of one row's 64-column slice from the exact sums in run[]
// (column parameters as for store_slice_float).
__device__ __forceinline__ void store_slice(const GemmEpilogue& ep, int64_t row, int64_t col0, int64_t N,
                                            const int32_t (&run)[SLICE], int32_t zA, float sA, const int32_t* pc,
                                            const float* ps, const float* pb) {
  const bool full = col0 + SLICE <= N;
  if (ep.out_mode == OUT_S32) {
    int32_t* C = static_cast<int32_t*>(ep.C) + row * ep.ldc + col0;
    const bool vec = full && (ep.ldc % 4 == 0) && (reinterpret_cast<uintptr_t>(ep.C) & 15) == 0;
#pragma unroll
    for (int j = 0; j < SLICE; j += 4) {
      const int4 c = *reinterpret_cast<const int4*>(pc + j);
      const int32_t v[4] = {run[j] - zA * c.x, run[j + 1] - zA * c.y, run[j + 2] - zA * c.z, run[j + 3] - zA * c.w};
      if (vec) {
        *reinterpret_cast<int4*>(C + j) = make_int4(v[0], v[1], v[2], v[3]);
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (col0 + j + u < N) C[j + u] = v[u];
      }
    }
    return;
  }
  const bool bf16 = ep.out_mode == OUT_BF16;
  const bool vec = full && (bf16 ? (ep.ldc % 8 == 0) : (ep.ldc % 4 == 0)) &&
                   (reinterpret_cast<uintptr_t>(ep.C) & 15) == 0;
#define I8Q_SLICE(A, B) store_slice_float<A, B>(ep, row, col0, N, run, zA, sA, pc, ps, pb, vec)
  if (bf16) {
    if (ep.act == I8Q_ACT_GELU) I8Q_SLICE(I8Q_ACT_GELU, true);
    else if (ep.act == I8Q_ACT_RELU) I8Q_SLICE(I8Q_ACT_RELU, true);
    else I8Q_SLICE(I8Q_ACT_IDENTITY, true);
  } else {
    if (ep.act == I8Q_ACT_GELU) I8Q_SLICE(I8Q_ACT_GELU, false);
    else if (ep.act == I8Q_ACT_RELU) I8Q_SLICE(I8Q_ACT_RELU, false);
    else I8Q_SLICE(I8Q_ACT_IDENTITY, false);
  }
#undef I8Q_SLICE
}

// The same slice for bf16 outputs, stored by TMA: the warp's 32 rows
// (row0 .. row0 + 31, lane = row) go out in 16-column chunks through the
// warp's 1 KB staging buffer (32 rows x 32 bytes, dense), one bulk store
// per chunk issued by lane 0 once the previous one has read the buffer.
// Rows and columns past the tensor are clipped by the store itself.  The
// chunk loop is rolled (the sums shift down by 16 after each chunk, which
// consumes run[]): the unrolled form's larger code ran 1 % slower.
template <int ACT>
__device__ __forceinline__ void store_slice_tma(const CUtensorMap* tmC, int64_t M, int64_t N, int64_t row0,
                                                int64_t col0, int lane, int32_t (&run)[SLICE], int32_t zA,
                                                float sA, const int32_t* pc, const float* ps, const float* pb,
                                                uint8_t* stg) {
  const uint32_t stg_s = smem_u32(stg);
#pragma unroll 1
  for (int ch = 0; ch < SLICE / 16; ++ch) {
    uint32_t wd[8];
#pragma unroll
    for (int hg = 0; hg < 2; ++hg) {
      float2 o[4];
      epi8<ACT, true>(run, hg * 8, zA, sA, pc + ch * 16, ps + ch * 16, pb + ch * 16, o);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const __nv_bfloat162 hv = __float22bfloat162_rn(o[u]);
        wd[hg * 4 + u] = *reinterpret_cast<const uint32_t*>(&hv);
      }
    }
#pragma unroll
    for (int i = 0; i < SLICE - 16; ++i) run[i] = run[i + 16];
    if (lane == 0) bulk_wait_read();
    __syncwarp();
    uint4* d = reinterpret_cast<uint4*>(stg + lane * 32);
    d[0] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
    d[1] = make_uint4(wd[4], wd[5], wd[6], wd[7]);
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    __syncwarp();
    if (lane == 0) {
      const int64_t x = col0 + ch * 16;
      if (x < N && row0 < M) {
        tma_store_2d(tmC, stg_s, (int)x, (int)row0);
        bulk_commit();
      }
    }
  }
}

// The same slice for fp32 outputs: 8-column chunks (32 rows x 32 bytes)
// through the warp's staging buffer, one bulk store each.
template <int ACT>
__device__ __forceinline__ void store_slice_tma_f32(const CUtensorMap* tmC, int64_t M, int64_t N, int64_t row0,
                                                    int64_t col0, int lane, const int32_t (&run)[SLICE], int32_t zA,
                                                    float sA, const int32_t* pc, const float* ps, const float* pb,
                                                    uint8_t* stg) {
  const uint32_t stg_s = smem_u32(stg);
#pragma unroll
  for (int ch = 0; ch < SLICE / 8; ++ch) {
    float2 o[4];
    epi8<ACT, false>(run, ch * 8, zA, sA, pc, ps, pb, o);
    if (lane == 0) bulk_wait_read();
    __syncwarp();
    uint4* d = reinterpret_cast<uint4*>(stg + lane * 32);
    d[0] = make_uint4(__float_as_uint(o[0].x), __float_as_uint(o[0].y), __float_as_uint(o[1].x),
                      __float_as_uint(o[1].y));
    d[1] = make_uint4(__float_as_uint(o[2].x), __float_as_uint(o[2].y), __float_as_uint(o[3].x),
                      __float_as_uint(o[3].y));
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    __syncwarp();
    if (lane == 0) {
      const int64_t x = col0 + ch * 8;
      if (x < N && row0 < M) {
        tma_store_2d(tmC, stg_s, (int)x, (int)row0);
        bulk_commit();
      }
    }
  }
}

// Epilogue of one row's 64-column slice for the 8-bit-code products (see
// QgEpilogue): column parameters pg (g), pe (e), pb (bsc), pz (bias) from
// shared memory; rs, dr, ar: the row's rowsum, d and asc.
__device__ __forceinline__ void store_slice_qg(const QgEpilogue& qg, int64_t row, int64_t col0, int64_t N,
                                               const int32_t (&run)[SLICE], int32_t rs, int32_t dr, float ar,
                                               const int32_t* pg, const int32_t* pe, const float* pb,
                                               const float* pz) {
  const bool full = col0 + SLICE <= N;
  const int32_t* crow = (qg.C && !qg.c_col) ? qg.C + row * qg.c_si : nullptr;
  const bool has_bias = qg.bias != nullptr;
  auto value_at = [&](int j) -> float {
    // wrapping int32 arithmetic: the exact sum fits int32
    uint32_t a = (uint32_t)run[j] + (uint32_t)rs * (uint32_t)pg[j] + (uint32_t)dr * (uint32_t)pe[j];
    if (qg.c_col) a += (uint32_t)__float_as_int(pz[j]);
    if (crow && col0 + j < N) a += (uint32_t)__ldg(crow + (col0 + j) * qg.c_sj);
    float v = __fmul_rn(__int2float_rn((int32_t)a), __fmul_rn(ar, pb[j]));
    if (has_bias) v = __fadd_rn(v, pz[j]);
    return v;
  };
  if (qg.ytype == I8Q_F32) {
    float* Y = static_cast<float*>(qg.Y) + row * qg.ldy + col0;
    const bool vec = full && (qg.ldy % 4 == 0) && (reinterpret_cast<uintptr_t>(qg.Y) & 15) == 0;
#pragma unroll
    for (int j = 0; j < SLICE; j += 4) {
      float o[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) o[u] = value_at(j + u);
      if (vec) {
        *reinterpret_cast<float4*>(Y + j) = make_float4(o[0], o[1], o[2], o[3]);
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (col0 + j + u < N) Y[j + u] = o[u];
      }
    }
    return;
  }
  const int zp = qg.y_zero_point;
  const float lo = (qg.ytype == I8Q_U8 ? 0.0f : -128.0f) - (float)zp;
  const float hi = (qg.ytype == I8Q_U8 ? 255.0f : 127.0f) - (float)zp;
  uint8_t* Y = static_cast<uint8_t*>(qg.Y) + row * qg.ldy + col0;
  const bool vec = full && (qg.ldy % 16 == 0) && (reinterpret_cast<uintptr_t>(qg.Y) & 15) == 0;
#pragma unroll
  for (int j = 0; j < SLICE; j += 16) {
    uint32_t b[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) b[u] = quot_code_bits(value_at(j + u), qg.y_scale, qg.y_rcp, lo, hi, zp);
    if (vec) {
      *reinterpret_cast<uint4*>(Y + j) =
          make_uint4(pack_low_bytes(b[0], b[1], b[2], b[3]), pack_low_bytes(b[4], b[5], b[6], b[7]),
                     pack_low_bytes(b[8], b[9], b[10], b[11]), pack_low_bytes(b[12], b[13], b[14], b[15]));
    } else {
#pragma unroll
      for (int u = 0; u < 16; ++u)
        if (col0 + j + u < N) Y[j + u] = (uint8_t)b[u];
    }
  }
}

// The 8-bit-code products' slice stored by TMA (fp32 Y in 8-column chunks,
// 8-bit Y in 32-column chunks, 32 bytes per row either way) through the
// warp's staging buffer, as store_slice_tma.  Rows past M hold zeros in
// their parameters (never stored: the store clips them).
__device__ __forceinline__ void store_slice_qg_tma(const QgEpilogue& qg, const CUtensorMap* tmY, int64_t M,
                                                   int64_t N, int64_t row0, int64_t col0, int lane,
                                                   const int32_t (&run)[SLICE], int32_t rs, int32_t dr, float ar,
                                                   const int32_t* pg, const int32_t* pe, const float* pb,
                                                   const float* pz, uint8_t* stg) {
  const int64_t row = row0 + lane;
  const int32_t* crow = (qg.C && !qg.c_col && row < M) ? qg.C + row * qg.c_si : nullptr;
  const bool has_bias = qg.bias != nullptr;
  auto value_at = [&](int j) -> float {
    uint32_t a = (uint32_t)run[j] + (uint32_t)rs * (uint32_t)pg[j] + (uint32_t)dr * (uint32_t)pe[j];
    if (qg.c_col) a += (uint32_t)__float_as_int(pz[j]);
    if (crow && col0 + j < N) a += (uint32_t)__ldg(crow + (col0 + j) * qg.c_sj);
    float v = __fmul_rn(__int2float_rn((int32_t)a), __fmul_rn(ar, pb[j]));
    if (has_bias) v = __fadd_rn(v, pz[j]);
    return v;
  };
  const uint32_t stg_s = smem_u32(stg);
  auto put = [&](const uint32_t (&wd)[8], int64_t x) {
    if (lane == 0) bulk_wait_read();
    __syncwarp();
    uint4* d = reinterpret_cast<uint4*>(stg + lane * 32);
    d[0] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
    d[1] = make_uint4(wd[4], wd[5], wd[6], wd[7]);
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    __syncwarp();
    if (lane == 0 && x < N && row0 < M) {
      tma_store_2d(tmY, stg_s, (int)x, (int)row0);
      bulk_commit();
    }
  };
  if (qg.ytype == I8Q_F32) {
#pragma unroll
    for (int j = 0; j < SLICE; j += 8) {
      uint32_t wd[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) wd[u] = __float_as_uint(value_at(j + u));
      put(wd, col0 + j);
    }
    return;
  }
  const int zp = qg.y_zero_point;
  const float lo = (qg.ytype == I8Q_U8 ? 0.0f : -128.0f) - (float)zp;
  const float hi = (qg.ytype == I8Q_U8 ? 255.0f : 127.0f) - (float)zp;
#pragma unroll
  for (int j = 0; j < SLICE; j += 32) {
    uint32_t wd[8];
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      uint32_t b[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) b[u] = quot_code_bits(value_at(j + 4 * w + u), qg.y_scale, qg.y_rcp, lo, hi, zp);
      wd[w] = pack_low_bytes(b[0], b[1], b[2], b[3]);
    }
    put(wd, col0 + j);
  }
}

// Stage one epilogue warp's column parameters for the tile (read back after
// the K loop).
template <int EPI>
__device__ __forceinline__ void stage_params(const TcParams& p, int64_t col0, int lane, int32_t* pc, float* ps,
                                             float* pb, float* pd) {
  for (int j = lane; j < SLICE; j += 32) {
    const int64_t c = col0 + j;
    const bool in = c < p.N;
    if constexpr (EPI == EPI_DYN) {
      pc[j] = in ? __ldg(p.ep.colsum + c) : 0;
      ps[j] = in ? __ldg(p.ep.scaleB + c) : 0.0f;
      pb[j] = (in && p.ep.bias) ? __ldg(p.ep.bias + c) : 0.0f;
    } else {
      pc[j] = in ? __ldg(p.qg.g + c) : 0;
      reinterpret_cast<int32_t*>(ps)[j] = in ? __ldg(p.qg.e + c) : 0;
      pb[j] = in ? __ldg(p.qg.bsc + c) : 0.0f;
      if (p.qg.c_col)  // the row-independent C, as int32 bits in the bias slot
        reinterpret_cast<int32_t*>(pd)[j] = in ? __ldg(p.qg.C + c * p.qg.c_sj) : 0;
      else
        pd[j] = (in && p.qg.bias) ? __ldg(p.qg.bias + c) : 0.0f;
    }
  }
}

// The epilogue of one row of the tile from its exact sums.
template <int EPI>
__device__ __forceinline__ void finish_row(const TcParams& p, int64_t row, int64_t col0, const int32_t (&run)[SLICE],
                                           const int32_t* pc, const float* ps, const float* pb, const float* pd) {
  if constexpr (EPI == EPI_DYN) {
    const float sA = __ldg(p.ep.scaleA + row);
    // A entered as uA - 128: sum_k (uA - zA) iB = run - (zA - 128) colsum
    const int32_t zA = __ldg(p.ep.zeroA + row) - 128;
    store_slice(p.ep, row, col0, p.N, run, zA, sA, pc, ps, pb);
  } else {
    store_slice_qg(p.qg, row, col0, p.N, run, __ldg(p.qg.rowsum + row), __ldg(p.qg.d + row * p.qg.d_stride),
                   __ldg(p.qg.asc + row * p.qg.asc_stride), pc, reinterpret_cast<const int32_t*>(ps), pb, pd);
  }
}

template <int EPI>
__global__ void __launch_bounds__(THREADS, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned, indexed from the shared array itself so that accesses stay shared-space
  uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* params = smem + STAGES * STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(params + PARAM_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t smem0 = smem_u32(smem);
  auto sA = [&](int s) { return smem0 + (uint32_t)(s * STAGE_BYTES); };
  auto sB = [&](int s) { return smem0 + (uint32_t)(s * STAGE_BYTES + A_STAGE); };
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto empty = [&](int s) { return smem_u32(bars + STAGES + s); };
  auto accf = [&](int b) { return smem_u32(bars + 2 * STAGES + b); };
  auto acce = [&](int b) { return smem_u32(bars + 2 * STAGES + 2 + b); };
  const uint32_t fin = smem_u32(bars + 2 * STAGES + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf(b), 1);
      mbar_init(acce(b), NUM_EPI_WARPS);
    }
    mbar_init(fin, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int KT = p.KT, CS = p.CS;
  const int nchunks = (KT + CS - 1) / CS;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        int mt, nt;
        tile_coords(tile, p.tiles_m, p.tiles_n, mt, nt);
        for (int kt = 0; kt < KT; ++kt, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
          if (!wait_bar(empty(s), ph ^ 1u, abort_flag, p.status, ST_TIMEOUT_PRODUCER)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full(s), STAGE_BYTES);
          tma_load_2d(sA(s), &tmA, full(s), kt * BK, mt * BM);
          tma_load_2d(sB(s), &tmB, full(s), kt * BK, nt * BN);
        }
      }
      if (!ok) {
        // let the copies already issued land before the CTA exits
        for (int j = max(0, it - STAGES); j < it; ++j) {
          unsigned long long t0 = global_ns();
          while (!mbar_try_wait(full(j % STAGES), (uint32_t)(j / STAGES) & 1u))
            if (global_ns() - t0 > WAIT_LIMIT_NS) {
              atomicOr(p.status, ST_TIMEOUT_DRAIN);
              break;
            }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      int it = 0, chunk = 0;
      bool ok = true;
      uint32_t d = tmem_base;
      if (KT % STAGES == 0) {
        // every tile starts at stage 0: the K loop unrolled by the ring's
        // length, stage indices and descriptor offsets constant (as in the
        // pair kernel)
        const uint64_t a0 = desc_sw128(sA(0)), b0 = desc_sw128(sB(0));
        constexpr uint64_t STAGE_STEP = STAGE_BYTES >> 4, K_STEP = 32 >> 4;
        uint32_t ph = 0;
        int kc = 0;
        for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
          for (int kt0 = 0; ok && kt0 < KT; kt0 += STAGES) {
#pragma unroll
            for (int j = 0; j < STAGES; ++j) {
              if (kc == 0) {
                const int b = chunk & 1;
                if (!wait_bar(acce(b), ((uint32_t)(chunk >> 1) & 1u) ^ 1u, abort_flag, p.status, ST_TIMEOUT_MMA)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                d = tmem_base + (uint32_t)(b * BN);
              }
              if (!wait_bar(full(j), ph, abort_flag, p.status, ST_TIMEOUT_MMA)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t ad = a0 + (uint64_t)j * STAGE_STEP, bd = b0 + (uint64_t)j * STAGE_STEP;
#pragma unroll
              for (int k = 0; k < BK / 16; ++k)
                tc_mma(d, ad + k * K_STEP, bd + k * K_STEP, IDESC, (kc == 0 && k == 0) ? 0u : 1u);
              tc_commit(empty(j));
              if (++kc == CS || kt0 + j == KT - 1) {
                tc_commit(accf(chunk & 1));
                ++chunk;
                kc = 0;
              }
            }
            ph ^= 1u;
          }
        }
      }
      for (int tile = blockIdx.x; ok && KT % STAGES != 0 && tile < p.num_tiles; tile += gridDim.x) {
        for (int kt = 0; kt < KT; ++kt, ++it) {
          const int kc = kt % CS;
          if (kc == 0) {
            const int b = chunk & 1;
            if (!wait_bar(acce(b), ((uint32_t)(chunk >> 1) & 1u) ^ 1u, abort_flag, p.status, ST_TIMEOUT_MMA)) {
              ok = false;
              break;
            }
            tc_fence_after();
            d = tmem_base + (uint32_t)(b * BN);
          }
          const int s = it % STAGES;
          if (!wait_bar(full(s), (uint32_t)(it / STAGES) & 1u, abort_flag, p.status, ST_TIMEOUT_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t ad = desc_sw128(sA(s) + (uint32_t)(k * 32));
            const uint64_t bd = desc_sw128(sB(s) + (uint32_t)(k * 32));
            tc_mma(d, ad, bd, IDESC, (kc == 0 && k == 0) ? 0u : 1u);
          }
          tc_commit(empty(s));
          if (kc == CS - 1 || kt == KT - 1) {
            tc_commit(accf(chunk & 1));
            ++chunk;
          }
        }
      }
      // all MMAs issued by this thread complete before TMEM is released
      tc_commit(fin);
      unsigned long long t0 = global_ns();
      while (!mbar_try_wait(fin, 0))
        if (global_ns() - t0 > WAIT_LIMIT_NS) {
          atomicOr(p.status, ST_TIMEOUT_DRAIN);
          break;
        }
    }
  } else {
    // ---------------- drain + epilogue ----------------
    const int q = warp & 3;               // TMEM lane quadrant of this warp (its 32 rows)
    const int slice = (warp - 2) >> 2;    // which 64 of the 256 columns
    int32_t* pc = reinterpret_cast<int32_t*>(params) + (warp - 2) * SLICE * 4;
    float* ps = reinterpret_cast<float*>(pc + SLICE);
    float* pb = ps + SLICE;
    float* pd = pb + SLICE;
    int chunk = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
      int mt, nt;
      tile_coords(tile, p.tiles_m, p.tiles_n, mt, nt);
      const int64_t col0 = (int64_t)nt * BN + slice * SLICE;
      // stage this slice's column parameters (read back after the K loop)
      stage_params<EPI>(p, col0, lane, pc, ps, pb, pd);
      int32_t run[SLICE];
#pragma unroll
      for (int j = 0; j < SLICE; ++j) run[j] = 0;
      for (int c = 0; c < nchunks; ++c, ++chunk) {
        const int b = chunk & 1;
        // every lane waits; the outcome is made warp-uniform before the
        // warp-collective TMEM loads
        const bool got = wait_bar(accf(b), (uint32_t)(chunk >> 1) & 1u, abort_flag, p.status, ST_TIMEOUT_EPILOGUE);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * BN + slice * SLICE);
#pragma unroll
        for (int j = 0; j < SLICE / 16; j += 2) {
          uint32_t r0[16], r1[16];
          tmem_ld16(taddr + (uint32_t)(j * 16), r0);
          tmem_ld16(taddr + (uint32_t)(j * 16 + 16), r1);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            run[j * 16 + i] += __float2int_rn(__uint_as_float(r0[i]));
            run[j * 16 + 16 + i] += __float2int_rn(__uint_as_float(r1[i]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce(b));
      }
      if (!ok) break;
      __syncwarp();
      const int64_t row = (int64_t)mt * BM + q * 32 + lane;
      if (row < p.M) finish_row<EPI>(p, row, col0, run, pc, ps, pb, pd);
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---- CTA-pair kernel -------------------------------------------------------
// A cluster of two CTAs computes 256 x 256 output tiles with one
// tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16) per 16 K elements:
// CTA r of the pair holds rows 128r..128r+127 of the A tile and rows
// 128r..128r+127 of the B tile (output columns) in its shared memory, and
// the accumulator rows 128r.. in its TMEM.  Per SM this halves the bytes the
// tensor core reads from shared memory and the bytes TMA writes there per
// multiply-add, compared with the 128 x 256 single-CTA tile, where the two
// together exceed the shared-memory bandwidth before the tensor pipe is full.
// Roles as in the single-CTA kernel; the even CTA of the pair (the leader)
// issues the MMAs and owns the stage-full and accumulator-empty barriers:
// both CTAs' TMA loads complete on the leader's stage barrier, and both
// CTAs' epilogue warps arrive on its accumulator-empty barrier.  The MMA
// commits arrive on the stage-empty and accumulator-full barriers of both
// CTAs (multicast).
constexpr int PBM = 256, PBN = 256;
constexpr int HALF_ROWS = 128;
constexpr int P_STAGES = 4;
constexpr int P_A_STAGE = HALF_ROWS * BK * 2;  // 16 KB
constexpr int P_B_STAGE = HALF_ROWS * BK * 2;  // 16 KB
constexpr int P_STAGE_BYTES = P_A_STAGE + P_B_STAGE;
constexpr int P_NUM_BARS = 2 * P_STAGES + 4 + 1;
constexpr int P_STG_BYTES = NUM_EPI_WARPS * 1024;  // per-warp staging of bf16 C (32 rows x 32 bytes)
constexpr int P_SMEM_BYTES = 1024 + P_STAGES * P_STAGE_BYTES + PARAM_BYTES + P_STG_BYTES + P_NUM_BARS * 8 + 16;
constexpr int P_GROUP_M = 16;
constexpr uint32_t IDESC_PAIR = idesc_bf16(PBM, PBN);
static_assert(P_SMEM_BYTES <= 227 * 1024, "shared memory of the pair kernel");

__device__ __forceinline__ void tile_coords_g(int tile, int tiles_m, int tiles_n, int group, int& mt, int& nt) {
  const int per_group = group * tiles_n;
  const int g = tile / per_group;
  const int first = g * group;
  const int gsize = min(tiles_m - first, group);
  const int r = tile - g * per_group;
  mt = first + r % gsize;
  nt = r / gsize;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;\n" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t num_clusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;\n" : "=r"(r));
  return r;
}

// TMA_C: outputs stored by TMA through per-warp staging (1: the 8-bit-code
// products' Y, or bf16 C of EPI_DYN; 2: fp32 C of EPI_DYN); 0: stored
// directly.
template <int EPI, int TMA_C = 0>
__global__ void __launch_bounds__(THREADS, 1)
gemm_tc_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned, indexed from the shared array itself so that accesses stay shared-space
  uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* params = smem + P_STAGES * P_STAGE_BYTES;
  uint8_t* stg_all = params + PARAM_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(stg_all + P_STG_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + P_NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t smem0 = smem_u32(smem);
  auto sA = [&](int s) { return smem0 + (uint32_t)(s * P_STAGE_BYTES); };
  auto sB = [&](int s) { return smem0 + (uint32_t)(s * P_STAGE_BYTES + P_A_STAGE); };
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto empty = [&](int s) { return smem_u32(bars + P_STAGES + s); };
  auto accf = [&](int b) { return smem_u32(bars + 2 * P_STAGES + b); };
  auto acce = [&](int b) { return smem_u32(bars + 2 * P_STAGES + 2 + b); };
  const uint32_t fin = smem_u32(bars + 2 * P_STAGES + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int cid = (int)cluster_id_x(), ncl = (int)num_clusters_x();
  if (threadIdx.x == 0) {
    for (int s = 0; s < P_STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf(b), 1);
      mbar_init(acce(b), 2 * NUM_EPI_WARPS);
    }
    mbar_init(fin, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  // the peer's barriers are initialised before any remote arrival or copy
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int KT = p.KT, CS = p.CS;
  const int nchunks = (KT + CS - 1) / CS;

  if (warp == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    if (lane == 0) {
      int it = 0, s = 0;
      uint32_t ph = 0;  // phase parity of stage s
      bool ok = true;
      const uint32_t full0 = map_shared_rank(full(0), 0);  // the leader's stage barriers
      for (int tile = cid; ok && tile < p.num_tiles; tile += ncl) {
        int mt, nt;
        tile_coords_g(tile, p.tiles_m, p.tiles_n, P_GROUP_M, mt, nt);
        const int ya = mt * PBM + (int)rank * HALF_ROWS, yb = nt * PBN + (int)rank * HALF_ROWS;
        for (int kt = 0; kt < KT; ++kt, ++it) {
          if (!wait_bar<true>(empty(s), ph ^ 1u, abort_flag, p.status, ST_TIMEOUT_PRODUCER)) {
            ok = false;
            break;
          }
          const uint32_t fb = full0 + (uint32_t)(s * 8);
          if (leader) mbar_arrive_expect_tx(full(s), 2 * P_STAGE_BYTES);
          tma_load_2d_pair(sA(s), &tmA, fb, kt * BK, ya);
          tma_load_2d_pair(sB(s), &tmB, fb, kt * BK, yb);
          if (++s == P_STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // Wait until the MMAs have released every stage: the last commits
      // arrive on this CTA's stage-empty barriers, which must not outlive it.
      if (ok) {
        for (int j = it; j < it + P_STAGES; ++j)
          if (!wait_bar<true>(empty(j % P_STAGES), ((uint32_t)(j / P_STAGES) & 1u) ^ 1u, abort_flag, p.status,
                              ST_TIMEOUT_DRAIN))
            break;
      } else if (leader) {
        for (int j = max(0, it - P_STAGES); j < it; ++j) {
          unsigned long long t0 = global_ns();
          while (!mbar_try_wait_cluster(full(j % P_STAGES), (uint32_t)(j / P_STAGES) & 1u))
            if (global_ns() - t0 > WAIT_LIMIT_NS) {
              atomicOr(p.status, ST_TIMEOUT_DRAIN);
              break;
            }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (leader CTA) ----------------
    if (leader && lane == 0) {
      // Kept lean: this one thread feeds the tensor pipe and shares its
      // sub-partition with epilogue warps, so stage, phase and chunk are
      // counters and the descriptors advance by addition (the start-address
      // field holds address / 16; the sums stay inside shared memory).
      int s = 0, kc = 0, chunk = 0;
      uint32_t ph = 0, cph = 0;  // stage phase; accumulator-buffer phase
      bool ok = true;
      uint32_t d = tmem_base;
      const uint64_t a0 = desc_sw128(sA(0)), b0 = desc_sw128(sB(0));
      constexpr uint64_t STAGE_STEP = P_STAGE_BYTES >> 4, K_STEP = 32 >> 4;
      if (KT % P_STAGES == 0) {
        // every tile starts at stage 0: the K loop unrolled by the ring's
        // length, stage indices and descriptor offsets constant (the issue
        // loop of one thread sets the pace of these MMAs; unrolled, the
        // kernel ran 9 % faster than with a six-stage ring and counters)
        for (int tile = cid; ok && tile < p.num_tiles; tile += ncl) {
          for (int kt0 = 0; ok && kt0 < KT; kt0 += P_STAGES) {
#pragma unroll
            for (int j = 0; j < P_STAGES; ++j) {
              if (kc == 0) {
                const int b = chunk & 1;
                if (!wait_bar<true>(acce(b), cph ^ 1u, abort_flag, p.status, ST_TIMEOUT_MMA)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                d = tmem_base + (uint32_t)(b * PBN);
              }
              if (!wait_bar<true>(full(j), ph, abort_flag, p.status, ST_TIMEOUT_MMA)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t ad = a0 + (uint64_t)j * STAGE_STEP, bd = b0 + (uint64_t)j * STAGE_STEP;
              tc_mma_pair(d, ad, bd, IDESC_PAIR, kc == 0 ? 0u : 1u);
#pragma unroll
              for (int k = 1; k < BK / 16; ++k) tc_mma_pair(d, ad + k * K_STEP, bd + k * K_STEP, IDESC_PAIR, 1u);
              tc_commit_pair_mc(empty(j), 0x3);
              if (++kc == CS || kt0 + j == KT - 1) {
                tc_commit_pair_mc(accf(chunk & 1), 0x3);
                ++chunk;
                kc = 0;
                if ((chunk & 1) == 0) cph ^= 1u;
              }
            }
            ph ^= 1u;
          }
        }
      }
      for (int tile = cid; ok && KT % P_STAGES != 0 && tile < p.num_tiles; tile += ncl) {
        for (int kt = 0; kt < KT; ++kt) {
          if (kc == 0) {
            const int b = chunk & 1;
            if (!wait_bar<true>(acce(b), cph ^ 1u, abort_flag, p.status, ST_TIMEOUT_MMA)) {
              ok = false;
              break;
            }
            tc_fence_after();
            d = tmem_base + (uint32_t)(b * PBN);
          }
          if (!wait_bar<true>(full(s), ph, abort_flag, p.status, ST_TIMEOUT_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = a0 + (uint64_t)s * STAGE_STEP, bd = b0 + (uint64_t)s * STAGE_STEP;
          tc_mma_pair(d, ad, bd, IDESC_PAIR, kc == 0 ? 0u : 1u);
#pragma unroll
          for (int k = 1; k < BK / 16; ++k) tc_mma_pair(d, ad + k * K_STEP, bd + k * K_STEP, IDESC_PAIR, 1u);
          tc_commit_pair_mc(empty(s), 0x3);
          if (++kc == CS || kt == KT - 1) {
            tc_commit_pair_mc(accf(chunk & 1), 0x3);
            ++chunk;
            kc = 0;
            if ((chunk & 1) == 0) cph ^= 1u;
          }
          if (++s == P_STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // all MMAs issued by this thread complete before either CTA releases
      // its TMEM or its shared memory
      tc_commit_pair_mc(fin, 0x1);
      unsigned long long t0 = global_ns();
      while (!mbar_try_wait_cluster(fin, 0))
        if (global_ns() - t0 > WAIT_LIMIT_NS) {
          atomicOr(p.status, ST_TIMEOUT_DRAIN);
          break;
        }
    }
  } else {
    // ---------------- drain + epilogue (both CTAs) ----------------
    const int q = warp & 3;
    const int slice = (warp - 2) >> 2;
    int32_t* pc = reinterpret_cast<int32_t*>(params) + (warp - 2) * SLICE * 4;
    float* ps = reinterpret_cast<float*>(pc + SLICE);
    float* pb = ps + SLICE;
    float* pd = pb + SLICE;
    const uint32_t acce_leader0 = map_shared_rank(acce(0), 0), acce_leader1 = map_shared_rank(acce(1), 0);
    int chunk = 0;
    bool ok = true;
    for (int tile = cid; ok && tile < p.num_tiles; tile += ncl) {
      int mt, nt;
      tile_coords_g(tile, p.tiles_m, p.tiles_n, P_GROUP_M, mt, nt);
      const int64_t col0 = (int64_t)nt * PBN + slice * SLICE;
      stage_params<EPI>(p, col0, lane, pc, ps, pb, pd);
      int32_t run[SLICE];
#pragma unroll
      for (int j = 0; j < SLICE; ++j) run[j] = 0;
      for (int c = 0; c < nchunks; ++c, ++chunk) {
        const int b = chunk & 1;
        const bool got =
            wait_bar<true>(accf(b), (uint32_t)(chunk >> 1) & 1u, abort_flag, p.status, ST_TIMEOUT_EPILOGUE);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * PBN + slice * SLICE);
#pragma unroll
        for (int j = 0; j < SLICE / 16; j += 2) {
          uint32_t r0[16], r1[16];
          tmem_ld16(taddr + (uint32_t)(j * 16), r0);
          tmem_ld16(taddr + (uint32_t)(j * 16 + 16), r1);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            run[j * 16 + i] += __float2int_rn(__uint_as_float(r0[i]));
            run[j * 16 + 16 + i] += __float2int_rn(__uint_as_float(r1[i]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(b ? acce_leader1 : acce_leader0);
      }
      if (!ok) break;
      __syncwarp();
      const int64_t row0 = (int64_t)mt * PBM + (int64_t)rank * HALF_ROWS + q * 32, row = row0 + lane;
      if constexpr (EPI == EPI_QG && TMA_C) {
        const bool in = row < p.M;
        const int32_t rs = in ? __ldg(p.qg.rowsum + row) : 0;
        const int32_t dr = in ? __ldg(p.qg.d + row * p.qg.d_stride) : 0;
        const float ar = in ? __ldg(p.qg.asc + row * p.qg.asc_stride) : 0.0f;
        store_slice_qg_tma(p.qg, &tmC, p.M, p.N, row0, col0, lane, run, rs, dr, ar, pc,
                           reinterpret_cast<const int32_t*>(ps), pb, pd, stg_all + (warp - 2) * 1024);
        __syncwarp();
        continue;
      }
      if constexpr (EPI == EPI_DYN && TMA_C == 1) {
        {
          const bool in = row < p.M;
          const float sA = in ? __ldg(p.ep.scaleA + row) : 0.0f;
          const int32_t zA = in ? __ldg(p.ep.zeroA + row) - 128 : 0;  // A entered as uA - 128
          uint8_t* stg = stg_all + (warp - 2) * 1024;
          if (p.ep.act == I8Q_ACT_GELU)
            store_slice_tma<I8Q_ACT_GELU>(&tmC, p.M, p.N, row0, col0, lane, run, zA, sA, pc, ps, pb, stg);
          else if (p.ep.act == I8Q_ACT_RELU)
            store_slice_tma<I8Q_ACT_RELU>(&tmC, p.M, p.N, row0, col0, lane, run, zA, sA, pc, ps, pb, stg);
          else
            store_slice_tma<I8Q_ACT_IDENTITY>(&tmC, p.M, p.N, row0, col0, lane, run, zA, sA, pc, ps, pb, stg);
          __syncwarp();
          continue;
        }
      }
      if constexpr (EPI == EPI_DYN && TMA_C == 2) {
        const bool in = row < p.M;
        const float sA = in ? __ldg(p.ep.scaleA + row) : 0.0f;
        const int32_t zA = in ? __ldg(p.ep.zeroA + row) - 128 : 0;  // A entered as uA - 128
        uint8_t* stg = stg_all + (warp - 2) * 1024;
        if (p.ep.act == I8Q_ACT_GELU)
          store_slice_tma_f32<I8Q_ACT_GELU>(&tmC, p.M, p.N, row0, col0, lane, run, zA, sA, pc, ps, pb, stg);
        else if (p.ep.act == I8Q_ACT_RELU)
          store_slice_tma_f32<I8Q_ACT_RELU>(&tmC, p.M, p.N, row0, col0, lane, run, zA, sA, pc, ps, pb, stg);
        else
          store_slice_tma_f32<I8Q_ACT_IDENTITY>(&tmC, p.M, p.N, row0, col0, lane, run, zA, sA, pc, ps, pb, stg);
        __syncwarp();
        continue;
      }
      if (row < p.M) finish_row<EPI>(p, row, col0, run, pc, ps, pb, pd);
      __syncwarp();
    }
    // the bulk stores are complete before the CTA leaves
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  // the leader's MMAs into this CTA's TMEM and its arrivals here are done
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// Clusters of two CTAs of the pair kernel that fit on the current device
// at once (0 when none do; -1 on a CUDA error), computed once per
// instantiation and device.
template <int EPI>
int pair_max_clusters() {
  static int n[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return fail(I8Q_ERR_CUDA, "gemm_tc: no device"), -1;
  const int rc = once_per_device((const void*)&n, [](void* p) -> int {
    int* out = static_cast<int*>(p);
    cudaError_t err = cudaFuncSetAttribute(gemm_tc_pair_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           P_SMEM_BYTES);
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(gemm_tc_pair_kernel<EPI, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 P_SMEM_BYTES);
    if constexpr (EPI == EPI_DYN)
      if (err == cudaSuccess)
        err = cudaFuncSetAttribute(gemm_tc_pair_kernel<EPI, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   P_SMEM_BYTES);
    if (err != cudaSuccess) return cuda_fail(err, "gemm_tc: pair kernel setup");
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)(2 * sm_count()));
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = P_SMEM_BYTES;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int c = 0;
    err = cudaOccupancyMaxActiveClusters(&c, gemm_tc_pair_kernel<EPI>, &cfg);
    if (err != cudaSuccess) return cuda_fail(err, "gemm_tc: pair kernel occupancy");
    *out = c;
    return I8Q_OK;
  }, n + dev);
  return rc ? -1 : n[dev];
}

// Shared launch of both kernels for either epilogue kind.  prof1 / prof2
// name the single-CTA and pair launches in the kernel timing.
template <int EPI>
int launch_tc_impl(const __nv_bfloat16* uA, const __nv_bfloat16* iBt, int64_t M, int64_t N, int64_t Kp,
                   int max_abs_product_log2, const TcParams& base, cudaStream_t s, const char* prof1,
                   const char* prof2) {
  if (M <= 0 || N <= 0) return I8Q_OK;
  if (!uA || !iBt) return fail(I8Q_ERR_UNSUPPORTED, "gemm_tc: bf16 operands missing");
  if (Kp % BK != 0 || Kp > (int64_t)1 << 20) return fail(I8Q_ERR_UNSUPPORTED, "gemm_tc: Kp must be a multiple of 64");
  if (M > ((int64_t)1 << 31) - BM || N > ((int64_t)1 << 31) - BN) return fail(I8Q_ERR_UNSUPPORTED, "gemm_tc: too large");
  if ((reinterpret_cast<uintptr_t>(uA) | reinterpret_cast<uintptr_t>(iBt)) & 15)
    return fail(I8Q_ERR_UNSUPPORTED, "gemm_tc: operands must be 16-byte aligned");
  if (max_abs_product_log2 < 1 || max_abs_product_log2 > 17)
    return fail(I8Q_ERR_UNSUPPORTED, "gemm_tc: product bound out of range");
  // largest chunk of K steps whose partial sums stay below 2^24 in magnitude
  const int64_t chunk_k = ((int64_t)1 << 24) >> max_abs_product_log2;
  const int CS = (int)std::max<int64_t>(1, chunk_k / BK);
  uint32_t* status = device_status_word();
  if (!status) return fail(I8Q_ERR_CUDA, "gemm_tc: no device status word");
  const int ar = smem_attr((const void*)gemm_tc_kernel<EPI>, SMEM_BYTES);
  if (ar) return ar;
  TcParams p = base;
  p.M = M;
  p.N = N;
  p.KT = (int)(Kp / BK);
  p.CS = CS;
  p.status = status;

  // CTA pairs when there is at least a wave of 256 x 256 tiles;
  // I8Q_FORCE_CORE=tc1 / tc2 picks the single-CTA / pair kernel.
  const char* force = getenv("I8Q_FORCE_CORE");
  const int pair_clusters = pair_max_clusters<EPI>();
  if (pair_clusters < 0) return I8Q_ERR_CUDA;
  const int64_t pair_tiles = ceil_div(M, PBM) * ceil_div(N, PBN);
  bool use_pair = M >= PBM && pair_clusters > 0 && pair_tiles >= pair_clusters;
  if (force && std::string(force) == "tc1") use_pair = false;
  if (force && std::string(force) == "tc2") use_pair = pair_clusters > 0;
  int rc;
  if (use_pair) {
    CUtensorMap pA, pB;
    rc = make_map_2d(&pA, uA, M, Kp, HALF_ROWS, "gemm_tc");
    if (rc) return rc;
    rc = make_map_2d(&pB, iBt, N, Kp, HALF_ROWS, "gemm_tc");
    if (rc) return rc;
    p.tiles_m = (int)ceil_div(M, PBM);
    p.tiles_n = (int)ceil_div(N, PBN);
    p.num_tiles = p.tiles_m * p.tiles_n;
    const int clusters = std::min(p.num_tiles, pair_clusters);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)(2 * clusters));
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = P_SMEM_BYTES;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    I8Q_PROF(prof2, s);
    // bf16 or fp32 C of the dynamic inner product goes out by TMA when its
    // rows are 16-byte aligned
    CUtensorMap pC = pA;
    int tma_c = 0;
    if constexpr (EPI == EPI_DYN) {
      const bool bf = p.ep.out_mode == OUT_BF16;
      if ((bf || p.ep.out_mode == OUT_F32) && (p.ep.ldc * (bf ? 2 : 4)) % 16 == 0 &&
          (reinterpret_cast<uintptr_t>(p.ep.C) & 15) == 0 && M < ((int64_t)1 << 31) && N < ((int64_t)1 << 31) &&
          !getenv("I8Q_GEMM_DIRECT_STORE")) {
        rc = make_map_plain_2d(&pC, p.ep.C, bf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, N,
                               M, p.ep.ldc * (bf ? 2 : 4), bf ? 16 : 8, 32, "gemm_tc");
        if (rc) return rc;
        tma_c = bf ? 1 : 2;
      }
    }
    if constexpr (EPI == EPI_QG) {
      // fp32 or 8-bit Y of the 8-bit-code products, likewise
      const int esz = p.qg.ytype == I8Q_F32 ? 4 : 1;
      if ((p.qg.ldy * esz) % 16 == 0 && (reinterpret_cast<uintptr_t>(p.qg.Y) & 15) == 0 && M < ((int64_t)1 << 31) &&
          N < ((int64_t)1 << 31) && !getenv("I8Q_GEMM_DIRECT_STORE")) {
        rc = make_map_plain_2d(&pC, p.qg.Y,
                               esz == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_UINT8, N, M,
                               p.qg.ldy * esz, 32 / esz, 32, "gemm_tc");
        if (rc) return rc;
        tma_c = 1;
      }
    }
    if constexpr (EPI == EPI_DYN) {
      if (tma_c == 2) {
        I8Q_CUDA_TRY(cudaLaunchKernelEx(&cfg, gemm_tc_pair_kernel<EPI, 2>, pA, pB, pC, p));
        I8Q_LAUNCH_CHECK("gemm_tc_pair_kernel");
        return I8Q_OK;
      }
    }
    if (tma_c) {
      I8Q_CUDA_TRY(cudaLaunchKernelEx(&cfg, gemm_tc_pair_kernel<EPI, 1>, pA, pB, pC, p));
      I8Q_LAUNCH_CHECK("gemm_tc_pair_kernel");
      return I8Q_OK;
    }
    I8Q_CUDA_TRY(cudaLaunchKernelEx(&cfg, gemm_tc_pair_kernel<EPI, 0>, pA, pB, pC, p));
    I8Q_LAUNCH_CHECK("gemm_tc_pair_kernel");
    return I8Q_OK;
  }
  CUtensorMap mA, mB;
  rc = make_map_2d(&mA, uA, M, Kp, BM, "gemm_tc");
  if (rc) return rc;
  rc = make_map_2d(&mB, iBt, N, Kp, BN, "gemm_tc");
  if (rc) return rc;
  p.tiles_m = (int)ceil_div(M, BM);
  p.tiles_n = (int)ceil_div(N, BN);
  p.num_tiles = p.tiles_m * p.tiles_n;
  const int grid = std::min(p.num_tiles, sm_count());
  I8Q_PROF(prof1, s);
  gemm_tc_kernel<EPI><<<grid, THREADS, SMEM_BYTES, s>>>(mA, mB, p);
  I8Q_LAUNCH_CHECK("gemm_tc_kernel");
  return I8Q_OK;
}

}  // namespace

int launch_gemm_tc(const __nv_bfloat16* uA, const __nv_bfloat16* iBt, int64_t M, int64_t N, int64_t Kp,
                   int max_abs_product_log2, const GemmEpilogue& ep, cudaStream_t s) {
  TcParams p{};
  p.ep = ep;
  return launch_tc_impl<EPI_DYN>(uA, iBt, M, N, Kp, max_abs_product_log2, p, s, "gemm_tc", "gemm_tc_pair");
}

int launch_qgemm_tc(const __nv_bfloat16* Ac, const __nv_bfloat16* Bc, int64_t M, int64_t N, int64_t Kp,
                    int max_abs_product_log2, const QgEpilogue& qg, cudaStream_t s) {
  TcParams p{};
  p.qg = qg;
  return launch_tc_impl<EPI_QG>(Ac, Bc, M, N, Kp, max_abs_product_log2, p, s, "qgemm_tc", "qgemm_tc_pair");
}

}  // namespace i8q
