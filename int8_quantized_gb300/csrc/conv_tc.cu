// conv_tc.cu -- QLinearConv (onnx-light docs, "QLinearConv") for group 1,
// stride 1, dilation 1 as an implicit GEMM on the bf16 tensor pipe
// (tcgen05.mma kind::f16), exact in integers.
//
// Two small passes centre the operands, exactly, in bf16:
//   xc = x - x_zero_point      NHWC  [N][H][W][Cp]      (|xc| <= 255)
//   wc = w - w_zero_point[m]   [M][kH][kW][Cp]          (|wc| <= 255)
// with Cp = C rounded up to 64 and zeros beyond C.  Then, for an output tile
// of 128 output channels x R output rows (R * OW pixels),
//   acc[m, p] = sum over taps (kh, kw) and 64-channel slabs of
//               wc[m, kh, kw, c] * xc[n, oh + kh - pad_top, ow + kw - pad_left, c]
// The x slab of one tap is one 4-D TMA box {64 channels, OW, R, 1} at
// (c0, kw - pad_left, oh0 + kh - pad_top, n); coordinates outside the input
// read 0, which is exactly the padding of QLinearConv (a padded position is
// real 0, i.e. x_zero_point, so xc = 0 there).  Products are within
// max|xc| * max|wc|, so fp32 chunks of CS K-steps stay exact (partial sums at
// most 2^24) and are drained into int32 as in the GEMM core.  The epilogue
// requantizes each output,
//   y = saturate(rint(((float)(acc + B[m]) * (x_scale * w_scale[m])) / y_scale) + y_zero_point),
// and stores NCHW bytes: thread = output channel, its slice = consecutive
// pixels of one output row.
#include <type_traits>

#include "tcgen05.cuh"

namespace i8q {
namespace {

using namespace tc;

constexpr int BM = 128, BK = 64, STAGES = 4;
constexpr int NUM_EPI_WARPS = 16;
constexpr int THREADS = 64 + NUM_EPI_WARPS * 32;
constexpr int TMEM_COLS = 512;
constexpr int NUM_BARS = 2 * STAGES + 4 + 1;

constexpr uint32_t ST_TIMEOUT_PRODUCER = 1u << 4;
constexpr uint32_t ST_TIMEOUT_MMA = 1u << 5;
constexpr uint32_t ST_TIMEOUT_EPILOGUE = 1u << 6;
constexpr uint32_t ST_TIMEOUT_DRAIN = 1u << 7;

template <int TN>
struct ConvTile {
  static constexpr int A_STAGE = BM * BK * 2;
  static constexpr int B_STAGE = TN * BK * 2;
  static constexpr int STAGE_BYTES = A_STAGE + B_STAGE;
  static constexpr int SL = TN / 4;  // pixels per epilogue warp
  // staging of the codes of 32 channels x TN pixels per TMEM lane quadrant,
  // for the bulk store of y (1024-byte aligned groups)
  static constexpr int STG_GROUP = ((32 * TN + 1023) / 1024) * 1024;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + 4 * STG_GROUP + NUM_BARS * 8 + 16;
  static_assert(STAGE_BYTES % 1024 == 0, "stages must keep 1024-byte alignment");
  static_assert(TN % 32 == 0 && TN <= 256, "tile width");
};

struct ConvParams {
  int M, CC, taps, kW, pt, pl, OH, OW, R, NB;
  int tiles_m, row_groups, num_tiles;
  int KT;
  int xmax;            // max |x - x_zero_point| over the input type
  const void* wzp;     // w zero points (w's type), n_wzp of them; null = 0
  int n_wzp, wsigned;
  float x_scale, y_scale, qlo_z, qhi_z;  // qlo_z = qlo - y_zp, qhi_z = qhi - y_zp
  int y_zp;
  const int32_t* bias;
  const float* w_scale;
  int per_channel;
  uint8_t* y;  // NCHW bytes (uint8 or int8 codes)
  uint32_t* status;
  int tma_y;   // y stored by bulk tensor copies through shared memory (R * OW == TN)
};

// Tiled TMA store of a 3-D box from this CTA's shared memory (dense rows)
// to the tensor at (x, y, z), in the calling thread's bulk group.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];\n" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y), "r"(z)
               : "memory");
}

__device__ __forceinline__ void conv_tile_coords(int tile, const ConvParams& p, int& mt, int& rg, int& n) {
  mt = tile % p.tiles_m;
  const int rest = tile / p.tiles_m;
  rg = rest % p.row_groups;
  n = rest / p.row_groups;
}

template <int TN>
__global__ void __launch_bounds__(THREADS, 1)
conv_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
               const __grid_constant__ CUtensorMap tmY, ConvParams p) {
  using T = ConvTile<TN>;
  constexpr uint32_t IDESC = idesc_bf16(BM, TN);
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned, indexed from the shared array itself so that accesses stay shared-space
  uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* stg_all = smem + STAGES * T::STAGE_BYTES;  // 4 groups of T::STG_GROUP bytes
  uint64_t* bars = reinterpret_cast<uint64_t*>(stg_all + 4 * T::STG_GROUP);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t smem0 = smem_u32(smem);
  auto sA = [&](int s) { return smem0 + (uint32_t)(s * T::STAGE_BYTES); };
  auto sB = [&](int s) { return smem0 + (uint32_t)(s * T::STAGE_BYTES + T::A_STAGE); };
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto empty = [&](int s) { return smem_u32(bars + STAGES + s); };
  auto accf = [&](int b) { return smem_u32(bars + 2 * STAGES + b); };
  auto acce = [&](int b) { return smem_u32(bars + 2 * STAGES + 2 + b); };
  const uint32_t fin = smem_u32(bars + 2 * STAGES + 4);
  __shared__ int wmax_w[THREADS / 32];  // per warp: max |w - w_zero_point| bound

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
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
    asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmX)) : "memory");
    if (p.tma_y) asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&tmY)) : "memory");
  }
  {
    const int lo = p.wsigned ? -128 : 0, hi = p.wsigned ? 127 : 255;
    int wm = p.wzp ? 0 : max(-lo, hi);
    for (int i = threadIdx.x; p.wzp && i < p.n_wzp; i += THREADS) {
      const int z = p.wsigned ? (int)static_cast<const int8_t*>(p.wzp)[i] : (int)static_cast<const uint8_t*>(p.wzp)[i];
      wm = max(wm, max(z - lo, hi - z));
    }
    wm = __reduce_max_sync(0xffffffffu, wm);
    if (lane == 0) wmax_w[warp] = wm;
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int KT = p.KT;
  // K steps per exact fp32 chunk: every partial sum of CS * 64 products
  // stays within 2^24 when CS * 64 * max|xc| * max|wc| <= 2^24, with
  // max|wc| = max over the zero points of their distance to the ends of
  // w's type (the warps' maxima were merged across the barrier above)
  int wmax = 0;
#pragma unroll 1
  for (int i = 0; i < THREADS / 32; ++i) wmax = max(wmax, wmax_w[i]);
  const int CS = max(1, (int)((int64_t(1) << 24) / ((int64_t)BK * p.xmax * max(wmax, 1))));
  const int nchunks = (KT + CS - 1) / CS;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      // counters instead of division: stage st / round parity ph, and the
      // K step's 64-channel slab cch, filter column kw and row kh
      int it = 0;
      uint32_t st = 0, ph = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
        int mt, rg, n;
        conv_tile_coords(tile, p, mt, rg, n);
        int cch = 0, kw = 0, kh = 0;
        for (int kt = 0; kt < KT; ++kt, ++it) {
          if (!wait_bar(empty(st), ph ^ 1u, abort_flag, p.status, ST_TIMEOUT_PRODUCER)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full(st), T::STAGE_BYTES);
          tma_load_2d(sA(st), &tmW, full(st), kt * BK, mt * BM);
          tma_load_4d(sB(st), &tmX, full(st), cch * BK, kw - p.pl, rg * p.R + kh - p.pt, n);
          if (++cch == p.CC) {
            cch = 0;
            if (++kw == p.kW) {
              kw = 0;
              ++kh;
            }
          }
          if (++st == (uint32_t)STAGES) {
            st = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) {
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
      // counters instead of division; descriptors advanced by addition
      // (start address >> 4)
      const uint64_t adesc0 = desc_sw128(sA(0)), bdesc0 = desc_sw128(sB(0));
      uint32_t st = 0, ph = 0;
      int chunk = 0;
      bool ok = true;
      uint32_t d = tmem_base;
      if (KT % STAGES == 0) {
        // every tile starts at stage 0: the K loop unrolled by the ring's
        // length, so that each stage's descriptors are the base plus a
        // constant and the stage index is static (a leaner issue loop)
        for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
          int kc = 0;
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
                d = tmem_base + (uint32_t)(b * TN);
              }
              if (!wait_bar(full(j), ph, abort_flag, p.status, ST_TIMEOUT_MMA)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t soff = (uint64_t)(((uint32_t)j * (uint32_t)T::STAGE_BYTES) >> 4);
              const uint32_t acc = kc == 0 ? 0u : 1u;
#pragma unroll
              for (int k = 0; k < BK / 16; ++k)
                tc_mma(d, adesc0 + soff + (uint64_t)(2 * k), bdesc0 + soff + (uint64_t)(2 * k), IDESC,
                       (k == 0) ? acc : 1u);
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
        int kc = 0;
        for (int kt = 0; kt < KT; ++kt) {
          if (kc == 0) {
            const int b = chunk & 1;
            if (!wait_bar(acce(b), ((uint32_t)(chunk >> 1) & 1u) ^ 1u, abort_flag, p.status, ST_TIMEOUT_MMA)) {
              ok = false;
              break;
            }
            tc_fence_after();
            d = tmem_base + (uint32_t)(b * TN);
          }
          if (!wait_bar(full(st), ph, abort_flag, p.status, ST_TIMEOUT_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t soff = (uint64_t)((st * (uint32_t)T::STAGE_BYTES) >> 4);
          const uint32_t acc = kc == 0 ? 0u : 1u;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            tc_mma(d, adesc0 + soff + (uint64_t)(2 * k), bdesc0 + soff + (uint64_t)(2 * k), IDESC,
                   (k == 0) ? acc : 1u);
          tc_commit(empty(st));
          if (++kc == CS || kt == KT - 1) {
            tc_commit(accf(chunk & 1));
            ++chunk;
            kc = 0;
          }
          if (++st == (uint32_t)STAGES) {
            st = 0;
            ph ^= 1u;
          }
        }
      }
      tc_commit(fin);
      unsigned long long t0 = global_ns();
      while (!mbar_try_wait(fin, 0))
        if (global_ns() - t0 > WAIT_LIMIT_NS) {
          atomicOr(p.status, ST_TIMEOUT_DRAIN);
          break;
        }
    }
  } else {
    // ---------------- drain + requantizing epilogue ----------------
    constexpr int SL = T::SL;
    const int q = warp & 3;             // TMEM lanes 32q.. = output channels of this warp
    const int slice = (warp - 2) >> 2;  // pixels [slice*SL, slice*SL + SL) of the tile
    int chunk = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
      int mt, rg, n;
      conv_tile_coords(tile, p, mt, rg, n);
      int32_t run[SL];
#pragma unroll
      for (int j = 0; j < SL; ++j) run[j] = 0;
      for (int c = 0; c < nchunks; ++c, ++chunk) {
        const int b = chunk & 1;
        const bool got = wait_bar(accf(b), (uint32_t)(chunk >> 1) & 1u, abort_flag, p.status, ST_TIMEOUT_EPILOGUE);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * TN + slice * SL);
#pragma unroll
        for (int j = 0; j < SL / 8; j += 2) {
          uint32_t r0[8], r1[8];
          tmem_ld8(taddr + (uint32_t)(j * 8), r0);
          if (j + 1 < SL / 8) tmem_ld8(taddr + (uint32_t)(j * 8 + 8), r1);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            run[j * 8 + i] += __float2int_rn(__uint_as_float(r0[i]));
            if (j + 1 < SL / 8) run[j * 8 + 8 + i] += __float2int_rn(__uint_as_float(r1[i]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce(b));
      }
      const int m = mt * BM + q * 32 + lane;
      if (p.tma_y) {
        // the four slices of quadrant q (warps q + 2 .. q + 14 step 4) stage
        // their 32 channels x SL codes as one dense 32 x TN box, stored by
        // one bulk tensor copy (coalesced rows of the NCHW planes)
        uint8_t* stg = stg_all + q * T::STG_GROUP;
        const uint32_t group_bar = 1u + (uint32_t)q;
        if (ok && slice == 0 && lane == 0) bulk_wait_read();  // the previous tile's store has read the buffer
        // barrier over the quadrant's 128 threads, which also agree on ok
        // (so that they leave the tile loop together)
        uint32_t all_ok;
        asm volatile(
            "{\n .reg .pred p, r;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred r, %2, 128, p;\n selp.u32 %0, 1, 0, r;\n}\n"
            : "=r"(all_ok)
            : "r"((uint32_t)ok), "r"(group_bar)
            : "memory");
        if (!all_ok) {
          ok = false;
          break;
        }
        const int32_t bm = (m < p.M && p.bias) ? __ldg(p.bias + m) : 0;
        const float mul = __fmul_rn(p.x_scale, __ldg(p.w_scale + (p.per_channel ? min(m, p.M - 1) : 0)));
        uint8_t* dst = stg + lane * TN + slice * SL;
#pragma unroll
        for (int j = 0; j < SL; j += 8) {
          uint32_t code[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            float v = __fmul_rn(__int2float_rn(run[j + u] + bm), mul);
            v = __fdiv_rn(v, p.y_scale);
            code[u] = rint_code_bits(v, p.qlo_z, p.qhi_z, p.y_zp);
          }
          *reinterpret_cast<uint2*>(dst + j) = make_uint2(pack_low_bytes(code[0], code[1], code[2], code[3]),
                                                          pack_low_bytes(code[4], code[5], code[6], code[7]));
        }
        asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
        asm volatile("bar.sync %0, 128;\n" ::"r"(group_bar) : "memory");
        if (slice == 0 && lane == 0) {
          // rows past OH and channels past M fall outside the tensor: not written
          tma_store_3d(&tmY, smem_u32(stg), rg * p.R * p.OW, mt * BM + q * 32, n);
          bulk_commit();
        }
        __syncwarp();
        continue;
      }
      if (!ok) break;
      if (m < p.M) {
        const int32_t bm = p.bias ? __ldg(p.bias + m) : 0;
        const float mul = __fmul_rn(p.x_scale, __ldg(p.w_scale + (p.per_channel ? m : 0)));
        uint8_t* yrow = p.y + ((int64_t)n * p.M + m) * p.OH * p.OW;
        const int p0 = slice * SL;
        if (SL == p.OW && (p.OW & 7) == 0 && (reinterpret_cast<uintptr_t>(p.y) & 7) == 0) {
          // the slice is exactly one output row: 8-byte stores
          const int oh = rg * p.R + slice;
          if (oh < p.OH) {
            uint8_t* dst = yrow + (int64_t)oh * p.OW;
#pragma unroll
            for (int j = 0; j < SL; j += 8) {
              uint32_t code[8];
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                float v = __fmul_rn(__int2float_rn(run[j + u] + bm), mul);
                v = __fdiv_rn(v, p.y_scale);
                code[u] = rint_code_bits(v, p.qlo_z, p.qhi_z, p.y_zp);
              }
              *reinterpret_cast<uint2*>(dst + j) = make_uint2(pack_low_bytes(code[0], code[1], code[2], code[3]),
                                                              pack_low_bytes(code[4], code[5], code[6], code[7]));
            }
          }
        } else {
          int oh = rg * p.R + p0 / p.OW, ow = p0 % p.OW;
#pragma unroll
          for (int j = 0; j < SL; ++j) {
            if (oh < p.OH) {
              float v = __fmul_rn(__int2float_rn(run[j] + bm), mul);
              v = __fdiv_rn(v, p.y_scale);
              yrow[(int64_t)oh * p.OW + ow] = (uint8_t)rint_code_bits(v, p.qlo_z, p.qhi_z, p.y_zp);
            }
            if (++ow == p.OW) {
              ow = 0;
              ++oh;
            }
          }
        }
      }
      __syncwarp();
    }
    // the bulk stores are complete before the CTA leaves
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---- operand preparation -------------------------------------------------------

// xc[n][h][w][c] = x[n][c][h][w] - xz (bf16), zero for c >= C.  One block per
// (n, h, 64-channel slab); the slab is transposed through shared memory in
// chunks of 32 columns.
template <typename XT>
__global__ void __launch_bounds__(256)
center_x_nhwc(const XT* __restrict__ x, int C, int H, int W, int Cp, int xz, __nv_bfloat16* __restrict__ xc) {
  __shared__ float tile[64][33];
  const int n = blockIdx.z, h = blockIdx.y, c0 = blockIdx.x * 64;
  const int t = threadIdx.x;
  for (int w0 = 0; w0 < W; w0 += 32) {
    for (int cc = t / 32; cc < 64; cc += 8) {
      const int c = c0 + cc, w = w0 + (t & 31);
      float v = 0.0f;
      if (c < C && w < W) v = (float)((int)x[(((int64_t)n * C + c) * H + h) * W + w] - xz);
      tile[cc][t & 31] = v;
    }
    __syncthreads();
    // each thread writes 8 channels (16 bytes) of one column
    for (int i = t; i < 32 * 8; i += 256) {
      const int wl = i / 8, cg = (i % 8) * 8, w = w0 + wl;
      if (w < W) {
        uint32_t pk[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t lo = __float_as_uint(tile[cg + 2 * u][wl]) >> 16;
          const uint32_t hi = __float_as_uint(tile[cg + 2 * u + 1][wl]) & 0xffff0000u;
          pk[u] = lo | hi;
        }
        *reinterpret_cast<uint4*>(xc + (((int64_t)n * H + h) * W + w) * Cp + c0 + cg) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
    }
    __syncthreads();
  }
}

// Same result, one CTA per (n, h): the whole NHWC row xc[n][h][:][:] is
// W * Cp * 2 contiguous bytes.  Inputs land in shared memory as [w][c] with
// a row stride of Cp + 8 halfwords (16-byte aligned rows, read back as 16-byte
// vectors) and, within a row, 4-pair groups of channels XOR-swizzled by the
// 8-pixel piece (w / 8) so the stores of one warp spread over the banks;
// then they leave in 16-byte pieces of the contiguous output row.
__device__ __forceinline__ int center_swz(int w) { return ((w >> 3) & 7) << 2; }  // in channel pairs

template <typename XT>
__global__ void __launch_bounds__(256, 6)
center_x_row(const XT* __restrict__ x, int C, int H, int W, int Cp, int xz, __nv_bfloat16* __restrict__ xc) {
  extern __shared__ __align__(16) uint16_t rowt[];  // W x (Cp + 8)
  const int n = blockIdx.y, h = blockIdx.x;
  const int ld = Cp + 8, ldw = ld / 2;
  const XT* xr = x + ((int64_t)n * C * H + h) * W;  // + c * H * W + w
  uint32_t* rw = reinterpret_cast<uint32_t*>(rowt);
  if ((W & 7) == 0 && ((int64_t)H * W) % 8 == 0 && (reinterpret_cast<uintptr_t>(xr) & 7) == 0) {
    // 8-byte pieces of two adjacent channel rows per work item (their codes
    // meet in 32-bit shared stores), four items in flight per thread
    const int cw = W / 8, pairs = Cp / 2, total = pairs * cw;
    const uint32_t flip = std::is_signed<XT>::value ? 0x80808080u : 0u;  // signed codes as unsigned + 128
    const int xzu = std::is_signed<XT>::value ? xz + 128 : xz;
    // code b as the fp32 1.5 * 2^23 + b (one byte permute), minus 1.5 * 2^23 + xz:
    // exactly b - xz (|b - xz| <= 255), whose bf16 is the top half
    const float zf = __int_as_float(0x4B400000 + xzu);
    // (pair, piece) of item idx = base + tid + u * blockDim.x, advanced
    // without division
    const int dq = blockDim.x / cw, dr = blockDim.x - dq * cw;
    int cpn = threadIdx.x / cw, pcn = threadIdx.x - cpn * cw;
    for (int base = 0; base < total; base += 4 * blockDim.x) {
      uint2 v[4][2];
      int cp[4], ww[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const bool live = base + (int)threadIdx.x + u * (int)blockDim.x < total;
        cp[u] = live ? cpn : pairs;
        ww[u] = pcn * 8;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int c = 2 * cpn + h2;
          v[u][h2] = (live && c < C) ? __ldg(reinterpret_cast<const uint2*>(xr + (int64_t)c * H * W + ww[u]))
                                     : make_uint2(0, 0);
        }
        cpn += dq;
        pcn += dr;
        if (pcn >= cw) {
          pcn -= cw;
          ++cpn;
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (cp[u] >= pairs) continue;
        uint32_t* dst = rw + ww[u] * ldw + (cp[u] ^ center_swz(ww[u]));
        const uint32_t a[2] = {v[u][0].x ^ flip, v[u][0].y ^ flip}, b[2] = {v[u][1].x ^ flip, v[u][1].y ^ flip};
        if (2 * cp[u] + 1 < C) {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const uint32_t sel = 0x7640u + (e & 3);
            const float f0 = __fsub_rn(__uint_as_float(__byte_perm(a[e >> 2], 0x4B400000u, sel)), zf);
            const float f1 = __fsub_rn(__uint_as_float(__byte_perm(b[e >> 2], 0x4B400000u, sel)), zf);
            dst[e * ldw] = __byte_perm(__float_as_uint(f0), __float_as_uint(f1), 0x7632);
          }
        } else {  // channel padding: zeros beyond C
          const bool in0 = 2 * cp[u] < C;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const uint32_t sel = 0x7640u + (e & 3);
            const float f0 = in0 ? __fsub_rn(__uint_as_float(__byte_perm(a[e >> 2], 0x4B400000u, sel)), zf) : 0.0f;
            dst[e * ldw] = __float_as_uint(f0) >> 16;
          }
        }
      }
    }
  } else {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    for (int c = warp; c < Cp; c += nwarps)
      for (int w = lane; w < W; w += 32) {
        float v = 0.0f;
        if (c < C) v = (float)((int)xr[(int64_t)c * H * W + w] - xz);
        rowt[w * ld + (c ^ (center_swz(w) << 1))] = (uint16_t)(__float_as_uint(v) >> 16);  // exact: |v| <= 255
      }
  }
  __syncthreads();
  uint4* dst = reinterpret_cast<uint4*>(xc + ((int64_t)n * H + h) * W * Cp);
  const int per_w = Cp / 8;
  const int sq = blockDim.x / per_w, sr = blockDim.x - sq * per_w;
  int w = threadIdx.x / per_w, g8 = threadIdx.x - w * per_w;  // pixel, 8-channel group of qi
  for (int qi = threadIdx.x; qi < W * per_w; qi += blockDim.x) {
    dst[qi] = *reinterpret_cast<const uint4*>(rw + w * ldw + ((g8 * 4) ^ center_swz(w)));
    w += sq;
    g8 += sr;
    if (g8 >= per_w) {
      g8 -= per_w;
      ++w;
    }
  }
}

// wc[m][kh][kw][c] = w[m][c][kh][kw] - wz[m] (bf16), zero for c >= C.  One
// thread per (m, tap, 8 channels): 8 strided byte reads, one 16-byte store;
// threads first, first + stride, ... of the M * taps * Cp / 8 items.
template <typename WT>
__device__ __forceinline__ void center_w_items(const WT* __restrict__ w, const WT* __restrict__ wz, int per_channel,
                                               int M, int C, int taps, int Cp, __nv_bfloat16* __restrict__ wc,
                                               int64_t first, int64_t stride) {
  const int groups = Cp / 8;
  const int64_t total = (int64_t)M * taps * groups;
  for (int64_t i = first; i < total; i += stride) {
    const int g = (int)(i % groups);
    const int r = (int)(i / groups);  // m * taps + tap
    const int m = r / taps, tap = r - m * taps;
    const int z = wz ? (int)wz[per_channel ? m : 0] : 0;
    const WT* src = w + (int64_t)m * C * taps + tap;
    uint32_t pk[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = g * 8 + 2 * u;
      // exact: |w - z| <= 255; bf16 = top half of the fp32 value
      const float v0 = c < C ? (float)((int)src[(int64_t)c * taps] - z) : 0.0f;
      const float v1 = c + 1 < C ? (float)((int)src[(int64_t)(c + 1) * taps] - z) : 0.0f;
      pk[u] = __byte_perm(__float_as_uint(v0), __float_as_uint(v1), 0x7632u);
    }
    *reinterpret_cast<uint4*>(wc + (int64_t)r * Cp + g * 8) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
}

template <typename WT>
__global__ void center_w(const WT* __restrict__ w, const WT* __restrict__ wz, int per_channel, int M, int C, int taps,
                         int Cp, __nv_bfloat16* __restrict__ wc) {
  center_w_items(w, wz, per_channel, M, C, taps, Cp, wc, (int64_t)blockIdx.x * blockDim.x + threadIdx.x,
                 (int64_t)gridDim.x * blockDim.x);
}

// Both operands in one launch, for rows of whole 8-byte pieces (W % 8 == 0,
// H * W % 8 == 0, 8-byte aligned x): blocks [0, wblocks) centre the filter
// as center_w; each later block of two warps centres two input rows, warp
// r taking row n * H + h = 2 * (block - wblocks) + r whole.  Lane l takes
// the channels 8l .. 8l + 7 of each 256-channel slab and walks the row two
// 8-pixel pieces at a time: sixteen 8-byte reads in flight (one per channel
// row and piece; the lane reads each channel row's sectors whole, one piece
// after the other), then per pixel the eight codes turned into bf16 pairs
// and one 16-byte store, the warp writing each pixel's 512 contiguous bytes
// of xc.  A code b becomes the fp32 1.5 * 2^23 + b by one byte permute;
// subtracting 1.5 * 2^23 + xz (paired) leaves b - xz exactly, whose bf16 is
// the top half.  Channels C .. Cp - 1 read as the code xz and so come out 0.
template <typename XT, typename WT>
__global__ void __launch_bounds__(64, 8)
center_ops_pix(const XT* __restrict__ x, int N, int C, int H, int W, int Cp, int xz, __nv_bfloat16* __restrict__ xc,
               const WT* __restrict__ w, const WT* __restrict__ wzp, int per_channel, int M, int taps,
               __nv_bfloat16* __restrict__ wc, int wblocks) {
  if ((int)blockIdx.x < wblocks) {
    center_w_items(w, wzp, per_channel, M, C, taps, Cp, wc, (int64_t)blockIdx.x * blockDim.x + threadIdx.x,
                   (int64_t)wblocks * blockDim.x);
    return;
  }
  const int64_t row = 2 * ((int64_t)blockIdx.x - wblocks) + (threadIdx.x >> 5);  // n * H + h
  if (row >= (int64_t)N * H) return;
  const int64_t n = row / H, h = row - n * H;
  const int lane = (int)threadIdx.x & 31;
  const int64_t plane = (int64_t)H * W;
  constexpr bool XS = std::is_signed<XT>::value;
  const uint32_t flip = XS ? 0x80808080u : 0u;  // signed codes as unsigned + 128
  const int xzu = XS ? xz + 128 : xz;
  const uint32_t zrow = (uint32_t)xzu * 0x01010101u;
  const float zf = __int_as_float(0x4B400000 + xzu);
  const XT* xrow = x + (n * C * H + h) * W;  // + c * plane + w
  __nv_bfloat16* orow = xc + row * W * Cp;
  for (int c0 = 8 * lane; c0 < Cp; c0 += 256) {
    for (int w0 = 0; w0 < W; w0 += 16) {
      const bool two = w0 + 8 < W;
      uint32_t r[2][8][2];
#pragma unroll
      for (int k = 0; k < 2; ++k)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (c0 + i < C && (k == 0 || two)) {
            const uint2 v = __ldg(reinterpret_cast<const uint2*>(xrow + (int64_t)(c0 + i) * plane + w0 + 8 * k));
            r[k][i][0] = v.x ^ flip;
            r[k][i][1] = v.y ^ flip;
          } else {
            r[k][i][0] = r[k][i][1] = zrow;
          }
        }
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        if (k == 1 && !two) break;
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          const uint32_t sel = 0x7640u + (p & 3);
          uint32_t o[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float b0 = __uint_as_float(__byte_perm(r[k][2 * q][p >> 2], 0x4B400000u, sel));
            const float b1 = __uint_as_float(__byte_perm(r[k][2 * q + 1][p >> 2], 0x4B400000u, sel));
            const float2 f = fma2_rn(make_float2(b0, b1), make_float2(1.0f, 1.0f), make_float2(-zf, -zf));
            o[q] = __byte_perm(__float_as_uint(f.x), __float_as_uint(f.y), 0x7632);
          }
          *reinterpret_cast<uint4*>(orow + (int64_t)(w0 + 8 * k + p) * Cp + c0) = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
    }
  }
}

template <typename XT, typename WT>
void launch_center_pix(cudaStream_t s, const void* x, int64_t N, int64_t C, int64_t H, int64_t W, int64_t Cp,
                       int x_zp, __nv_bfloat16* xc, const void* w, const void* w_zp, int per_channel, int64_t M,
                       int taps, __nv_bfloat16* wc, int wblocks) {
  const unsigned grid = (unsigned)(wblocks + ceil_div(N * H, 2));
  center_ops_pix<XT, WT><<<grid, 64, 0, s>>>((const XT*)x, (int)N, (int)C, (int)H, (int)W, (int)Cp, x_zp, xc,
                                             (const WT*)w, (const WT*)w_zp, per_channel, (int)M, taps, wc, wblocks);
}

size_t a256(size_t v) { return (v + 255) & ~size_t(255); }

// Output rows per tile so that R * OW is a multiple of 32 and at most 256.
int pick_rows(int64_t OW, int64_t OH) {
  int best = 0;
  for (int r = 1; r * OW <= 256; ++r)
    if ((r * OW) % 32 == 0) best = r;
  (void)OH;
  return best;
}

}  // namespace

// Scratch bytes of the tensor-core path, or 0 when the shape does not take it.
size_t conv_tc_workspace(int64_t N, int64_t C, int64_t H, int64_t W, int64_t M, int64_t Cg, int64_t kH, int64_t kW,
                         int64_t OH, int64_t OW, int64_t group, int64_t sh, int64_t sw, int64_t dh, int64_t dw) {
  if (group != 1 || sh != 1 || sw != 1 || dh != 1 || dw != 1 || Cg != C) return 0;
  const char* f = getenv("I8Q_FORCE_CONV");
  if (f && std::string(f) == "direct") return 0;
  const int R = pick_rows(OW, OH);
  if (R == 0 || R * OW != 224) return 0;  // the tile width instantiated
  if (OW > W || C > 65536 || M > 65535 || N > 65535) return 0;
  const int64_t Cp = round_up(C, 64);
  return a256((size_t)(N * H * W * Cp * 2)) + a256((size_t)(M * kH * kW * Cp * 2));
}

int launch_conv_tc(const void* x, int xtype, int64_t N, int64_t C, int64_t H, int64_t W, float x_scale, int x_zp,
                   const void* w, int wtype, int64_t M, int64_t kH, int64_t kW, const float* w_scale,
                   const void* w_zp, int per_channel, float y_scale, int y_zp, int ytype, const int32_t* B,
                   int64_t pt, int64_t pl, int64_t OH, int64_t OW, void* y, void* workspace, cudaStream_t s) {
  const int R = pick_rows(OW, OH);
  const int64_t Cp = round_up(C, 64);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  __nv_bfloat16* xc = reinterpret_cast<__nv_bfloat16*>(ws);
  __nv_bfloat16* wc = reinterpret_cast<__nv_bfloat16*>(ws + a256((size_t)(N * H * W * Cp * 2)));
  const int taps = (int)(kH * kW);
  uint32_t* status = device_status_word();
  if (!status) return fail(I8Q_ERR_CUDA, "qlinearconv: no device status word");
  {
    I8Q_PROF("conv_center_operands", s);
    const size_t row_smem = (size_t)W * (Cp + 8) * 2;
    const int64_t tw = M * taps * (Cp / 8);
    const bool pix = W % 8 == 0 && (H * W) % 8 == 0 && (reinterpret_cast<uintptr_t>(x) & 7) == 0 &&
                     ceil_div(N * H, 2) + (int64_t)sm_count() * 8 < ((int64_t)1 << 31) &&
                     !getenv("I8Q_CONV_CENTER_ROW");
    if (pix) {
      // the filter takes two of the eight 2-warp blocks an SM holds at first, the rows the rest
      const int wblocks = (int)std::min<int64_t>(ceil_div(tw, 64), (int64_t)sm_count() * 2);
      if (xtype == I8Q_U8 && wtype == I8Q_U8)
        launch_center_pix<uint8_t, uint8_t>(s, x, N, C, H, W, Cp, x_zp, xc, w, w_zp, per_channel, M, taps, wc,
                                             wblocks);
      else if (xtype == I8Q_U8)
        launch_center_pix<uint8_t, int8_t>(s, x, N, C, H, W, Cp, x_zp, xc, w, w_zp, per_channel, M, taps, wc,
                                            wblocks);
      else if (wtype == I8Q_U8)
        launch_center_pix<int8_t, uint8_t>(s, x, N, C, H, W, Cp, x_zp, xc, w, w_zp, per_channel, M, taps, wc,
                                            wblocks);
      else
        launch_center_pix<int8_t, int8_t>(s, x, N, C, H, W, Cp, x_zp, xc, w, w_zp, per_channel, M, taps, wc,
                                           wblocks);
      I8Q_LAUNCH_CHECK("conv operand centering");
    } else if (row_smem <= 200 * 1024) {
      if (xtype == I8Q_U8) {
        const int ar = smem_attr((const void*)center_x_row<uint8_t>, 200 * 1024);
        if (ar) return ar;
        center_x_row<uint8_t><<<dim3((unsigned)H, (unsigned)N), 256, row_smem, s>>>((const uint8_t*)x, (int)C, (int)H,
                                                                                   (int)W, (int)Cp, x_zp, xc);
      } else {
        const int ar = smem_attr((const void*)center_x_row<int8_t>, 200 * 1024);
        if (ar) return ar;
        center_x_row<int8_t><<<dim3((unsigned)H, (unsigned)N), 256, row_smem, s>>>((const int8_t*)x, (int)C, (int)H,
                                                                                 (int)W, (int)Cp, x_zp, xc);
      }
    } else {
      dim3 gx((unsigned)(Cp / 64), (unsigned)H, (unsigned)N);
      if (xtype == I8Q_U8)
        center_x_nhwc<uint8_t><<<gx, 256, 0, s>>>((const uint8_t*)x, (int)C, (int)H, (int)W, (int)Cp, x_zp, xc);
      else
        center_x_nhwc<int8_t><<<gx, 256, 0, s>>>((const int8_t*)x, (int)C, (int)H, (int)W, (int)Cp, x_zp, xc);
    }
    if (!pix) {
      const int gw = (int)std::min<int64_t>(ceil_div(tw, 256), (int64_t)sm_count() * 8);
      if (wtype == I8Q_U8)
        center_w<uint8_t><<<gw, 256, 0, s>>>((const uint8_t*)w, (const uint8_t*)w_zp, per_channel, (int)M, (int)C,
                                             taps, (int)Cp, wc);
      else
        center_w<int8_t><<<gw, 256, 0, s>>>((const int8_t*)w, (const int8_t*)w_zp, per_channel, (int)M, (int)C, taps,
                                            (int)Cp, wc);
      I8Q_LAUNCH_CHECK("conv operand centering");
    }
  }
  CUtensorMap mW, mX;
  int rc = make_map_2d(&mW, wc, M, (int64_t)taps * Cp, BM, "qlinearconv");
  if (rc) return rc;
  {
    cuuint64_t dims[4] = {(cuuint64_t)Cp, (cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)N};
    cuuint64_t strides[3] = {(cuuint64_t)(Cp * 2), (cuuint64_t)(W * Cp * 2), (cuuint64_t)(H * W * Cp * 2)};
    cuuint32_t box[4] = {64u, (cuuint32_t)OW, (cuuint32_t)R, 1u};
    rc = make_tensor_map(&mX, xc, 4, dims, strides, box, "qlinearconv");
    if (rc) return rc;
  }
  // |xc| <= max distance of x_zp to its type's ends; |wc| <= 255
  const int xmax = xtype == I8Q_U8 ? std::max(x_zp, 255 - x_zp) : std::max(x_zp + 128, 127 - x_zp);
  constexpr int TN = 224;
  using T = ConvTile<TN>;
  const int ar = smem_attr((const void*)conv_tc_kernel<TN>, T::SMEM_BYTES);
  if (ar) return ar;
  ConvParams p;
  p.M = (int)M;
  p.CC = (int)(Cp / 64);
  p.taps = taps;
  p.kW = (int)kW;
  p.pt = (int)pt;
  p.pl = (int)pl;
  p.OH = (int)OH;
  p.OW = (int)OW;
  p.R = R;
  p.NB = (int)N;
  p.tiles_m = (int)ceil_div(M, BM);
  p.row_groups = (int)ceil_div(OH, R);
  p.num_tiles = p.tiles_m * p.row_groups * (int)N;
  p.KT = taps * p.CC;
  p.xmax = std::max(xmax, 1);
  p.wzp = w_zp;
  p.n_wzp = per_channel ? (int)M : 1;
  p.wsigned = wtype == I8Q_S8 ? 1 : 0;
  p.x_scale = x_scale;
  p.y_scale = y_scale;
  const float qlo = ytype == I8Q_U8 ? 0.0f : -128.0f, qhi = ytype == I8Q_U8 ? 255.0f : 127.0f;
  p.qlo_z = qlo - (float)y_zp;
  p.qhi_z = qhi - (float)y_zp;
  p.y_zp = y_zp;
  p.bias = B;
  p.w_scale = w_scale;
  p.per_channel = per_channel;
  p.y = static_cast<uint8_t*>(y);
  p.status = status;
  // y as [N][M][OH * OW] bytes for bulk stores of 32 channels x TN pixels:
  // when a tile is whole rows filling TN and the planes and y are 16-byte
  // aligned
  CUtensorMap mY = mX;
  p.tma_y = 0;
  if ((int64_t)R * OW == TN && (OH * OW) % 16 == 0 && (reinterpret_cast<uintptr_t>(y) & 15) == 0 &&
      OH * OW < ((int64_t)1 << 31) && !getenv("I8Q_CONV_DIRECT_STORE")) {
    auto fn = tc::encode_fn();
    if (!fn) return fail(I8Q_ERR_CUDA, "qlinearconv: cuTensorMapEncodeTiled unavailable");
    cuuint64_t dims[3] = {(cuuint64_t)(OH * OW), (cuuint64_t)M, (cuuint64_t)N};
    cuuint64_t strides[2] = {(cuuint64_t)(OH * OW), (cuuint64_t)(M * OH * OW)};
    cuuint32_t box[3] = {(cuuint32_t)TN, 32u, 1u};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(&mY, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3u, y, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
      return fail(I8Q_ERR_CUDA, "qlinearconv: cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")");
    p.tma_y = 1;
  }
  const int grid = std::min(p.num_tiles, sm_count());
  I8Q_PROF("qlinearconv_tc", s);
  conv_tc_kernel<TN><<<grid, THREADS, T::SMEM_BYTES, s>>>(mW, mX, mY, p);
  I8Q_LAUNCH_CHECK("conv_tc_kernel");
  return I8Q_OK;
}

}  // namespace i8q
