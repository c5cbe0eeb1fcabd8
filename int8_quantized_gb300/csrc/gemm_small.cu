// gemm_small.cu -- the dynamic quantized inner product (Simd
// "SynetDynamicQuantizedInnerProduct16b", Detailed Description) for
// products too small to fill tensor-core tiles, such as 64 x 128 x 256.
//
// One launch does the whole Forward after B is prepared: each CTA takes four
// rows of A, quantizes them per row to uint8 in shared memory (the same
// arithmetic as the row quantization kernels, and it writes uA, scaleA,
// zeroA out once), then forms
//   sum[i,j] = sum_k uA[i,k] * iB[k,j]  -  zeroA[i] * colsum[j]
// with dp4a (four uint8 x int8 products per instruction, int32 exact) and
// applies the epilogue.  On this GPU the warp-level int8 mma.sync is slow
// (about 4x the latency of the bf16 form), so the SIMT dot product is the
// faster integer path for work that cannot use the tcgen05 tiles.
//
// Thread layout: 128 threads = 32 columns x 4 K-slices per pass; K-slice s
// reads the 16-byte chunks s, s+4, ... of the iB row and the four A rows,
// the slices are summed with two shuffles, and lane slice s then owns row s
// of the four for the epilogue.
#include "common.cuh"

namespace i8q {
namespace {

constexpr int RB = 4;         // rows of A per CTA (one warp quantizes each)
constexpr int KSL = 4;        // K-slices per column
constexpr int COLS = 32;      // columns per pass
constexpr int THREADS = COLS * KSL;
constexpr int64_t kMaxKp = 8192;  // RB * Kp bytes of shared memory

static_assert(RB == KSL, "lane slice s writes row s");
static_assert(THREADS == 32 * RB, "one warp per row in the quantization");

__device__ __forceinline__ int32_t dp4a_u8s8(uint32_t a, uint32_t b, int32_t c) {
  int32_t d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ float load_f32(const float* p) { return __ldg(p); }
__device__ __forceinline__ float load_f32(const __nv_bfloat16* p) { return __bfloat162float(*p); }

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
__global__ void __launch_bounds__(THREADS)
small_qgemm_kernel(const T* __restrict__ A, int64_t M, int64_t K, int64_t Kp, const int8_t* __restrict__ iBt,
                   int64_t N, uint8_t* __restrict__ uA, float* __restrict__ scaleA, int32_t* __restrict__ zeroA,
                   GemmEpilogue ep) {
  extern __shared__ __align__(16) uint8_t su[];  // RB rows x Kp codes
  __shared__ float s_scale[RB];
  __shared__ int s_zero[RB];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t r0 = (int64_t)blockIdx.x * RB;

  // ---- quantize row r0 + warp into shared memory -------------------------
  {
    const int64_t row = r0 + warp;
    uint8_t* dst = su + (int64_t)warp * Kp;
    const bool writer = blockIdx.y == 0;
    if (row < M) {
      const T* a = A + row * K;
      float mn = 0.0f, mx = 0.0f;
      for (int64_t k = lane; k < K; k += 32) {
        const float v = load_f32(a + k);
        mn = fminf(mn, v);
        mx = fmaxf(mx, v);
      }
      mn = warp_min(mn);
      mx = warp_max(mx);
      float s;
      int z;
      row_scale_zero(mn, mx, s, z);
      const float lo_z = (float)(-z), hi_z = (float)(255 - z);
      for (int64_t k = lane; k < Kp; k += 32) {
        const uint8_t c = k < K ? (uint8_t)row_code(load_f32(a + k), s, lo_z, hi_z, z) : (uint8_t)0;
        dst[k] = c;
        if (writer) uA[row * Kp + k] = c;
      }
      if (lane == 0) {
        s_scale[warp] = s;
        s_zero[warp] = z;
        if (writer) {
          scaleA[row] = s;
          zeroA[row] = z;
        }
      }
    } else {
      for (int64_t k = lane; k < Kp; k += 32) dst[k] = 0;
      if (lane == 0) {
        s_scale[warp] = 1.0f;
        s_zero[warp] = 0;
      }
    }
  }
  __syncthreads();

  // ---- integer sums and epilogue ----------------------------------------
  const int ks = tid % KSL, cl = tid / KSL;
  const int64_t chunks = Kp / 16;
  const int64_t row = r0 + ks;
  const float sA = s_scale[ks];
  const int32_t zA = s_zero[ks];
  for (int64_t j0 = (int64_t)blockIdx.y * COLS; j0 < N; j0 += (int64_t)gridDim.y * COLS) {
    const int64_t j = j0 + cl;
    int32_t acc[RB] = {0, 0, 0, 0};
    if (j < N) {
      const uint4* b = reinterpret_cast<const uint4*>(iBt + j * Kp);
#pragma unroll 4
      for (int64_t c = ks; c < chunks; c += KSL) {
        const uint4 bw = __ldg(b + c);
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          const uint4 aw = *reinterpret_cast<const uint4*>(su + r * Kp + c * 16);
          int32_t t = acc[r];
          t = dp4a_u8s8(aw.x, bw.x, t);
          t = dp4a_u8s8(aw.y, bw.y, t);
          t = dp4a_u8s8(aw.z, bw.z, t);
          t = dp4a_u8s8(aw.w, bw.w, t);
          acc[r] = t;
        }
      }
    }
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], 1);
      acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], 2);
    }
    if (j >= N || row >= M) continue;
    const int32_t sum = ks == 0 ? acc[0] : ks == 1 ? acc[1] : ks == 2 ? acc[2] : acc[3];
    const int32_t v = sum - zA * __ldg(ep.colsum + j);
    const int64_t o = row * ep.ldc + j;
    if (ep.out_mode == OUT_S32) {
      static_cast<int32_t*>(ep.C)[o] = v;
      continue;
    }
    const float b = ep.bias ? __ldg(ep.bias + j) : 0.0f;
    const float sB = __ldg(ep.scaleB + j);
    if (ep.out_mode == OUT_BF16)
      static_cast<__nv_bfloat16*>(ep.C)[o] = __float2bfloat16_rn(dequant_epilogue_bf16out(v, sA, sB, b, ep.act));
    else
      static_cast<float*>(ep.C)[o] = dequant_epilogue(v, sA, sB, b, ep.act);
  }
}

}  // namespace

int64_t small_max_kp() { return kMaxKp; }

int launch_gemm_small(const void* A, int typeA, int64_t M, int64_t K, int64_t Kp, const int8_t* iBt, int64_t N,
                      uint8_t* uA, float* scaleA, int32_t* zeroA, const GemmEpilogue& ep, cudaStream_t s) {
  if (M <= 0 || N <= 0) return I8Q_OK;
  if (Kp % 64 != 0 || Kp > kMaxKp || K > Kp) return fail(I8Q_ERR_UNSUPPORTED, "gemm_small: Kp must be <= 8192");
  if (reinterpret_cast<uintptr_t>(iBt) & 15) return fail(I8Q_ERR_UNSUPPORTED, "gemm_small: iBt must be 16-byte aligned");
  const int64_t gx = ceil_div(M, RB);
  if (gx > 0x7fffffff) return fail(I8Q_ERR_UNSUPPORTED, "gemm_small: M too large");
  // enough CTAs to cover the SMs twice, splitting the columns when there are
  // few row blocks
  const int64_t groups = ceil_div(N, COLS);
  const int64_t gy = std::min<int64_t>(std::min<int64_t>(groups, 65535),
                                       std::max<int64_t>(1, ceil_div(2 * (int64_t)sm_count(), gx)));
  const dim3 grid((unsigned)gx, (unsigned)gy);
  const size_t smem = (size_t)RB * (size_t)Kp;
  I8Q_PROF("gemm_small", s);
  if (typeA == I8Q_BF16)
    small_qgemm_kernel<__nv_bfloat16><<<grid, THREADS, smem, s>>>(static_cast<const __nv_bfloat16*>(A), M, K, Kp,
                                                                   iBt, N, uA, scaleA, zeroA, ep);
  else
    small_qgemm_kernel<float><<<grid, THREADS, smem, s>>>(static_cast<const float*>(A), M, K, Kp, iBt, N, uA, scaleA,
                                                           zeroA, ep);
  I8Q_LAUNCH_CHECK("small_qgemm_kernel");
  return I8Q_OK;
}

}  // namespace i8q
