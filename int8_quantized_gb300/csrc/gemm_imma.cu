// gemm_imma.cu -- integer GEMM core on the warp-level int8 tensor
// instruction (mma.sync m16n8k32, uint8 x int8 -> int32), the only 8-bit
// integer tensor-core form sm_103a accepts.  It serves small products (M or
// N below one tensor-core tile) and is the reference point for the int8
// tensor peak.
//
// It computes the integer step of the Simd dynamic quantized inner product
// ("sum += (uA[i,k] - zeroA[i]) * iB[k,j]") as
//   sum = sum_k uA[i,k] * iB[k,j]  -  zeroA[i] * colsum(iB)[j]
// exactly in int32, then the fused epilogue (dequantize, bias, activation,
// store).  Tiles: 128 x 128 x 64 per CTA, 8 warps of 64 x 32, a 4-stage
// cp.async ring in shared memory with an XOR swizzle on 16-byte chunks so
// ldmatrix reads are bank-conflict free.
#include "common.cuh"

namespace i8q {
namespace {

constexpr int BM = 128, BN = 128, BK = 64, STAGES = 4, THREADS = 256;
constexpr int STAGE_BYTES = (BM + BN) * BK;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_u8s8(int32_t (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.u8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// byte offset of 16-byte chunk c of row r in a BK = 64-byte-row tile
__device__ __forceinline__ int swz(int r, int c) { return r * BK + ((c ^ ((r >> 1) & 3)) << 4); }

__device__ __forceinline__ void store_out(const GemmEpilogue& ep, int64_t r, int64_t c, int64_t N, int32_t v0,
                                          int32_t v1, float sA, int32_t zA) {
  // two adjacent columns c, c+1 of row r
  if (c >= N) return;
  const bool two = c + 1 < N;
  int32_t a0 = v0 - zA * __ldg(ep.colsum + c);
  int32_t a1 = two ? v1 - zA * __ldg(ep.colsum + c + 1) : 0;
  if (ep.out_mode == OUT_S32) {
    int32_t* C = static_cast<int32_t*>(ep.C) + r * ep.ldc + c;
    C[0] = a0;
    if (two) C[1] = a1;
    return;
  }
  const bool bf16 = ep.out_mode == OUT_BF16;
  float b0 = ep.bias ? __ldg(ep.bias + c) : 0.0f;
  float o0 = bf16 ? dequant_epilogue_bf16out(a0, sA, __ldg(ep.scaleB + c), b0, ep.act)
                  : dequant_epilogue(a0, sA, __ldg(ep.scaleB + c), b0, ep.act);
  float o1 = 0.0f;
  if (two) {
    float b1 = ep.bias ? __ldg(ep.bias + c + 1) : 0.0f;
    o1 = bf16 ? dequant_epilogue_bf16out(a1, sA, __ldg(ep.scaleB + c + 1), b1, ep.act)
              : dequant_epilogue(a1, sA, __ldg(ep.scaleB + c + 1), b1, ep.act);
  }
  const bool vec = two && ((ep.ldc & 1) == 0) && ((c & 1) == 0) && (reinterpret_cast<uintptr_t>(ep.C) & 7) == 0;
  if (ep.out_mode == OUT_F32) {
    float* C = static_cast<float*>(ep.C) + r * ep.ldc + c;
    if (vec) {
      *reinterpret_cast<float2*>(C) = make_float2(o0, o1);
    } else {
      C[0] = o0;
      if (two) C[1] = o1;
    }
  } else {
    __nv_bfloat16* C = static_cast<__nv_bfloat16*>(ep.C) + r * ep.ldc + c;
    if (vec) {
      *reinterpret_cast<__nv_bfloat162*>(C) = __floats2bfloat162_rn(o0, o1);
    } else {
      C[0] = __float2bfloat16_rn(o0);
      if (two) C[1] = __float2bfloat16_rn(o1);
    }
  }
}

__global__ void __launch_bounds__(THREADS)
gemm_imma_kernel(const uint8_t* __restrict__ uA, const int8_t* __restrict__ iBt, int64_t M, int64_t N, int64_t Kp,
                 GemmEpilogue ep) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int warp_m = warp >> 2, warp_n = warp & 3;
  const int64_t m0 = (int64_t)blockIdx.y * BM, n0 = (int64_t)blockIdx.x * BN;
  const int KT = (int)(Kp / BK);

  auto load_stage = [&](int stage, int kt) {
    uint8_t* sA = smem + stage * STAGE_BYTES;
    uint8_t* sB = sA + BM * BK;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int idx = tid + i * THREADS;  // 0..511: row = idx/4, chunk = idx%4
      const int r = idx >> 2, c = idx & 3;
      const int64_t ga = m0 + r, gb = n0 + r;
      const uint8_t* pa = uA + (ga < M ? ga : M - 1) * Kp + (int64_t)kt * BK + c * 16;
      const int8_t* pb = iBt + (gb < N ? gb : N - 1) * Kp + (int64_t)kt * BK + c * 16;
      cp_async16(smem_u32(sA + swz(r, c)), pa, ga < M ? 16 : 0);
      cp_async16(smem_u32(sB + swz(r, c)), pb, gb < N ? 16 : 0);
    }
  };

  int32_t acc[4][4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[i][j][q] = 0;

#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < KT) load_stage(s, s);
    cp_async_commit();
  }

  for (int kt = 0; kt < KT; ++kt) {
    cp_async_wait<STAGES - 2>();
    __syncthreads();
    {
      const int nk = kt + STAGES - 1;
      if (nk < KT) load_stage(nk % STAGES, nk);
      cp_async_commit();
    }
    const uint8_t* sA = smem + (kt % STAGES) * STAGE_BYTES;
    const uint8_t* sB = sA + BM * BK;
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      uint32_t af[4][4], bf[4][2];
#pragma unroll
      for (int mi = 0; mi < 4; ++mi) {
        const int r = warp_m * 64 + mi * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int c = kk * 2 + (lane >> 4);
        ldmatrix_x4(smem_u32(sA + swz(r, c)), af[mi][0], af[mi][1], af[mi][2], af[mi][3]);
      }
#pragma unroll
      for (int nj = 0; nj < 2; ++nj) {
        const int r = warp_n * 32 + nj * 16 + (lane & 7) + (lane >> 4) * 8;
        const int c = kk * 2 + ((lane >> 3) & 1);
        ldmatrix_x4(smem_u32(sB + swz(r, c)), bf[2 * nj][0], bf[2 * nj][1], bf[2 * nj + 1][0], bf[2 * nj + 1][1]);
      }
#pragma unroll
      for (int mi = 0; mi < 4; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) mma_u8s8(acc[mi][ni], af[mi], bf[ni][0], bf[ni][1]);
    }
  }
  cp_async_wait<0>();

  const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
  for (int mi = 0; mi < 4; ++mi) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t r = m0 + warp_m * 64 + mi * 16 + g + h * 8;
      if (r >= M) continue;
      const float sA = __ldg(ep.scaleA + r);
      const int32_t zA = __ldg(ep.zeroA + r);
#pragma unroll
      for (int ni = 0; ni < 4; ++ni) {
        const int64_t c = n0 + warp_n * 32 + ni * 8 + 2 * t4;
        store_out(ep, r, c, N, acc[mi][ni][2 * h], acc[mi][ni][2 * h + 1], sA, zA);
      }
    }
  }
}

}  // namespace

int launch_gemm_imma(const uint8_t* uA, const int8_t* iBt, int64_t M, int64_t N, int64_t Kp, const GemmEpilogue& ep,
                     cudaStream_t s) {
  if (M <= 0 || N <= 0) return I8Q_OK;
  if (Kp % BK != 0) return fail(I8Q_ERR_INVALID_ARG, "gemm_imma: Kp must be a multiple of 64");
  const int ar = smem_attr((const void*)gemm_imma_kernel, SMEM_BYTES);
  if (ar) return ar;
  if (ceil_div(M, BM) > 65535) return fail(I8Q_ERR_UNSUPPORTED, "gemm_imma: M too large");
  dim3 grid((unsigned)ceil_div(N, BN), (unsigned)ceil_div(M, BM));
  I8Q_PROF("gemm_imma", s);
  gemm_imma_kernel<<<grid, THREADS, SMEM_BYTES, s>>>(uA, iBt, M, N, Kp, ep);
  I8Q_LAUNCH_CHECK("gemm_imma_kernel");
  return I8Q_OK;
}

}  // namespace i8q
