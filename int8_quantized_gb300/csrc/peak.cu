// peak.cu -- throughput probe of the int8 tensor instruction available on
// sm_103a (mma.sync m16n8k32 u8 x s8 -> s32).  Every warp issues
// back-to-back MMAs on register operands with 8 independent accumulators;
// the result is the dense int8 tensor peak this GPU offers to a kernel, the
// denominator of "% of INT8 tensor peak".
#include "common.cuh"

namespace i8q {
namespace {

__device__ __forceinline__ void mma_u8s8_peak(int32_t (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.u8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(256) imma_peak_kernel(int64_t iters, int32_t* out) {
  uint32_t a[4] = {threadIdx.x * 0x01010101u, 0x02020202u, 0x03030303u ^ threadIdx.x, 0x04040404u};
  const uint32_t b0 = 0x01020304u ^ blockIdx.x, b1 = 0x05060708u;
  int32_t acc[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[j][q] = 0;
  for (int64_t i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < 8; ++j) mma_u8s8_peak(acc[j], a, b0, b1);
  }
  int32_t s = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) s += acc[j][0] + acc[j][1] + acc[j][2] + acc[j][3];
  if (s == 0x7fffffff) out[0] = s;  // keeps the loop live; never true in practice
}

}  // namespace
}  // namespace i8q

using namespace i8q;

extern "C" int i8q_measure_int8_mma_peak(int64_t iters, void* stream, double* tops) {
  if (!tops || iters <= 0) return fail(I8Q_ERR_INVALID_ARG, "measure_int8_mma_peak: bad arguments");
  cudaStream_t s = as_stream(stream);
  int32_t* out = nullptr;
  I8Q_CUDA_TRY(cudaMalloc(&out, sizeof(int32_t)));
  cudaEvent_t e0, e1;
  I8Q_CUDA_TRY(cudaEventCreate(&e0));
  I8Q_CUDA_TRY(cudaEventCreate(&e1));
  const int blocks = sm_count() * 4, threads = 256;
  imma_peak_kernel<<<blocks, threads, 0, s>>>(iters / 8 + 1, out);  // warm-up
  I8Q_CUDA_TRY(cudaEventRecord(e0, s));
  imma_peak_kernel<<<blocks, threads, 0, s>>>(iters, out);
  I8Q_CUDA_TRY(cudaEventRecord(e1, s));
  I8Q_CUDA_TRY(cudaEventSynchronize(e1));
  float ms = 0.0f;
  I8Q_CUDA_TRY(cudaEventElapsedTime(&ms, e0, e1));
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  cudaFree(out);
  const double warps = (double)blocks * threads / 32.0;
  const double ops = warps * (double)iters * 8.0 * (2.0 * 16 * 8 * 32);
  *tops = ops / (ms * 1e-3) / 1e12;
  return I8Q_OK;
}
