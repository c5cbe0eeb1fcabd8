// noalloc.cu -- the dynamic quantized inner product in one call that
// allocates no memory.
//
// Who needs it: code that runs inside a host application which owns every
// byte of device memory through its own pool and does not let plugins call
// cudaMalloc (an inference server's custom-op plugin, say), and code on a
// latency-critical path that cannot afford cudaMalloc/cudaFree, which may
// synchronize the device.  Such a caller cannot create a context (Init
// allocates) or hand Forward a scratch buffer it allocated itself.
//
// This entry point takes A, an int8 B with its per-column scales, the bias
// and C from the caller, and keeps every intermediate (the uint8 copy of A
// with its row scales and zero points, B transposed to K-contiguous rows and
// its column sums) in one file-scope device array of fixed size.  Every GPU
// that loads the library holds that array until the process exits.
#include <mutex>

#include "common.cuh"

namespace i8q {
namespace {

constexpr size_t kStaticScratchBytes = I8Q_QGEMM_STATIC_SCRATCH_BYTES;

static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_static_mu;
uint8_t* g_static_ptr[kMaxDev] = {nullptr};

// Device address of g_static_scratch on the current device.  In host code
// the symbol is only a host-side stand-in, so the address comes from the
// runtime, once per device, with that device current.
int static_scratch(uint8_t** out) {
  int dev = 0;
  I8Q_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDev) return fail(I8Q_ERR_UNSUPPORTED, "qgemm_dyn_static: device index out of range");
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || !p) return cuda_fail(e, "cudaGetSymbolAddress(g_static_scratch)");
    g_static_ptr[dev] = static_cast<uint8_t*>(p);
  }
  *out = g_static_ptr[dev];
  return I8Q_OK;
}

size_t a256(size_t v) { return (v + 255) & ~size_t(255); }

}  // namespace
}  // namespace i8q

using namespace i8q;

extern "C" size_t i8q_qgemm_dyn_static_scratch_bytes(size_t M, size_t N, size_t K) {
  const size_t Kp = (size_t)round_up((int64_t)K, 64);
  return a256(M * Kp) + a256(M * 4) + a256(M * 4) + a256(N * Kp) + a256(N * 4);
}

extern "C" size_t i8q_qgemm_dyn_static_scratch_capacity(void) { return kStaticScratchBytes; }

extern "C" int i8q_qgemm_dyn_static(size_t M, size_t N, size_t K, int typeA, const void* A, const int8_t* B,
                                    const float* scaleB, const float* bias, int activation, int typeC, void* C,
                                    void* stream) {
  if (M == 0 || N == 0 || K == 0) return fail(I8Q_ERR_INVALID_ARG, "qgemm_dyn_static: M, N, K must be >= 1");
  if (K > 65536) return fail(I8Q_ERR_UNSUPPORTED, "qgemm_dyn_static: K > 65536 (int32 sums could overflow)");
  if (typeA != I8Q_F32 && typeA != I8Q_BF16) return fail(I8Q_ERR_INVALID_ARG, "qgemm_dyn_static: typeA must be F32 or BF16");
  if (typeC != I8Q_F32 && typeC != I8Q_BF16) return fail(I8Q_ERR_INVALID_ARG, "qgemm_dyn_static: typeC must be F32 or BF16");
  if (activation < I8Q_ACT_IDENTITY || activation > I8Q_ACT_GELU)
    return fail(I8Q_ERR_UNSUPPORTED, "qgemm_dyn_static: unknown activation");
  if (!A || !B || !scaleB || !C) return fail(I8Q_ERR_INVALID_ARG, "qgemm_dyn_static: A, B, scaleB and C are required");
  const size_t need = i8q_qgemm_dyn_static_scratch_bytes(M, N, K);
  if (need > kStaticScratchBytes)
    return fail(I8Q_ERR_UNSUPPORTED, "qgemm_dyn_static: needs " + std::to_string(need) + " bytes of scratch, more than the " +
                                         std::to_string(kStaticScratchBytes) + "-byte static array");
  uint8_t* base = nullptr;
  int rc = static_scratch(&base);
  if (rc) return rc;
  const int64_t Kp = round_up((int64_t)K, 64);
  size_t o = 0;
  uint8_t* uA = base + o;
  o += a256(M * (size_t)Kp);
  float* scaleA = reinterpret_cast<float*>(base + o);
  o += a256(M * 4);
  int32_t* zeroA = reinterpret_cast<int32_t*>(base + o);
  o += a256(M * 4);
  int8_t* iBt = reinterpret_cast<int8_t*>(base + o);
  o += a256(N * (size_t)Kp);
  int32_t* colsum = reinterpret_cast<int32_t*>(base + o);
  cudaStream_t s = as_stream(stream);
  // every byte read below is written first in this call: the repack writes
  // iBt over all Kp columns and every column sum; the row quantization (on
  // its own, or inside the fused small-product kernel) writes uA over all Kp
  // columns (zero beyond K)
  rc = launch_repack_cols_s8(B, (int64_t)K, (int64_t)N, (int64_t)N, iBt, nullptr, Kp, colsum, s);
  if (rc) return rc;
  GemmEpilogue ep{zeroA, scaleA, colsum, scaleB, bias, activation, typeC == I8Q_BF16 ? OUT_BF16 : OUT_F32, C,
                  (int64_t)N};
  // the same rule as a context's choice: small products (Kp <= 8192 and
  // at most 2^27 multiply-adds) on the fused dp4a kernel, larger ones on the
  // row kernel and the int8 mma.sync core (the tensor-pipe path would need
  // bf16 copies of both operands, twice the scratch)
  const double macs = (double)M * (double)N * (double)Kp;
  if (Kp <= small_max_kp() && macs <= (double)(1 << 27))
    return launch_gemm_small(A, typeA, (int64_t)M, (int64_t)K, Kp, iBt, (int64_t)N, uA, scaleA, zeroA, ep, s);
  rc = launch_quantize_rows(A, typeA, (int64_t)M, (int64_t)K, (int64_t)K, uA, nullptr, Kp, scaleA, zeroA, s);
  if (rc) return rc;
  return launch_gemm_imma(uA, iBt, (int64_t)M, (int64_t)N, Kp, ep, s);
}
