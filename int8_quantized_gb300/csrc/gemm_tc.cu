// gemm_tc.cu -- exact-integer GEMM on the bf16 tensor pipe (tcgen05).
#include "common.cuh"

namespace i8q {

int launch_gemm_tc(const __nv_bfloat16* uA, const __nv_bfloat16* iBt, int64_t M, int64_t N, int64_t Kp,
                   int max_abs_product_log2, const GemmEpilogue& ep, cudaStream_t s) {
  (void)uA; (void)iBt; (void)M; (void)N; (void)Kp; (void)max_abs_product_log2; (void)ep; (void)s;
  return fail(I8Q_ERR_UNSUPPORTED, "gemm_tc: not built");
}

}  // namespace i8q
