// Instantiations of the tensor-core GEMM for nv_bfloat16 inputs, CTA pairs.
#include "gemm_tc.cuh"

namespace rpp {

cudaError_t gemm_dispatch_float_bf16_cl2(int bn, int epi, rpp_dtype out_dtype, rpp_dtype res_dtype, const CUtensorMap& ta,
                                  const CUtensorMap& tb, const gemm::GemmParams& p, int gr, cudaStream_t stream) {
  return gemm::dispatch_float<__nv_bfloat16, 2>(bn, epi, out_dtype, res_dtype, ta, tb, p, gr, stream);
}

}  // namespace rpp
