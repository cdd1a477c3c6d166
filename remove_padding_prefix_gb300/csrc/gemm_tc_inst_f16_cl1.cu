// Instantiations of the tensor-core GEMM for half inputs, single CTAs.
#include "gemm_tc.cuh"

namespace rpp {

cudaError_t gemm_dispatch_float_f16_cl1(int bn, int epi, rpp_dtype out_dtype, rpp_dtype res_dtype, const CUtensorMap& ta,
                                  const CUtensorMap& tb, const gemm::GemmParams& p, int gr, cudaStream_t stream) {
  return gemm::dispatch_float<__half, 1>(bn, epi, out_dtype, res_dtype, ta, tb, p, gr, stream);
}

}  // namespace rpp
