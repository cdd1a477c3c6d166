// Instantiations of the exact int8 GEMM (bf16-held codes, one or four K chunks).
#include "gemm_tc.cuh"

namespace rpp {

cudaError_t gemm_dispatch_int(int nch, int bn, int epi, const CUtensorMap& ta, const CUtensorMap& tb,
                              const gemm::GemmParams& p, int gr, cudaStream_t stream) {
  if (nch == 1) return gemm::dispatch_int<1>(bn, epi, ta, tb, p, gr, stream);
  return gemm::dispatch_int<4>(bn, epi, ta, tb, p, gr, stream);
}

}  // namespace rpp
