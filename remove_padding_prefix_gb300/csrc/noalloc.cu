// Allocation-free variant of the int8 GEMM with int32 output.
//
// rpp_gemm_i8_i32 needs scratch memory: the int8 operands are re-encoded as bf16 for
// the tensor cores, and the caller provides the buffer.  Some callers have no way to
// provide one -- a plugin inside a host framework that owns all device memory and
// hands out no allocator, a real-time path that must not call cudaMalloc (it can
// synchronise the device and stall other streams), or a foreign-function caller that
// cannot manage the lifetime of device buffers.  For them this file keeps the scratch
// in a fixed-size array in device global memory that is part of the library itself.
//
// Costs and limits a user should know:
//  * every GPU that loads the library holds the array (kNoAllocScratchBytes) until the
//    process exits;
//  * problems whose re-encoded operands need more than that are rejected with
//    RPP_EWORKSPACE before anything is launched;
//  * all calls share the one array and it keeps whatever the previous call left; every
//    byte a call reads is written earlier by the same call, so nothing needs clearing,
//    but two calls whose kernels overlap on the GPU (different streams, no ordering
//    between them) race on the array and give wrong results;
//  * every call looks up the array's device address on the current device with
//    cudaGetSymbolAddress (cheap, no stream work), so the address stays right after a
//    cudaDeviceReset or a context change; the first call on a device also loads the
//    library's device code there, so make that first call outside any stream capture.
#include "kernels.h"

namespace rpp {
namespace {

constexpr size_t kNoAllocScratchBytes = RPP_GEMM_I8_NOALLOC_SCRATCH_BYTES;

// In host code this name stands for a host-side shadow of the symbol, not a device
// address: only the address returned by cudaGetSymbolAddress may be handed to kernels.
static __device__ __align__(256) uint8_t g_i8_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array in the current device's context.  Looked up on
// every call rather than cached: after a cudaDeviceReset the module is loaded again and
// the array may sit at another address.
cudaError_t scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_i8_noalloc_scratch);
  if (e != cudaSuccess) return e;
  if (!p) return cudaErrorInvalidSymbol;
  *out = p;
  return cudaSuccess;
}

inline size_t round256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

}  // namespace
}  // namespace rpp

extern "C" rpp_status rpp_gemm_i8_i32_noalloc(const int8_t* aq, const int8_t* wq_t, int32_t* acc, int M, int N,
                                              int K, int32_t* err, rpp_stream stream) {
  using namespace rpp;
  if (!aq || !wq_t || !acc || M <= 0 || N <= 0 || K <= 0) return RPP_EINVAL;
  if (K % 16 || N % 16 || K > 4096) return RPP_EUNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(acc) & 15u) != 0) return RPP_EINVAL;
  const size_t a_bytes = round256(static_cast<size_t>(M) * K * 2);
  const size_t w_bytes = round256(static_cast<size_t>(N) * K * 2);
  if (a_bytes + w_bytes > kNoAllocScratchBytes) return RPP_EWORKSPACE;
  void* base = nullptr;
  const cudaError_t ea = scratch_address(&base);
  if (ea != cudaSuccess) return status_from_cuda(ea);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* a_codes = base;
  void* w_codes = static_cast<uint8_t*>(base) + a_bytes;
  cudaError_t e = launch_i8_to_bf16(aq, a_codes, static_cast<long long>(M) * K, s);
  if (e == cudaSuccess) e = launch_i8_to_bf16(wq_t, w_codes, static_cast<long long>(N) * K, s);
  if (e == cudaSuccess) {
    TcGemmArgs g{};
    g.a = a_codes;
    g.w_t = w_codes;
    g.out = acc;
    g.M_max = M;
    g.N = N;
    g.K = K;
    g.in_dtype = RPP_BF16;
    g.out_dtype = RPP_F32;
    g.epi = EPI_I32;
    g.err = err;
    e = launch_gemm_tc(g, s);
  }
  return status_from_cuda(e);   // the same mapping as rpp_gemm_i8_i32
}
