// Swin stage downsampling, first half: the 2 x 2 neighbourhood gather fused into the
// LayerNorm over the concatenated 4C channels.
//
// The NVIDIA Swin talk shows the network as stages at falling resolution with a
// downsampling step between them (a resolution pyramid, like a CNN's); the standard
// patch merging is taken for that step.  Output token (py, px) of an image concatenates
// input tokens (2py, 2px), (2py+1, 2px), (2py, 2px+1), (2py+1, 2px+1) -- block k of the
// 4C channels comes from row offset k & 1 and column offset k >> 1 -- and normalises
// the 4C values (biased variance, fp32 statistics, two passes over registers).  The
// bias-free 4C -> 2C map that follows is the tensor-core GEMM.
//
// One warp per output token: lane l holds 16-byte vectors l, l + 32, ... of the
// concatenated row, each read straight from its source token (no concatenated copy is
// ever stored unnormalised).
#include "kernels.h"

namespace rpp {

namespace {

template <typename T, int VPL>
__global__ void __launch_bounds__(256) patch_merge_ln_kernel(const T* __restrict__ x, int B, int I, int C,
                                                             const float* __restrict__ gamma,
                                                             const float* __restrict__ beta, float eps,
                                                             T* __restrict__ out, int32_t* err) {
  pdl_wait();
  pdl_trigger();
  constexpr int EPV = 8;               // 16-bit elements per 16-byte vector
  const int V = C / 2;                 // vectors per output row (4C / 8)
  // LayerNorm parameters staged once per block (4C floats each)
  extern __shared__ float pm_smem[];
  float* s_gamma = pm_smem;
  float* s_beta = pm_smem + 4 * C;
  for (int i = threadIdx.x; i < 4 * C; i += blockDim.x) {
    s_gamma[i] = __ldg(gamma + i);
    s_beta[i] = __ldg(beta + i);
  }
  // other blocks may set the error word at any time: one thread reads it and the
  // whole block follows that reading through the barrier below
  __shared__ int s_quit;
  if (threadIdx.x == 0) s_quit = device_error_set(err) ? 1 : 0;
  __syncthreads();
  if (s_quit) return;
  const int Ih = I / 2;
  const unsigned per_img = static_cast<unsigned>(Ih) * Ih;
  const unsigned rows = static_cast<unsigned>(B) * per_img;   // the host keeps this below 2^31
  const int vpc = C / EPV;             // vectors per source token
  const int lane = lane_id();
  // a lane owns the same vectors of every row: vector v of the concatenated row is
  // block k = v / vpc, read from row offset k & 1, column offset k >> 1 of the 2 x 2
  // neighbourhood; those source offsets are fixed for the whole loop
  int voff[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int v = lane + 32 * i;
    const int k = v < V ? v / vpc : 0;
    voff[i] = ((k & 1) * I + (k >> 1)) * C + (v - k * vpc) * EPV;
  }
  const unsigned warps = gridDim.x * (blockDim.x >> 5);
  for (unsigned j = blockIdx.x * (blockDim.x >> 5) + warp_id(); j < rows; j += warps) {
    const unsigned b = j / per_img;
    const unsigned rem = j - b * per_img;
    const unsigned py = rem / Ih, px = rem - py * Ih;
    const T* base = x + ((static_cast<long long>(b) * I + 2 * py) * I + 2 * px) * C;
    uint4 rv[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      rv[i] = lane + 32 * i < V ? *reinterpret_cast<const uint4*>(base + voff[i]) : make_uint4(0u, 0u, 0u, 0u);
    float f[VPL][EPV];
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      unpack16<T>(rv[i], f[i]);
#pragma unroll
      for (int e = 0; e < EPV; ++e) sum += f[i][e];   // zero for vectors past the row
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float mean = sum / static_cast<float>(4 * C);
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      if (lane + 32 * i < V) {
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
          const float d = f[i][e] - mean;
          ss += d * d;
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float rstd = rsqrtf(ss / static_cast<float>(4 * C) + eps);
    T* orow = out + static_cast<long long>(j) * 4 * C;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int v = lane + 32 * i;
      if (v < V) {
        const float4* g4 = reinterpret_cast<const float4*>(s_gamma + v * EPV);
        const float4* b4 = reinterpret_cast<const float4*>(s_beta + v * EPV);
        const float4 g0 = g4[0], g1 = g4[1], b0 = b4[0], b1 = b4[1];
        const float gg[EPV] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        const float bb[EPV] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
        float o8[EPV];
#pragma unroll
        for (int e = 0; e < EPV; ++e) o8[e] = (f[i][e] - mean) * rstd * gg[e] + bb[e];
        *reinterpret_cast<uint4*>(orow + v * EPV) = pack16<T>(o8);
      }
    }
  }
}

template <typename T, int VPL>
cudaError_t pm_launch(const void* x, int B, int I, int C, const float* gamma, const float* beta, float eps, void* out,
                      int32_t* err, cudaStream_t stream) {
  const long long rows = static_cast<long long>(B) * (I / 2) * (I / 2);
  const size_t smem = 8 * static_cast<size_t>(C) * sizeof(float);
  // grid-strided rows: one wave of resident blocks, no partial last wave
  static int cached_C = -1, cached_per_sm = 0;
  if (cached_C != C) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, patch_merge_ln_kernel<T, VPL>, 256, smem) != cudaSuccess || n < 1)
      n = 2;
    cached_per_sm = n;
    cached_C = C;
  }
  const int per_sm = cached_per_sm;
  long long blocks = (rows + 7) / 8;
  const long long cap = static_cast<long long>(num_sms()) * per_sm;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_pdl(patch_merge_ln_kernel<T, VPL>, dim3(static_cast<unsigned>(blocks)), dim3(256), smem, stream,
                    static_cast<const T*>(x), B, I, C, gamma, beta, eps, static_cast<T*>(out), err);
}

template <typename T>
cudaError_t pm_dispatch(const void* x, int B, int I, int C, const float* gamma, const float* beta, float eps,
                        void* out, int32_t* err, cudaStream_t stream) {
  const int vpl = (C / 2 + 31) / 32;   // 4C / 8 vectors over 32 lanes
  if (vpl <= 1) return pm_launch<T, 1>(x, B, I, C, gamma, beta, eps, out, err, stream);
  if (vpl <= 2) return pm_launch<T, 2>(x, B, I, C, gamma, beta, eps, out, err, stream);
  if (vpl <= 3) return pm_launch<T, 3>(x, B, I, C, gamma, beta, eps, out, err, stream);
  if (vpl <= 4) return pm_launch<T, 4>(x, B, I, C, gamma, beta, eps, out, err, stream);
  if (vpl <= 6) return pm_launch<T, 6>(x, B, I, C, gamma, beta, eps, out, err, stream);
  if (vpl <= 8) return pm_launch<T, 8>(x, B, I, C, gamma, beta, eps, out, err, stream);
  if (vpl <= 12) return pm_launch<T, 12>(x, B, I, C, gamma, beta, eps, out, err, stream);
  return cudaErrorNotSupported;
}

}  // namespace

bool patch_merge_supported(int C, int I) { return C > 0 && C % 8 == 0 && C <= 768 && I > 0 && I % 2 == 0; }

cudaError_t launch_patch_merge_ln(const void* x, int B, int I, int C, rpp_dtype dtype, const float* gamma,
                                  const float* beta, float eps, void* out, int32_t* err, cudaStream_t stream) {
  if (!patch_merge_supported(C, I)) return cudaErrorNotSupported;
  if (B <= 0) return cudaSuccess;
  if (static_cast<long long>(B) * (I / 2) * (I / 2) > 0x7fffffffLL) return cudaErrorNotSupported;   // 32-bit row index
  if (dtype == RPP_F16) return pm_dispatch<__half>(x, B, I, C, gamma, beta, eps, out, err, stream);
  if (dtype == RPP_BF16) return pm_dispatch<__nv_bfloat16>(x, B, I, C, gamma, beta, eps, out, err, stream);
  return cudaErrorNotSupported;
}

}  // namespace rpp
