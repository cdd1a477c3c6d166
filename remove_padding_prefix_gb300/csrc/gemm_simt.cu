// fp32 GEMM on the CUDA cores for fp32 layers (the tensor cores have no fp32-in,
// fp32-exact mode; tf32 would change the arithmetic).  Same contract and epilogues as
// the tcgen05 GEMM: out[M, N] = epilogue(A[M, K] @ W[N, K]^T).
//
// 64 x 64 output tile per 256-thread CTA, K staged through shared memory 16 at a time,
// each thread accumulating a 4 x 4 block in registers.
#include "kernels.h"

namespace rpp {

namespace {

constexpr int kT = 64;
constexpr int kK = 16;

template <int EPI>
__global__ void __launch_bounds__(256) gemm_f32_kernel(const float* __restrict__ A, const float* __restrict__ W,
                                                       const float* __restrict__ bias, const float* residual,
                                                       float* out, int M_max, const int32_t* rows, int N, int K,
                                                       int32_t* err) {
  pdl_wait();
  pdl_trigger();
  if (device_error_set(err)) return;
  int M = rows ? *rows : M_max;
  if (M > M_max || M < 0) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) set_device_error(err, RPP_DERR_ROWS);
    return;
  }
  const int m0 = blockIdx.y * kT;
  const int n0 = blockIdx.x * kT;
  if (m0 >= M) return;
  __shared__ float As[kK][kT + 4];
  __shared__ float Ws[kK][kT + 4];
  const int tx = threadIdx.x % 16;   // n direction
  const int ty = threadIdx.x / 16;   // m direction
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += kK) {
    // 64 rows x 16 k of A and W: 1024 floats each, 4 per thread (one float4)
    {
      const int r = threadIdx.x / 4;
      const int kk = (threadIdx.x % 4) * 4;
      float4 av = make_float4(0.f, 0.f, 0.f, 0.f), wv = make_float4(0.f, 0.f, 0.f, 0.f);
      if (m0 + r < M && k0 + kk < K) av = *reinterpret_cast<const float4*>(A + static_cast<long long>(m0 + r) * K + k0 + kk);
      if (n0 + r < N && k0 + kk < K) wv = *reinterpret_cast<const float4*>(W + static_cast<long long>(n0 + r) * K + k0 + kk);
      As[kk + 0][r] = av.x; As[kk + 1][r] = av.y; As[kk + 2][r] = av.z; As[kk + 3][r] = av.w;
      Ws[kk + 0][r] = wv.x; Ws[kk + 1][r] = wv.y; Ws[kk + 2][r] = wv.z; Ws[kk + 3][r] = wv.w;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kK; ++kk) {
      float a[4], w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = Ws[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], w[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= M) continue;
    const int n = n0 + tx * 4;
    if (n >= N) continue;
    const float4 b = *reinterpret_cast<const float4*>(bias + n);
    float v[4] = {acc[i][0] + b.x, acc[i][1] + b.y, acc[i][2] + b.z, acc[i][3] + b.w};
    if constexpr (EPI == RPP_EPI_BIAS_GELU) {
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = gelu_erf(v[j]);
    }
    if constexpr (EPI == RPP_EPI_BIAS_RESIDUAL) {
      const float4 r = *reinterpret_cast<const float4*>(residual + static_cast<long long>(m) * N + n);
      v[0] += r.x; v[1] += r.y; v[2] += r.z; v[3] += r.w;
    }
    *reinterpret_cast<float4*>(out + static_cast<long long>(m) * N + n) = make_float4(v[0], v[1], v[2], v[3]);
  }
}

}  // namespace

cudaError_t launch_gemm_f32(const float* a, const float* w_t, const float* bias, const float* residual, float* out,
                            int M_max, const int32_t* rows, int N, int K, int epi, int32_t* err,
                            cudaStream_t stream) {
  dim3 grid((N + kT - 1) / kT, (M_max + kT - 1) / kT);
  if (grid.y == 0) grid.y = 1;
  switch (epi) {
    case RPP_EPI_BIAS:
      return launch_pdl(gemm_f32_kernel<RPP_EPI_BIAS>, grid, dim3(256), 0, stream, a, w_t, bias, residual, out, M_max,
                        rows, N, K, err);
    case RPP_EPI_BIAS_GELU:
      return launch_pdl(gemm_f32_kernel<RPP_EPI_BIAS_GELU>, grid, dim3(256), 0, stream, a, w_t, bias, residual, out,
                        M_max, rows, N, K, err);
    case RPP_EPI_BIAS_RESIDUAL:
      return launch_pdl(gemm_f32_kernel<RPP_EPI_BIAS_RESIDUAL>, grid, dim3(256), 0, stream, a, w_t, bias, residual,
                        out, M_max, rows, N, K, err);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace rpp
