// One-time preprocessing and int8 helper kernels.
//
// NVIDIA Swin talk, §3: inference allows computing once, ahead of time, what every
// forward pass would otherwise recompute -- here the weight reformat (the QKV weights
// concatenated into one K-major matrix so one GEMM feeds the attention kernel),
// fp32 copies of biases and LayerNorm parameters, and the per-output-channel int8
// weight quantisation; plus the activation quantiser whose codes feed the int8 GEMM.
#include "kernels.h"

namespace rpp {

namespace {

template <typename T>
__device__ __forceinline__ float load_f32(const void* p, long long i) {
  return to_f32(static_cast<const T*>(p)[i]);
}

__device__ __forceinline__ float load_any(const void* p, rpp_dtype dt, long long i) {
  if (dt == RPP_F16) return load_f32<__half>(p, i);
  if (dt == RPP_BF16) return load_f32<__nv_bfloat16>(p, i);
  return load_f32<float>(p, i);
}

// dst[n, k] (row stride dst_ld elements) = src[k, n]; 32 x 32 tiles through shared memory
template <typename E>
__global__ void transpose_kernel(const E* __restrict__ src, int K, int N, E* __restrict__ dst, int dst_ld) {
  __shared__ E tile[32][33];
  const int k0 = blockIdx.y * 32, n0 = blockIdx.x * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int k = k0 + i, n = n0 + threadIdx.x;
    if (k < K && n < N) tile[i][threadIdx.x] = src[static_cast<long long>(k) * N + n];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int n = n0 + i, k = k0 + threadIdx.x;
    if (k < K && n < N) dst[static_cast<long long>(n) * dst_ld + k] = tile[threadIdx.x][i];
  }
}

// s_w[n] = fp32(max_k |W[k, n]| / 127), 1 for an all-zero column
__global__ void weight_scale_kernel(const void* w, rpp_dtype dt, int K, int N, float* s_w) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  float m = 0.f;
  for (int k = 0; k < K; ++k) m = fmaxf(m, fabsf(load_any(w, dt, static_cast<long long>(k) * N + n)));
  s_w[n] = m > 0.f ? __fdiv_rn(m, 127.0f) : 1.0f;
}

// q[n, k] = clamp(rne(fp32(W[k, n] / s_w[n])), -127, 127), written K-major (int8 and/or bf16 codes)
__global__ void weight_quant_kernel(const void* w, rpp_dtype dt, int K, int N, const float* s_w, int8_t* wq_t,
                                    __nv_bfloat16* wq_t_bf16) {
  __shared__ float tile[32][33];
  const int k0 = blockIdx.y * 32, n0 = blockIdx.x * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int k = k0 + i, n = n0 + threadIdx.x;
    if (k < K && n < N) tile[i][threadIdx.x] = load_any(w, dt, static_cast<long long>(k) * N + n);
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int n = n0 + i, k = k0 + threadIdx.x;
    if (k < K && n < N) {
      const float t = __fdiv_rn(tile[threadIdx.x][i], s_w[n]);
      float q = rintf(t);
      q = fminf(fmaxf(q, -127.f), 127.f);
      const long long o = static_cast<long long>(n) * K + k;
      if (wq_t) wq_t[o] = static_cast<int8_t>(static_cast<int>(q));
      if (wq_t_bf16) wq_t_bf16[o] = __float2bfloat16_rn(q);
    }
  }
}

template <typename T>
__global__ void codes_bf16_kernel(const T* __restrict__ x, const float* scale, __nv_bfloat16* __restrict__ codes,
                                  int M_max, const int32_t* rows, int H, int32_t* err) {
  pdl_wait();
  pdl_trigger();
  if (device_error_set(err)) return;
  int M = rows ? *rows : M_max;
  if (M > M_max || M < 0) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_device_error(err, RPP_DERR_ROWS);
    return;
  }
  const float inv_s = __fdiv_rn(1.0f, *scale);
  const long long n = static_cast<long long>(M) * H;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float t = __fmul_rn(to_f32(x[i]), inv_s);
    const float q = fminf(fmaxf(rintf(t), -127.f), 127.f);
    codes[i] = __float2bfloat16_rn(q);
  }
}

__global__ void i8_to_bf16_kernel(const int8_t* __restrict__ src, __nv_bfloat16* __restrict__ dst, long long n) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x)
    dst[i] = __float2bfloat16_rn(static_cast<float>(src[i]));
}

__global__ void to_f32_kernel(const void* src, rpp_dtype dt, long long n, float* dst) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x)
    dst[i] = load_any(src, dt, i);
}

int grid_for(long long n, int threads, int per_sm) {
  long long b = (n + threads - 1) / threads;
  const long long cap = static_cast<long long>(num_sms()) * per_sm;
  if (b > cap) b = cap;
  return b < 1 ? 1 : static_cast<int>(b);
}

}  // namespace

cudaError_t launch_transpose_to_kmajor(const void* w, int K, int N, int elem_bytes, void* dst, int dst_ld,
                                       cudaStream_t stream) {
  dim3 grid((N + 31) / 32, (K + 31) / 32), block(32, 8);
  if (elem_bytes == 2)
    transpose_kernel<uint16_t><<<grid, block, 0, stream>>>(static_cast<const uint16_t*>(w), K, N,
                                                           static_cast<uint16_t*>(dst), dst_ld);
  else if (elem_bytes == 4)
    transpose_kernel<uint32_t><<<grid, block, 0, stream>>>(static_cast<const uint32_t*>(w), K, N,
                                                           static_cast<uint32_t*>(dst), dst_ld);
  else if (elem_bytes == 1)
    transpose_kernel<uint8_t><<<grid, block, 0, stream>>>(static_cast<const uint8_t*>(w), K, N,
                                                          static_cast<uint8_t*>(dst), dst_ld);
  else
    return cudaErrorNotSupported;
  return cudaGetLastError();
}

cudaError_t launch_quantize_weight(const void* w, int K, int N, rpp_dtype dtype, int8_t* wq_t, void* wq_t_bf16,
                                   float* s_w, cudaStream_t stream) {
  weight_scale_kernel<<<(N + 127) / 128, 128, 0, stream>>>(w, dtype, K, N, s_w);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 grid((N + 31) / 32, (K + 31) / 32), block(32, 8);
  weight_quant_kernel<<<grid, block, 0, stream>>>(w, dtype, K, N, s_w, wq_t, static_cast<__nv_bfloat16*>(wq_t_bf16));
  return cudaGetLastError();
}

cudaError_t launch_quantize_codes_bf16(const void* x, const float* scale, void* codes, int M_max, const int32_t* rows,
                                       int H, rpp_dtype dtype, int32_t* err, cudaStream_t stream) {
  const int g = grid_for(static_cast<long long>(M_max) * H, 256, 8);
  auto* c = static_cast<__nv_bfloat16*>(codes);
  const dim3 grid(static_cast<unsigned>(g));
  switch (dtype) {
    case RPP_F16:
      return launch_pdl(codes_bf16_kernel<__half>, grid, dim3(256), 0, stream, static_cast<const __half*>(x), scale, c,
                        M_max, rows, H, err);
    case RPP_BF16:
      return launch_pdl(codes_bf16_kernel<__nv_bfloat16>, grid, dim3(256), 0, stream,
                        static_cast<const __nv_bfloat16*>(x), scale, c, M_max, rows, H, err);
    case RPP_F32:
      return launch_pdl(codes_bf16_kernel<float>, grid, dim3(256), 0, stream, static_cast<const float*>(x), scale, c,
                        M_max, rows, H, err);
    default: return cudaErrorNotSupported;
  }
}

cudaError_t launch_i8_to_bf16(const int8_t* src, void* dst, long long n, cudaStream_t stream) {
  i8_to_bf16_kernel<<<grid_for(n, 256, 8), 256, 0, stream>>>(src, static_cast<__nv_bfloat16*>(dst), n);
  return cudaGetLastError();
}

cudaError_t launch_to_f32(const void* src, rpp_dtype dtype, long long n, float* dst, cudaStream_t stream) {
  to_f32_kernel<<<grid_for(n, 256, 4), 256, 0, stream>>>(src, dtype, n, dst);
  return cudaGetLastError();
}

}  // namespace rpp
