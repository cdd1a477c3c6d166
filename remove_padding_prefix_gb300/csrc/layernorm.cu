// Row LayerNorm with register arrays, plus the per-tensor int8 quantiser and the
// max-abs reduction used by calibration.
//
// Design (NVIDIA Swin talk, §3: register arrays sized by template parameters with
// constant indices, a strided element-to-thread assignment so that neighbouring
// threads touch neighbouring 16-byte vectors, vector types to cut memory
// instructions): a group of G lanes owns one row; each lane keeps VPL 16-byte vectors
// of the row in registers, so the row is read from HBM once and written once.  Mean
// and variance are two-pass over the registers (biased variance, fp32), reductions
// are xor-shuffles inside the group.  Optional outputs: int8 codes of the normalised
// row (the FC1 input of the int8 layer) and a running max-abs (calibration).
#include "kernels.h"

namespace rpp {

namespace {

__device__ __forceinline__ int8_t quantize_one(float v, float inv_s) {
  const float t = __fmul_rn(v, inv_s);          // one IEEE fp32 multiply
  int q = __float2int_rn(t);                    // round half to even
  q = q > 127 ? 127 : (q < -127 ? -127 : q);
  return static_cast<int8_t>(q);
}

// four residual values of a 16-bit or fp32 row segment (kind: 1 fp32, 2 fp16, 3 bf16)
__device__ __forceinline__ void load_res4(const void* base, int kind, long long off, float* f) {
  if (kind == 1) {
    const float4 r = *reinterpret_cast<const float4*>(static_cast<const float*>(base) + off);
    f[0] = r.x; f[1] = r.y; f[2] = r.z; f[3] = r.w;
  } else {
    const uint2 r = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(base) + off);
    if (kind == 2) {
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&r.x));
      const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&r.y));
      f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    } else {
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.x));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.y));
      f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    }
  }
}

__device__ __forceinline__ void atomic_max_nonneg(float* addr, float v) {
  // non-negative floats order like their bit patterns
  atomicMax(reinterpret_cast<int*>(addr), __float_as_int(v));
}

// EPV floats -> EPV elements of TOut at p (16 or 8 bytes)
template <typename TOut, int EPV>
__device__ __forceinline__ void store_vec(TOut* p, const float* o) {
  if constexpr (sizeof(TOut) * EPV == 16) {
    *reinterpret_cast<uint4*>(p) = pack16<TOut>(o);
  } else {
    static_assert(sizeof(TOut) == 2 && EPV == 4, "8-byte store of four 16-bit values");
    uint2 v;
    if constexpr (std::is_same<TOut, __half>::value) {
      __half2 a = __floats2half2_rn(o[0], o[1]), b = __floats2half2_rn(o[2], o[3]);
      v.x = *reinterpret_cast<uint32_t*>(&a);
      v.y = *reinterpret_cast<uint32_t*>(&b);
    } else {
      __nv_bfloat162 a = __floats2bfloat162_rn(o[0], o[1]), b = __floats2bfloat162_rn(o[2], o[3]);
      v.x = *reinterpret_cast<uint32_t*>(&a);
      v.y = *reinterpret_cast<uint32_t*>(&b);
    }
    *reinterpret_cast<uint2*>(p) = v;
  }
}

template <typename T, typename TOut, int G, int VPL>
__global__ void __launch_bounds__(256) layernorm_kernel(const T* __restrict__ x, const float* __restrict__ gamma,
                                                        const float* __restrict__ beta, TOut* y, int M_max,
                                                        const int32_t* rows, int H, float eps,
                                                        __nv_bfloat16* __restrict__ q_out, const float* q_scale,
                                                        float* amax, float* __restrict__ y32, int n_in,
                                                        long long in_stride, const float* __restrict__ add_bias,
                                                        const void* __restrict__ residual, int res_kind,
                                                        int32_t* err) {
  if (device_error_set(err)) return;
  int M = rows ? *rows : M_max;
  if (M > M_max || M < 0) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_device_error(err, RPP_DERR_ROWS);
    return;
  }
  constexpr int EPV = Vec<T>::N;
  constexpr int GPW = 32 / G;   // groups (rows) per warp
  const int lane = lane_id();
  const int gl = lane % G;      // lane inside the group
  const int gw = lane / G;      // group inside the warp
  const int warps_total = gridDim.x * (blockDim.x >> 5);
  const int wglob = blockIdx.x * (blockDim.x >> 5) + warp_id();
  float inv_s = 0.f;
  if (q_out) inv_s = __fdiv_rn(1.0f, *q_scale);
  float local_amax = 0.f;

  for (int row0 = wglob * GPW; row0 < M; row0 += warps_total * GPW) {
    const int row = row0 + gw;
    const bool valid = row < M;
    float v[VPL][EPV];
    const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<long long>(valid ? row : 0) * H);
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      uint4 raw = make_uint4(0u, 0u, 0u, 0u);
      if (valid) raw = xr[i * G + gl];
      unpack16<T>(raw, v[i]);
    }
    // split-K partial sums of the preceding GEMM: add the other slices of this row
    for (int sl = 1; sl < n_in; ++sl) {
      const uint4* xs = reinterpret_cast<const uint4*>(x + sl * in_stride + static_cast<long long>(valid ? row : 0) * H);
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        float f[EPV];
        uint4 raw = make_uint4(0u, 0u, 0u, 0u);
        if (valid) raw = xs[i * G + gl];
        unpack16<T>(raw, f);
#pragma unroll
        for (int j = 0; j < EPV; ++j) v[i][j] += f[j];
      }
    }
    // the GEMM's bias and the residual branch, split off the GEMM and added here
    if (add_bias) {
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int col0 = (i * G + gl) * EPV;
#pragma unroll
        for (int j = 0; j < EPV; j += 4) {
          const float4 b4 = *reinterpret_cast<const float4*>(add_bias + col0 + j);
          v[i][j] += b4.x; v[i][j + 1] += b4.y; v[i][j + 2] += b4.z; v[i][j + 3] += b4.w;
        }
      }
    }
    if (residual && valid) {
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const long long off = static_cast<long long>(row) * H + (i * G + gl) * EPV;
#pragma unroll
        for (int j = 0; j < EPV; j += 4) {
          float f[4];
          load_res4(residual, res_kind, off + j, f);
          v[i][j] += f[0]; v[i][j + 1] += f[1]; v[i][j + 2] += f[2]; v[i][j + 3] += f[3];
        }
      }
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
#pragma unroll
      for (int j = 0; j < EPV; ++j) s += v[i][j];
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float mean = s / static_cast<float>(H);
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
#pragma unroll
      for (int j = 0; j < EPV; ++j) {
        const float d = v[i][j] - mean;
        ss += d * d;
      }
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float rstd = rsqrtf(ss / static_cast<float>(H) + eps);
    if (valid) {
      TOut* yr = y + static_cast<long long>(row) * H;
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int col0 = (i * G + gl) * EPV;
        float o[EPV];
#pragma unroll
        for (int j = 0; j < EPV; j += 4) {
          const float4 g4 = *reinterpret_cast<const float4*>(gamma + col0 + j);
          const float4 b4 = *reinterpret_cast<const float4*>(beta + col0 + j);
          o[j + 0] = (v[i][j + 0] - mean) * rstd * g4.x + b4.x;
          o[j + 1] = (v[i][j + 1] - mean) * rstd * g4.y + b4.y;
          o[j + 2] = (v[i][j + 2] - mean) * rstd * g4.z + b4.z;
          o[j + 3] = (v[i][j + 3] - mean) * rstd * g4.w + b4.w;
        }
        store_vec<TOut, EPV>(yr + col0, o);
        if (y32) {   // fp32 copy of the normalised row (the next residual add reads it)
          float* yf = y32 + static_cast<long long>(row) * H + col0;
#pragma unroll
          for (int j = 0; j < EPV; j += 4) *reinterpret_cast<float4*>(yf + j) = make_float4(o[j], o[j + 1], o[j + 2], o[j + 3]);
        }
        if (q_out) {   // int8 codes of the normalised row, held in bf16 (exact)
          float qv[EPV];
#pragma unroll
          for (int j = 0; j < EPV; ++j) qv[j] = static_cast<float>(quantize_one(o[j], inv_s));
          store_vec<__nv_bfloat16, EPV>(q_out + static_cast<long long>(row) * H + col0, qv);
        }
        if (amax) {
#pragma unroll
          for (int j = 0; j < EPV; ++j) local_amax = fmaxf(local_amax, fabsf(o[j]));
        }
      }
    }
  }
  if (amax) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) local_amax = fmaxf(local_amax, __shfl_xor_sync(0xffffffffu, local_amax, o));
    if (lane == 0) atomic_max_nonneg(amax, local_amax);
  }
}

// per-tensor symmetric int8 quantisation of [M, H] (8 elements per thread step)
template <typename T>
__global__ void quantize_kernel(const T* __restrict__ x, const float* scale, int8_t* __restrict__ q, int M_max,
                                const int32_t* rows, int H, int32_t* err) {
  if (device_error_set(err)) return;
  int M = rows ? *rows : M_max;
  if (M > M_max || M < 0) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_device_error(err, RPP_DERR_ROWS);
    return;
  }
  const float inv_s = __fdiv_rn(1.0f, *scale);
  const long long n8 = static_cast<long long>(M) * H / 8;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    float f[8];
    if constexpr (sizeof(T) == 2) {
      unpack16<T>(reinterpret_cast<const uint4*>(x)[i], f);
    } else {
      unpack16<T>(reinterpret_cast<const uint4*>(x)[2 * i], f);
      unpack16<T>(reinterpret_cast<const uint4*>(x)[2 * i + 1], f + 4);
    }
    int8_t qv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) qv[j] = quantize_one(f[j], inv_s);
    reinterpret_cast<uint2*>(q)[i] = *reinterpret_cast<const uint2*>(qv);
  }
}

// max |x| over [M, H] (8 elements per thread step), accumulated into *amax
template <typename T>
__global__ void amax_kernel(const T* __restrict__ x, int M_max, const int32_t* rows, int H, float* amax,
                            int32_t* err) {
  if (device_error_set(err)) return;
  int M = rows ? *rows : M_max;
  if (M > M_max || M < 0) M = 0;
  const long long n8 = static_cast<long long>(M) * H / 8;
  float m = 0.f;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    float f[8];
    if constexpr (sizeof(T) == 2) {
      unpack16<T>(reinterpret_cast<const uint4*>(x)[i], f);
    } else {
      unpack16<T>(reinterpret_cast<const uint4*>(x)[2 * i], f);
      unpack16<T>(reinterpret_cast<const uint4*>(x)[2 * i + 1], f + 4);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(f[j]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane_id() == 0) atomic_max_nonneg(amax, m);
}

template <typename T, typename TOut, int G, int VPL>
cudaError_t ln_launch(const void* x, const float* gamma, const float* beta, void* y, int M_max, const int32_t* rows,
                      int H, float eps, __nv_bfloat16* q_out, const float* q_scale, float* amax, float* y32,
                      int n_in, long long in_stride, const float* add_bias, const void* residual, int res_kind,
                      int32_t* err, cudaStream_t stream) {
  const int threads = 256;
  const int rows_per_block = (threads / 32) * (32 / G);
  long long blocks = (static_cast<long long>(M_max) + rows_per_block - 1) / rows_per_block;
  const long long cap = static_cast<long long>(num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  layernorm_kernel<T, TOut, G, VPL><<<static_cast<int>(blocks), threads, 0, stream>>>(
      static_cast<const T*>(x), gamma, beta, static_cast<TOut*>(y), M_max, rows, H, eps, q_out, q_scale, amax, y32,
      n_in, in_stride, add_bias, residual, res_kind, err);
  return cudaGetLastError();
}

template <typename T, typename TOut>
cudaError_t ln_dispatch(const void* x, const float* gamma, const float* beta, void* y, int M_max, const int32_t* rows,
                        int H, float eps, __nv_bfloat16* q_out, const float* q_scale, float* amax, float* y32,
                        int n_in, long long in_stride, const float* add_bias, const void* residual, int res_kind,
                        int32_t* err, cudaStream_t stream) {
  const int V = H / Vec<T>::N;   // 16-byte vectors per row
#define RPP_LN_CASE(G_, VPL_)                                                                                  \
  if (V == (G_) * (VPL_))                                                                                      \
    return ln_launch<T, TOut, G_, VPL_>(x, gamma, beta, y, M_max, rows, H, eps, q_out, q_scale, amax, y32, n_in, \
                                        in_stride, add_bias, residual, res_kind, err, stream);
  RPP_LN_CASE(32, 1) RPP_LN_CASE(32, 2) RPP_LN_CASE(32, 3) RPP_LN_CASE(32, 4)
  RPP_LN_CASE(32, 5) RPP_LN_CASE(32, 6) RPP_LN_CASE(32, 8) RPP_LN_CASE(32, 12) RPP_LN_CASE(32, 16)
  RPP_LN_CASE(16, 1) RPP_LN_CASE(16, 3) RPP_LN_CASE(8, 1) RPP_LN_CASE(8, 3) RPP_LN_CASE(8, 5)
  RPP_LN_CASE(4, 1) RPP_LN_CASE(4, 3) RPP_LN_CASE(4, 5) RPP_LN_CASE(2, 1) RPP_LN_CASE(2, 3) RPP_LN_CASE(1, 1)
  RPP_LN_CASE(1, 3)
#undef RPP_LN_CASE
  return cudaErrorNotSupported;
}

}  // namespace

bool layernorm_supported(int H, rpp_dtype dtype) {
  const int epv = dtype == RPP_F32 ? 4 : 8;
  if (H % epv) return false;
  const int V = H / epv;
  static const int kCases[][2] = {{32, 1}, {32, 2}, {32, 3}, {32, 4}, {32, 5}, {32, 6}, {32, 8}, {32, 12},
                                  {32, 16}, {16, 1}, {16, 3}, {8, 1},  {8, 3},  {8, 5},  {4, 1},  {4, 3},
                                  {4, 5},   {2, 1},  {2, 3},  {1, 1},  {1, 3}};
  for (const auto& c : kCases)
    if (c[0] * c[1] == V) return true;
  return false;
}

cudaError_t launch_layernorm(const void* x, const float* gamma, const float* beta, void* y, int M_max,
                             const int32_t* rows, int H, float eps, rpp_dtype in_dtype, rpp_dtype out_dtype,
                             void* q_codes, const float* q_scale, float* amax, float* y32, int32_t* err,
                             cudaStream_t stream, int n_in, long long in_stride, const float* add_bias,
                             const void* residual, rpp_dtype res_dtype) {
  if (n_in > 1 && in_dtype != RPP_F32) return cudaErrorNotSupported;
  const int res_kind = !residual ? 0 : (res_dtype == RPP_F32 ? 1 : (res_dtype == RPP_F16 ? 2 : 3));
  __nv_bfloat16* q_out = static_cast<__nv_bfloat16*>(q_codes);
  using BF = __nv_bfloat16;
  if (in_dtype == out_dtype) {
    switch (in_dtype) {
      case RPP_F32: return ln_dispatch<float, float>(x, gamma, beta, y, M_max, rows, H, eps, q_out, q_scale, amax, y32, n_in, in_stride, add_bias, residual, res_kind, err, stream);
      case RPP_F16: return ln_dispatch<__half, __half>(x, gamma, beta, y, M_max, rows, H, eps, q_out, q_scale, amax, y32, n_in, in_stride, add_bias, residual, res_kind, err, stream);
      case RPP_BF16: return ln_dispatch<BF, BF>(x, gamma, beta, y, M_max, rows, H, eps, q_out, q_scale, amax, y32, n_in, in_stride, add_bias, residual, res_kind, err, stream);
      default: return cudaErrorNotSupported;
    }
  }
  if (in_dtype == RPP_F32 && out_dtype == RPP_F16)
    return ln_dispatch<float, __half>(x, gamma, beta, y, M_max, rows, H, eps, q_out, q_scale, amax, y32, n_in, in_stride, add_bias, residual, res_kind, err, stream);
  if (in_dtype == RPP_F32 && out_dtype == RPP_BF16)
    return ln_dispatch<float, BF>(x, gamma, beta, y, M_max, rows, H, eps, q_out, q_scale, amax, y32, n_in, in_stride, add_bias, residual, res_kind, err, stream);
  return cudaErrorNotSupported;
}

cudaError_t launch_quantize(const void* x, const float* scale, int8_t* q, int M_max, const int32_t* rows, int H,
                            rpp_dtype dtype, int32_t* err, cudaStream_t stream) {
  const long long n8 = static_cast<long long>(M_max) * H / 8;
  long long blocks = (n8 + 255) / 256;
  const long long cap = static_cast<long long>(num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  switch (dtype) {
    case RPP_F32:
      quantize_kernel<float><<<static_cast<int>(blocks), 256, 0, stream>>>(static_cast<const float*>(x), scale, q,
                                                                            M_max, rows, H, err);
      break;
    case RPP_F16:
      quantize_kernel<__half><<<static_cast<int>(blocks), 256, 0, stream>>>(static_cast<const __half*>(x), scale, q,
                                                                             M_max, rows, H, err);
      break;
    case RPP_BF16:
      quantize_kernel<__nv_bfloat16><<<static_cast<int>(blocks), 256, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(x), scale, q, M_max, rows, H, err);
      break;
    default: return cudaErrorNotSupported;
  }
  return cudaGetLastError();
}

cudaError_t launch_amax(const void* x, int M_max, const int32_t* rows, int H, rpp_dtype dtype, float* amax,
                        int32_t* err, cudaStream_t stream) {
  const long long n8 = static_cast<long long>(M_max) * H / 8;
  long long blocks = (n8 + 255) / 256;
  const long long cap = static_cast<long long>(num_sms()) * 4;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  switch (dtype) {
    case RPP_F32:
      amax_kernel<float><<<static_cast<int>(blocks), 256, 0, stream>>>(static_cast<const float*>(x), M_max, rows, H,
                                                                        amax, err);
      break;
    case RPP_F16:
      amax_kernel<__half><<<static_cast<int>(blocks), 256, 0, stream>>>(static_cast<const __half*>(x), M_max, rows,
                                                                         H, amax, err);
      break;
    case RPP_BF16:
      amax_kernel<__nv_bfloat16><<<static_cast<int>(blocks), 256, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(x), M_max, rows, H, amax, err);
      break;
    default: return cudaErrorNotSupported;
  }
  return cudaGetLastError();
}

}  // namespace rpp
