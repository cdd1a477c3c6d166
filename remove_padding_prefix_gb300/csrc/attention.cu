// Fused multi-head attention over packed variable-length sequences: the entry point
// and the fp32 kernel (fp16 / bf16 run on the tensor cores, attention_tc.cu).
//
// NVIDIA Swin talk, §3: batch GEMM, softmax and batch GEMM merged into one fMHA kernel,
// with the head transposes absorbed into the kernel's reads and writes.  Kuaishou
// article, Fig. 10: attention is the kernel that needs the sequence boundaries after
// padding removal, so it reads them from cu_seqlens and touches valid tokens only.
//
// The fp32 kernel (fp32 layers): one thread per query row, K and V tiles staged
// through shared memory, online softmax.  Keys past the sequence end are excluded.
#include "kernels.h"

namespace rpp {

namespace {

constexpr int kD = 64;   // head dim

// fp32 attention for fp32 layers: one thread per query row, keys staged through smem
constexpr int kF32Rows = 64;
__global__ void __launch_bounds__(kF32Rows) attention_varlen_f32_kernel(const float* __restrict__ qkv,
                                                                        const int32_t* __restrict__ cu, int T_max,
                                                                        int max_len, int nh,
                                                                        float* __restrict__ out, float scale,
                                                                        int32_t* err) {
  pdl_wait();
  pdl_trigger();
  // other CTAs of this launch may set the error word at any time: one thread reads it
  // and the whole CTA follows that one reading (all threads return here, or none)
  __shared__ int s_quit;
  if (threadIdx.x == 0) s_quit = device_error_set(err) ? 1 : 0;
  __syncthreads();
  if (s_quit) return;
  const int b = blockIdx.z;
  const int h = blockIdx.y;
  const int q0 = blockIdx.x * kF32Rows;
  const int c0 = cu[b];
  const int c1 = cu[b + 1];
  const int len = c1 - c0;
  if (c0 < 0 || len < 0 || c1 > T_max || len > max_len) {
    if (threadIdx.x == 0) set_device_error(err, len > max_len ? RPP_DERR_LENGTH : RPP_DERR_ROWS);
    return;
  }
  if (q0 >= len) return;
  __shared__ float sK[kF32Rows][kD + 1];
  __shared__ float sV[kF32Rows][kD];
  const int H = nh * kD;
  const long long ld = 3LL * H;
  const int qi = q0 + threadIdx.x;
  const bool qvalid = qi < len;
  float q[kD], o[kD];
  const float* qrow = qkv + static_cast<long long>(c0 + (qvalid ? qi : 0)) * ld + h * kD;
#pragma unroll
  for (int c = 0; c < kD; ++c) {
    q[c] = qrow[c] * scale;
    o[c] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  for (int k0 = 0; k0 < len; k0 += kF32Rows) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < kF32Rows * kD; idx += kF32Rows) {
      const int r = idx / kD, c = idx % kD;
      const bool ok = k0 + r < len;
      const float* row = qkv + static_cast<long long>(c0 + (ok ? k0 + r : 0)) * ld;
      sK[r][c] = ok ? row[H + h * kD + c] : 0.f;
      sV[r][c] = ok ? row[2 * H + h * kD + c] : 0.f;
    }
    __syncthreads();
    const int nk = min(kF32Rows, len - k0);
    for (int j = 0; j < nk; ++j) {
      float sc = 0.f;
#pragma unroll
      for (int c = 0; c < kD; ++c) sc = fmaf(q[c], sK[j][c], sc);
      const float mn = fmaxf(m, sc);
      const float corr = expf(m - mn);
      const float p = expf(sc - mn);
      l = l * corr + p;
#pragma unroll
      for (int c = 0; c < kD; ++c) o[c] = fmaf(p, sV[j][c], o[c] * corr);
      m = mn;
    }
  }
  if (qvalid) {
    float* orow = out + static_cast<long long>(c0 + qi) * H + h * kD;
    const float inv = 1.f / l;
#pragma unroll
    for (int c = 0; c < kD; c += 4)
      *reinterpret_cast<float4*>(orow + c) = make_float4(o[c] * inv, o[c + 1] * inv, o[c + 2] * inv, o[c + 3] * inv);
  }
}

}  // namespace

cudaError_t launch_attention_varlen(const void* qkv, const int32_t* cu, int B, int T_max, int max_len, int nh, int d,
                                    rpp_dtype dtype, void* out, int32_t* err, cudaStream_t stream) {
  if (d != kD) return cudaErrorNotSupported;
  if (B <= 0 || max_len <= 0) return cudaSuccess;
  const float scale = 1.0f / sqrtf(static_cast<float>(d));
  if (dtype == RPP_F32) {
    dim3 grid((max_len + kF32Rows - 1) / kF32Rows, nh, B);
    return launch_pdl(attention_varlen_f32_kernel, grid, dim3(kF32Rows), 0, stream, static_cast<const float*>(qkv), cu,
                      T_max, max_len, nh, static_cast<float*>(out), scale, err);
  }
  if (dtype == RPP_F16 || dtype == RPP_BF16) {
    if (attention_sched_supported(B, max_len))
      return launch_attention_sched(qkv, cu, B, T_max, max_len, nh, dtype, out, err, stream);
    return launch_attention_tc(qkv, cu, B, T_max, max_len, nh, dtype, out, err, stream);
  }
  return cudaErrorNotSupported;
}

}  // namespace rpp
