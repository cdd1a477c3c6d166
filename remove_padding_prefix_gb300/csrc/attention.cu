// Fused multi-head attention over packed variable-length sequences.
//
// NVIDIA Swin talk, §3: batch GEMM, softmax and batch GEMM merged into one fMHA kernel,
// with the head transposes absorbed into the kernel's reads and writes.  Kuaishou
// article, Fig. 10: attention is the kernel that needs the sequence boundaries after
// padding removal, so it reads them from cu_seqlens and touches valid tokens only.
//
// One CTA = one (query tile of 64 rows, head, sequence); 4 warps x 16 query rows.
// Q, K, V tiles are read straight out of the token-major QKV GEMM output (row t holds
// Q | K | V, head h at columns h*d) with cp.async into XOR-swizzled shared memory; K/V
// tiles of 64 keys are double-buffered.  S = Q K^T and O += P V use
// mma.sync.m16n8k16 with fp32 accumulation; the softmax is online (running row max
// and sum, exp2 with the 1/sqrt(d) scale folded in), its row reductions are
// xor-shuffles inside each quad of lanes.  The normalised output goes back through
// shared memory and leaves as 16-byte stores into the token-major [T, nh*d] output.
// Keys past the sequence end are excluded (score -inf).
#include "kernels.h"

namespace rpp {

namespace {

constexpr int kD = 64;      // head dim
constexpr int kBMq = 64;    // query rows per CTA
constexpr int kBNk = 64;    // keys per iteration
constexpr int kWarps = 4;

__device__ __forceinline__ uint32_t swz(int r, int chunk) {   // byte offset inside a 64 x 64 x 2B tile
  return static_cast<uint32_t>(r * 128 + ((chunk ^ (r & 7)) << 4));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

template <typename T>
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1);
template <>
__device__ __forceinline__ void mma16816<__half>(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <>
__device__ __forceinline__ void mma16816<__nv_bfloat16>(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <typename T> __device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <> __device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
template <> __device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// load a 64-row x 64-col tile (rows [row0, row0+64) of a [*, ld] matrix at column col0),
// rows >= row_end are zero-filled; 128 threads, 4 x 16-byte chunks each
template <typename T>
__device__ __forceinline__ void load_tile(uint8_t* s, const T* g, long long ld, int row0, int row_end, int col0,
                                          int tid) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int id = tid + i * 128;
    const int r = id >> 3;
    const int c = id & 7;
    const bool ok = row0 + r < row_end;
    const T* src = g + static_cast<long long>(ok ? row0 + r : row0) * ld + col0 + c * 8;
    cp_async_16(s + swz(r, c), src, ok);
  }
}

template <typename T>
__global__ void __launch_bounds__(128) attention_varlen_kernel(const T* __restrict__ qkv,
                                                               const int32_t* __restrict__ cu, int T_max,
                                                               int max_len, int nh, T* __restrict__ out,
                                                               float scale_log2, int32_t* err) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.z;
  const int h = blockIdx.y;
  const int q0 = blockIdx.x * kBMq;
  // the error word and the sequence bounds are read together (one round trip)
  const int c0 = cu[b];
  const int c1 = cu[b + 1];
  if (device_error_set(err)) return;
  const int len = c1 - c0;
  if (c0 < 0 || len < 0 || c1 > T_max || len > max_len) {
    if (threadIdx.x == 0) set_device_error(err, len > max_len ? RPP_DERR_LENGTH : RPP_DERR_ROWS);
    return;
  }
  if (q0 >= len) return;

  __shared__ __align__(128) uint8_t sQ[kBMq * kD * 2];
  __shared__ __align__(128) uint8_t sK[2][kBNk * kD * 2];
  __shared__ __align__(128) uint8_t sV[2][kBNk * kD * 2];

  const int H = nh * kD;
  const long long ld = 3LL * H;
  const T* base = qkv + static_cast<long long>(c0) * ld;
  const int tid = threadIdx.x;
  const int warp = warp_id();
  const int lane = lane_id();
  const int nkb = (len + kBNk - 1) / kBNk;

  load_tile<T>(sQ, base, ld, q0, len, h * kD, tid);
  load_tile<T>(sK[0], base, ld, 0, len, H + h * kD, tid);
  load_tile<T>(sV[0], base, ld, 0, len, 2 * H + h * kD, tid);
  cp_async_commit();

  uint32_t qf[4][4];
  float o[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m_r[2] = {-INFINITY, -INFINITY};
  float l_r[2] = {0.f, 0.f};

  const uint32_t sQa = smem_u32(sQ);
  for (int kb = 0; kb < nkb; ++kb) {
    if (kb + 1 < nkb) {
      load_tile<T>(sK[(kb + 1) & 1], base, ld, (kb + 1) * kBNk, len, H + h * kD, tid);
      load_tile<T>(sV[(kb + 1) & 1], base, ld, (kb + 1) * kBNk, len, 2 * H + h * kD, tid);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (kb == 0) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int r = warp * 16 + (lane & 15);
        const int ch = kk * 2 + (lane >> 4);
        ldsm_x4(sQa + swz(r, ch), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
      }
    }
    const uint32_t sKa = smem_u32(sK[kb & 1]);
    const uint32_t sVa = smem_u32(sV[kb & 1]);
    // ---- S = Q K^T for this warp's 16 rows x 64 keys
    float s[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {   // pairs of 8-key tiles
        uint32_t b0, b1, b2, b3;
        const int r = np * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int ch = kk * 2 + ((lane >> 3) & 1);
        ldsm_x4(sKa + swz(r, ch), b0, b1, b2, b3);
        mma16816<T>(s[2 * np], qf[kk], b0, b1);
        mma16816<T>(s[2 * np + 1], qf[kk], b2, b3);
      }
    }
    // ---- online softmax (scores scaled into the log2 domain)
    const int kbase = kb * kBNk;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int key = kbase + j * 8 + 2 * (lane & 3);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool valid = key + (e & 1) < len;
        s[j][e] = valid ? s[j][e] * scale_log2 : -INFINITY;
      }
      mx[0] = fmaxf(mx[0], fmaxf(s[j][0], s[j][1]));
      mx[1] = fmaxf(mx[1], fmaxf(s[j][2], s[j][3]));
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
    }
    float alpha[2], mnew[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mnew[i] = fmaxf(m_r[i], mx[i]);
      const float mref = mnew[i] == -INFINITY ? 0.f : mnew[i];
      alpha[i] = exp2f(m_r[i] - mref);
      m_r[i] = mnew[i];
      mnew[i] = mref;
    }
    float rs[2] = {0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      s[j][0] = exp2f(s[j][0] - mnew[0]);
      s[j][1] = exp2f(s[j][1] - mnew[0]);
      s[j][2] = exp2f(s[j][2] - mnew[1]);
      s[j][3] = exp2f(s[j][3] - mnew[1]);
      rs[0] += s[j][0] + s[j][1];
      rs[1] += s[j][2] + s[j][3];
    }
    l_r[0] = l_r[0] * alpha[0] + rs[0];
    l_r[1] = l_r[1] * alpha[1] + rs[1];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      o[j][0] *= alpha[0];
      o[j][1] *= alpha[0];
      o[j][2] *= alpha[1];
      o[j][3] *= alpha[1];
    }
    // ---- O += P V
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {   // 16 keys per step
      uint32_t pa[4];
      pa[0] = pack2<T>(s[2 * kk][0], s[2 * kk][1]);
      pa[1] = pack2<T>(s[2 * kk][2], s[2 * kk][3]);
      pa[2] = pack2<T>(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[3] = pack2<T>(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int dp = 0; dp < 4; ++dp) {   // pairs of 8-wide d tiles
        uint32_t b0, b1, b2, b3;
        const int r = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int ch = dp * 2 + (lane >> 4);
        ldsm_x4_t(sVa + swz(r, ch), b0, b1, b2, b3);
        mma16816<T>(o[2 * dp], pa, b0, b1);
        mma16816<T>(o[2 * dp + 1], pa, b2, b3);
      }
    }
    __syncthreads();
  }
  // ---- normalise, stage through shared memory (this warp's 16 rows of sQ), store
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    l_r[i] += __shfl_xor_sync(0xffffffffu, l_r[i], 1);
    l_r[i] += __shfl_xor_sync(0xffffffffu, l_r[i], 2);
    l_r[i] = l_r[i] > 0.f ? 1.f / l_r[i] : 0.f;
  }
  const int rA = warp * 16 + (lane >> 2);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t lo = pack2<T>(o[j][0] * l_r[0], o[j][1] * l_r[0]);
    const uint32_t hi = pack2<T>(o[j][2] * l_r[1], o[j][3] * l_r[1]);
    *reinterpret_cast<uint32_t*>(sQ + swz(rA, j) + (lane & 3) * 4) = lo;
    *reinterpret_cast<uint32_t*>(sQ + swz(rA + 8, j) + (lane & 3) * 4) = hi;
  }
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int id = lane + i * 32;
    const int r = warp * 16 + (id >> 3);
    const int c = id & 7;
    const int q = q0 + r;
    if (q < len) {
      const uint4 v = *reinterpret_cast<const uint4*>(sQ + swz(r, c));
      *reinterpret_cast<uint4*>(out + static_cast<long long>(c0 + q) * H + h * kD + c * 8) = v;
    }
  }
}

// fp32 attention for fp32 layers: one thread per query row, keys staged through smem
constexpr int kF32Rows = 64;
__global__ void __launch_bounds__(kF32Rows) attention_varlen_f32_kernel(const float* __restrict__ qkv,
                                                                        const int32_t* __restrict__ cu, int T_max,
                                                                        int max_len, int nh,
                                                                        float* __restrict__ out, float scale,
                                                                        int32_t* err) {
  pdl_wait();
  pdl_trigger();
  if (device_error_set(err)) return;
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
  if (dtype == RPP_F16 || dtype == RPP_BF16)
    return launch_attention_tc(qkv, cu, B, T_max, max_len, nh, dtype, out, err, stream);
  dim3 grid((max_len + kBMq - 1) / kBMq, nh, B);
  const float scale_log2 = scale * 1.4426950408889634f;
  if (dtype == RPP_F16) {
    return launch_pdl(attention_varlen_kernel<__half>, grid, dim3(kWarps * 32), 0, stream,
                      static_cast<const __half*>(qkv), cu, T_max, max_len, nh, static_cast<__half*>(out), scale_log2,
                      err);
  }
  if (dtype == RPP_BF16) {
    return launch_pdl(attention_varlen_kernel<__nv_bfloat16>, grid, dim3(kWarps * 32), 0, stream,
                      static_cast<const __nv_bfloat16*>(qkv), cu, T_max, max_len, nh,
                      static_cast<__nv_bfloat16*>(out), scale_log2, err);
  }
  return cudaErrorNotSupported;
}

}  // namespace rpp
