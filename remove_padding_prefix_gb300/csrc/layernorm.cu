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

constexpr int kMaxSlices = 4;   // split-K partial sums a LayerNorm input may consist of

__device__ __forceinline__ int8_t quantize_one(float v, float inv_s) {
  const float t = __fmul_rn(v, inv_s);          // one IEEE fp32 multiply
  int q = __float2int_rn(t);                    // round half to even
  q = q > 127 ? 127 : (q < -127 ? -127 : q);
  return static_cast<int8_t>(q);
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

// One row (group of G lanes) per iteration.  All of the row's global loads -- the
// input (and the split-K slices), the residual -- are issued before any arithmetic,
// so a row costs one memory round trip; gamma, beta and the GEMM bias live in shared
// memory, loaded once per CTA.  In padded-output mode the grid walks the padded
// [B, L] slots: a valid slot normalises its packed row and writes it in place, a pad
// slot is written as zeros (the padding rebuild of the last layer, fused).
// Shared-memory position (in float4 units) of the 4 parameters starting at column 4 q.
// Lane gl of a group reads, for its vector i and quarter j4, the float4 at
// (i EPV/4 + j4) G + gl: the lanes of a group read consecutive float4s, so one
// 16-byte shared load per quarter is free of bank conflicts.
template <int G, int EPV>
__device__ __forceinline__ int param_slot(int q) {
  constexpr int E4 = EPV / 4;
  const int vec = q / E4;   // = i G + gl
  return ((vec / G) * E4 + q % E4) * G + vec % G;
}

template <typename T, typename TOut, int G, int VPL, int NS>
__global__ void __launch_bounds__(128) layernorm_kernel(LnArgs a) {
  const int H = a.H;
  constexpr int EPV = Vec<T>::N;
  // gamma, beta and the bias are layer weights, never written by the launch just
  // before this one: their reads are issued before the grid-dependency wait, so they
  // overlap the tail of the preceding kernel.  H = G VPL EPV exactly (the host
  // dispatch), so each thread stages kPre float4 quarters of each vector.
  constexpr int kQ = G * VPL * EPV / 4;
  constexpr int kPre = (kQ + 127) / 128;
  float4 pg[kPre], pb[kPre], pc[kPre];
#pragma unroll
  for (int k = 0; k < kPre; ++k) {
    const int q = threadIdx.x + k * 128;
    if (q < kQ) {
      pg[k] = __ldg(reinterpret_cast<const float4*>(a.gamma) + q);
      pb[k] = __ldg(reinterpret_cast<const float4*>(a.beta) + q);
      pc[k] = a.add_bias ? __ldg(reinterpret_cast<const float4*>(a.add_bias) + q) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  pdl_wait();
  pdl_trigger();
  const bool err_set = device_error_set(a.err);
  int M = a.rows ? *a.rows : a.M_max;
  extern __shared__ float4 ln_smem4[];
  float4* s_gamma = ln_smem4;
  float4* s_beta = ln_smem4 + kQ;
  float4* s_bias = ln_smem4 + 2 * kQ;
#pragma unroll
  for (int k = 0; k < kPre; ++k) {
    const int q = threadIdx.x + k * 128;
    if (q < kQ) {
      const int slot = param_slot<G, EPV>(q);
      s_gamma[slot] = pg[k];
      s_beta[slot] = pb[k];
      s_bias[slot] = pc[k];
    }
  }
  if (err_set) return;
  if (M > a.M_max || M < 0) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_device_error(a.err, RPP_DERR_ROWS);
    return;
  }
  __syncthreads();

  constexpr int GPW = 32 / G;   // groups (rows) per warp
  const T* x = static_cast<const T*>(a.x);
  TOut* y = static_cast<TOut*>(a.y);
  const int lane = lane_id();
  const int gl = lane % G;      // lane inside the group
  const int gw = lane / G;      // group inside the warp
  const int warps_total = gridDim.x * (blockDim.x >> 5);
  const int wglob = blockIdx.x * (blockDim.x >> 5) + warp_id();
  const bool padded = a.pad_cu != nullptr;
  const long long n_iter = padded ? static_cast<long long>(a.pad_B) * a.pad_L : M;
  float inv_s = 0.f;
  if (a.q_codes) inv_s = __fdiv_rn(1.0f, *a.q_scale);
  float local_amax = 0.f;

  // packed row normalised for loop position itx (-1: none)
  auto src_of = [&](long long itx) -> int {
    if (itx >= n_iter) return -1;
    if (!padded) return static_cast<int>(itx);
    // 32-bit division: the host keeps pad_B * pad_L below 2^31
    const unsigned b = static_cast<unsigned>(itx) / static_cast<unsigned>(a.pad_L);
    const int p = static_cast<int>(static_cast<unsigned>(itx) - b * static_cast<unsigned>(a.pad_L));
    const int c0 = a.pad_cu[b];
    return p < a.pad_cu[b + 1] - c0 ? c0 + p : -1;
  };
  // residual adds are taken only with fp32 input (the host rejects the rest): 16-bit
  // instantiations carry no residual registers
  constexpr bool kRes = std::is_same<T, float>::value;
  // 16-bit input (one slice, no residual): the next row's vectors are requested before
  // this row's arithmetic, two rows in flight per group
  constexpr bool kPf = !kRes && NS == 1;
  const long long stride_it = static_cast<long long>(warps_total) * GPW;
  uint4 nx[kPf ? VPL : 1];
  if constexpr (kPf) {
    const int s0 = src_of(static_cast<long long>(wglob) * GPW + gw);
    const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<long long>(s0 >= 0 ? s0 : 0) * H);
#pragma unroll
    for (int i = 0; i < VPL; ++i) nx[i] = s0 >= 0 ? xr[i * G + gl] : make_uint4(0u, 0u, 0u, 0u);
  }

  for (long long it0 = static_cast<long long>(wglob) * GPW; it0 < n_iter; it0 += stride_it) {
    const long long it = it0 + gw;
    const int src = src_of(it);                        // packed row normalised by this group
    const long long dst = it < n_iter ? it : -1;       // output row
    const bool valid = src >= 0;
    // ---- loads: input and its split-K slices (NS > 1), residual -- all issued together
    uint4 rx[NS][VPL];
    uint4 rr[kRes ? VPL : 1][kRes ? EPV / 4 : 1];
    if constexpr (kPf) {
#pragma unroll
      for (int i = 0; i < VPL; ++i) rx[0][i] = nx[i];
      const int sn = src_of(it + stride_it);
      const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<long long>(sn >= 0 ? sn : 0) * H);
#pragma unroll
      for (int i = 0; i < VPL; ++i) nx[i] = sn >= 0 ? xr[i * G + gl] : make_uint4(0u, 0u, 0u, 0u);
    } else {
#pragma unroll
      for (int sl = 0; sl < NS; ++sl) {
        if (sl == 0 || sl < a.n_in) {
          const uint4* xr =
              reinterpret_cast<const uint4*>(x + sl * a.in_stride + static_cast<long long>(valid ? src : 0) * H);
#pragma unroll
          for (int i = 0; i < VPL; ++i) rx[sl][i] = valid ? xr[i * G + gl] : make_uint4(0u, 0u, 0u, 0u);
        }
      }
    }
    const bool has_res = kRes && a.residual != nullptr && valid;
    if constexpr (kRes) {
    if (has_res) {
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
#pragma unroll
        for (int j = 0; j < EPV / 4; ++j) {
          const long long off = static_cast<long long>(src) * H + (i * G + gl) * EPV + 4 * j;
          if (a.res_kind == 1) {
            rr[i][j] = *reinterpret_cast<const uint4*>(static_cast<const float*>(a.residual) + off);
          } else {
            const uint2 t = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(a.residual) + off);
            rr[i][j] = make_uint4(t.x, t.y, 0u, 0u);
          }
        }
      }
    }
    }
    float v[VPL][EPV];
#pragma unroll
    for (int i = 0; i < VPL; ++i) unpack16<T>(rx[0][i], v[i]);
    // split-K partial sums of the preceding GEMM: the other slices of this row (those
    // beyond the NS loaded up front, one round trip each)
#pragma unroll
    for (int sl = 1; sl < NS; ++sl) {
      if (sl < a.n_in) {
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
          float f[EPV];
          unpack16<T>(rx[sl][i], f);
#pragma unroll
          for (int j = 0; j < EPV; ++j) v[i][j] += f[j];
        }
      }
    }
    for (int sl = NS; sl < a.n_in; ++sl) {
      const uint4* xs =
          reinterpret_cast<const uint4*>(x + sl * a.in_stride + static_cast<long long>(valid ? src : 0) * H);
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        float f[EPV];
        unpack16<T>(valid ? xs[i * G + gl] : make_uint4(0u, 0u, 0u, 0u), f);
#pragma unroll
        for (int j = 0; j < EPV; ++j) v[i][j] += f[j];
      }
    }
    // the GEMM's bias and the residual branch, split off the GEMM and added here
    if (a.add_bias) {
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
#pragma unroll
        for (int j4 = 0; j4 < EPV / 4; ++j4) {
          const float4 b4 = s_bias[(i * (EPV / 4) + j4) * G + gl];
          v[i][4 * j4 + 0] += b4.x; v[i][4 * j4 + 1] += b4.y; v[i][4 * j4 + 2] += b4.z; v[i][4 * j4 + 3] += b4.w;
        }
      }
    }
    if constexpr (kRes) {
    if (has_res) {
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
#pragma unroll
        for (int j = 0; j < EPV / 4; ++j) {
          float f[4];
          const uint4 t = rr[i][j];
          if (a.res_kind == 1) {
            f[0] = __uint_as_float(t.x); f[1] = __uint_as_float(t.y);
            f[2] = __uint_as_float(t.z); f[3] = __uint_as_float(t.w);
          } else if (a.res_kind == 2) {
            const float2 p0 = __half22float2(*reinterpret_cast<const __half2*>(&t.x));
            const float2 p1 = __half22float2(*reinterpret_cast<const __half2*>(&t.y));
            f[0] = p0.x; f[1] = p0.y; f[2] = p1.x; f[3] = p1.y;
          } else {
            const float2 p0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&t.x));
            const float2 p1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&t.y));
            f[0] = p0.x; f[1] = p0.y; f[2] = p1.x; f[3] = p1.y;
          }
          v[i][4 * j + 0] += f[0]; v[i][4 * j + 1] += f[1]; v[i][4 * j + 2] += f[2]; v[i][4 * j + 3] += f[3];
        }
      }
    }
    }
    // ---- statistics (biased variance, two passes over the registers)
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
#pragma unroll
      for (int j = 0; j < EPV; ++j) sum += v[i][j];
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float mean = sum / static_cast<float>(H);
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
    const float rstd = rsqrtf(ss / static_cast<float>(H) + a.eps);
    if (dst < 0) continue;
    TOut* yr = y + dst * H;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const int col0 = (i * G + gl) * EPV;
      float o[EPV];
      if (valid) {
#pragma unroll
        for (int j4 = 0; j4 < EPV / 4; ++j4) {
          const float4 g4 = s_gamma[(i * (EPV / 4) + j4) * G + gl];
          const float4 b4 = s_beta[(i * (EPV / 4) + j4) * G + gl];
          o[4 * j4 + 0] = (v[i][4 * j4 + 0] - mean) * rstd * g4.x + b4.x;
          o[4 * j4 + 1] = (v[i][4 * j4 + 1] - mean) * rstd * g4.y + b4.y;
          o[4 * j4 + 2] = (v[i][4 * j4 + 2] - mean) * rstd * g4.z + b4.z;
          o[4 * j4 + 3] = (v[i][4 * j4 + 3] - mean) * rstd * g4.w + b4.w;
        }
      } else {
#pragma unroll
        for (int j = 0; j < EPV; ++j) o[j] = 0.f;   // pad slot of the padded output
      }
      store_vec<TOut, EPV>(yr + col0, o);
      if (!valid) continue;
      if (a.y32) {   // fp32 copy of the normalised row (the next residual add reads it)
        float* yf = a.y32 + dst * H + col0;
#pragma unroll
        for (int j = 0; j < EPV; j += 4)
          *reinterpret_cast<float4*>(yf + j) = make_float4(o[j], o[j + 1], o[j + 2], o[j + 3]);
      }
      if (a.q_codes) {   // int8 codes of the normalised row, held in bf16 (exact)
        float qv[EPV];
#pragma unroll
        for (int j = 0; j < EPV; ++j) qv[j] = static_cast<float>(quantize_one(o[j], inv_s));
        store_vec<__nv_bfloat16, EPV>(static_cast<__nv_bfloat16*>(a.q_codes) + dst * H + col0, qv);
      }
      if (a.amax) {
#pragma unroll
        for (int j = 0; j < EPV; ++j) local_amax = fmaxf(local_amax, fabsf(o[j]));
      }
    }
  }
  if (a.amax) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) local_amax = fmaxf(local_amax, __shfl_xor_sync(0xffffffffu, local_amax, o));
    if (lane == 0) atomic_max_nonneg(a.amax, local_amax);
  }
}

// per-tensor symmetric int8 quantisation of [M, H] (8 elements per thread step)
template <typename T>
__global__ void quantize_kernel(const T* __restrict__ x, const float* scale, int8_t* __restrict__ q, int M_max,
                                const int32_t* rows, int H, int32_t* err) {
  pdl_wait();
  pdl_trigger();
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
  pdl_wait();
  pdl_trigger();
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

// ---------------------------------------------------------------- streaming rows
// LayerNorm of rows that arrive complete (the pre-LayerNorm sums that the proj and FC2
// GEMMs write with bias and residual already added: fp16 in 16-bit layers, fp32 in bf16
// layers): no slices, bias or residual to add.  One warp per row with H = 32 VPL EPV
// (lane l holds the 16-byte vectors l, l + 32, ...), the next row's vectors in flight
// while this one is normalised, and the arithmetic on packed fp32 pairs (one f32x2
// instruction per two elements).  Statistics as in the general kernel: fp32, two passes
// over the registers, biased variance.  Optional fp32 or fp16 copy of the output, and the
// padded-output mode of the general kernel.
constexpr int kLnsThreads = 256;

template <typename TIn, typename TOut, int VPL>
__global__ void __launch_bounds__(kLnsThreads) ln_stream_kernel(LnArgs a) {
  constexpr int EPV = Vec<TIn>::N;   // elements per 16-byte vector: 8 (16-bit) or 4 (fp32)
  constexpr int E4 = EPV / 4;        // float4 quarters per vector
  constexpr int H = 32 * VPL * EPV;
  constexpr int kQ = H / 4;          // float4 quarters of a parameter vector
  constexpr int kPre = (kQ + kLnsThreads - 1) / kLnsThreads;
  constexpr int kWarps = kLnsThreads / 32;
  // gamma and beta are layer weights, not written by the preceding launch: read before
  // the grid-dependency wait
  float4 pg[kPre], pb[kPre];
#pragma unroll
  for (int k = 0; k < kPre; ++k) {
    const int qd = threadIdx.x + k * kLnsThreads;
    if (qd < kQ) {
      pg[k] = __ldg(reinterpret_cast<const float4*>(a.gamma) + qd);
      pb[k] = __ldg(reinterpret_cast<const float4*>(a.beta) + qd);
    }
  }
  pdl_wait();
  pdl_trigger();
  const bool err_set = device_error_set(a.err);
  const int M = a.rows ? *a.rows : a.M_max;
  __shared__ float4 s_g[kQ], s_b[kQ];
#pragma unroll
  for (int k = 0; k < kPre; ++k) {
    const int qd = threadIdx.x + k * kLnsThreads;
    if (qd < kQ) {
      const int slot = param_slot<32, EPV>(qd);
      s_g[slot] = pg[k];
      s_b[slot] = pb[k];
    }
  }
  if (err_set) return;
  if (M > a.M_max || M < 0) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_device_error(a.err, RPP_DERR_ROWS);
    return;
  }
  __syncthreads();

  const TIn* x = static_cast<const TIn*>(a.x);
  TOut* y = static_cast<TOut*>(a.y);
  const int lane = lane_id();
  const bool padded = a.pad_cu != nullptr;
  // the host keeps pad_B * pad_L below 2^31
  const unsigned n_iter = padded ? static_cast<unsigned>(a.pad_B) * static_cast<unsigned>(a.pad_L)
                                 : static_cast<unsigned>(M);
  const unsigned stride = gridDim.x * kWarps;
  auto src_of = [&](unsigned itx) -> int {   // packed row normalised for loop position itx (-1: none)
    if (itx >= n_iter) return -1;
    if (!padded) return static_cast<int>(itx);
    const unsigned b = itx / static_cast<unsigned>(a.pad_L);
    const int p = static_cast<int>(itx - b * static_cast<unsigned>(a.pad_L));
    const int c0 = a.pad_cu[b];
    return p < a.pad_cu[b + 1] - c0 ? c0 + p : -1;
  };
  auto load_row = [&](int src, uint4* r) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<size_t>(src >= 0 ? src : 0) * H);
#pragma unroll
    for (int i = 0; i < VPL; ++i) r[i] = src >= 0 ? xr[i * 32 + lane] : make_uint4(0u, 0u, 0u, 0u);
  };
  constexpr int NP = VPL * EPV / 2;   // fp32 pairs per lane
  unsigned it = blockIdx.x * kWarps + warp_id();
  int src = src_of(it);
  uint4 nx[VPL];
  load_row(src, nx);
  for (; it < n_iter; it += stride) {
    uint64_t v[NP];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      float f[EPV];
      unpack16<TIn>(nx[i], f);
#pragma unroll
      for (int h = 0; h < EPV / 2; ++h) v[i * (EPV / 2) + h] = f2_pack(f[2 * h], f[2 * h + 1]);
    }
    const int src_next = src_of(it + stride);
    load_row(src_next, nx);
    TOut* yr = y + static_cast<size_t>(it) * H;
    if (src < 0) {   // pad slot of the padded output
      constexpr int OV = sizeof(TOut) * EPV / 16 > 0 ? sizeof(TOut) * EPV / 16 : 1;   // 16-byte stores per vector
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        if constexpr (sizeof(TOut) * EPV >= 16) {
#pragma unroll
          for (int u = 0; u < OV; ++u)
            reinterpret_cast<uint4*>(yr + (i * 32 + lane) * EPV)[u] = make_uint4(0u, 0u, 0u, 0u);
        } else {
          *reinterpret_cast<uint2*>(yr + (i * 32 + lane) * EPV) = make_uint2(0u, 0u);
        }
      }
      src = src_next;
      continue;
    }
    uint64_t s2a = v[0], s2b = v[1];
#pragma unroll
    for (int k = 2; k < NP; k += 2) {
      s2a = f2_add(s2a, v[k]);
      s2b = f2_add(s2b, v[k + 1]);
    }
    s2a = f2_add(s2a, s2b);
    float sum = f2_lo(s2a) + f2_hi(s2a);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float mean = sum * (1.0f / H);
    const uint64_t nm = f2_pack(-mean, -mean);
    uint64_t q2a = 0ull, q2b = 0ull;
#pragma unroll
    for (int k = 0; k < NP; k += 2) {
      v[k] = f2_add(v[k], nm);
      v[k + 1] = f2_add(v[k + 1], nm);
      q2a = f2_fma(v[k], v[k], q2a);
      q2b = f2_fma(v[k + 1], v[k + 1], q2b);
    }
    q2a = f2_add(q2a, q2b);
    float ss = f2_lo(q2a) + f2_hi(q2a);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float rstd = rsqrtf(ss * (1.0f / H) + a.eps);
    const uint64_t r2 = f2_pack(rstd, rstd);
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      float o[EPV];
#pragma unroll
      for (int j4 = 0; j4 < E4; ++j4) {
        const float4 g4 = s_g[(i * E4 + j4) * 32 + lane];
        const float4 b4 = s_b[(i * E4 + j4) * 32 + lane];
        const int k0 = i * (EPV / 2) + 2 * j4;
        const uint64_t o0 = f2_fma(v[k0], f2_mul(f2_pack(g4.x, g4.y), r2), f2_pack(b4.x, b4.y));
        const uint64_t o1 = f2_fma(v[k0 + 1], f2_mul(f2_pack(g4.z, g4.w), r2), f2_pack(b4.z, b4.w));
        o[4 * j4 + 0] = f2_lo(o0); o[4 * j4 + 1] = f2_hi(o0);
        o[4 * j4 + 2] = f2_lo(o1); o[4 * j4 + 3] = f2_hi(o1);
      }
      const int col0 = (i * 32 + lane) * EPV;
      store_vec<TOut, EPV>(yr + col0, o);
      if (a.y32) {
        float* yf = a.y32 + static_cast<size_t>(it) * H + col0;
#pragma unroll
        for (int j = 0; j < EPV; j += 4)
          *reinterpret_cast<float4*>(yf + j) = make_float4(o[j], o[j + 1], o[j + 2], o[j + 3]);
      }
      if (a.y16) store_vec<__half, EPV>(a.y16 + static_cast<size_t>(it) * H + col0, o);
    }
    src = src_next;
  }
}

template <typename TIn, typename TOut, int VPL>
cudaError_t ln_stream_launch(const LnArgs& a, cudaStream_t stream) {
  constexpr int kWarps = kLnsThreads / 32;
  const long long n_iter = a.pad_cu ? static_cast<long long>(a.pad_B) * a.pad_L : a.M_max;
  long long blocks = (n_iter + kWarps - 1) / kWarps;
  static int per_sm = 0;   // one wave of resident blocks: the row loop is grid-strided
  if (per_sm == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, ln_stream_kernel<TIn, TOut, VPL>, kLnsThreads, 0) !=
            cudaSuccess || n < 1)
      n = 2;
    per_sm = n;
  }
  const long long cap = static_cast<long long>(num_sms()) * per_sm;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_pdl(ln_stream_kernel<TIn, TOut, VPL>, dim3(static_cast<unsigned>(blocks)), dim3(kLnsThreads), 0,
                    stream, a);
}

// vectors per lane of a supported row width (H = 32 VPL EPV), else 0
int ln_stream_vpl(int H, rpp_dtype in) {
  const int epv = in == RPP_F32 ? 4 : 8;
  if (H % (32 * epv)) return 0;
  const int v = H / (32 * epv);
  return (v == 1 || v == 2 || v == 3 || v == 4 || v == 6 || v == 8) ? v : 0;
}

template <typename TIn, typename TOut>
cudaError_t ln_stream_dispatch(const LnArgs& a, cudaStream_t stream) {
  switch (ln_stream_vpl(a.H, a.in_dtype)) {
    case 1: return ln_stream_launch<TIn, TOut, 1>(a, stream);
    case 2: return ln_stream_launch<TIn, TOut, 2>(a, stream);
    case 3: return ln_stream_launch<TIn, TOut, 3>(a, stream);
    case 4: return ln_stream_launch<TIn, TOut, 4>(a, stream);
    case 6: return ln_stream_launch<TIn, TOut, 6>(a, stream);
    case 8: return ln_stream_launch<TIn, TOut, 8>(a, stream);
    default: return cudaErrorNotSupported;
  }
}

bool ln_stream_applies(const LnArgs& a) {
  return a.out_dtype != RPP_F32 && a.n_in == 1 && !a.residual && !a.add_bias && !a.q_codes && !a.amax &&
         ln_stream_vpl(a.H, a.in_dtype) > 0;
}

// max |x| of each part of [M, W] rows cut into column parts of width part_w (at most
// three: the Q, K and V parts of the QKV projection), accumulated into amax[part]
template <typename T>
__global__ void amax_parts_kernel(const T* __restrict__ x, int M_max, const int32_t* rows, int W, int part_w,
                                  float* amax, int32_t* err) {
  pdl_wait();
  pdl_trigger();
  if (device_error_set(err)) return;
  int M = rows ? *rows : M_max;
  if (M > M_max || M < 0) M = 0;
  const long long n8 = static_cast<long long>(M) * W / 8;
  const int vpr = W / 8;   // vectors per row
  float m0 = 0.f, m1 = 0.f, m2 = 0.f;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    float f[8];
    if constexpr (sizeof(T) == 2) {
      unpack16<T>(reinterpret_cast<const uint4*>(x)[i], f);
    } else {
      unpack16<T>(reinterpret_cast<const uint4*>(x)[2 * i], f);
      unpack16<T>(reinterpret_cast<const uint4*>(x)[2 * i + 1], f + 4);
    }
    float m = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(f[j]));
    const int part = static_cast<int>(i % vpr) * 8 / part_w;   // part_w % 8 == 0: a vector lies in one part
    if (part == 0) m0 = fmaxf(m0, m);
    else if (part == 1) m1 = fmaxf(m1, m);
    else m2 = fmaxf(m2, m);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
    m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
    m2 = fmaxf(m2, __shfl_xor_sync(0xffffffffu, m2, o));
  }
  if (lane_id() == 0) {
    const int np = W / part_w;
    atomic_max_nonneg(amax, m0);
    if (np > 1) atomic_max_nonneg(amax + 1, m1);
    if (np > 2) atomic_max_nonneg(amax + 2, m2);
  }
}

template <typename T, typename TOut, int G, int VPL, int NS>
cudaError_t ln_launch(const LnArgs& a, cudaStream_t stream) {
  const int threads = 128;
  const int rows_per_block = (threads / 32) * (32 / G);
  const long long n_iter = a.pad_cu ? static_cast<long long>(a.pad_B) * a.pad_L : a.M_max;
  long long blocks = (n_iter + rows_per_block - 1) / rows_per_block;
  // the row loop is grid-strided: one wave of resident blocks covers any row count
  // without a partial last wave
  static int per_sm = 0;
  if (per_sm == 0) {
    int n = 0;
    const size_t smem_row = 3 * static_cast<size_t>(G) * VPL * Vec<T>::N * sizeof(float);   // = smem below
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, layernorm_kernel<T, TOut, G, VPL, NS>, threads, smem_row) !=
            cudaSuccess || n < 1)
      n = 4;
    per_sm = n;
  }
  const long long cap = static_cast<long long>(num_sms()) * per_sm;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const size_t smem = 3 * static_cast<size_t>(a.H) * sizeof(float);
  return launch_pdl(layernorm_kernel<T, TOut, G, VPL, NS>, dim3(static_cast<unsigned>(blocks)), dim3(threads), smem,
                    stream, a);
}

template <typename T, typename TOut>
cudaError_t ln_dispatch(const LnArgs& a, cudaStream_t stream) {
  const int V = a.H / Vec<T>::N;   // 16-byte vectors per row
  // split-K slices (fp32 input only) take the variant that loads all of them at once,
  // where the registers allow (up to 8 vectors per lane)
#define RPP_LN_CASE(G_, VPL_)                                                              \
  if (V == (G_) * (VPL_)) {                                                                \
    if constexpr (std::is_same<T, float>::value && (VPL_) <= 8) {                          \
      if (a.n_in > 2) return ln_launch<T, TOut, G_, VPL_, kMaxSlices>(a, stream);         \
      if (a.n_in == 2) return ln_launch<T, TOut, G_, VPL_, 2>(a, stream);                 \
    }                                                                                      \
    return ln_launch<T, TOut, G_, VPL_, 1>(a, stream);                                     \
  }
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

cudaError_t launch_layernorm(const LnArgs& args, cudaStream_t stream) {
  LnArgs a = args;
  if (a.n_in > 1 && a.in_dtype != RPP_F32) return cudaErrorNotSupported;
  if (a.n_in < 1) return cudaErrorInvalidValue;
  a.res_kind = !a.residual ? 0 : (a.res_dtype == RPP_F32 ? 1 : (a.res_dtype == RPP_F16 ? 2 : 3));
  if (a.residual && a.in_dtype != RPP_F32) return cudaErrorNotSupported;   // residual adds use 4-element groups
  if (a.pad_cu && (a.pad_B <= 0 || a.pad_L <= 0)) return cudaErrorInvalidValue;
  if (a.pad_cu && static_cast<long long>(a.pad_B) * a.pad_L > 0x7fffffffLL) return cudaErrorNotSupported;
  using BF = __nv_bfloat16;
  if (ln_stream_applies(a)) {
    if (a.in_dtype == RPP_F16 && a.out_dtype == RPP_F16) return ln_stream_dispatch<__half, __half>(a, stream);
    if (a.in_dtype == RPP_F16 && a.out_dtype == RPP_BF16) return ln_stream_dispatch<__half, BF>(a, stream);
    if (a.in_dtype == RPP_BF16 && a.out_dtype == RPP_BF16) return ln_stream_dispatch<BF, BF>(a, stream);
    if (a.in_dtype == RPP_F32 && a.out_dtype == RPP_BF16) return ln_stream_dispatch<float, BF>(a, stream);
    if (a.in_dtype == RPP_F32 && a.out_dtype == RPP_F16) return ln_stream_dispatch<float, __half>(a, stream);
  }
  if (a.in_dtype == a.out_dtype) {
    switch (a.in_dtype) {
      case RPP_F32: return ln_dispatch<float, float>(a, stream);
      case RPP_F16: return ln_dispatch<__half, __half>(a, stream);
      case RPP_BF16: return ln_dispatch<BF, BF>(a, stream);
      default: return cudaErrorNotSupported;
    }
  }
  if (a.in_dtype == RPP_F16 && a.out_dtype == RPP_BF16) return ln_dispatch<__half, BF>(a, stream);
  if (a.in_dtype == RPP_F32 && a.out_dtype == RPP_F16) return ln_dispatch<float, __half>(a, stream);
  if (a.in_dtype == RPP_F32 && a.out_dtype == RPP_BF16) return ln_dispatch<float, BF>(a, stream);
  return cudaErrorNotSupported;
}

cudaError_t launch_quantize(const void* x, const float* scale, int8_t* q, int M_max, const int32_t* rows, int H,
                            rpp_dtype dtype, int32_t* err, cudaStream_t stream) {
  const long long n8 = static_cast<long long>(M_max) * H / 8;
  long long blocks = (n8 + 255) / 256;
  const long long cap = static_cast<long long>(num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const dim3 grid(static_cast<unsigned>(blocks));
  switch (dtype) {
    case RPP_F32:
      return launch_pdl(quantize_kernel<float>, grid, dim3(256), 0, stream, static_cast<const float*>(x), scale, q, M_max, rows, H, err);
    case RPP_F16:
      return launch_pdl(quantize_kernel<__half>, grid, dim3(256), 0, stream, static_cast<const __half*>(x), scale, q, M_max, rows, H, err);
    case RPP_BF16:
      return launch_pdl(quantize_kernel<__nv_bfloat16>, grid, dim3(256), 0, stream, static_cast<const __nv_bfloat16*>(x),
                        scale, q, M_max, rows, H, err);
    default: return cudaErrorNotSupported;
  }
}

cudaError_t launch_amax(const void* x, int M_max, const int32_t* rows, int H, rpp_dtype dtype, float* amax,
                        int32_t* err, cudaStream_t stream) {
  const long long n8 = static_cast<long long>(M_max) * H / 8;
  long long blocks = (n8 + 255) / 256;
  const long long cap = static_cast<long long>(num_sms()) * 4;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const dim3 grid(static_cast<unsigned>(blocks));
  switch (dtype) {
    case RPP_F32:
      return launch_pdl(amax_kernel<float>, grid, dim3(256), 0, stream, static_cast<const float*>(x), M_max, rows, H, amax, err);
    case RPP_F16:
      return launch_pdl(amax_kernel<__half>, grid, dim3(256), 0, stream, static_cast<const __half*>(x), M_max, rows, H, amax, err);
    case RPP_BF16:
      return launch_pdl(amax_kernel<__nv_bfloat16>, grid, dim3(256), 0, stream, static_cast<const __nv_bfloat16*>(x),
                        M_max, rows, H, amax, err);
    default: return cudaErrorNotSupported;
  }
}

cudaError_t launch_amax_parts(const void* x, int M_max, const int32_t* rows, int W, int part_w, rpp_dtype dtype,
                              float* amax, int32_t* err, cudaStream_t stream) {
  if (part_w <= 0 || part_w % 8 || W % part_w || W / part_w > 3) return cudaErrorInvalidValue;
  const long long n8 = static_cast<long long>(M_max) * W / 8;
  long long blocks = (n8 + 255) / 256;
  const long long cap = static_cast<long long>(num_sms()) * 4;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const dim3 grid(static_cast<unsigned>(blocks));
  switch (dtype) {
    case RPP_F16:
      return launch_pdl(amax_parts_kernel<__half>, grid, dim3(256), 0, stream, static_cast<const __half*>(x), M_max,
                        rows, W, part_w, amax, err);
    case RPP_BF16:
      return launch_pdl(amax_parts_kernel<__nv_bfloat16>, grid, dim3(256), 0, stream,
                        static_cast<const __nv_bfloat16*>(x), M_max, rows, W, part_w, amax, err);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace rpp
