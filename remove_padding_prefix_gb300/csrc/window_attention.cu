// Shifted-window attention with the cyclic shift, window partition, window reverse
// and unshift folded into the kernel's loads and stores, plus the relative-position
// bias lookup done once in preprocessing.
//
// NVIDIA Swin talk: §1 (window attention, cyclic window shift, relative position
// bias), §2 (window shift / partition / merge are pure index mappings; the training
// timeline spent 4.6 % in roll kernels alone), §3 (bias lookup moved to
// preprocessing; batch GEMM + softmax + batch GEMM in one fMHA kernel with the
// transposes in its I/O; the 49-token windows padded to a multiple of 8).
//
// One CTA (4 warps) processes one head of one window.  For window
// (image, wy, wx) token t = ty*w + tx sits at (y, x) = (wy*w + ty, wx*w + tx) in the
// shifted frame and reads raster row ((y + s) mod I, (x + s) mod I); the output row
// is written back to the same raster row, which performs reverse + unshift.  The
// 49 rows are padded to 64 inside shared memory only (padding rows stay zero); warp w
// owns query rows 16w..16w+15.  S = Q K^T and O = P V use mma.sync.m16n8k16 with fp32
// accumulation; scores get the bias and, for shifted blocks, exclusion of pairs from
// different regions of the shifted frame (per axis: c < I-w, c < I-s, else).
#include "kernels.h"

namespace rpp {

namespace {

constexpr int kWD = 32;     // head dim
constexpr int kWRows = 64;  // padded window rows

// 64-byte rows (32 x 16-bit): chunk c of row r lives at chunk c ^ ((r >> 1) & 3)
__device__ __forceinline__ uint32_t swz64(int r, int c) {
  return static_cast<uint32_t>(r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
}

__device__ __forceinline__ void ldsm_x4w(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4w_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

template <typename T>
__device__ __forceinline__ void mma_w(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  if constexpr (sizeof(T) == 2 && std::is_same<T, __half>::value) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

template <typename T>
__device__ __forceinline__ uint32_t pack2w(float lo, float hi) {
  if constexpr (std::is_same<T, __half>::value) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

__device__ __forceinline__ int region(int c, int I, int w, int s) { return c < I - w ? 0 : (c < I - s ? 1 : 2); }

// One CTA (4 warps) per head and a strided set of windows (persistent over windows):
// each thread builds, once, its 32 scores' bias (from the preprocessed fp32 table, in
// log2 units; -inf for padding keys) and, for shifted blocks, the region-mask bits of
// the four window kinds (interior, last window row, last window column, corner: only
// windows touching the wrap seam mix regions).  Per window the score epilogue is then
// one FMA and a select per element.  The next window's rows are gathered (cp.async)
// into the second of two shared-memory buffers while the current one is computed.
template <typename T>
__global__ void __launch_bounds__(128, 4) window_attention_kernel(const T* __restrict__ qkv,
                                                                  const float* __restrict__ bias,
                                                                  T* __restrict__ out, int I, int w, int s, int nh,
                                                                  long long n_win, float scale_log2, int32_t* err) {
  pdl_wait();
  pdl_trigger();
  constexpr int TILE = kWRows * kWD * 2;   // bytes of one 64 x 32 tile
  __shared__ __align__(128) uint8_t sQKV[2][3 * TILE];
  __shared__ int sRow[2][kWRows];          // raster rows of the window's tokens
  const int C = nh * kWD;
  const int N = w * w;
  const int h = blockIdx.x;
  const int nWs = I / w;
  const int nW = nWs * nWs;
  const int tid = threadIdx.x;
  const int warp = warp_id();
  const int lane = lane_id();
  const int rA = warp * 16 + (lane >> 2);   // this thread's two query rows: rA, rA + 8
  const float log2e = 1.4426950408889634f;

  // ---- per-thread constants: bias of its 32 scores and the mask bits of the four kinds
  const float* bh = bias + static_cast<long long>(h) * N * N;
  float bv[8][4];
  uint32_t mask[4] = {0u, 0u, 0u, 0u};   // bit 4j+e: pair excluded in window kind k
#pragma unroll
  for (int j = 0; j < 8; ++j) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int t = rA + ((e >> 1) << 3);
      const int u = j * 8 + 2 * (lane & 3) + (e & 1);
      bv[j][e] = u >= N ? -INFINITY : (t < N ? __ldg(bh + t * N + u) * log2e : 0.f);
      if (s > 0 && t < N && u < N) {
        // region labels in the shifted frame for a window in the last row (ky = 1) or
        // column (kx = 1) of windows; elsewhere every token is in region 0
        const int tyy = I - w + t / w, txx = I - w + t % w;
        const int uyy = I - w + u / w, uxx = I - w + u % w;
#pragma unroll
        for (int k = 1; k < 4; ++k) {
          const bool ky = k & 2, kx = k & 1;
          const int lt = 3 * (ky ? region(tyy, I, w, s) : 0) + (kx ? region(txx, I, w, s) : 0);
          const int lu = 3 * (ky ? region(uyy, I, w, s) : 0) + (kx ? region(uxx, I, w, s) : 0);
          if (lt != lu) mask[k] |= 1u << (4 * j + e);
        }
      }
    }
  }
  if (device_error_set(err)) return;

  // padding rows (N..63) of Q, K and V are zero in both buffers (V's must be: P = 0
  // there, and 0 * junk could be NaN); the gathers never write them
  for (int i = tid; i < 2 * 3 * (kWRows - N) * 4; i += blockDim.x) {
    const int bt = i / ((kWRows - N) * 4);   // buffer * 3 + tile
    const int r = N + (i / 4) % (kWRows - N);
    *reinterpret_cast<uint4*>(sQKV[bt / 3] + (bt % 3) * TILE + swz64(r, i & 3)) = make_uint4(0u, 0u, 0u, 0u);
  }

  auto window_rows = [&](int buf, long long wid) {   // threads tid < N
    if (tid < N) {
      const int img = static_cast<int>(wid / nW);
      const int wr = static_cast<int>(wid - static_cast<long long>(img) * nW);
      const int wy = wr / nWs, wx = wr - (wr / nWs) * nWs;
      int ys = wy * w + tid / w + s, xs = wx * w + tid % w + s;
      if (ys >= I) ys -= I;
      if (xs >= I) xs -= I;
      sRow[buf][tid] = img * I * I + ys * I + xs;
    }
  };
  auto gather = [&](int buf) {   // this head's Q, K, V rows: N rows x 3 parts x 4 chunks
    for (int i = tid; i < N * 12; i += blockDim.x) {
      const int r = i / 12;
      const int cc = i - r * 12;
      const int part = cc >> 2;
      const T* src = qkv + static_cast<long long>(sRow[buf][r]) * (3 * C) + part * C + h * kWD + (cc & 3) * 8;
      cp_async_16(sQKV[buf] + part * TILE + swz64(r, cc & 3), src, true);
    }
    cp_async_commit();
  };

  long long wid = blockIdx.y;
  if (wid < n_win) {
    window_rows(0, wid);
    __syncthreads();
    gather(0);
  }
  for (int it = 0; wid < n_win; ++it, wid += gridDim.y) {
    const int buf = it & 1;
    const long long nxt = wid + gridDim.y;
    if (nxt < n_win) {   // prefetch the next window into the other buffer
      window_rows(buf ^ 1, nxt);
      __syncthreads();
      gather(buf ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const int wr = static_cast<int>(wid % nW);
    const int kind = s > 0 ? 2 * (wr / nWs == nWs - 1) + (wr % nWs == nWs - 1) : 0;
    const uint32_t mk = mask[0] | (kind == 1 ? mask[1] : 0u) | (kind == 2 ? mask[2] : 0u) | (kind == 3 ? mask[3] : 0u);

    const uint32_t sQa = smem_u32(sQKV[buf]);
    const uint32_t sKa = sQa + TILE;
    const uint32_t sVa = sQa + 2 * TILE;
    uint32_t qf[2][4];
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const int r = warp * 16 + (lane & 15);
      ldsm_x4w(sQa + swz64(r, kk * 2 + (lane >> 4)), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
    }
    float sc[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b0, b1, b2, b3;
        const int r = np * 16 + (lane & 7) + ((lane >> 4) << 3);
        ldsm_x4w(sKa + swz64(r, kk * 2 + ((lane >> 3) & 1)), b0, b1, b2, b3);
        mma_w<T>(sc[2 * np], qf[kk], b0, b1);
        mma_w<T>(sc[2 * np + 1], qf[kk], b2, b3);
      }
    }
    // scores -> log2 domain with bias and region mask; softmax over the N keys
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float v = fmaf(sc[j][e], scale_log2, bv[j][e]);
        sc[j][e] = (mk >> (4 * j + e)) & 1u ? -INFINITY : v;
      }
      mx[0] = fmaxf(mx[0], fmaxf(sc[j][0], sc[j][1]));
      mx[1] = fmaxf(mx[1], fmaxf(sc[j][2], sc[j][3]));
    }
    float sum[2] = {0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      sc[j][0] = ex2_approx(sc[j][0] - mx[0]);
      sc[j][1] = ex2_approx(sc[j][1] - mx[0]);
      sc[j][2] = ex2_approx(sc[j][2] - mx[1]);
      sc[j][3] = ex2_approx(sc[j][3] - mx[1]);
      sum[0] += sc[j][0] + sc[j][1];
      sum[1] += sc[j][2] + sc[j][3];
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      sum[i] += __shfl_xor_sync(0xffffffffu, sum[i], 1);
      sum[i] += __shfl_xor_sync(0xffffffffu, sum[i], 2);
      sum[i] = 1.f / sum[i];   // >= 1: the row's maximum contributes 2^0
    }
    float o[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      pa[0] = pack2w<T>(sc[2 * kk][0], sc[2 * kk][1]);
      pa[1] = pack2w<T>(sc[2 * kk][2], sc[2 * kk][3]);
      pa[2] = pack2w<T>(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
      pa[3] = pack2w<T>(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
      for (int dp = 0; dp < 2; ++dp) {
        uint32_t b0, b1, b2, b3;
        const int r = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        ldsm_x4w_t(sVa + swz64(r, dp * 2 + (lane >> 4)), b0, b1, b2, b3);
        mma_w<T>(o[2 * dp], pa, b0, b1);
        mma_w<T>(o[2 * dp + 1], pa, b2, b3);
      }
    }
    // normalised output over this warp's own Q rows, then scattered back to the raster rows
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t lo = pack2w<T>(o[j][0] * sum[0], o[j][1] * sum[0]);
      const uint32_t hi = pack2w<T>(o[j][2] * sum[1], o[j][3] * sum[1]);
      *reinterpret_cast<uint32_t*>(sQKV[buf] + swz64(rA, j) + (lane & 3) * 4) = lo;
      *reinterpret_cast<uint32_t*>(sQKV[buf] + swz64(rA + 8, j) + (lane & 3) * 4) = hi;
    }
    __syncthreads();
    for (int i = tid; i < N * 4; i += blockDim.x) {
      const int r = i >> 2;
      const int cc = i & 3;
      const uint4 v = *reinterpret_cast<const uint4*>(sQKV[buf] + swz64(r, cc));
      *reinterpret_cast<uint4*>(out + static_cast<long long>(sRow[buf][r]) * C + h * kWD + cc * 8) = v;
    }
    __syncthreads();   // this buffer (and its rows) may be refilled next
  }
}

__global__ void swin_bias_kernel(const void* table, int table_dtype, int w, int nh, float* bias) {
  const int N = w * w;
  const int total = nh * N * N;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const int h = i / (N * N);
    const int t = (i / N) % N;
    const int u = i % N;
    const int ty = t / w, tx = t % w, uy = u / w, ux = u % w;
    const int idx = (ty - uy + w - 1) * (2 * w - 1) + (tx - ux + w - 1);
    float v;
    if (table_dtype == RPP_F16) v = __half2float(static_cast<const __half*>(table)[idx * nh + h]);
    else if (table_dtype == RPP_BF16) v = __bfloat162float(static_cast<const __nv_bfloat16*>(table)[idx * nh + h]);
    else v = static_cast<const float*>(table)[idx * nh + h];
    bias[i] = v;
  }
}

template <typename T>
cudaError_t wa_launch(int B, const void* qkv, const float* bias, void* out, int nh, int I, int w, int s, int32_t* err,
                      cudaStream_t stream) {
  const long long windows = static_cast<long long>(B) * (I / w) * (I / w);
  if (windows > 0x7fffffffLL || nh > 1024) return cudaErrorNotSupported;
  if (windows == 0) return cudaSuccess;
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(kWD));
  // persistent over windows: exactly as many CTAs as fit on the GPU at once (a CTA
  // more would run alone after the others), split across the heads
  static int per_sm = 0;
  if (per_sm == 0) {
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, window_attention_kernel<T>, 128, 0);
    if (e != cudaSuccess || per_sm < 1) per_sm = 1;
  }
  long long per_head = static_cast<long long>(num_sms()) * per_sm / nh;
  if (per_head < 1) per_head = 1;
  if (per_head > windows) per_head = windows;
  if (per_head > 65535) per_head = 65535;
  dim3 grid(nh, static_cast<unsigned>(per_head));
  return launch_pdl(window_attention_kernel<T>, grid, dim3(128), 0, stream, static_cast<const T*>(qkv), bias,
                    static_cast<T*>(out), I, w, s, nh, windows, scale_log2, err);
}

}  // namespace

bool window_attention_supported(int C, int nh, int w, int I, int s) {
  return nh > 0 && C == nh * kWD && w > 0 && w * w <= kWRows && I % w == 0 && s >= 0 && s < w;
}

cudaError_t launch_window_attention(int B, const void* qkv, const float* bias, void* out, int C, int nh, int I, int w,
                                    int s, rpp_dtype dtype, int32_t* err, cudaStream_t stream) {
  if (!window_attention_supported(C, nh, w, I, s)) return cudaErrorNotSupported;
  if (B <= 0) return cudaSuccess;
  if (dtype == RPP_F16) return wa_launch<__half>(B, qkv, bias, out, nh, I, w, s, err, stream);
  if (dtype == RPP_BF16) return wa_launch<__nv_bfloat16>(B, qkv, bias, out, nh, I, w, s, err, stream);
  return cudaErrorNotSupported;
}

cudaError_t launch_swin_bias(const void* table, rpp_dtype table_dtype, int w, int nh, float* bias,
                             cudaStream_t stream) {
  const int total = nh * w * w * w * w;
  swin_bias_kernel<<<(total + 255) / 256, 256, 0, stream>>>(table, table_dtype, w, nh, bias);
  return cudaGetLastError();
}

}  // namespace rpp
