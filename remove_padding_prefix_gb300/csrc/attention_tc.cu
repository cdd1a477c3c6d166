// Variable-length fused multi-head attention on the 5th-generation tensor cores
// (head size 64, fp16 or bf16).
//
// The Swin talk (§3) runs fMHA as batch GEMM + softmax + batch GEMM with the head
// transposes folded into its I/O, and the Kuaishou article (Fig. 10) runs attention
// on the padding-free packed batch, one sequence at a time.  Here one CTA takes 128
// queries of one head of one sequence and walks that sequence's keys in 128-key tiles:
//
//   warp 0      TMA producer: the Q tile once, then K and V tiles (128 rows x 64
//               columns, 128-byte swizzle) straight from the token-major [T, 3H] QKV
//               rows (the head transpose is the load's column offset).  K_{j+1} loads
//               as soon as S_j is computed and V_{j+1} as soon as P_j V_j is, so each
//               load overlaps a softmax; one buffer each keeps the CTA at 80 KB of
//               shared memory (two CTAs per SM).
//   warp 1      allocates tensor memory and issues, from one thread, S = Q K^T
//               (M = 128, N = 128, K = 64) into tensor memory, and after the softmax
//               has written P, O_j = P V_j (M = 128, N = 64, K = 128; V is read
//               N-major from its token-major tile).
//   warps 2..9  softmax, two threads per query row (64 keys and 32 output columns
//               each; the pair exchanges row maxima through shared memory): S from
//               tensor memory (tcgen05.ld), scale and key mask, running max and sum
//               (the online softmax), P = 2^(s - max) rounded to the input type into
//               shared memory (swizzled K-major, the A operand of the PV MMA).  O
//               accumulates in tensor memory over the key tiles; the reference maximum
//               is moved (and O and the sum rescaled) only when a tile's maximum exceeds
//               it by more than 8 in log2 units, so P stays below 2^8.  At the end O / sum
//               is written to the packed output row.
//
// Keys past the sequence's end are excluded (their scores become -inf before the max,
// so P is exactly 0 there); V rows past the end of a partial last tile are zeroed in
// shared memory before the PV MMA, so whatever lies beyond the sequence in the QKV
// buffer (another sequence, or unwritten capacity) never reaches the output.  Query
// rows past the end are computed and not stored.  Every mbarrier wait is bounded.
#include "kernels.h"

namespace rpp {

namespace {

constexpr int kQT = 128;                  // queries per CTA
constexpr int kKT = 128;                  // keys per tile
constexpr int kDh = 64;                   // head size
constexpr int kAttnThreads = 320;         // warp 0 TMA, warp 1 MMA, warps 2..9 softmax
constexpr uint32_t kTileBytes = 128 * kDh * 2;   // one 128 x 64 tile of Q, K or V
constexpr uint32_t kPBytes = kQT * kKT * 2;      // P: two 64-key column blocks of 16 KB
constexpr uint32_t kTmemCols = 256;       // S: columns [0, 128); O_j: [128, 192)
constexpr size_t kRedBytes = 3 * 256 * sizeof(float);   // row max (two tile parities) and row sum exchange
constexpr size_t kAttnSmem = 1024 + kTileBytes * 3 + kPBytes + kRedBytes + 256;

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

template <typename T> struct AbFmtOf;
template <> struct AbFmtOf<__half> { static constexpr int v = 0; };
template <> struct AbFmtOf<__nv_bfloat16> { static constexpr int v = 1; };

template <typename T>
__device__ __forceinline__ uint32_t pack2(float a, float b);
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <typename T>
__global__ void __launch_bounds__(kAttnThreads, 2) attention_tc_kernel(const __grid_constant__ CUtensorMap tm,
                                                                    const int32_t* __restrict__ cu, int T_max,
                                                                    int max_len, int nh, T* __restrict__ out,
                                                                    float scale_log2, int32_t* err) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.z;
  const int h = blockIdx.y;
  const int q0 = blockIdx.x * kQT;
  const int c0 = cu[b];
  const int c1 = cu[b + 1];
  // other CTAs of this launch may set the error word at any time: one thread reads it
  // and the whole CTA follows that one reading (all threads return here, or none)
  __shared__ int s_quit;
  if (threadIdx.x == 0) s_quit = device_error_set(err) ? 1 : 0;
  __syncthreads();
  if (s_quit) return;
  const int len = c1 - c0;
  if (c0 < 0 || len < 0 || c1 > T_max || len > max_len) {
    if (threadIdx.x == 0) set_device_error(err, len > max_len ? RPP_DERR_LENGTH : RPP_DERR_ROWS);
    return;
  }
  if (q0 >= len) return;
  const int nkb = (len + kKT - 1) / kKT;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + kTileBytes;
  uint8_t* sV = sK + kTileBytes;
  uint8_t* sP = sV + kTileBytes;
  float* s_red = reinterpret_cast<float*>(sP + kPBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sP + kPBytes + kRedBytes);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = bars + 2;
  uint64_t* v_full = bars + 3;
  uint64_t* v_empty = bars + 4;
  uint64_t* s_full = bars + 5;
  uint64_t* p_full = bars + 6;
  uint64_t* o_full = bars + 7;
  uint64_t* drain = bars + 8;
  uint64_t* ex_tile = bars + 9;     // [4] per lane quadrant: the row-max exchange of a tile
  uint64_t* ex_end = bars + 13;     // [4] per lane quadrant: the row-sum exchange at the end
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 17);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id();
  const int lane = lane_id();
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(k_full, 1);
    mbar_init(k_empty, 1);
    mbar_init(v_full, 1);
    mbar_init(v_empty, 1);
    mbar_init(s_full, 1);
    mbar_init(p_full, 256);
    mbar_init(o_full, 1);
    mbar_init(drain, 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(&ex_tile[i], 64);
      mbar_init(&ex_end[i], 64);
    }
    *abort_flag = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&tm);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int H = nh * kDh;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      bool ok = true;
      mbar_arrive_expect_tx(q_full, kTileBytes);
      tma_load_2d(sQ, &tm, q_full, h * kDh, c0 + q0);
      int jk = 0, jv = 0;   // K and V tiles issued
      for (; jv < nkb && ok; ++jv) {
        // K_j once S_{j-1} has read K_{j-1}; V_j once P_{j-1} V_{j-1} has read V_{j-1}
        if (!mbar_wait_bounded(k_empty, (jk & 1) ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(k_full, kTileBytes);
        tma_load_2d(sK, &tm, k_full, H + h * kDh, c0 + jk * kKT);
        ++jk;
        if (!mbar_wait_bounded(v_empty, (jv & 1) ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(v_full, kTileBytes);
        tma_load_2d(sV, &tm, v_full, 2 * H + h * kDh, c0 + jv * kKT);
      }
      if (!ok) {
        set_device_error(err, RPP_DERR_TIMEOUT);
        *abort_flag = 1;
      }
      // copies still in flight land before the CTA can exit
      mbar_wait_bounded(q_full, 0, nullptr);
      if (jk > 0) mbar_wait_bounded(k_full, (jk - 1) & 1, nullptr);
      if (jv > 0) mbar_wait_bounded(v_full, (jv - 1) & 1, nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr int fmt = AbFmtOf<T>::v;
      constexpr uint32_t IDESC_S = idesc_f16(fmt, kQT, kKT);
      constexpr uint32_t IDESC_O = idesc_f16(fmt, kQT, kDh) | (1u << 16);   // B (= V) N-major
      const uint32_t d_s = tmem_base;
      const uint32_t d_o = tmem_base + kKT;
      bool ok = mbar_wait_bounded(q_full, 0, abort_flag) && mbar_wait_bounded(k_full, 0, abort_flag);
      const uint64_t qdesc = sw128_kmajor_desc(smem_u32(sQ));
      const uint64_t kdesc = sw128_kmajor_desc(smem_u32(sK));
      auto issue_s = [&]() {
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < kDh / 16; ++k) tc_mma_f16(d_s, qdesc + 2u * k, kdesc + 2u * k, IDESC_S, k ? 1u : 0u);
        tc_commit(s_full);
        tc_commit(k_empty);
      };
      if (ok) issue_s();
      for (int j = 0; j < nkb && ok; ++j) {
        ok = mbar_wait_bounded(p_full, j & 1, abort_flag) && mbar_wait_bounded(v_full, j & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint64_t vdesc = sw128_kmajor_desc(smem_u32(sV));
#pragma unroll
        for (int k = 0; k < kKT / 16; ++k) {
          // P: K-major, 64-key column blocks of 16 KB, +32 bytes per 16 keys inside one;
          // V: N-major, 16 keys = two 8-row swizzle atoms = +2048 bytes
          const uint64_t pdesc = sw128_kmajor_desc(smem_u32(sP + (k >> 2) * (kPBytes / 2))) + 2u * (k & 3);
          tc_mma_f16(d_o, pdesc, vdesc + 128u * k, IDESC_O, (j | k) ? 1u : 0u);   // O accumulates over tiles
        }
        tc_commit(o_full);
        tc_commit(v_empty);
        if (j + 1 < nkb) {
          if (!mbar_wait_bounded(k_full, (j + 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          issue_s();
        }
      }
      if (!ok) {
        set_device_error(err, RPP_DERR_TIMEOUT);
        *abort_flag = 1;
      }
      tc_commit(drain);
      mbar_wait_bounded(drain, 0, nullptr);
    }
  } else {
    // ------------------------------------------------------------ softmax
    // two warps per tensor-memory lane quadrant: thread (row r, half hf) owns S columns
    // [64 hf, 64 hf + 64) and output columns [32 hf, 32 hf + 32) of query row r
    const int q = warp & 3;
    const int hf = (warp - 2) >> 2;
    const int r = q * 32 + lane;                  // query row of the tile
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    float m = neg_inf(), l = 0.f;                  // reference maximum (log2 units) and row sum
    bool ok = true;
    for (int j = 0; j < nkb; ++j) {
      const int nvalid = min(kKT, len - j * kKT);   // keys of this tile inside the sequence
      // S_j complete; the MMAs before it (P_{j-1} V_{j-1}) too, so P's buffer is free
      // and O holds every earlier tile
      int w = mbar_wait_bounded(s_full, j & 1, abort_flag) ? 1 : 0;
      if (!__all_sync(0xffffffffu, w)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t v[64];
      tmem_ld_32x32b_x32(t_lane + hf * 64, v);
      tmem_ld_32x32b_x32(t_lane + hf * 64 + 32, v + 32);
      tmem_ld_wait();
      const bool full = nvalid == kKT;
      if (!full) {   // keys past the sequence: -inf
#pragma unroll
        for (int e = 0; e < 64; ++e)
          if (hf * 64 + e >= nvalid) v[e] = 0xff800000u;
      }
      float mx;
      {   // eight independent partial maxima, then a tree: no 64-long dependency chain
        float pm[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) pm[t] = __uint_as_float(v[t]);
#pragma unroll
        for (int e = 8; e < 64; ++e) pm[e & 7] = fmaxf(pm[e & 7], __uint_as_float(v[e]));
        mx = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])), fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
      }
      // exchange with the other half of the row (bounded wait on the pair's barrier)
      s_red[(j & 1) * 256 + hf * 128 + r] = mx;
      mbar_arrive(&ex_tile[q]);
      w = mbar_wait_bounded(&ex_tile[q], j & 1, abort_flag) ? 1 : 0;
      if (!__all_sync(0xffffffffu, w)) {
        ok = false;
        break;
      }
      mx = fmaxf(mx, s_red[(j & 1) * 256 + (hf ^ 1) * 128 + r]) * scale_log2;   // the row's tile maximum
      // Lazy rescaling: the reference maximum moves only when the tile's exceeds it by
      // more than 8 (P stays below 2^8); then O (in tensor memory) and the row sum are
      // rescaled.  Both threads of a row see the same values and decide alike.  The
      // decision is per row, but the tensor-memory loads and stores are warp-collective:
      // when any row of the warp rescales, the whole warp runs them (scale 1 for rows
      // that keep their maximum -- exact), so no lane skips a collective instruction
      // whatever the rows hold (query rows past the sequence end hold arbitrary data).
      if (j == 0) {
        m = mx;
      } else {
        const bool move = mx > m + 8.0f;
        if (__any_sync(0xffffffffu, move)) {
          const float alpha = move ? ex2_approx(m - mx) : 1.0f;
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            uint32_t ov[16];
            tmem_ld_32x32b_x16(t_lane + kKT + hf * 32 + c * 16, ov);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st_32x32b_x16(t_lane + kKT + hf * 32 + c * 16, ov);
            tmem_st_wait_tied16(ov);   // the store reads ov until it completes
          }
          tmem_st_wait();
          if (move) {
            l *= alpha;
            m = mx;
          }
        }
      }
      // P = 2^(s - m) for this half's 64 keys (one 64-key column block of P)
      float ps[4] = {0.f, 0.f, 0.f, 0.f};   // independent partial sums
      uint8_t* prow = sP + hf * (kPBytes / 2) + r * 128;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        uint32_t pk[4];
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2) {
          const int e = 8 * u + 2 * e2;
          const float p0 = ex2_approx(fmaf(__uint_as_float(v[e]), scale_log2, -m));
          const float p1 = ex2_approx(fmaf(__uint_as_float(v[e + 1]), scale_log2, -m));
          ps[e2] += p0 + p1;
          pk[e2] = pack2<T>(p0, p1);
        }
        // 16-byte chunk u of the row sits at chunk u ^ (r & 7) (the 128-byte swizzle)
        *reinterpret_cast<uint4*>(prow + ((u ^ (r & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      l += (ps[0] + ps[1]) + (ps[2] + ps[3]);      // this half's share of the row sum
      if (!full) {
        // a partial last tile: zero the V rows past the sequence (0 * NaN would be NaN)
        w = mbar_wait_bounded(v_full, j & 1, abort_flag) ? 1 : 0;
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        if (r >= nvalid) {
          uint4* vrow = reinterpret_cast<uint4*>(sV + r * 128) + hf * 4;
#pragma unroll
          for (int u = 0; u < 4; ++u) vrow[u] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();   // P (and the zeroed V rows) visible to the tensor core
      tc_fence_before();
      mbar_arrive(p_full);
    }
    // the pair's two halves of the row sum
    if (ok) {
      s_red[512 + hf * 128 + r] = l;
      mbar_arrive(&ex_end[q]);
      const int w = mbar_wait_bounded(&ex_end[q], 0, abort_flag) ? 1 : 0;
      ok = __all_sync(0xffffffffu, w) != 0;
      l += s_red[512 + (hf ^ 1) * 128 + r];
    }
    if (ok) {
      const int w = mbar_wait_bounded(o_full, (nkb - 1) & 1, abort_flag) ? 1 : 0;
      ok = __all_sync(0xffffffffu, w) != 0;
    }
    if (!ok) {
      if (lane == 0) {
        set_device_error(err, RPP_DERR_TIMEOUT);
        *abort_flag = 1;
      }
    } else {
      tc_fence_after();
      uint32_t ov[32];
      tmem_ld_32x32b_x32(t_lane + kKT + hf * 32, ov);
      tmem_ld_wait();
      if (q0 + r < len) {
        const float inv = 1.0f / l;
        uint4* orow = reinterpret_cast<uint4*>(out + static_cast<long long>(c0 + q0 + r) * H + h * kDh + hf * 32);
#pragma unroll
        for (int u = 0; u < kDh / 16; ++u) {
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(ov[8 * u + e]) * inv;
          orow[u] = make_uint4(pack2<T>(f[0], f[1]), pack2<T>(f[2], f[3]), pack2<T>(f[4], f[5]), pack2<T>(f[6], f[7]));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_attention_tc(const void* qkv, const int32_t* cu, int B, int T_max, int max_len, int nh,
                                rpp_dtype dtype, void* out, int32_t* err, cudaStream_t stream) {
  if (B <= 0 || max_len <= 0 || T_max <= 0) return cudaSuccess;
  if (dtype != RPP_F16 && dtype != RPP_BF16) return cudaErrorNotSupported;
  const int H = nh * kDh;
  CUtensorMap tm;
  const CUtensorMapDataType dt = dtype == RPP_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  if (!make_tmap_2d(&tm, qkv, dt, 2, T_max, 3 * H, 128, kDh, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(kDh));
  dim3 grid((max_len + kQT - 1) / kQT, nh, B);
  if (dtype == RPP_F16) {
    static bool attr = false;
    if (!attr) {
      cudaError_t e = cudaFuncSetAttribute(attention_tc_kernel<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(kAttnSmem));
      if (e != cudaSuccess) return e;
      attr = true;
    }
    return launch_pdl(attention_tc_kernel<__half>, grid, dim3(kAttnThreads), kAttnSmem, stream, tm, cu, T_max,
                      max_len, nh, static_cast<__half*>(out), scale_log2, err);
  }
  static bool attr_bf = false;
  if (!attr_bf) {
    cudaError_t e = cudaFuncSetAttribute(attention_tc_kernel<__nv_bfloat16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kAttnSmem));
    if (e != cudaSuccess) return e;
    attr_bf = true;
  }
  return launch_pdl(attention_tc_kernel<__nv_bfloat16>, grid, dim3(kAttnThreads), kAttnSmem, stream, tm, cu, T_max,
                    max_len, nh, static_cast<__nv_bfloat16*>(out), scale_log2, err);
}

}  // namespace rpp
