// GEMM + bias + residual + LayerNorm in one kernel (the encoder layer's proj -> LN1 and
// FC2 -> LN2, 16-bit activations, hidden size H = 256, 512, 768 or 1024):
//
//   y = LayerNorm(A[M, K] @ W[H, K]^T + bias + residual) * gamma + beta     (per row)
//
// The NVIDIA Swin talk (§3) splits the bias off the GEMM and fuses it, with the residual,
// into the LayerNorm that follows; the Kuaishou article (Fig. 6) fuses the elementwise
// work into the GEMMs.  Here the LayerNorm moves into the GEMM's epilogue, so the
// pre-LayerNorm sum never leaves the chip: it stays fp32 in tensor memory between the
// accumulation and the normalisation.
//
// Work split: a thread-block cluster of 2 x (H / 256) CTAs takes a 256-row block of the
// output.  The cluster's CTAs form H / 256 CTA pairs; pair p computes columns
// [256 p, 256 p + 256) with cta_group::2 MMAs (M = 256 across the pair, N = 256, K = 16):
// each CTA of a pair loads its 128 rows of A and half (128 rows) of the W tile into its
// own shared memory, every copy completes on the even CTA's barrier, the even CTA issues
// the MMAs and each CTA receives its 128 accumulator rows in its own tensor memory (fp32,
// double-buffered so the epilogue of one row block overlaps the MMAs of the next).
// Clusters are persistent over row blocks.
//
//   warp 0      TMA producer: per K block, the A tile and half of the W tile (128-byte
//               swizzle), in a 5-stage ring; then four more blocks that add the residual
//               inside the MMAs: the residual's 64-column tiles of this pair's columns
//               against 64-column slices of a 256 x 256 identity (exact: each product is
//               a residual value times 1 or 0).
//   warp 1      allocates tensor memory (collectively for the pair); in the even CTA,
//               issues the MMAs from one thread; commits reach both CTAs' barriers.
//   warps 2..9  epilogue, two per tensor-memory lane quadrant (32 rows each; 128 of the
//               pair's 256 columns each), three passes over tensor memory:
//                 A  acc + bias: the warp's mean over its 128 columns
//                 B  the warp's sum of squared deviations from that mean (M2)
//                 C  (v - mean) * rstd * gamma + beta -> 16-bit output rows (and an
//                    optional fp16 copy, the next residual of a bf16 layer), staged in
//                    shared memory and written with TMA bulk-tensor stores
//               Between B and C the CTAs that hold the same 128 rows (one per pair)
//               agree on the row statistics: every thread stores its (mean, M2) into
//               each of those CTAs' shared memory (st.shared::cluster), fences at cluster
//               scope, and one lane per warp arrives on each CTA's exchange mbarrier;
//               each thread then waits (bounded, acquire at cluster scope) and combines
//               the 2 x (H / 256) pairs of its row pairwise (Chan, Golub and LeVeque):
//               the mean of the means, M2 = sum of the M2s plus n times the squared
//               deviations of the means.  Biased variance, fp32.
//
// Rows past the device row count M are computed and never stored (a row block that
// reaches past M is stored row by row).  Every mbarrier wait is bounded; a wait that
// gives up records RPP_DERR_TIMEOUT, raises the CTA's abort flag and the CTA drains its
// copies and MMAs, frees its tensor memory and leaves.
#include <cstring>

#include "kernels.h"

namespace rpp {

namespace {

constexpr int kBM = 128;                         // rows per CTA (256 per pair)
constexpr int kBN = 256;                         // columns per pair
constexpr int kBK = 64;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr uint32_t kABytes = kBM * kBK * 2;      // 16 KB
constexpr uint32_t kBHalf = (kBN / 2) * kBK * 2;  // 16 KB: this CTA's half of the W tile
constexpr uint32_t kStageTx = 2 * (kABytes + kBHalf);   // both CTAs' copies, on the even CTA's barrier
constexpr int kStages = 5;
constexpr uint32_t kTmemCols = 512;              // two 256-column accumulators
constexpr int kMaxPairs = 4;                     // H <= 1024
constexpr uint32_t kStageBlock = 32 * 32 * 2;    // one warp's 32 x 32 output block

// shared memory (bytes from the 1024-aligned base)
constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffB = kStages * kABytes;
constexpr uint32_t kOffStg = kOffB + kStages * kBHalf;                 // [8 warps] staging blocks
constexpr uint32_t kOffPar = kOffStg + kEpiWarps * kStageBlock;        // bias, gamma, beta: 3 x 256 floats
constexpr uint32_t kOffX = kOffPar + 3 * kBN * 4;   // [2 parities][kMaxPairs][2 halves][128 rows] x (mean, M2)
constexpr uint32_t kOffBar = kOffX + 2 * kMaxPairs * 2 * kBM * 8;
constexpr uint32_t kOffMisc = kOffBar + (2 * kStages + 4 + 2) * 8;
constexpr size_t kSmem = 1024 + kOffMisc + 64;
static_assert(kSmem <= 232448, "shared memory per CTA");

struct Params {
  int M_max;
  const int32_t* rows;     // device row count, or null (M = M_max)
  int K;
  const float* bias;       // [H]
  const float* gamma;      // [H]
  const float* beta;       // [H]
  float eps;
  void* out;               // [M_max, H] of T
  __half* out_f16;         // optional fp16 copy of out
  int32_t* err;
};

template <typename T> struct Fmt;
template <> struct Fmt<__half> { static constexpr int v = 0; };
template <> struct Fmt<__nv_bfloat16> { static constexpr int v = 1; };

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// bounded wait, acquire at cluster scope (the waited-for writes come from other CTAs)
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((i & 31u) == 0) {
      if (abort_flag && *abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
  }
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// this thread's 32 values of its row into the warp's 32 x 32 staging block: rows of 64
// bytes, 16-byte chunk c of row r at chunk c ^ ((r >> 1) & 3) (the TMA 64-byte swizzle);
// eight consecutive lanes cover all 32 banks
template <typename TO>
__device__ __forceinline__ void stage_row16(uint8_t* stage, int r, const float* y) {
  const int x = (r >> 1) & 3;
#pragma unroll
  for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4*>(stage + r * 64 + ((c ^ x) << 4)) = pack16<TO>(y + 8 * c);
}

template <typename T, bool RES_F16>
__global__ void __launch_bounds__(kThreads, 1)
gemm_ln_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmR, const __grid_constant__ CUtensorMap tmI,
               const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmO16, Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem + kOffA;
  uint8_t* sB = smem + kOffB;
  uint8_t* sStg = smem + kOffStg;
  float* s_bias = reinterpret_cast<float*>(smem + kOffPar);
  float* s_gamma = s_bias + kBN;
  float* s_beta = s_gamma + kBN;
  float* xs = reinterpret_cast<float*>(smem + kOffX);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* xbar = tempty + 2;       // the row-statistics exchange
  uint64_t* drain = xbar + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  int* cl_info = reinterpret_cast<int*>(smem + kOffMisc + 8);   // [M, skip, tmem base, mismatch]

  const int warp = warp_id();
  const int lane = lane_id();
  const uint32_t ncta = cluster_nctarank();      // 2 x (H / 256)
  const uint32_t rank = cluster_ctarank();
  const uint32_t hrow = rank & 1u;               // which 128 rows of the pair's 256
  const uint32_t lead = rank & ~1u;              // the pair's even CTA: issues the MMAs
  const bool leader = hrow == 0;
  const uint16_t pair_mask = static_cast<uint16_t>(3u << lead);
  const uint32_t npairs = ncta >> 1;
  const int cid = blockIdx.x / ncta;             // cluster index
  const int ncl = gridDim.x / ncta;              // clusters in the grid
  const int H = kBN * static_cast<int>(npairs);
  const int n0 = kBN * static_cast<int>(rank >> 1);   // the pair's first column

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);    // only the even CTA's is used
      mbar_init(&empty[s], 1);   // released by the even CTA's multicast commit
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * kEpiWarps);   // both CTAs' epilogue warps, on the even CTA's
    }
    mbar_init(xbar, kEpiWarps * npairs);      // one arrival per epilogue warp of each same-row CTA
    mbar_init(drain, 1);
    *abort_flag = 0;
    cl_info[3] = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmR);
    tma_prefetch_desc(&tmI);
    tma_prefetch_desc(&tmO);
    if (p.out_f16) tma_prefetch_desc(&tmO16);
  }
  if (warp == 1) {
    tmem_alloc_cg<2>(tmem_slot, kTmemCols);
    tmem_relinquish_cg<2>();
  }
  // this pair's columns of bias, gamma and beta (parameters, never written by a kernel
  // that lets its dependents start early)
  for (int i = threadIdx.x; i < kBN; i += kThreads) {
    s_bias[i] = __ldg(p.bias + n0 + i);
    s_gamma[i] = __ldg(p.gamma + n0 + i);
    s_beta[i] = __ldg(p.beta + n0 + i);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  pdl_trigger();

  // One decision for the cluster (every CTA walks the same row blocks): rank 0 reads the
  // error word and the row count and publishes them into every CTA's shared memory.  The
  // first barrier also orders every CTA's barrier inits before remote use.  The odd CTA
  // of each pair checks that the collective allocation gave both the same columns.
  cluster_sync();
  if (rank == 0 && threadIdx.x == 0) {
    bool skip = device_error_set(p.err);
    int M = p.M_max;
    if (p.rows) {
      M = *p.rows;
      if (M > p.M_max || M < 0) {
        set_device_error(p.err, RPP_DERR_ROWS);
        skip = true;
      }
    }
    for (uint32_t r = 0; r < ncta; ++r) {
      st_shared_remote(cl_info, r, static_cast<uint32_t>(M));
      st_shared_remote(cl_info + 1, r, skip ? 1u : 0u);
    }
  }
  if (leader && threadIdx.x == 0) st_shared_remote(cl_info + 2, rank + 1, tmem_base);
  cluster_sync();
  if (!leader && threadIdx.x == 0 && static_cast<uint32_t>(cl_info[2]) != tmem_base) {
    set_device_error(p.err, RPP_DERR_TMEM);
    for (uint32_t r = 0; r < ncta; ++r) st_shared_remote(cl_info + 3, r, 1u);
  }
  cluster_sync();
  const int M = cl_info[0];
  const int num_m = (cl_info[1] || cl_info[3]) ? 0 : (M + 2 * kBM - 1) / (2 * kBM);   // 256-row blocks
  const int num_k = (p.K + kBK - 1) / kBK;
  // K blocks past num_k add the residual: its 256 x 256 tile times the 256 x 256 identity
  constexpr int kResBlocks = kBN / kBK;
  const int num_kt = num_k + kResBlocks;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (each CTA of a pair)
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      const uint32_t fb0 = cluster_addr(&full[0], lead);
      for (int u = cid; u < num_m && ok; u += ncl) {
        const int m0 = u * 2 * kBM + static_cast<int>(hrow) * kBM;
        for (int kb = 0; kb < num_kt; ++kb, ++it) {
          const uint32_t s = it % kStages;
          const uint32_t ph = (it / kStages) & 1u;
          if (!mbar_wait_bounded(&empty[s], ph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(&full[s], kStageTx);
          const uint32_t fb = fb0 + s * 8;
          if (kb < num_k) {
            tma_load_2d_pair(sA + s * kABytes, &tmA, fb, kb * kBK, m0);
            tma_load_2d_pair(sB + s * kBHalf, &tmB, fb, kb * kBK, n0 + static_cast<int>(hrow) * (kBN / 2));
          } else {   // residual columns n0 + 64 kr .. and the matching half of the identity slice
            const int kr = kb - num_k;
            tma_load_2d_pair(sA + s * kABytes, &tmR, fb, n0 + kr * kBK, m0);
            tma_load_2d_pair(sB + s * kBHalf, &tmI, fb, kr * kBK, static_cast<int>(hrow) * (kBN / 2));
          }
        }
      }
      if (!ok) {
        set_device_error(p.err, RPP_DERR_TIMEOUT);
        *abort_flag = 1;
      }
      // the even CTA waits (bounded) for the copies still in flight (its partner's too:
      // they complete on its barriers); the pair meets at the final cluster barrier
      if (leader) {
        const uint32_t first = it > kStages ? it - kStages : 0;
        for (uint32_t j = first; j < it; ++j) mbar_wait_bounded(&full[j % kStages], (j / kStages) & 1u, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (the even CTA's)
    if (lane == 0 && leader) {
      constexpr uint32_t IDESC = idesc_f16(Fmt<T>::v, 2 * kBM, kBN);
      constexpr uint32_t IDESC_R = idesc_f16(RES_F16 ? 0 : Fmt<T>::v, 2 * kBM, kBN);   // residual x identity
      uint32_t it = 0, acc_it = 0;
      bool ok = true;
      for (int u = cid; u < num_m && ok; u += ncl, ++acc_it) {
        const uint32_t a = acc_it & 1u;
        if (!mbar_wait_bounded(&tempty[a], ((acc_it >> 1) & 1u) ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < num_kt; ++kb, ++it) {
          const uint32_t s = it % kStages;
          if (!mbar_wait_bounded(&full[s], (it / kStages) & 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = sw128_kmajor_desc(smem_u32(sA + s * kABytes));
          const uint64_t bdesc = sw128_kmajor_desc(smem_u32(sB + s * kBHalf));
          const uint32_t idesc = kb < num_k ? IDESC : IDESC_R;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            tc_mma_f16_cg<2>(tmem_base + a * kBN, adesc + 2u * k, bdesc + 2u * k, idesc, (kb | k) ? 1u : 0u);
          tc_commit_cg<2>(&empty[s], pair_mask);   // the stage is free in both CTAs
        }
        if (ok) tc_commit_cg<2>(&tfull[a], pair_mask);
      }
      if (!ok) {
        set_device_error(p.err, RPP_DERR_TIMEOUT);
        *abort_flag = 1;
      }
      tc_commit_cg<2>(drain, static_cast<uint16_t>(1u << lead));
      mbar_wait_bounded(drain, 0, nullptr);
    }
  } else {
    // ------------------------------------------------------------ epilogue: bias, LayerNorm, store
    const int q = warp & 3;                 // lane quadrant: rows 32 q .. 32 q + 31 of this CTA's 128
    const int hh = (warp - 2) >> 2;         // columns [128 hh, 128 hh + 128) of the pair's 256
    const int r = q * 32 + lane;
    const int c0 = 128 * hh;
    const float inv_h = 1.0f / static_cast<float>(H);
    uint8_t* stage = sStg + (warp - 2) * kStageBlock;
    uint32_t acc_it = 0, nx = 0;
    bool ok = true, pending = false;
    // this warp's (mean, M2) of its 128 columns of row r -> every CTA holding the same rows
    // (one per pair); the row's mean and M2 over all H columns come back (Chan, Golub and
    // LeVeque's pairwise combination: equal counts n = 128, so mean = the average of the
    // partial means and M2 = sum M2_i + n sum (mean_i - mean)^2)
    auto exchange = [&](float mean_w, float m2_w, float& mean, float& m2) -> bool {
      const uint32_t par = nx & 1u;
      float* slot = xs + (((par * kMaxPairs + (rank >> 1)) * 2 + hh) * kBM + r) * 2;
      for (uint32_t j = 0; j < npairs; ++j) {
        const uint32_t ra = cluster_addr(slot, 2 * j + hrow);
        asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(ra), "f"(mean_w), "f"(m2_w) : "memory");
      }
      asm volatile("fence.acq_rel.cluster;" ::: "memory");   // this lane's remote stores before the arrival
      __syncwarp();
      if (lane == 0)
        for (uint32_t j = 0; j < npairs; ++j) mbar_arrive_cluster_relaxed(cluster_addr(xbar, 2 * j + hrow));
      const bool got = mbar_wait_cluster_bounded(xbar, par, abort_flag);
      ++nx;
      if (!__all_sync(0xffffffffu, got ? 1 : 0)) return false;
      const int n = 2 * static_cast<int>(npairs);
      const float2* pr = reinterpret_cast<const float2*>(xs) + (par * kMaxPairs * 2) * kBM + r;
      float msum = 0.f;
      for (int i = 0; i < n; ++i) msum += pr[i * kBM].x;
      mean = msum / static_cast<float>(n);
      float acc = 0.f;
      for (int i = 0; i < n; ++i) {
        const float2 v = pr[i * kBM];
        const float dm = v.x - mean;
        acc += v.y + 128.0f * dm * dm;
      }
      m2 = acc;
      return true;
    };
    for (int u = cid; u < num_m; u += ncl, ++acc_it) {
      const uint32_t a = acc_it & 1u;
      int w = 1;
      if (lane == 0) w = mbar_wait_bounded(&tfull[a], (acc_it >> 1) & 1u, abort_flag) ? 1 : 0;
      w = __shfl_sync(0xffffffffu, w, 0);
      if (!w) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int m0 = u * 2 * kBM + static_cast<int>(hrow) * kBM;   // this CTA's first row
      const int row = m0 + r;
      const bool row_ok = row < M;
      const bool full_tile = m0 + kBM <= M;
      const uint32_t t_acc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + a * kBN + c0;
      // pass A: this warp's sum of acc + bias (the residual is already in acc)
      float s1 = 0.f;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(t_acc + 32 * c, v);
        tmem_ld_wait_tied32(v);
        const float4* b4 = reinterpret_cast<const float4*>(s_bias + c0 + 32 * c);
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float4 b = b4[e];
          ps[0] += __uint_as_float(v[4 * e]) + b.x;
          ps[1] += __uint_as_float(v[4 * e + 1]) + b.y;
          ps[2] += __uint_as_float(v[4 * e + 2]) + b.z;
          ps[3] += __uint_as_float(v[4 * e + 3]) + b.w;
        }
        s1 += (ps[0] + ps[1]) + (ps[2] + ps[3]);
      }
      const float mean_w = s1 * (1.0f / 128.0f);
      // pass B: squared deviations from this warp's own mean
      float m2_w = 0.f;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(t_acc + 32 * c, v);
        tmem_ld_wait_tied32(v);
        const float4* b4 = reinterpret_cast<const float4*>(s_bias + c0 + 32 * c);
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float4 b = b4[e];
          const float d0 = __uint_as_float(v[4 * e]) + b.x - mean_w;
          const float d1 = __uint_as_float(v[4 * e + 1]) + b.y - mean_w;
          const float d2 = __uint_as_float(v[4 * e + 2]) + b.z - mean_w;
          const float d3 = __uint_as_float(v[4 * e + 3]) + b.w - mean_w;
          ps[0] = fmaf(d0, d0, ps[0]);
          ps[1] = fmaf(d1, d1, ps[1]);
          ps[2] = fmaf(d2, d2, ps[2]);
          ps[3] = fmaf(d3, d3, ps[3]);
        }
        m2_w += (ps[0] + ps[1]) + (ps[2] + ps[3]);
      }
      float mean, m2;
      if (!exchange(mean_w, m2_w, mean, m2)) {
        ok = false;
        break;
      }
      const float rstd = rsqrtf(m2 * inv_h + p.eps);
      // pass C: normalise, scale, shift; full row blocks leave through the staging block
      // and TMA stores, a block that reaches past M row by row
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(t_acc + 32 * c, v);
        tmem_ld_wait_tied32(v);
        float y[32];
        const int col = c0 + 32 * c;
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 b = *reinterpret_cast<const float4*>(s_bias + col + e);
          const float4 g = *reinterpret_cast<const float4*>(s_gamma + col + e);
          const float4 be = *reinterpret_cast<const float4*>(s_beta + col + e);
          y[e] = fmaf((__uint_as_float(v[e]) + b.x - mean) * rstd, g.x, be.x);
          y[e + 1] = fmaf((__uint_as_float(v[e + 1]) + b.y - mean) * rstd, g.y, be.y);
          y[e + 2] = fmaf((__uint_as_float(v[e + 2]) + b.z - mean) * rstd, g.z, be.z);
          y[e + 3] = fmaf((__uint_as_float(v[e + 3]) + b.w - mean) * rstd, g.w, be.w);
        }
        if (full_tile) {
#pragma unroll 1
          for (int o = 0; o < (p.out_f16 ? 2 : 1); ++o) {
            if (pending) {   // the previous store has finished reading the staging block
              if (lane == 0) bulk_wait_read0();
              __syncwarp();
            }
            if (o == 0) stage_row16<T>(stage, lane, y);
            else stage_row16<__half>(stage, lane, y);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(o == 0 ? &tmO : &tmO16, stage, n0 + col, m0 + q * 32);
              bulk_commit();
            }
            pending = true;
          }
        } else if (row_ok) {
          const long long off = static_cast<long long>(row) * H + n0 + col;
          uint4* op = reinterpret_cast<uint4*>(static_cast<T*>(p.out) + off);
#pragma unroll
          for (int j = 0; j < 4; ++j) op[j] = pack16<T>(y + 8 * j);
          if (p.out_f16) {
            uint4* hp = reinterpret_cast<uint4*>(p.out_f16 + off);
#pragma unroll
            for (int j = 0; j < 4; ++j) hp[j] = pack16<__half>(y + 8 * j);
          }
        }
      }
      // the accumulator buffer is free for the MMAs of a later row block (on the even CTA)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(cluster_addr(&tempty[a], lead));
    }
    if (pending && lane == 0) bulk_wait0();   // stores complete before the CTA leaves
    __syncwarp();
    if (!ok && lane == 0) {
      set_device_error(p.err, RPP_DERR_TIMEOUT);
      *abort_flag = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  // the cluster frees its tensor memory together: no copy, commit, remote store or
  // arrival of another CTA is still aimed at this one
  cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_cg<2>(tmem_base, kTmemCols);
  }
}

template <typename T, bool RES_F16>
cudaError_t launch_typed(const CUtensorMap* maps, const Params& p, int H, int rows_hint, cudaStream_t stream) {
  auto kern = gemm_ln_kernel<T, RES_F16>;
  const int ncta = 2 * (H / kBN);
  static int max_clusters[2 * kMaxPairs + 1] = {0};
  static bool attr = false;
  if (!attr) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmem));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  if (!max_clusters[ncta]) {
    cudaLaunchConfig_t oc{};
    oc.gridDim = dim3(static_cast<unsigned>(num_sms() / ncta * ncta));
    oc.blockDim = dim3(kThreads);
    oc.dynamicSmemBytes = kSmem;
    cudaLaunchAttribute oa[1];
    oa[0].id = cudaLaunchAttributeClusterDimension;
    oa[0].val.clusterDim.x = ncta;
    oa[0].val.clusterDim.y = 1;
    oa[0].val.clusterDim.z = 1;
    oc.attrs = oa;
    oc.numAttrs = 1;
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, kern, &oc);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorNotSupported;
    max_clusters[ncta] = n;
  }
  const int units = (rows_hint + 2 * kBM - 1) / (2 * kBM);
  int clusters = units < max_clusters[ncta] ? units : max_clusters[ncta];
  if (clusters < 1) clusters = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * ncta));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  at[1].id = cudaLaunchAttributeClusterDimension;
  at[1].val.clusterDim.x = ncta;
  at[1].val.clusterDim.y = 1;
  at[1].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], p);
}

}  // namespace

bool gemm_ln_supported(int H, int K, rpp_dtype dtype) {
  return (dtype == RPP_F16 || dtype == RPP_BF16) && H % kBN == 0 && H / kBN >= 1 && H / kBN <= kMaxPairs &&
         K % 8 == 0 && K > 0;
}

cudaError_t launch_gemm_ln(const GemmLnArgs& g, cudaStream_t stream) {
  if (!gemm_ln_supported(g.H, g.K, g.dtype)) return cudaErrorNotSupported;
  if (g.res_f16 && g.dtype == RPP_F16) return cudaErrorInvalidValue;   // fp16 layers pass the residual as T
  if (!g.ident) return cudaErrorInvalidValue;
  const CUtensorMapDataType dt = g.dtype == RPP_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUtensorMapDataType rdt = g.res_f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : dt;
  CUtensorMap maps[6];
  std::memset(maps, 0, sizeof(maps));
  constexpr CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
  if (!make_tmap_2d(&maps[0], g.a, dt, 2, g.M_max, g.K, kBM, kBK, sw)) return cudaErrorInvalidValue;
  if (!make_tmap_2d(&maps[1], g.w_t, dt, 2, g.H, g.K, kBN / 2, kBK, sw)) return cudaErrorInvalidValue;
  if (!make_tmap_2d(&maps[2], g.residual, rdt, 2, g.M_max, g.H, kBM, kBK, sw)) return cudaErrorInvalidValue;
  if (!make_tmap_2d(&maps[3], g.ident, rdt, 2, kBN, kBN, kBN / 2, kBK, sw)) return cudaErrorInvalidValue;
  // outputs: 32 x 32 boxes with the 64-byte swizzle of the staging rows
  if (!make_tmap_2d(&maps[4], g.out, dt, 2, g.M_max, g.H, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B)) return cudaErrorInvalidValue;
  if (g.out_f16 && !make_tmap_2d(&maps[5], g.out_f16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, g.M_max, g.H, 32, 32,
                                 CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  Params p{g.M_max, g.rows, g.K, g.bias, g.gamma, g.beta, g.eps, g.out, g.out_f16, g.err};
  const int hint = (g.rows_hint > 0 && g.rows_hint < g.M_max) ? g.rows_hint : g.M_max;
  if (g.dtype == RPP_BF16)
    return g.res_f16 ? launch_typed<__nv_bfloat16, true>(maps, p, g.H, hint, stream)
                     : launch_typed<__nv_bfloat16, false>(maps, p, g.H, hint, stream);
  return launch_typed<__half, false>(maps, p, g.H, hint, stream);
}

}  // namespace rpp
