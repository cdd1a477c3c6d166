// Tensor-core GEMM kernel template and its launch/dispatch templates (instantiated by the
// gemm_tc_inst_*.cu translation units, one per input type and cluster size, so that the
// instantiations compile in parallel; gemm_tc.cu holds the host-side tile choice).
#pragma once
#include <cstring>
#include "kernels.h"

namespace rpp {
namespace gemm {


constexpr int kBM = 128;
constexpr int kBK = 64;   // 64 x 16-bit = 128 bytes = one swizzle row
// epilogue warps: 16 for the arithmetic-heavy bias + GELU epilogue (four per
// tensor-memory lane quadrant: its per-element math is issue-bound), 8 for the others
template <int EPI>
constexpr int epi_warps() {
  return EPI == RPP_EPI_BIAS_GELU ? 16 : 8;
}
template <int EPI>
constexpr bool kHoistBias = EPI == RPP_EPI_BIAS || EPI == RPP_EPI_BIAS_GELU;
template <int EPI>
constexpr int gemm_threads() {
  return 64 + 32 * epi_warps<EPI>();
}
constexpr int kChunkBlocks = 16;   // 16 x 64 = 1024 K per exact integer chunk
constexpr size_t kSmemLimit = 232448;   // 227 KB per CTA
constexpr uint16_t kPairMask = 0x3;      // both CTAs of a pair
constexpr int kPairTmemCols = 512;       // tensor-memory columns a CTA pair allocates at most

struct GemmParams {
  int M_max;
  const int32_t* rows;   // device row count or null
  int N;
  int K;
  const float* bias;
  const void* residual;
  void* out;
  const float* a_scale;
  const float* w_scale;
  const float* q_scale;
  int32_t* err;
  int splits;               // K splits per tile (1 = none)
  long long split_stride;   // elements between the fp32 partial slices
  unsigned long long wait_ns;   // limit of the pipeline's bounded waits (the drains keep the default)
  int stall;                // test hook: the producer issues no loads, so the waits run out
};

constexpr uint32_t pow2_cols(uint32_t c) {
  return c <= 32 ? 32 : c <= 64 ? 64 : c <= 128 ? 128 : c <= 256 ? 256 : 512;
}

template <typename T> struct AbFmt;
template <> struct AbFmt<__half> { static constexpr int v = 0; };
template <> struct AbFmt<__nv_bfloat16> { static constexpr int v = 1; };

// epilogues whose full 32 x 32 blocks leave through the TMA store path (all of them)
template <int EPI>
constexpr bool tma_store_epi() {
  return true;
}
// 16-byte vectors of residual per 32 columns
template <typename TRes>
constexpr int res_vecs32() {
  return 32 * static_cast<int>(sizeof(TRes)) / 16;
}
template <int EPI>
constexpr bool is_int_epi() {
  return (EPI >= EPI_I32 && EPI <= EPI_DQ_BIAS_GELU_Q) || EPI == EPI_DQ_BIAS_Q3;
}

// TMA store of a 2D box from shared memory (bulk group)
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until at most N of this thread's bulk store groups are still reading shared memory
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Epilogue arithmetic on NV columns of this thread's row (v holds the accumulator;
// for int8 epilogues the exact integer sum converted to float).
template <int EPI>
constexpr bool has_bias() {
  return EPI == RPP_EPI_BIAS || EPI == RPP_EPI_BIAS_GELU || EPI == RPP_EPI_BIAS_RESIDUAL || EPI == EPI_DQ_BIAS ||
         EPI == EPI_DQ_BIAS_GELU_Q || EPI == EPI_DQ_BIAS_Q3;
}

template <typename TOut, typename TRes, int EPI, int NV>
__device__ __forceinline__ void epi_math(const GemmParams& p, float* v, int row, int n, bool first, float a_s,
                                         float inv_q, const uint4* rres = nullptr, const float4* bpre = nullptr) {
  if constexpr (EPI == EPI_I32 || EPI == EPI_ACC) return;
  if constexpr (EPI == EPI_DQ_BIAS || EPI == EPI_DQ_ACC || EPI == EPI_DQ_BIAS_GELU_Q || EPI == EPI_DQ_BIAS_Q3) {
    const float4* s4 = reinterpret_cast<const float4*>(p.w_scale + n);
#pragma unroll
    for (int j = 0; j < NV / 4; ++j) {
      const float4 ss = __ldg(s4 + j);
      v[4 * j + 0] *= a_s * ss.x;
      v[4 * j + 1] *= a_s * ss.y;
      v[4 * j + 2] *= a_s * ss.z;
      v[4 * j + 3] *= a_s * ss.w;
    }
  }
  if constexpr (has_bias<EPI>()) {
    if (first) {
      const float4* b4 = reinterpret_cast<const float4*>(p.bias + n);
#pragma unroll
      for (int j = 0; j < NV / 4; ++j) {
        const float4 bb = bpre ? bpre[j] : __ldg(b4 + j);
        v[4 * j + 0] += bb.x;
        v[4 * j + 1] += bb.y;
        v[4 * j + 2] += bb.z;
        v[4 * j + 3] += bb.w;
      }
    }
  }
  if constexpr (EPI == RPP_EPI_BIAS_GELU || EPI == EPI_DQ_BIAS_GELU_Q) {
#pragma unroll
    for (int j = 0; j < NV; ++j) v[j] = gelu_erf<(EPI == RPP_EPI_BIAS_GELU && sizeof(TOut) == 2) ? 5 : 7>(v[j]);
  }
  if constexpr (EPI == EPI_DQ_BIAS_GELU_Q) {
#pragma unroll
    for (int j = 0; j < NV; ++j) v[j] = code_of(v[j], inv_q);
  }
  if constexpr (EPI == EPI_DQ_BIAS_Q3) {   // NV columns never straddle a third (N / 3 % 32 == 0)
    const float iq = __fdiv_rn(1.0f, __ldg(p.q_scale + n / (p.N / 3)));
#pragma unroll
    for (int j = 0; j < NV; ++j) v[j] = code_of(v[j], iq);
  }
  if constexpr (EPI == RPP_EPI_BIAS_RESIDUAL) {
    if (first) {
      constexpr int RPV = Vec<TRes>::N;
      const uint4* rr =
          rres ? rres
               : reinterpret_cast<const uint4*>(static_cast<const TRes*>(p.residual) + static_cast<long long>(row) * p.N + n);
#pragma unroll
      for (int j = 0; j < NV / RPV; ++j) {
        float f[RPV];
        unpack16<TRes>(rr[j], f);
#pragma unroll
        for (int e = 0; e < RPV; ++e) v[RPV * j + e] += f[e];
      }
    }
  }
}

// tensor memory -> registers: NV fp32 columns, or for int8 epilogues the exact sum of
// the K-chunk partials (each an integer below 2^24)
template <int EPI, int NCH, int ACC, int NV>
__device__ __forceinline__ void load_acc(uint32_t base, int nch, float* v, int* acc) {
  uint32_t r[NV];
  if constexpr (NV == 32) tmem_ld_32x32b_x32(base, r); else tmem_ld_32x32b_x16(base, r);
  tmem_ld_wait();
  if constexpr (is_int_epi<EPI>()) {
#pragma unroll
    for (int j = 0; j < NV; ++j) acc[j] = __float2int_rn(__uint_as_float(r[j]));
    for (int ch = 1; ch < nch; ++ch) {
      if constexpr (NV == 32) tmem_ld_32x32b_x32(base + ch * ACC, r); else tmem_ld_32x32b_x16(base + ch * ACC, r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < NV; ++j) acc[j] += __float2int_rn(__uint_as_float(r[j]));
    }
#pragma unroll
    for (int j = 0; j < NV; ++j) v[j] = static_cast<float>(acc[j]);
  } else {
#pragma unroll
    for (int j = 0; j < NV; ++j) v[j] = __uint_as_float(r[j]);
  }
}

// per-row 16-byte stores of NV columns (ragged tiles, tails, residual epilogue)
template <typename TOut, int EPI, int NV>
__device__ __forceinline__ void store_row(const GemmParams& p, const float* v, const int* acc, int row, int n,
                                          int split) {
  if constexpr (EPI == EPI_I32) {
    int4* o = reinterpret_cast<int4*>(static_cast<int32_t*>(p.out) + static_cast<long long>(row) * p.N + n);
#pragma unroll
    for (int j = 0; j < NV / 4; ++j) o[j] = make_int4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
  } else {
    constexpr int EPV = Vec<TOut>::N;
    uint4* o = reinterpret_cast<uint4*>(static_cast<TOut*>(p.out) + split * p.split_stride +
                                        static_cast<long long>(row) * p.N + n);
#pragma unroll
    for (int j = 0; j < NV / EPV; ++j) o[j] = pack16<TOut>(v + EPV * j);
  }
}

// Write this thread's row (32 values) into the swizzled 32 x 32 staging block: rows of
// 32 * sizeof(TOut) bytes; 16-byte chunk c of row r sits at chunk c ^ f(r), which is
// the TMA 64-byte swizzle (2-byte types, 64-byte rows) or 128-byte swizzle (4-byte
// types, 128-byte rows).  Eight consecutive lanes cover all 32 banks: no conflicts.
template <typename TOut, int EPI>
__device__ __forceinline__ void stage_row(uint8_t* stage, int r, const float* v, const int* acc) {
  if constexpr (sizeof(TOut) == 2) {
    const int x = (r >> 1) & 3;
#pragma unroll
    for (int c = 0; c < 4; ++c)
      *reinterpret_cast<uint4*>(stage + r * 64 + ((c ^ x) << 4)) = pack16<TOut>(v + 8 * c);
  } else {
    const int x = r & 7;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint4 w;
      if constexpr (EPI == EPI_I32)
        w = make_uint4(static_cast<uint32_t>(acc[4 * c]), static_cast<uint32_t>(acc[4 * c + 1]),
                       static_cast<uint32_t>(acc[4 * c + 2]), static_cast<uint32_t>(acc[4 * c + 3]));
      else
        w = pack16<float>(v + 4 * c);
      *reinterpret_cast<uint4*>(stage + r * 128 + ((c ^ x) << 4)) = w;
    }
  }
}

// one pipeline stage: the 128-row A tile and this CTA's part of the W tile (all of it,
// or half of it in a CTA pair)
constexpr size_t stage_bytes(int bn, int cl) { return kBM * kBK * 2 + ((bn / cl * kBK * 2 + 1023) & ~1023); }
constexpr size_t smem_bytes(int bn, int cl, int stages, size_t epi_total) {
  return 1024 + stages * stage_bytes(bn, cl) + epi_total + 256;
}
// staging blocks per epilogue warp: two for 2-byte outputs with 8 epilogue warps (a
// block is refilled while the store of the other is still reading it), else one
template <typename TOut, int EPI>
constexpr int epi_bufs() {
  return (sizeof(TOut) == 2 && epi_warps<EPI>() == 8) ? 2 : 1;
}
template <typename TOut, int EPI>
constexpr size_t epi_stage_total() {
  return tma_store_epi<EPI>() ? epi_warps<EPI>() * epi_bufs<TOut, EPI>() * 32 * 32 * sizeof(TOut) : 0;
}
// pipeline depth: as many stages (<= 8) as fit next to the epilogue staging blocks
template <typename TOut, int BN, int EPI, int CL>
constexpr int stages_for() {
  const size_t avail = kSmemLimit - 1024 - 256 - epi_stage_total<TOut, EPI>();
  const size_t s = avail / stage_bytes(BN, CL);
  return s > 8 ? 8 : static_cast<int>(s);
}

template <typename TIn, typename TOut, typename TRes, int BN, int STAGES, int EPI, int NCH, int CL>
__global__ void __launch_bounds__(gemm_threads<EPI>(), 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmC, GemmParams p) {
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M = 128");
  static_assert(CL == 1 || CL == 2, "one CTA or a CTA pair");
  constexpr uint32_t A_BYTES = kBM * kBK * 2;
  constexpr uint32_t B_PART = BN / CL * kBK * 2;   // bytes of the W tile held by this CTA
  static_assert(CL == 1 || B_PART % 1024 == 0, "each CTA's half of the W tile is whole 8-row swizzle atoms");
  constexpr uint32_t B_BYTES_AL = (B_PART + 1023u) & ~1023u;
  // bytes the (leader's) full barrier of a stage waits for: every CTA's A tile and W part
  constexpr uint32_t STAGE_TX = CL * (A_BYTES + B_PART);
  constexpr int ACC = (BN + 31) / 32 * 32;               // columns per accumulator region
  constexpr int TMEM_LIMIT = CL == 1 ? 512 : kPairTmemCols;
  constexpr int NBUF = (2 * NCH * ACC <= TMEM_LIMIT) ? 2 : 1;  // accumulator buffers in tensor memory
  static_assert(NCH * ACC <= TMEM_LIMIT, "tensor memory columns");
  constexpr uint32_t TMEM_COLS = pow2_cols(NBUF * NCH * ACC);
  constexpr uint32_t IDESC = idesc_f16(AbFmt<TIn>::v, kBM * CL, BN);   // M = 256 across a CTA pair
  constexpr bool kTma = tma_store_epi<EPI>();
  constexpr uint32_t EPI_STAGE = kTma ? 32 * 32 * sizeof(TOut) : 0;   // one staging block
  constexpr int EPI_BUFS = epi_bufs<TOut, EPI>();
  constexpr int EW = epi_warps<EPI>();
  constexpr int WPQ = EW / 4;   // epilogue warps per tensor-memory lane quadrant

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled tiles
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint8_t* sEpi = sB + STAGES * B_BYTES_AL;   // EW x EPI_BUFS staging blocks (1024-aligned)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sEpi + EW * EPI_BUFS * EPI_STAGE);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // [M, skip, tensor-memory base] as decided by CTA rank 0 of the pair; [3]: mismatch seen
  int* cl_info = const_cast<int*>(abort_flag) + 1;

  const int warp = warp_id();
  const int lane = lane_id();
  const uint32_t rank = CL > 1 ? cluster_ctarank() : 0u;
  const int cid = blockIdx.x / CL;         // pair (cluster) index
  const int ncl = gridDim.x / CL;          // pairs in the grid
  const bool leader = rank == 0;           // issues the MMAs of the pair

  // Stages whose W part was issued before the programmatic-launch wait (unpaired
  // GEMMs): the weights are never written by a kernel that lets its dependents start
  // early, so this CTA's first unit's first W boxes can be in flight while the
  // preceding kernel drains; its A boxes follow after the wait.
  int npre = 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);     // in a pair only the leader's is used
      mbar_init(&empty[s], 1);    // released by the (leader's) MMA commit
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], CL * EW);   // one arrival per epilogue warp of the pair
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    cl_info[3] = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if constexpr (kTma) tma_prefetch_desc(&tmC);
    if (CL == 1 && !p.stall) {
      // unit cid: column block (cid / S) % num_n, K blocks [kb0, kb1) (independent of M)
      const int nk = (p.K + kBK - 1) / kBK;
      const int kps0 = (nk + p.splits - 1) / p.splits;
      const int t0 = cid / p.splits;
      const int kb0 = (cid - t0 * p.splits) * kps0;
      const int kb1 = min(nk, kb0 + kps0);
      const int n0 = (t0 % (p.N / BN)) * BN;
      npre = kb1 > kb0 ? min(kb1 - kb0, STAGES) : 0;
      for (int s = 0; s < npre; ++s) {
        mbar_expect_tx(&full[s], B_PART);
        tma_load_2d(sB + s * B_BYTES_AL, &tmB, &full[s], (kb0 + s) * kBK, n0);
      }
    }
  }
  if (warp == 1) {
    tmem_alloc_cg<CL>(tmem_slot, TMEM_COLS);
    tmem_relinquish_cg<CL>();
  }
  if (CL > 1 && threadIdx.x == 32) {
    // The weights are never written by the preceding kernel: warm L2 with this CTA's
    // first weight boxes while that kernel drains.  The (tile, split) order puts the
    // column block of unit `cid` at (unit / S) % num_n regardless of M.
    const int nn = p.N / BN;
    const int nk = (p.K + kBK - 1) / kBK;
    const int kps0 = (nk + p.splits - 1) / p.splits;
    const int t0 = cid / p.splits;
    const int kb0 = (cid - t0 * p.splits) * kps0;
    const int n0 = (t0 % nn) * BN + static_cast<int>(rank) * (BN / CL);
    const int kb1 = min(nk, kb0 + min(kps0, STAGES));
    for (int kb = kb0; kb < kb1; ++kb) tma_prefetch_l2_2d(&tmB, kb * kBK, n0);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // everything below may read what the preceding kernel wrote
  pdl_wait();
  pdl_trigger();

  int M = p.M_max;
  bool skip = false;
  if (CL == 1 || rank == 0) {
    skip = device_error_set(p.err);
    if (p.rows) {
      M = *p.rows;
      if (M > p.M_max || M < 0) {
        if (threadIdx.x == 0) set_device_error(p.err, RPP_DERR_ROWS);
        skip = true;
      }
    }
  }
  if constexpr (CL > 1) {
    // One decision for the pair (both CTAs must run the same units): rank 0 publishes
    // M and skip into both CTAs' shared memory.  The first barrier also makes the
    // leader's mbarrier inits visible before the partner's loads signal them.
    cluster_sync();
    if (rank == 0 && threadIdx.x == 0) {
      for (uint32_t r = 0; r < CL; ++r) {
        st_shared_remote(cl_info, r, static_cast<uint32_t>(M));
        st_shared_remote(cl_info + 1, r, skip ? 1u : 0u);
        st_shared_remote(cl_info + 2, r, tmem_base);
      }
    }
    cluster_sync();
    M = cl_info[0];
    skip = cl_info[1] != 0;
    // the leader's MMAs write both CTAs' tensor memory at the leader's column address:
    // the collective allocation must have given both CTAs the same one
    if (rank != 0 && threadIdx.x == 0 && static_cast<uint32_t>(cl_info[2]) != tmem_base) {
      set_device_error(p.err, RPP_DERR_TMEM);
      for (uint32_t r = 0; r < CL; ++r) st_shared_remote(cl_info + 3, r, 1u);
    }
    cluster_sync();
    if (cl_info[3]) skip = true;
  }
  const int num_m = skip ? 0 : (M + kBM - 1) / kBM;
  const int num_mc = (num_m + CL - 1) / CL;     // row-tile groups (one 128-row tile per CTA of a pair)
  const int num_n = p.N / BN;
  const int num_k = (p.K + kBK - 1) / kBK;
  const int S = p.splits;
  const int kps = (num_k + S - 1) / S;          // K blocks per split
  const int total = num_mc * num_n * S;         // work units of a pair: (row-tile group, column tile, split)
  // row tile of this CTA in unit u's group; the last group of an odd count has an
  // empty second tile (its rows are >= M: loaded, computed, never stored)
  auto m_tile = [&](int u) { return ((u / S) / num_n) * CL + static_cast<int>(rank); };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      // (test hook) no loads at all: the consumers' bounded waits run out
      for (int unit = p.stall ? total : cid; unit < total && ok; unit += ncl) {
        const int tile = unit / S;
        const int kb0 = (unit - tile * S) * kps;
        const int kb1 = min(num_k, kb0 + kps);
        const int m0 = m_tile(unit) * kBM;
        const int n0 = (tile % num_n) * BN;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const uint32_t s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1u;
          if (static_cast<int>(it) < npre) {   // first pass, W part already in flight
            mbar_arrive_expect_tx(&full[s], A_BYTES);
            tma_load_2d(sA + s * A_BYTES, &tmA, &full[s], kb * kBK, m0);
            continue;
          }
          if (!mbar_wait_bounded(&empty[s], ph ^ 1u, abort_flag, p.wait_ns)) {
            ok = false;
            break;
          }
          if constexpr (CL == 1) {
            mbar_arrive_expect_tx(&full[s], STAGE_TX);
            tma_load_2d(sA + s * A_BYTES, &tmA, &full[s], kb * kBK, m0);
            tma_load_2d(sB + s * B_BYTES_AL, &tmB, &full[s], kb * kBK, n0);
          } else {
            // both CTAs load their A tile and their half of the W tile into their own
            // shared memory; every copy completes on the leader's full barrier
            if (leader) mbar_arrive_expect_tx(&full[s], STAGE_TX);
            const uint32_t fb = cluster_addr(&full[s], 0);
            tma_load_2d_pair(sA + s * A_BYTES, &tmA, fb, kb * kBK, m0);
            tma_load_2d_pair(sB + s * B_BYTES_AL, &tmB, fb, kb * kBK, n0 + static_cast<int>(rank) * (BN / CL));
          }
        }
      }
      if (!ok) {
        set_device_error(p.err, RPP_DERR_TIMEOUT);
        *abort_flag = 1;
      }
      // early W boxes of a unit this CTA does not have (fewer rows than the grid was
      // sized for, or an error raised upstream): complete those phases without A
      for (; static_cast<int>(it) < npre; ++it) mbar_arrive(&full[it % STAGES]);
      // wait (bounded) for the copies still in flight: the last min(it, STAGES) loads
      // (a pair's partner: the leader waits for them, and the pair meets at the end)
      if (leader) {
        const uint32_t first = it > STAGES ? it - STAGES : 0;
        for (uint32_t j = first; j < it; ++j) mbar_wait_bounded(&full[j % STAGES], (j / STAGES) & 1u, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (the leader's)
    if (lane == 0 && leader) {
      // The issuing thread's loop is on the tensor pipe's critical path: the stage and its
      // phase advance incrementally, and a stage only moves the start-address field
      // (16-byte units) of the first stage's descriptors.
      uint32_t s = 0, ph = 0, acc_it = 0;
      const uint64_t adesc0 = sw128_kmajor_desc(smem_u32(sA));
      const uint64_t bdesc0 = sw128_kmajor_desc(smem_u32(sB));
      bool ok = true;
      for (int unit = cid; unit < total && ok; unit += ncl, ++acc_it) {
        const int tile = unit / S;
        const int kb0 = (unit - tile * S) * kps;
        const int kb1 = min(num_k, kb0 + kps);
        const uint32_t a = NBUF == 2 ? (acc_it & 1u) : 0u;
        const uint32_t aph = NBUF == 2 ? ((acc_it >> 1) & 1u) : (acc_it & 1u);
        if (!mbar_wait_bounded(&tempty[a], aph ^ 1u, abort_flag, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = kb0; kb < kb1; ++kb) {
          const int chunk = NCH > 1 ? (kb - kb0) / kChunkBlocks : 0;
          const int kb_in = (kb - kb0) - chunk * kChunkBlocks;
          const uint32_t d_tmem = tmem_base + (a * NCH + chunk) * ACC;
          if (!mbar_wait_bounded(&full[s], ph, abort_flag, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = adesc0 + s * (A_BYTES >> 4);
          const uint64_t bdesc = bdesc0 + s * (B_BYTES_AL >> 4);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            // +32 bytes along K inside the swizzled 128-byte row = +2 in the address field
            tc_mma_f16_cg<CL>(d_tmem, adesc + 2u * k, bdesc + 2u * k, IDESC, (kb_in | k) != 0 ? 1u : 0u);
          }
          // the stage is free in every CTA of the pair once these MMAs are done
          tc_commit_cg<CL>(&empty[s], kPairMask);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (ok) tc_commit_cg<CL>(&tfull[a], kPairMask);
      }
      if (!ok) {
        set_device_error(p.err, RPP_DERR_TIMEOUT);
        *abort_flag = 1;
      }
      // all MMAs issued by this thread complete before tensor memory is released
      tc_commit_cg<CL>(drain, 1u);
      mbar_wait_bounded(drain, 0, nullptr);
    }
  } else {
    // ------------------------------------------------------------ epilogue warps
    const int q = warp & 3;               // tensor-memory lane quadrant of this warp
    const int part = (warp - 2) >> 2;     // which of the WPQ warps of this quadrant
    const int r_in_tile = q * 32 + lane;
    uint8_t* stage0 = sEpi + (warp - 2) * EPI_BUFS * EPI_STAGE;
    int sb = 0;   // staging block of the next store
    float a_s = 1.f, inv_q = 0.f;
    if constexpr (EPI == EPI_DQ_BIAS || EPI == EPI_DQ_ACC || EPI == EPI_DQ_BIAS_GELU_Q || EPI == EPI_DQ_BIAS_Q3)
      a_s = *p.a_scale;
    if constexpr (EPI == EPI_DQ_BIAS_GELU_Q) inv_q = __fdiv_rn(1.0f, *p.q_scale);
    uint32_t acc_it = 0;
    bool pending_store = false;
    for (int unit = cid; unit < total; unit += ncl, ++acc_it) {
      const int tile = unit / S;
      const int split = unit - tile * S;
      const int kb0 = split * kps;
      const int kb1 = min(num_k, kb0 + kps);
      const int nch = NCH > 1 ? (kb1 - kb0 + kChunkBlocks - 1) / kChunkBlocks : 1;
      const uint32_t a = NBUF == 2 ? (acc_it & 1u) : 0u;
      const uint32_t aph = NBUF == 2 ? ((acc_it >> 1) & 1u) : (acc_it & 1u);
      // residual of this warp's first 32-column slice, requested before the accumulator wait
      constexpr int RV = res_vecs32<TRes>();
      uint4 rnext[RV];
      const int pre_m0 = m_tile(unit) * kBM;
      const int pre_n0 = (unit / S % num_n) * BN;
      const int pre_row = pre_m0 + r_in_tile;
      if constexpr (EPI == RPP_EPI_BIAS_RESIDUAL && BN >= 32) {
        if (pre_row < M && part < BN / 32) {
          const uint4* rr = reinterpret_cast<const uint4*>(static_cast<const TRes*>(p.residual) +
                                                           static_cast<long long>(pre_row) * p.N + pre_n0 + part * 32);
#pragma unroll
          for (int j = 0; j < RV; ++j) rnext[j] = rr[j];
        }
      }
      int ok = 1;
      if (lane == 0) ok = mbar_wait_bounded(&tfull[a], aph, abort_flag, p.wait_ns) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) {
          set_device_error(p.err, RPP_DERR_TIMEOUT);
          *abort_flag = 1;
        }
        break;
      }
      tc_fence_after();
      const int m0 = m_tile(unit) * kBM;
      const int n0 = (tile % num_n) * BN;
      const int row = m0 + r_in_tile;
      const bool row_ok = row < M;
      const bool full_tile = m0 + kBM <= M;
      const bool first = split == 0;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + (a * NCH) * ACC;
      if constexpr (BN >= 32) {
#pragma unroll 1
        for (int c = part; c < BN / 32; c += WPQ) {
          uint4 rcur[RV];
          if constexpr (EPI == RPP_EPI_BIAS_RESIDUAL) {
#pragma unroll
            for (int j = 0; j < RV; ++j) rcur[j] = rnext[j];
            if (row_ok && c + WPQ < BN / 32) {   // next slice's residual while this one is processed
              const uint4* rr = reinterpret_cast<const uint4*>(static_cast<const TRes*>(p.residual) +
                                                               static_cast<long long>(row) * p.N + n0 + (c + WPQ) * 32);
#pragma unroll
              for (int j = 0; j < RV; ++j) rnext[j] = rr[j];
            }
          }
          const uint4* rres = EPI == RPP_EPI_BIAS_RESIDUAL ? rcur : nullptr;
          const int n = n0 + c * 32;
          // the bias loads go out before the tensor-memory wait and overlap it
          float4 bpre[kHoistBias<EPI> ? 8 : 1];
          if constexpr (kHoistBias<EPI>) {
            if (first) {
#pragma unroll
              for (int j = 0; j < 8; ++j) bpre[j] = __ldg(reinterpret_cast<const float4*>(p.bias + n) + j);
            }
          }
          float v[32];
          int acc[32];
          load_acc<EPI, NCH, ACC, 32>(t_row + c * 32, nch, v, acc);
          if (kTma && full_tile) {
            epi_math<TOut, TRes, EPI, 32>(p, v, row, n, first, a_s, inv_q, rres, kHoistBias<EPI> ? bpre : nullptr);
            uint8_t* stage = stage0 + sb * EPI_STAGE;
            if (pending_store) {   // the store that last used this block has finished reading it
              if (lane == 0) bulk_wait_read<EPI_BUFS - 1>();
              __syncwarp();
            }
            stage_row<TOut, EPI>(stage, lane, v, acc);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmC, stage, n, split * p.M_max + m0 + q * 32);
              bulk_commit();
            }
            pending_store = true;
            sb = EPI_BUFS > 1 ? sb ^ 1 : 0;
          } else if (row_ok) {
            epi_math<TOut, TRes, EPI, 32>(p, v, row, n, first, a_s, inv_q, rres, kHoistBias<EPI> ? bpre : nullptr);
            store_row<TOut, EPI, 32>(p, v, acc, row, n, split);
          }
        }
      }
      if constexpr (BN % 32 == 16) {
        if (part == (BN / 32) % WPQ) {
          float v[16];
          int acc[16];
          load_acc<EPI, NCH, ACC, 16>(t_row + (BN - 16), nch, v, acc);
          if (row_ok) {
            const int n = n0 + BN - 16;
            epi_math<TOut, TRes, EPI, 16>(p, v, row, n, first, a_s, inv_q);
            store_row<TOut, EPI, 16>(p, v, acc, row, n, split);
          }
        }
      }
      // this warp is done with accumulator a (in a pair: tell the leader's barrier)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (CL == 1) mbar_arrive(&tempty[a]);
        else mbar_arrive_cluster_relaxed(cluster_addr(&tempty[a], 0));
      }
    }
    if (pending_store && lane == 0) bulk_wait0();   // stores complete before the CTA exits
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  // a pair frees its tensor memory together, once both CTAs' epilogues are done and
  // no copy or arrival of either CTA is still aimed at the other
  if constexpr (CL > 1) cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_cg<CL>(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side


template <typename T> struct MapType;
template <> struct MapType<__half> { static constexpr CUtensorMapDataType v = CU_TENSOR_MAP_DATA_TYPE_FLOAT16; };
template <> struct MapType<__nv_bfloat16> { static constexpr CUtensorMapDataType v = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16; };
template <> struct MapType<float> { static constexpr CUtensorMapDataType v = CU_TENSOR_MAP_DATA_TYPE_FLOAT32; };
template <> struct MapType<int32_t> { static constexpr CUtensorMapDataType v = CU_TENSOR_MAP_DATA_TYPE_INT32; };

template <typename TIn, typename TOut, typename TRes, int BN, int EPI, int NCH, int CL>
cudaError_t gemm_tc_launch(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p, int grid_rows,
                           cudaStream_t stream) {
  constexpr int STAGES = stages_for<TOut, BN, EPI, CL>();
  static_assert(STAGES >= 2, "pipeline depth");
  constexpr size_t SMEM = smem_bytes(BN, CL, STAGES, epi_stage_total<TOut, EPI>());
  static_assert(SMEM <= kSmemLimit, "shared memory per CTA");
  CUtensorMap tc;
  std::memset(&tc, 0, sizeof(tc));
  if constexpr (tma_store_epi<EPI>()) {
    // output as [splits * M_max, N]; 32 x 32 boxes, swizzle matching the staging rows
    const CUtensorMapSwizzle swz = sizeof(TOut) == 2 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    if (!make_tmap_2d(&tc, p.out, MapType<TOut>::v, sizeof(TOut), static_cast<long long>(p.splits) * p.M_max, p.N,
                      32, 32, swz))
      return cudaErrorInvalidValue;
  }
  auto kern = gemm_tc_kernel<TIn, TOut, TRes, BN, STAGES, EPI, NCH, CL>;
  static bool attr_set = false;
  static int max_clusters = 0;   // clusters of CL CTAs that fit on the GPU at once
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(SMEM));
    if (e != cudaSuccess) return e;
    if constexpr (CL > 1) {
      cudaLaunchConfig_t oc{};
      oc.gridDim = dim3(static_cast<unsigned>(num_sms() / CL * CL));
      oc.blockDim = dim3(gemm_threads<EPI>());
      oc.dynamicSmemBytes = SMEM;
      cudaLaunchAttribute oa[1];
      oa[0].id = cudaLaunchAttributeClusterDimension;
      oa[0].val.clusterDim.x = CL;
      oa[0].val.clusterDim.y = 1;
      oa[0].val.clusterDim.z = 1;
      oc.attrs = oa;
      oc.numAttrs = 1;
      e = cudaOccupancyMaxActiveClusters(&max_clusters, kern, &oc);
      if (e != cudaSuccess) return e;
    } else {
      max_clusters = num_sms();
    }
    attr_set = true;
  }
  if (max_clusters < 1) return cudaErrorNotSupported;
  const int num_m = (grid_rows + kBM - 1) / kBM;
  const long long units = static_cast<long long>((num_m + CL - 1) / CL) * (p.N / BN) * p.splits;
  int clusters = units < max_clusters ? static_cast<int>(units) : max_clusters;
  if (clusters < 1) clusters = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * CL));
  cfg.blockDim = dim3(gemm_threads<EPI>());
  cfg.dynamicSmemBytes = SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = CL;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = CL > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, p);
}

template <typename TIn, typename TOut, typename TRes, int EPI, int NCH, int CL = 1>
cudaError_t dispatch_bn(int bn, const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p, int gr,
                        cudaStream_t stream) {
  if constexpr (NCH == 1) {
    switch (bn) {
      case 256: return gemm_tc_launch<TIn, TOut, TRes, 256, EPI, 1, CL>(ta, tb, p, gr, stream);
      case 192: return gemm_tc_launch<TIn, TOut, TRes, 192, EPI, 1, CL>(ta, tb, p, gr, stream);
      case 144: return gemm_tc_launch<TIn, TOut, TRes, 144, EPI, 1, CL>(ta, tb, p, gr, stream);
      case 128: return gemm_tc_launch<TIn, TOut, TRes, 128, EPI, 1, CL>(ta, tb, p, gr, stream);
      case 96: return gemm_tc_launch<TIn, TOut, TRes, 96, EPI, 1, CL>(ta, tb, p, gr, stream);
      case 64: return gemm_tc_launch<TIn, TOut, TRes, 64, EPI, 1, CL>(ta, tb, p, gr, stream);
      case 48: return gemm_tc_launch<TIn, TOut, TRes, 48, EPI, 1, CL>(ta, tb, p, gr, stream);
      case 32: return gemm_tc_launch<TIn, TOut, TRes, 32, EPI, 1, CL>(ta, tb, p, gr, stream);
      case 16: return gemm_tc_launch<TIn, TOut, TRes, 16, EPI, 1, CL>(ta, tb, p, gr, stream);
      default: return cudaErrorNotSupported;
    }
  } else {
    static_assert(CL == 1, "the chunked integer GEMM runs unclustered");
    switch (bn) {   // NCH x BN <= 512 tensor-memory columns
      case 128: return gemm_tc_launch<TIn, TOut, TRes, 128, EPI, NCH, 1>(ta, tb, p, gr, stream);
      case 96: return gemm_tc_launch<TIn, TOut, TRes, 96, EPI, NCH, 1>(ta, tb, p, gr, stream);
      case 64: return gemm_tc_launch<TIn, TOut, TRes, 64, EPI, NCH, 1>(ta, tb, p, gr, stream);
      case 48: return gemm_tc_launch<TIn, TOut, TRes, 48, EPI, NCH, 1>(ta, tb, p, gr, stream);
      case 32: return gemm_tc_launch<TIn, TOut, TRes, 32, EPI, NCH, 1>(ta, tb, p, gr, stream);
      case 16: return gemm_tc_launch<TIn, TOut, TRes, 16, EPI, NCH, 1>(ta, tb, p, gr, stream);
      default: return cudaErrorNotSupported;
    }
  }
}

template <typename T, int CL>
cudaError_t dispatch_float(int bn, int epi, rpp_dtype out_dtype, rpp_dtype res_dtype, const CUtensorMap& ta,
                           const CUtensorMap& tb, const GemmParams& p, int gr, cudaStream_t stream) {
  switch (epi) {
    case RPP_EPI_BIAS: return dispatch_bn<T, T, T, RPP_EPI_BIAS, 1, CL>(bn, ta, tb, p, gr, stream);
    case RPP_EPI_BIAS_GELU: return dispatch_bn<T, T, T, RPP_EPI_BIAS_GELU, 1, CL>(bn, ta, tb, p, gr, stream);
    case RPP_EPI_BIAS_RESIDUAL:
      if (out_dtype == RPP_F32 && res_dtype == RPP_F32)
        return dispatch_bn<T, float, float, RPP_EPI_BIAS_RESIDUAL, 1, CL>(bn, ta, tb, p, gr, stream);
      if constexpr (!std::is_same<T, __half>::value) {
        if (out_dtype == RPP_F32 && res_dtype == RPP_F16)
          return dispatch_bn<T, float, __half, RPP_EPI_BIAS_RESIDUAL, 1, CL>(bn, ta, tb, p, gr, stream);
      }
      if (out_dtype == RPP_F32)
        return dispatch_bn<T, float, T, RPP_EPI_BIAS_RESIDUAL, 1, CL>(bn, ta, tb, p, gr, stream);
      if (out_dtype == RPP_F16 && res_dtype == RPP_F16)
        return dispatch_bn<T, __half, __half, RPP_EPI_BIAS_RESIDUAL, 1, CL>(bn, ta, tb, p, gr, stream);
      if (out_dtype == RPP_F16)
        return dispatch_bn<T, __half, T, RPP_EPI_BIAS_RESIDUAL, 1, CL>(bn, ta, tb, p, gr, stream);
      return dispatch_bn<T, T, T, RPP_EPI_BIAS_RESIDUAL, 1, CL>(bn, ta, tb, p, gr, stream);
    case EPI_ACC: return dispatch_bn<T, float, T, EPI_ACC, 1, CL>(bn, ta, tb, p, gr, stream);
    default: return cudaErrorNotSupported;
  }
}

template <int NCH>
cudaError_t dispatch_int(int bn, int epi, const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p, int gr,
                         cudaStream_t stream) {
  using BF = __nv_bfloat16;
  switch (epi) {
    case EPI_I32: return dispatch_bn<BF, int32_t, BF, EPI_I32, NCH>(bn, ta, tb, p, gr, stream);
    case EPI_DQ_BIAS: return dispatch_bn<BF, __half, __half, EPI_DQ_BIAS, NCH>(bn, ta, tb, p, gr, stream);
    case EPI_DQ_ACC: return dispatch_bn<BF, float, __half, EPI_DQ_ACC, NCH>(bn, ta, tb, p, gr, stream);
    case EPI_DQ_BIAS_GELU_Q: return dispatch_bn<BF, BF, BF, EPI_DQ_BIAS_GELU_Q, NCH>(bn, ta, tb, p, gr, stream);
    case EPI_DQ_BIAS_Q3: return dispatch_bn<BF, BF, BF, EPI_DQ_BIAS_Q3, NCH>(bn, ta, tb, p, gr, stream);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace gemm

// one entry per instantiation unit (gemm_tc_inst_*.cu)
cudaError_t gemm_dispatch_float_bf16_cl1(int bn, int epi, rpp_dtype out_dtype, rpp_dtype res_dtype,
                                         const CUtensorMap& ta, const CUtensorMap& tb, const gemm::GemmParams& p,
                                         int gr, cudaStream_t stream);
cudaError_t gemm_dispatch_float_bf16_cl2(int bn, int epi, rpp_dtype out_dtype, rpp_dtype res_dtype,
                                         const CUtensorMap& ta, const CUtensorMap& tb, const gemm::GemmParams& p,
                                         int gr, cudaStream_t stream);
cudaError_t gemm_dispatch_float_f16_cl1(int bn, int epi, rpp_dtype out_dtype, rpp_dtype res_dtype,
                                        const CUtensorMap& ta, const CUtensorMap& tb, const gemm::GemmParams& p,
                                        int gr, cudaStream_t stream);
cudaError_t gemm_dispatch_float_f16_cl2(int bn, int epi, rpp_dtype out_dtype, rpp_dtype res_dtype,
                                        const CUtensorMap& ta, const CUtensorMap& tb, const gemm::GemmParams& p,
                                        int gr, cudaStream_t stream);
cudaError_t gemm_dispatch_int(int nch, int bn, int epi, const CUtensorMap& ta, const CUtensorMap& tb,
                              const gemm::GemmParams& p, int gr, cudaStream_t stream);

}  // namespace rpp
