// Persistent variable-length multi-head attention on the 5th-generation tensor cores
// (head size 64, fp16 or bf16): the encoder layer's fMHA.
//
// The Swin talk (§3) runs fMHA as batch GEMM + softmax + batch GEMM in one kernel with
// the head transposes folded into its I/O; the Kuaishou article (Fig. 10) runs the
// attention on the padding-free packed batch, where it is the one kernel that needs
// the sequence bounds.  This kernel takes the sequence bounds from cu_seqlens and:
//
//  * Schedules work longest-first.  A work item is (sequence, head, 128-query tile);
//    its cost is the sequence's number of 128-key tiles.  Every CTA builds the same
//    item list from cu_seqlens in its prologue -- sequences grouped by tile count,
//    largest first, stable within a group -- and a persistent grid of two CTAs per SM
//    walks it round-robin.  The q-tiles of one (sequence, head) are neighbours in the
//    list, so the CTAs that share its K and V tiles run at the same time and read them
//    from L2.
//  * Keeps S, P and O in tensor memory: S = Q K^T (columns [0, 128)), P (the 16-bit
//    softmax numerators, columns [128, 192): 128 keys, two per 32-bit column) and O
//    (columns [192, 256)).  O += P V reads P straight from tensor memory (the A operand
//    of tcgen05.mma may live there), so P never goes through shared memory.
//  * Runs the softmax on eight warps, two per tensor-memory lane quadrant: each warp
//    owns 32 query rows and half of a tile's 128 keys.  A warp takes its half's row
//    maximum (tcgen05.ld, keys past the sequence masked), the two warps of a quadrant
//    exchange maxima through shared memory (bounded mbarrier wait), then each writes
//    2^(s - m) rounded to the input type into its half of P and keeps its half of the
//    fp32 row sum; the halves of the sum are added once per item.  The reference
//    maximum m moves only when a tile's maximum exceeds it by more than 8 (log2 units),
//    so P stays below 2^8; O and the sums are then rescaled in tensor memory.  Tensor-
//    memory loads and stores are warp-collective, so that decision is taken per warp
//    (scale 1 for rows that keep their maximum); both warps of a quadrant see the same
//    rows and maxima and decide alike.
//  * Overlaps: the MMA thread walks the CTA's tiles as one stream and issues S_{t+1}
//    before P_t V_t, also across items; K and V tiles are double-buffered and the next
//    item's Q tile loads while the current item finishes.  Partial tiles shrink the MMAs
//    to whole 16-key steps; warps whose 32 query rows all lie past the sequence skip the
//    softmax arithmetic.
//
// Keys past the sequence end get -inf before the maximum (P = 0 there); the V rows of
// the last 16-key step that lie past the end are zeroed in shared memory, so nothing
// beyond the sequence (another sequence, or unwritten capacity holding NaN) reaches a
// valid output.  Query rows past the end are computed and never stored.  Every
// mbarrier wait is bounded; a wait that gives up records RPP_DERR_TIMEOUT, raises the
// CTA's abort flag, and the CTA drains its copies and MMAs, frees tensor memory and
// exits.
#include "attention_common.cuh"

namespace rpp {

namespace {

using namespace attn;

constexpr int kThreads = 320;                  // warp 0 TMA, warp 1 MMA, warps 2..9 softmax
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0, kColP = 128, kColO = 192;

// shared-memory layout (bytes from the 1024-aligned base)
constexpr uint32_t kOffQ = 0;                  // [2] tiles
constexpr uint32_t kOffK = 2 * kTile;          // [2]
constexpr uint32_t kOffV = 4 * kTile;          // [2]
constexpr uint32_t kOffBar = 6 * kTile;        // 16 mbarriers
constexpr uint32_t kOffMisc = kOffBar + 16 * 8;   // tmem slot, abort flag, counts, more barriers
constexpr uint32_t kOffX = kOffMisc + 128;      // pair exchange: float [2 parities][2 halves][128 rows]
constexpr uint32_t kOffSched = kOffX + 2 * 2 * 128 * 4;   // the item list (sched_bytes(B))

size_t smem_bytes(int B) { return 1024 + kOffSched + sched_bytes(B); }

// I8: Q, K and V are int8 codes held in bf16 (exact), i8_scales = (s_q, s_k, s_v) in
// device memory, and every item takes two passes over its key tiles: the first computes
// only the row maxima and sums, the second writes P's codes clamp(rne(127 P), 0, 127)
// of the normalised softmax into tensor memory; S = Qc Kc^T and O = Pc Vc are then
// exact integers in the fp32 accumulators, and O is written as fp16 O s_v / 127.
// QO: O leaves as the int8 codes clamp(rne(O / s_o), -127, 127) held in bf16, s_o in
// device memory (the input quantisation of the output projection, fused).
template <typename T, bool I8, bool QO>
__global__ void __launch_bounds__(kThreads, 2)
attention_sched_kernel(const __grid_constant__ CUtensorMap tm, const int32_t* __restrict__ cu, int B, int T_max,
                       int max_len, int nh, int n_cls, void* __restrict__ out_v, float scale_log2,
                       const float* __restrict__ i8_scales, const float* __restrict__ out_scale, int32_t* err) {
  using TOut = typename std::conditional<QO, __nv_bfloat16, typename std::conditional<I8, __half, T>::type>::type;
  TOut* out = static_cast<TOut*>(out_v);
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* q_full = bars + 0;    // [2]
  uint64_t* q_empty = bars + 2;   // [2]
  uint64_t* k_full = bars + 4;    // [2]
  uint64_t* k_empty = bars + 6;   // [2]
  uint64_t* v_full = bars + 8;    // [2]
  uint64_t* v_empty = bars + 10;  // [2]
  uint64_t* s_full = bars + 12;   // S computed (commit)
  uint64_t* s_free = bars + 13;   // S read by the eight softmax warps
  uint64_t* p_full = bars + 14;   // P written by the eight softmax warps
  uint64_t* pv_done = bars + 15;  // O += P V completed (commit)
  uint64_t* o_free = reinterpret_cast<uint64_t*>(smem + kOffMisc + 32);   // O read out (eight warps)
  uint64_t* drain = reinterpret_cast<uint64_t*>(smem + kOffMisc + 40);
  uint64_t* xbar = reinterpret_cast<uint64_t*>(smem + kOffMisc + 48);   // [4] pair exchanges, per quadrant
  float* xval = reinterpret_cast<float*>(smem + kOffX);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  int* s_status = reinterpret_cast<int*>(smem + kOffMisc + 8);   // 0 ok, else the device error to record / quit
  const int warp = warp_id();
  const int lane = lane_id();

  // everything below reads what the preceding kernels wrote (the QKV rows, cu_seqlens)
  pdl_wait();
  pdl_trigger();

  if (threadIdx.x == 0) *abort_flag = 0;
  Sched sch;
  if (!build_items(cu, B, T_max, max_len, nh, n_cls, err, s_status, smem + kOffSched, sch)) return;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, 8);
    mbar_init(p_full, 8);
    mbar_init(pv_done, 1);
    mbar_init(o_free, 8);
    for (int i = 0; i < 4; ++i) mbar_init(&xbar[i], 2);
    mbar_init(drain, 1);
    fence_mbarrier_init();
    tma_prefetch_desc(&tm);
  }
  const int n_items = sch.item_off[0];
  if (static_cast<int>(blockIdx.x) >= n_items) return;   // uniform: nothing allocated yet
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int H = nh * kDh;
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sK = smem + kOffK;
  uint8_t* sV = smem + kOffV;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t nq = 0, nk = 0, nv = 0;
      bool ok = true;
      for (int g = blockIdx.x; g < n_items && ok; g += gridDim.x) {
        const Item it = decode(sch, g);
        {
          const uint32_t qb = nq & 1u;
          if (!mbar_wait_bounded(&q_empty[qb], ((nq >> 1) & 1u) ^ 1u, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(&q_full[qb], kTile);
          tma_load_2d(sQ + qb * kTile, &tm, &q_full[qb], it.h * kDh, it.c0 + it.q0);
          ++nq;
        }
        const int nt = I8 ? 2 * it.ntiles : it.ntiles;   // int8: K for both passes, V for the second
        for (int t = 0; t < nt; ++t) {
          const int j = t < it.ntiles ? t : t - it.ntiles;
          const uint32_t kb = nk & 1u;
          if (!mbar_wait_bounded(&k_empty[kb], ((nk >> 1) & 1u) ^ 1u, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(&k_full[kb], kTile);
          tma_load_2d(sK + kb * kTile, &tm, &k_full[kb], H + it.h * kDh, it.c0 + j * kT);
          ++nk;
          if (I8 && t < it.ntiles) continue;
          const uint32_t vb = nv & 1u;
          if (!mbar_wait_bounded(&v_empty[vb], ((nv >> 1) & 1u) ^ 1u, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(&v_full[vb], kTile);
          tma_load_2d(sV + vb * kTile, &tm, &v_full[vb], 2 * H + it.h * kDh, it.c0 + j * kT);
          ++nv;
        }
      }
      if (!ok) {
        set_device_error(err, RPP_DERR_TIMEOUT);
        *abort_flag = 1;
      }
      // the copies still in flight land before the CTA can exit: the last load into
      // each buffer (at most one outstanding phase per buffer)
      for (uint32_t i = nq > 2 ? nq - 2 : 0; i < nq; ++i) mbar_wait_bounded(&q_full[i & 1u], (i >> 1) & 1u, nullptr);
      for (uint32_t i = nk > 2 ? nk - 2 : 0; i < nk; ++i) mbar_wait_bounded(&k_full[i & 1u], (i >> 1) & 1u, nullptr);
      for (uint32_t i = nv > 2 ? nv - 2 : 0; i < nv; ++i) mbar_wait_bounded(&v_full[i & 1u], (i >> 1) & 1u, nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr int fmt = Fmt<T>::v;
      constexpr uint32_t IDESC_O = idesc_f16(fmt, kT, kDh) | (1u << 16);   // B (= V) MN-major
      const uint32_t d_s = tmem_base + kColS;
      const uint32_t d_o = tmem_base + kColO;
      const uint32_t a_p = tmem_base + kColP;
      uint32_t nq = 0, nk = 0, nv = 0, ns = 0, npv = 0, nit = 0;
      bool ok = true;
      // O += P_j V_j for tile j of the current item
      auto issue_pv = [&](const Item& it, int j) -> bool {
        if (!mbar_wait_bounded(p_full, npv & 1u, abort_flag)) return false;
        const uint32_t vb = nv & 1u;
        if (!mbar_wait_bounded(&v_full[vb], (nv >> 1) & 1u, abort_flag)) return false;
        if (j == 0 && nit > 0 && !mbar_wait_bounded(o_free, (nit - 1) & 1u, abort_flag)) return false;
        tc_fence_after();
        const int kvalid = min(kT, it.len - j * kT);
        const int ksteps = (kvalid + 15) >> 4;
        const uint64_t vdesc = sw128_kmajor_desc(smem_u32(sV + vb * kTile));
        for (int k = 0; k < ksteps; ++k)   // 16 keys: P columns +8, V rows +16 (two 8-row atoms, 2048 bytes)
          tc_mma_f16_tmem_a(d_o, a_p + 8u * k, vdesc + 128u * k, IDESC_O, (j | k) ? 1u : 0u);
        tc_commit(&v_empty[vb]);
        tc_commit(pv_done);
        ++nv;
        ++npv;
        return true;
      };
      // One stream of tiles across this CTA's items: S_{t+1} is issued before P_t V_t, also
      // when tile t + 1 belongs to the next item, so the next item's scores are ready by
      // the time the softmax warps have finished the current item.
      int gs = blockIdx.x, js = 0;                  // the S cursor: item index and tile
      Item its = decode(sch, gs);                   // (blockIdx.x < n_items here)
      bool has_s = true, pend = false;              // pend: a tile whose S is issued and P V is not
      Item itp = its;
      int jp = 0;
      uint64_t qdesc = 0;
      while (ok && (has_s || pend)) {
        if (has_s) {
          if (js == 0) {
            if (!mbar_wait_bounded(&q_full[nq & 1u], (nq >> 1) & 1u, abort_flag)) { ok = false; break; }
            qdesc = sw128_kmajor_desc(smem_u32(sQ + (nq & 1u) * kTile));
          }
          const int jk = (I8 && js >= its.ntiles) ? js - its.ntiles : js;   // key tile of this S
          const int nvalid = min(kT, its.len - jk * kT);
          const uint32_t idesc_s = idesc_f16(fmt, kT, (nvalid + 15) & ~15);
          const uint32_t kb = nk & 1u;
          if (!mbar_wait_bounded(&k_full[kb], (nk >> 1) & 1u, abort_flag)) { ok = false; break; }
          if (ns > 0 && !mbar_wait_bounded(s_free, (ns - 1) & 1u, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint64_t kdesc = sw128_kmajor_desc(smem_u32(sK + kb * kTile));
#pragma unroll
          for (int k = 0; k < kDh / 16; ++k) tc_mma_f16(d_s, qdesc + 2u * k, kdesc + 2u * k, idesc_s, k ? 1u : 0u);
          tc_commit(s_full);
          tc_commit(&k_empty[kb]);
          ++nk;
          ++ns;
          if (js == (I8 ? 2 * its.ntiles : its.ntiles) - 1) {
            tc_commit(&q_empty[nq & 1u]);
            ++nq;
          }
        }
        if (pend && !issue_pv(itp, jp)) { ok = false; break; }
        if (pend && jp == itp.ntiles - 1) ++nit;
        // the tile just issued waits for its P V (int8: second-pass tiles only)
        pend = has_s && (!I8 || js >= its.ntiles);
        if (has_s) {   // advance the S cursor
          if (pend) {
            itp = its;
            jp = js - (I8 ? its.ntiles : 0);
          }
          if (++js == (I8 ? 2 * its.ntiles : its.ntiles)) {
            js = 0;
            gs += gridDim.x;
            has_s = gs < n_items;
            if (has_s) its = decode(sch, gs);
          }
        }
      }
      if (!ok) {
        set_device_error(err, RPP_DERR_TIMEOUT);
        *abort_flag = 1;
      }
      // every MMA issued by this thread completes before tensor memory is released
      tc_commit(drain);
      mbar_wait_bounded(drain, 0, nullptr);
    }
  } else {
    // ------------------------------------------------------------ softmax: two warps per row block
    // Warps 2..9: lane quadrant q = warp & 3 holds query rows 32 q .. 32 q + 31 in tensor
    // memory; half hf = 0 (warps 2..5) takes keys [0, 64) of each tile, hf = 1 (warps
    // 6..9) keys [64, 128).  The two warps of a quadrant meet once per tile to agree on
    // the row maximum, and once per item to add their row sums.
    const int quad = warp & 3;
    const int hf = (warp - 2) >> 2;
    const int r = quad * 32 + lane;                  // query row of the item
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
    const uint32_t col_s = kColS + 64 * hf, col_p = kColP + 32 * hf, col_o = kColO + 32 * hf;
    uint32_t ns = 0, npv = 0, nit = 0, nx = 0;       // S tiles, P V products, items, pair exchanges
    bool ok = true;
    // exchange with the other warp of this quadrant: value v of row r in, the partner's out
    auto exchange = [&](float v, float& other) -> bool {
      const uint32_t par = nx & 1u;
      xval[(par * 2 + hf) * kT + r] = v;
      __syncwarp();
      if (lane == 0) mbar_arrive(&xbar[quad]);
      const int w = mbar_wait_bounded(&xbar[quad], par, abort_flag) ? 1 : 0;
      ++nx;
      if (!__all_sync(0xffffffffu, w)) return false;
      other = xval[(par * 2 + (hf ^ 1)) * kT + r];
      return true;
    };
    // scores are scaled by `scale` in log2 units: log2(e) / sqrt(d), times s_q s_k for codes
    float scale = scale_log2, o_scale = 0.f;
    if constexpr (I8) {
      scale = scale_log2 * __ldg(i8_scales) * __ldg(i8_scales + 1);
      o_scale = __ldg(i8_scales + 2) / 127.0f;
    }
    float inv_so = 0.f;   // 1 / s_o for the output codes
    if constexpr (QO) inv_so = __fdiv_rn(1.0f, __ldg(out_scale));
    // this half's row maximum of S (keys past the sequence: -inf), in raw score units
    auto half_max = [&](int nv_h) -> float {
      float pm[4] = {neg_inf(), neg_inf(), neg_inf(), neg_inf()};
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        if (32 * c < nv_h) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(t_lane + col_s + 32 * c, v);
          tmem_ld_wait_tied32(v);
          if (32 * c + 32 > nv_h) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (32 * c + e >= nv_h) v[e] = 0xff800000u;
          }
#pragma unroll
          for (int e = 0; e < 32; e += 8)
#pragma unroll
            for (int t = 0; t < 4; ++t)
              pm[t] = fmaxf(fmaxf(pm[t], __uint_as_float(v[e + t])), __uint_as_float(v[e + t + 4]));
        }
      }
      return fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3]));
    };
    // Second read of this half of S: 2^(s scale - m) for its keys, 32 per chunk, with
    // packed fp32 pairs for the scale and the sum (keys past the sequence give 0).
    // MODE 0: P rounded to the input type, written to tensor memory; returns the sum.
    // MODE 1: the sum only.  MODE 2: P's int8 codes clamp(rne(127 P inv_l), 0, 127).
    auto half_exp = [&](int nv_h, float m, float inv_l, auto mode_tag) -> float {
      constexpr int MODE = decltype(mode_tag)::value;
      const uint64_t sc2 = f2_pack(scale, scale);
      const uint64_t nm2 = f2_pack(-m, -m);
      uint64_t psum2[2] = {0ull, 0ull};
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        if (32 * c < nv_h) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(t_lane + col_s + 32 * c, v);
          tmem_ld_wait_tied32(v);
          if (32 * c + 32 > nv_h) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (32 * c + e >= nv_h) v[e] = 0xff800000u;
          }
#pragma unroll
          for (int e2 = 0; e2 < 16; ++e2) {   // pair e2 is written after keys 2 e2, 2 e2 + 1 are read
            const uint64_t x2 =
                f2_fma(f2_pack(__uint_as_float(v[2 * e2]), __uint_as_float(v[2 * e2 + 1])), sc2, nm2);
            float p0 = ex2_approx(f2_lo(x2));
            float p1 = ex2_approx(f2_hi(x2));
            if constexpr (MODE == 2) {
              p0 = fminf(rintf(p0 * inv_l * 127.0f), 127.0f);
              p1 = fminf(rintf(p1 * inv_l * 127.0f), 127.0f);
            } else {
              psum2[e2 & 1] = f2_add(psum2[e2 & 1], f2_pack(p0, p1));
            }
            if constexpr (MODE != 1) v[e2] = pack2<T>(p0, p1);
          }
          if constexpr (MODE != 1) {
            tmem_st_32x32b_x16(t_lane + col_p + 16 * c, v);
            tmem_st_wait_tied16(v);
          }
        }
      }
      return (f2_lo(psum2[0]) + f2_hi(psum2[0])) + (f2_lo(psum2[1]) + f2_hi(psum2[1]));
    };
    for (int g = blockIdx.x; g < n_items && ok; g += gridDim.x) {
      const Item it = decode(sch, g);
      const bool active = it.q0 + quad * 32 < it.len;   // the same for both warps of the quadrant
      float m = neg_inf(), l = 0.f;                     // l: this warp's half of the row sum
      float inv_l = 0.f;                                // int8: 1 / the whole row sum
      const int nt = I8 ? 2 * it.ntiles : it.ntiles;
      int jb = 0;                                       // P V products of this item so far
      for (int t = 0; t < nt; ++t) {
        const bool stats = I8 && t < it.ntiles;          // int8 first pass: maxima and sums only
        const int j = t < it.ntiles ? t : t - it.ntiles; // key tile
        const int nvalid = min(kT, it.len - j * kT);
        const int nv_h = min(64, max(0, nvalid - 64 * hf));   // keys of this half inside the sequence
        int w = mbar_wait_bounded(s_full, ns & 1u, abort_flag) ? 1 : 0;
        if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
        tc_fence_after();
        float mx = neg_inf();
        if (active && (!I8 || stats)) {
          mx = half_max(nv_h);
          float other;
          if (!exchange(mx, other)) { ok = false; break; }
          mx = fmaxf(mx, other) * scale;
        }
        // P and O: the previous P V must be done before P is rewritten or O rescaled (every
        // warp waits, active or not: p_full counts one arrival per warp, and a warp that
        // arrived for the next tile before another warp arrived for this one would
        // complete this tile's phase early)
        if (!stats && jb > 0) {
          w = mbar_wait_bounded(pv_done, (npv - 1) & 1u, abort_flag) ? 1 : 0;
          if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
          tc_fence_after();
        }
        if (active) {
          if constexpr (!I8) {
            if (j == 0) {
              m = mx;
            } else {
              // lazy rescaling, decided alike by both warps of the quadrant (same rows,
              // same maxima); the tensor-memory accesses are warp-collective
              const bool move = mx > m + 8.0f;
              if (__any_sync(0xffffffffu, move)) {
                const float alpha = move ? ex2_approx(m - mx) : 1.0f;
#pragma unroll 1
                for (int q2 = 0; q2 < 2; ++q2) {   // this warp's 32 columns of O
                  uint32_t ov[16];
                  tmem_ld_32x32b_x16(t_lane + col_o + 16 * q2, ov);
                  tmem_ld_wait_tied16(ov);
#pragma unroll
                  for (int e = 0; e < 16; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                  tmem_st_32x32b_x16(t_lane + col_o + 16 * q2, ov);
                  tmem_st_wait_tied16(ov);
                }
                if (move) {
                  l *= alpha;
                  m = mx;
                }
              }
            }
            l += half_exp(nv_h, m, 0.f, std::integral_constant<int, 0>{});
          } else if (stats) {
            // the reference maximum moves lazily as above (no O yet: only the sum rescales)
            if (j == 0) {
              m = mx;
            } else if (mx > m + 8.0f) {
              l *= ex2_approx(m - mx);
              m = mx;
            }
            l += half_exp(nv_h, m, 0.f, std::integral_constant<int, 1>{});
            if (j == it.ntiles - 1) {   // end of the first pass: the whole row sum
              float other;
              if (!exchange(l, other)) { ok = false; break; }
              inv_l = 1.0f / (l + other);
            }
          } else {
            half_exp(nv_h, m, inv_l, std::integral_constant<int, 2>{});
          }
        }
        // S has been read by this warp
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_free);
        ++ns;
        if (stats) continue;
        // the last 16-key step of a partial tile: zero the V rows past the sequence
        // (P is 0 there, but 0 * NaN would not be); one warp of each quadrant does it
        const int kpad = ((nvalid + 15) & ~15);
        if (hf == 0 && nvalid < kpad && r >= nvalid && r < kpad) {
          const uint32_t vb = npv & 1u;   // V tile j is the npv-th V load of this CTA
          if (mbar_wait_bounded(&v_full[vb], (npv >> 1) & 1u, abort_flag)) {
            uint8_t* vrow = sV + vb * kTile + r * 128;
#pragma unroll
            for (int u = 0; u < 8; ++u) *reinterpret_cast<uint4*>(vrow + (((u + r) & 7) << 4)) = make_uint4(0u, 0u, 0u, 0u);
            fence_proxy_async_smem();
          } else {
            ok = false;
          }
        }
        if (!__all_sync(0xffffffffu, ok ? 1 : 0)) { ok = false; break; }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);
        ++npv;
        ++jb;
      }
      if (!ok) break;
      // the item's O: wait for its last P V; float: add the two halves of the row sum and
      // scale by 1 / sum; int8: P was normalised, O scales by s_v / 127
      int w = mbar_wait_bounded(pv_done, (npv - 1) & 1u, abort_flag) ? 1 : 0;
      if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
      tc_fence_after();
      if (active) {
        float inv = o_scale;
        if constexpr (!I8) {
          float other;
          if (!exchange(l, other)) { ok = false; break; }
          inv = 1.0f / (l + other);
        }
        uint32_t ov[32];
        tmem_ld_32x32b_x32(t_lane + col_o, ov);
        tmem_ld_wait_tied32(ov);
        if (it.q0 + r < it.len) {
          uint4* orow = reinterpret_cast<uint4*>(out + static_cast<long long>(it.c0 + it.q0 + r) * H + it.h * kDh +
                                                 32 * hf);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              f[e] = __uint_as_float(ov[8 * u + e]) * inv;
              if constexpr (QO) f[e] = code_of(f[e], inv_so);
            }
            orow[u] = make_uint4(pack2<TOut>(f[0], f[1]), pack2<TOut>(f[2], f[3]), pack2<TOut>(f[4], f[5]),
                                 pack2<TOut>(f[6], f[7]));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free);
      ++nit;
    }
    if (!ok && lane == 0) {
      set_device_error(err, RPP_DERR_TIMEOUT);
      *abort_flag = 1;
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

bool attention_sched_supported(int B, int max_len) {
  return B >= 1 && B <= kMaxB && max_len >= 1 && (max_len + kT - 1) / kT <= kMaxCls;
}

namespace {

template <typename T, bool I8, bool QO>
cudaError_t launch_sched(const CUtensorMap& tm, const int32_t* cu, int B, int T_max, int max_len, int nh, void* out,
                         const float* i8_scales, const float* out_scale, int32_t* err, cudaStream_t stream) {
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(kDh));
  const int n_cls = (max_len + kT - 1) / kT;
  // persistent: two CTAs per SM, never more CTAs than the largest possible item count
  const long long max_items = static_cast<long long>(B) * nh * n_cls;
  const int grid = static_cast<int>(max_items < 2LL * num_sms() ? max_items : 2LL * num_sms());
  const size_t smem = smem_bytes(B);
  static size_t attr = 0;
  if (attr < smem) {
    cudaError_t e = cudaFuncSetAttribute(attention_sched_kernel<T, I8, QO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem_bytes(kMaxB)));
    if (e != cudaSuccess) return e;
    attr = smem_bytes(kMaxB);
  }
  return launch_pdl(attention_sched_kernel<T, I8, QO>, dim3(grid), dim3(kThreads), smem, stream, tm, cu, B, T_max,
                    max_len, nh, n_cls, out, scale_log2, i8_scales, out_scale, err);
}

}  // namespace

cudaError_t launch_attention_sched(const void* qkv, const int32_t* cu, int B, int T_max, int max_len, int nh,
                                   rpp_dtype dtype, void* out, int32_t* err, cudaStream_t stream,
                                   const float* i8_scales, const float* out_scale) {
  if (B <= 0 || max_len <= 0 || T_max <= 0) return cudaSuccess;
  if (dtype != RPP_F16 && dtype != RPP_BF16) return cudaErrorNotSupported;
  if (i8_scales && dtype != RPP_BF16) return cudaErrorNotSupported;   // codes are held in bf16
  if (!attention_sched_supported(B, max_len)) return cudaErrorNotSupported;
  const int H = nh * kDh;
  CUtensorMap tm;
  const CUtensorMapDataType dt = dtype == RPP_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  if (!make_tmap_2d(&tm, qkv, dt, 2, T_max, 3 * H, kT, kDh, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
  const float* q = i8_scales;
  const float* so = out_scale;
  if (q && so) return launch_sched<__nv_bfloat16, true, true>(tm, cu, B, T_max, max_len, nh, out, q, so, err, stream);
  if (q) return launch_sched<__nv_bfloat16, true, false>(tm, cu, B, T_max, max_len, nh, out, q, so, err, stream);
  if (dtype == RPP_F16) {
    if (so) return launch_sched<__half, false, true>(tm, cu, B, T_max, max_len, nh, out, q, so, err, stream);
    return launch_sched<__half, false, false>(tm, cu, B, T_max, max_len, nh, out, q, so, err, stream);
  }
  if (so) return launch_sched<__nv_bfloat16, false, true>(tm, cu, B, T_max, max_len, nh, out, q, so, err, stream);
  return launch_sched<__nv_bfloat16, false, false>(tm, cu, B, T_max, max_len, nh, out, q, so, err, stream);
}

}  // namespace rpp
