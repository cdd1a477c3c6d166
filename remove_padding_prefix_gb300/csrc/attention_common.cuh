// Pieces shared by the tensor-core varlen attention kernels: tile sizes, the
// longest-first item list built from cu_seqlens, 16-bit packing of P, and the MMA form
// whose A operand (P) lives in tensor memory.
//
// Work items are (sequence, head, 128-query tile); an item's cost is its sequence's
// number of 128-key tiles.  Every CTA builds the same list in its prologue: sequences
// grouped by tile count, largest first, stable within a group, items of a sequence in
// (head, q-tile) order.  The q-tiles of one (sequence, head) are neighbours, so the CTAs
// that share its K and V tiles run at the same time and read them from L2 (the Kuaishou
// article, Fig. 10: attention is the kernel that needs the sequence bounds of the
// padding-free batch).
#pragma once
#include "kernels.h"

namespace rpp {
namespace attn {

constexpr int kT = 128;                        // queries per item, keys per tile
constexpr int kDh = 64;                        // head size
constexpr uint32_t kTile = kT * kDh * 2;       // one 128 x 64 tile of Q, K or V (16 KB)
constexpr int kMaxCls = 64;                    // tiles per sequence: max_len <= 8192
constexpr int kMaxB = 2048;                    // sequences per batch

// shared-memory bytes of the item-list arrays: 4 int arrays of kMaxCls + 2, int16 perm[B],
// cu_seqlens int32[B + 1]
__host__ __device__ constexpr uint32_t perm_bytes(int B) { return (static_cast<uint32_t>(B) * 2u + 15u) & ~15u; }
__host__ __device__ constexpr uint32_t cls_bytes() { return 4u * (kMaxCls + 2) * 4u; }
__host__ __device__ constexpr uint32_t sched_bytes(int B) {
  return cls_bytes() + perm_bytes(B) + ((static_cast<uint32_t>(B + 1) * 4u + 15u) & ~15u);
}

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

template <typename T> struct Fmt;
template <> struct Fmt<__half> { static constexpr int v = 0; };
template <> struct Fmt<__nv_bfloat16> { static constexpr int v = 1; };

template <typename T>
__device__ __forceinline__ uint32_t pack2(float a, float b);   // a -> low half (the even key)
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

// D[tmem] (+)= A[tmem] * B[smem], kind::f16: A (M x K, one row per lane, two 16-bit
// elements per 32-bit column) from tensor memory
__device__ __forceinline__ void tc_mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

struct Sched {
  const int* item_off;   // [c]: first item of tile count c (c = n_cls .. 1), item_off[0] = total
  const int* seq_off;    // [c]: first position in perm of the sequences with c tiles
  const int16_t* perm;   // sequence indices, grouped
  const int* cu;         // cu_seqlens, copied into shared memory
  int n_cls, nh;
};
struct Item {
  int b, h, q0, c0, len, ntiles;
};
__device__ __forceinline__ Item decode(const Sched& s, int g) {
  int c = s.n_cls;
  while (c > 1 && g >= s.item_off[c - 1]) --c;   // classes laid out n_cls, n_cls - 1, ...: item_off decreasing in c
  // g lies in class c: [item_off[c], item_off[c - 1])
  const int idx = g - s.item_off[c];
  const int per_seq = s.nh * c;
  const int sq = idx / per_seq;
  const int rem = idx - sq * per_seq;
  Item it;
  it.b = s.perm[s.seq_off[c] + sq];
  it.h = rem / c;
  it.q0 = (rem - it.h * c) * kT;
  it.c0 = s.cu[it.b];
  it.len = s.cu[it.b + 1] - it.c0;
  it.ntiles = c;
  return it;
}

// Builds the item list in shared memory (`sched` points at sched_bytes(B) bytes).  Called
// by every thread of the CTA (it holds __syncthreads).  Returns false when the CTA must
// quit: an error word already set, or bad sequence bounds (recorded in err).
__device__ __forceinline__ bool build_items(const int32_t* __restrict__ cu, int B, int T_max, int max_len, int nh,
                                            int n_cls, int32_t* err, int* s_status, uint8_t* sched, Sched& out) {
  int* cls_cnt = reinterpret_cast<int*>(sched);
  int* seq_off = cls_cnt + (kMaxCls + 2);
  int* item_off = seq_off + (kMaxCls + 2);
  int* cursor = item_off + (kMaxCls + 2);
  int16_t* perm = reinterpret_cast<int16_t*>(sched + cls_bytes());
  int* s_cu = reinterpret_cast<int*>(sched + cls_bytes() + perm_bytes(B));
  const int nthreads = blockDim.x;
  if (threadIdx.x == 0) *s_status = device_error_set(err) ? -1 : 0;   // -1: quit without recording
  for (int c = threadIdx.x; c < kMaxCls + 2; c += nthreads) cls_cnt[c] = 0;
  __syncthreads();
  if (*s_status) return false;
  for (int b = threadIdx.x; b <= B; b += nthreads) s_cu[b] = __ldg(cu + b);
  __syncthreads();
  for (int b = threadIdx.x; b < B; b += nthreads) {
    const int c0 = s_cu[b], c1 = s_cu[b + 1], len = c1 - c0;
    if (c0 < 0 || len < 0 || c1 > T_max || len > max_len) {
      atomicCAS(s_status, 0, len > max_len ? RPP_DERR_LENGTH : RPP_DERR_ROWS);
    } else {
      atomicAdd(&cls_cnt[(len + kT - 1) / kT], 1);
    }
  }
  __syncthreads();
  if (*s_status) {
    if (threadIdx.x == 0 && *s_status > 0) set_device_error(err, *s_status);
    return false;
  }
  if (threadIdx.x == 0) {
    int so = 0, io = 0;
    for (int c = n_cls; c >= 1; --c) {   // largest tile count first
      seq_off[c] = so;
      item_off[c] = io;
      cursor[c] = so;
      so += cls_cnt[c];
      io += cls_cnt[c] * nh * c;
    }
    item_off[0] = io;   // the total, which is also where class 1 ends
  }
  __syncthreads();
  if (threadIdx.x < 32) {   // a stable grouping by tile count, 32 sequences at a time
    const int lane = threadIdx.x;
    for (int b0 = 0; b0 < B; b0 += 32) {
      const int b = b0 + lane;
      int c = -1;
      if (b < B) c = (s_cu[b + 1] - s_cu[b] + kT - 1) / kT;
      const unsigned peers = __match_any_sync(0xffffffffu, c);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      if (c > 0) perm[cursor[c] + rank] = static_cast<int16_t>(b);
      __syncwarp();
      if (c > 0 && rank == 0) cursor[c] += __popc(peers);
      __syncwarp();
    }
  }
  out = Sched{item_off, seq_off, perm, s_cu, n_cls, nh};
  return true;
}

}  // namespace attn
}  // namespace rpp
