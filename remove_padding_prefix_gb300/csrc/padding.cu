// Offset mask, padding removal and rebuild ('GPU底層優化 | 如何讓Transformer在GPU上跑得更快？',
// Fig. 9: an Offset Mask converts between the padded and the padding-removed batch).
//
// The offset builder is one CTA: a block-wide exclusive scan of the lengths followed
// by a cooperative fill of padding_offset.  Removal and rebuild are flat 16-byte
// vector copies over (row, vector) pairs with a grid-stride loop; the number of valid
// rows T = cu_seqlens[B] is read on the device so no host synchronisation is needed.
#include "kernels.h"

namespace rpp {

namespace {

constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kScanThreads) build_offsets_kernel(const int32_t* __restrict__ lengths, int B,
                                                                     int L, int32_t* __restrict__ cu,
                                                                     int32_t* __restrict__ padding_offset,
                                                                     int32_t* err) {
  pdl_wait();
  pdl_trigger();
  __shared__ int32_t warp_sums[kScanThreads / 32];
  __shared__ int32_t s_carry;
  const int tid = threadIdx.x;
  if (tid == 0) s_carry = 0;
  __syncthreads();
  // chunked block scan: each pass handles kScanThreads lengths
  for (int base = 0; base < B; base += kScanThreads) {
    const int b = base + tid;
    int32_t v = 0;
    if (b < B) {
      v = lengths[b];
      if (v < 0 || v > L) {
        set_device_error(err, RPP_DERR_LENGTH);
        v = v < 0 ? 0 : L;
      }
    }
    // inclusive warp scan
    int32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
      if ((tid & 31) >= o) x += y;
    }
    if ((tid & 31) == 31) warp_sums[tid >> 5] = x;
    __syncthreads();
    if (tid < 32) {
      int32_t w = warp_sums[tid];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
        if (tid >= o) w += y;
      }
      warp_sums[tid] = w;   // inclusive over warps
    }
    __syncthreads();
    const int32_t carry = s_carry;
    const int32_t incl = x + ((tid >> 5) ? warp_sums[(tid >> 5) - 1] : 0) + carry;
    if (b < B) cu[b + 1] = incl;
    if (b == 0) cu[0] = 0;
    __syncthreads();
    if (tid == kScanThreads - 1) s_carry = incl;
    __syncthreads();
  }
  __syncthreads();
  // padding_offset[i] = b*L - cu[b] for i in [cu[b], cu[b+1]); one pass over the (b, p) slots
  const long long slots = static_cast<long long>(B) * L;
  for (long long s = tid; s < slots; s += kScanThreads) {
    const int b = static_cast<int>(s / L);
    const int p = static_cast<int>(s - static_cast<long long>(b) * L);
    const int32_t c0 = cu[b];
    const int32_t len = cu[b + 1] - c0;
    if (p < len) padding_offset[c0 + p] = b * L - c0;
  }
}

// packed[i] = padded[i + po[i]] for i < T; VPR 16-byte vectors per row
__global__ void remove_padding_kernel(const uint4* __restrict__ padded, const int32_t* __restrict__ po,
                                      const int32_t* __restrict__ cu, int B, int T_max, int vpr,
                                      uint4* __restrict__ packed, int32_t* err) {
  pdl_wait();
  pdl_trigger();
  if (device_error_set(err)) return;
  int T = cu[B];
  if (T > T_max || T < 0) {
    set_device_error(err, RPP_DERR_ROWS);
    return;
  }
  const long long total = static_cast<long long>(T) * vpr;
  for (long long v = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; v < total;
       v += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int row = static_cast<int>(v / vpr);
    const int c = static_cast<int>(v - static_cast<long long>(row) * vpr);
    const int src_row = row + po[row];
    if (src_row < 0 || src_row >= T_max) {   // offsets inconsistent with cu_seqlens
      set_device_error(err, RPP_DERR_ROWS);
      continue;
    }
    packed[v] = __ldg(padded + static_cast<long long>(src_row) * vpr + c);
  }
}

// padded[b*L + p] = p < len_b ? packed[cu[b] + p] : 0
__global__ void rebuild_padding_kernel(const uint4* __restrict__ packed, const int32_t* __restrict__ cu, int B,
                                       int L, int vpr, uint4* __restrict__ padded, int32_t* err) {
  pdl_wait();
  pdl_trigger();
  if (device_error_set(err)) return;
  const long long total = static_cast<long long>(B) * L * vpr;
  for (long long v = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; v < total;
       v += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = v / vpr;
    const int c = static_cast<int>(v - row * vpr);
    const int b = static_cast<int>(row / L);
    const int p = static_cast<int>(row - static_cast<long long>(b) * L);
    const int32_t c0 = cu[b];
    const int32_t len = cu[b + 1] - c0;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (p < len) val = __ldg(packed + (static_cast<long long>(c0) + p) * vpr + c);
    padded[v] = val;
  }
}

// Offsets and removal in one launch (B <= kFusedMaxB): every CTA scans the lengths
// itself in shared memory -- B is small, so the redundant scan costs less than a
// second launch -- then copies its share of the valid padded rows to their packed
// slots and writes their padding offsets; CTA 0 also writes cu_seqlens.
constexpr int kFusedMaxB = 1024;
constexpr int kFusedThreads = 256;

__global__ void __launch_bounds__(kFusedThreads) offsets_remove_kernel(const int32_t* __restrict__ lengths, int B,
                                                                       int L, int vpr, const uint4* __restrict__ padded,
                                                                       int32_t* __restrict__ cu,
                                                                       int32_t* __restrict__ po,
                                                                       uint4* __restrict__ packed, int32_t* err) {
  pdl_wait();
  pdl_trigger();
  __shared__ int32_t s_cu[kFusedMaxB + 1];
  __shared__ int32_t s_warp[kFusedThreads / 32];
  const int tid = threadIdx.x;
  const bool err_before = device_error_set(err);   // read with the lengths, checked after the scan
  constexpr int PER = kFusedMaxB / kFusedThreads;   // lengths per thread
  int32_t v[PER];
  int32_t run = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int b = tid * PER + j;
    int32_t len = 0;
    if (b < B) {
      len = lengths[b];
      if (len < 0 || len > L) {
        if (blockIdx.x == 0) set_device_error(err, RPP_DERR_LENGTH);
        len = len < 0 ? 0 : L;
      }
    }
    run += len;
    v[j] = run;   // inclusive within the thread
  }
  // exclusive scan of the per-thread totals across the block
  int32_t x = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t t = __shfl_up_sync(0xffffffffu, x, o);
    if ((tid & 31) >= o) x += t;
  }
  if ((tid & 31) == 31) s_warp[tid >> 5] = x;
  __syncthreads();
  if (tid < 32) {
    int32_t w = tid < kFusedThreads / 32 ? s_warp[tid] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t t = __shfl_up_sync(0xffffffffu, w, o);
      if (tid >= o) w += t;
    }
    if (tid < kFusedThreads / 32) s_warp[tid] = w;
  }
  __syncthreads();
  const int32_t base = x - run + ((tid >> 5) ? s_warp[(tid >> 5) - 1] : 0);
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int b = tid * PER + j;
    if (b < B) s_cu[b + 1] = base + v[j];
  }
  if (tid == 0) s_cu[0] = 0;
  __syncthreads();
  if (blockIdx.x == 0)
    for (int b = tid; b <= B; b += kFusedThreads) cu[b] = s_cu[b];
  if (err_before) return;
  // one warp per packed row j: its sequence b is found by binary search in the scan,
  // the row's 16-byte vectors are read (up to 8 per lane in flight) and written
  const int T = s_cu[B];
  const int lane = tid & 31;
  const int warps = gridDim.x * (kFusedThreads / 32);
  for (int j = blockIdx.x * (kFusedThreads / 32) + (tid >> 5); j < T; j += warps) {
    int lo = 0, hi = B;   // largest b with s_cu[b] <= j (and s_cu[b + 1] > j)
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_cu[mid] <= j) lo = mid; else hi = mid;
    }
    const int b = lo;
    const int c0 = s_cu[b];
    const uint4* src = padded + (static_cast<long long>(b) * L + (j - c0)) * vpr;
    uint4* dst = packed + static_cast<long long>(j) * vpr;
    for (int c = lane; c < vpr; c += 32 * 8) {
      uint4 t[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (c + 32 * u < vpr) t[u] = __ldg(src + c + 32 * u);
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (c + 32 * u < vpr) dst[c + 32 * u] = t[u];
    }
    if (lane == 0) po[j] = b * L - c0;
  }
}

}  // namespace

bool offsets_remove_fusable(int B) { return B > 0 && B <= kFusedMaxB; }

cudaError_t launch_offsets_remove(const int32_t* lengths, int B, int L, int row_bytes, const void* padded,
                                  int32_t* cu, int32_t* po, void* packed, int32_t* err, cudaStream_t stream) {
  if (!offsets_remove_fusable(B)) return cudaErrorNotSupported;
  const int vpr = row_bytes / 16;
  // a warp per packed row, at most B * L rows
  long long blocks = (static_cast<long long>(B) * L + kFusedThreads / 32 - 1) / (kFusedThreads / 32);
  const long long cap = static_cast<long long>(num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_pdl(offsets_remove_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kFusedThreads), 0, stream,
                    lengths, B, L, vpr, static_cast<const uint4*>(padded), cu, po, static_cast<uint4*>(packed), err);
}

cudaError_t launch_build_offsets(const int32_t* lengths, int B, int L, int32_t* cu, int32_t* po, int32_t* err,
                                 cudaStream_t stream) {
  return launch_pdl(build_offsets_kernel, dim3(1), dim3(kScanThreads), 0, stream, lengths, B, L, cu, po, err);
}

cudaError_t launch_remove_padding(const void* padded, const int32_t* po, const int32_t* cu, int B, int L,
                                  int row_bytes, void* packed, int32_t* err, cudaStream_t stream) {
  const int vpr = row_bytes / 16;
  const long long total = static_cast<long long>(B) * L * vpr;
  const int threads = 256;
  long long blocks = (total + threads - 1) / threads;
  const long long cap = static_cast<long long>(num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_pdl(remove_padding_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream,
                    static_cast<const uint4*>(padded), po, cu, B, B * L, vpr, static_cast<uint4*>(packed), err);
}

cudaError_t launch_rebuild_padding(const void* packed, const int32_t* cu, int B, int L, int row_bytes,
                                   void* padded, int32_t* err, cudaStream_t stream) {
  const int vpr = row_bytes / 16;
  const long long total = static_cast<long long>(B) * L * vpr;
  const int threads = 256;
  long long blocks = (total + threads - 1) / threads;
  const long long cap = static_cast<long long>(num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_pdl(rebuild_padding_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream,
                    static_cast<const uint4*>(packed), cu, B, L, vpr, static_cast<uint4*>(padded), err);
}

}  // namespace rpp
