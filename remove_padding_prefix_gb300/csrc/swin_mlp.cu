// Swin MLP on the tensor cores, fused: out = y + FC2(GELU(FC1(h) + b1)) + b2 for the
// stage-1 width C = 96 (hidden F = 4C = 384), h the LayerNorm-2 output and y the block's
// running sum (the residual).
//
// NVIDIA Swin talk, §3: the MLP's bias + GELU and bias + residual are fused into the
// GEMMs.  Here the two GEMMs are fused with each other as well: a 128-token tile's
// hidden activation (128 x 384) goes from tensor memory through GELU into shared memory
// as the second GEMM's A operand and never reaches HBM.  Per token the kernel reads h
// and y once and writes out once (6 C bytes in 16-bit types), against 6 C + 4 F for the
// two separate GEMMs.
//
// Persistent, one CTA per SM, 2 + EW warps (EW = 16 epilogue warps; 8 warps of twice
// the columns measured 8% slower on the Swin-T stage-1 block):
//   warp 0      TMA: W1 once (before the programmatic-launch wait -- the weights are
//               not written by the preceding kernel), each tile's h rows, and W2 one
//               64-wide K panel at a time through a two-slot ring (from L2);
//   warp 1      MMA issue (one thread): FC1 of a tile in two halves of 192 hidden
//               columns, FC2 in six 64-wide K blocks;
//   warps 2..   epilogue: per 64-column block of the hidden activation, tensor memory
//               -> registers (the next block's load issued before this block's
//               arithmetic), + b1 (staged in shared memory), GELU, fp16/bf16 -> a
//               128-byte-swizzled K-major block in shared memory; per tile, the FC2
//               accumulator + b2 + y -> out, y's rows requested a half tile ahead.
// Shared memory (bytes): W1 as six MN-major panels [96 K rows x 64 N] (73 728), two
// W2 slots, each a K-major panel [96 N rows x 64 K] (24 576), the h tile as two K-major
// atoms (the TMA zero-fills columns 96..127, 32 768), and the whole tile's hidden
// activation as six 64-column blocks (98 304): the GELU of tile i + 1 never waits for
// FC2 of tile i to release a block it has not finished with.
// Tensor memory: FC1 accumulator in columns [0, 384), FC2 accumulator in [384, 480).
//
// Order of work (i = this CTA's tile counter), chosen so that every hand-off overlaps
// other work:
//   MMA:      FC2(i, 0..2) | FC1(i+1, half 0) | FC2(i, 3..5) | FC1(i+1, half 1)
//   epilogue: G(i+1, 0..2) | F(i) | G(i+1, 3..5)
//   TMA:      W2 panels of FC2(i, 0..2) | h of tile i + 1 | W2 panels of FC2(i, 3..5)
// where G(i, b) is the GELU of hidden block b of tile i and F(i) the final epilogue.
// FC1(i+1, half h) overwrites columns the epilogue finished reading in G(i, 3h..3h+2);
// F(i) needs FC2(i, 5), issued after G(i, 5) with three blocks of work in between;
// FC2(i+1, 0) waits until F(i) has read the FC2 accumulator.  Every wait is bounded.
#include "kernels.h"

namespace rpp {

namespace {

constexpr int kMC = 96;                        // C
constexpr int kMF = 384;                       // F = 4C
constexpr int kMBM = 128;                      // tokens per tile
constexpr int kMlpEW = 16;                     // epilogue warps (8 or 16)
constexpr uint32_t kPanel = kMC * 128;         // 96 rows x 128 bytes
constexpr uint32_t kW1Bytes = 6 * kPanel;
constexpr int kW2Slots = 2;
constexpr uint32_t kW2Bytes = kW2Slots * kPanel;
constexpr uint32_t kAtom = kMBM * 128;         // 128 rows x 128 bytes
constexpr uint32_t kABytes = 2 * kAtom;
constexpr int kHBufs = 6;
constexpr uint32_t kHBytes = kAtom;
constexpr uint32_t kB1Bytes = kMF * 4;          // b1 staged once (fp32)
constexpr size_t kMlpSmem = 1024 + kW1Bytes + kW2Bytes + kABytes + kHBufs * kHBytes + kB1Bytes + 256;
constexpr uint32_t kFc2Col = kMF;              // FC2 accumulator columns [384, 480)

template <typename T> struct MlpFmt;
template <> struct MlpFmt<__half> { static constexpr int v = 0; };
template <> struct MlpFmt<__nv_bfloat16> { static constexpr int v = 1; };

template <int EW>
constexpr int mlp_threads() { return 64 + 32 * EW; }

template <typename T, int EW>
__global__ void __launch_bounds__(mlp_threads<EW>(), 1)
swin_mlp_kernel(const __grid_constant__ CUtensorMap tmH, const __grid_constant__ CUtensorMap tmW1,
                const __grid_constant__ CUtensorMap tmW2, const float* __restrict__ b1, const float* __restrict__ b2,
                const T* __restrict__ resid, T* __restrict__ out, int M, int32_t* err) {
  constexpr int fmt = MlpFmt<T>::v;
  constexpr uint32_t IDESC_FC1 = idesc_f16(fmt, kMBM, 64) | (1u << 16);   // B (W1 panel) MN-major
  constexpr uint32_t IDESC_FC2 = idesc_f16(fmt, kMBM, kMC);
  static_assert(EW == 8 || EW == 16, "two or four epilogue warps per lane quadrant");
  constexpr int WPQ = EW / 4;    // epilogue warps per tensor-memory lane quadrant
  constexpr int CW = 64 / WPQ;   // hidden columns of a 64-wide block per warp

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sW1 = smem;
  uint8_t* sW2 = sW1 + kW1Bytes;
  uint8_t* sA = sW2 + kW2Bytes;
  uint8_t* sH = sA + kABytes;
  float* sB1 = reinterpret_cast<float*>(sH + kHBufs * kHBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sH + kHBufs * kHBytes + kB1Bytes);
  uint64_t* w_full = bars;        // W1 landed
  uint64_t* a_full = bars + 1;
  uint64_t* a_empty = bars + 2;
  uint64_t* s_full = bars + 3;    // [2] FC1 half done
  uint64_t* s_empty = bars + 5;   // [2] FC1 half read by the epilogue
  uint64_t* h_full = bars + 7;    // [6] hidden block written
  uint64_t* h_empty = bars + 13;  // [6] hidden block consumed by FC2
  uint64_t* o_full = bars + 19;
  uint64_t* o_empty = bars + 20;
  uint64_t* drain = bars + 21;
  uint64_t* p_full = bars + 22;   // [2] W2 slot loaded
  uint64_t* p_empty = bars + 24;  // [2] W2 slot consumed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 26);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_quit = const_cast<int*>(abort_flag) + 1;

  const int warp = warp_id();
  const int lane = lane_id();
  if (threadIdx.x == 0) {
    mbar_init(w_full, 1);
    mbar_init(a_full, 1);
    mbar_init(a_empty, 1);
    for (int h = 0; h < 2; ++h) {
      mbar_init(&s_full[h], 1);
      mbar_init(&s_empty[h], EW);
    }
    for (int b = 0; b < kHBufs; ++b) {
      mbar_init(&h_full[b], EW);
      mbar_init(&h_empty[b], 1);
    }
    mbar_init(o_full, 1);
    mbar_init(o_empty, EW);
    mbar_init(drain, 1);
    for (int k = 0; k < kW2Slots; ++k) {
      mbar_init(&p_full[k], 1);
      mbar_init(&p_empty[k], 1);
    }
    *abort_flag = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&tmH);
    tma_prefetch_desc(&tmW1);
    tma_prefetch_desc(&tmW2);
    // the weights are prepared data, never written by the preceding kernel
    mbar_arrive_expect_tx(w_full, kW1Bytes);
    for (int j = 0; j < 6; ++j) tma_load_2d(sW1 + j * kPanel, &tmW1, w_full, 64 * j, 0);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  for (int j = threadIdx.x; j < kMF; j += blockDim.x) sB1[j] = b1[j];   // prepared data
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) *s_quit = device_error_set(err) ? 1 : 0;
  __syncthreads();
  const int tiles = (M + kMBM - 1) / kMBM;
  const int n = *s_quit ? 0 : (static_cast<int>(blockIdx.x) < tiles
                                    ? (tiles - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                                          static_cast<int>(gridDim.x)
                                    : 0);
  auto tile_of = [&](int i) { return static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x); };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int na = 0, np = 0;   // h tiles and W2 panels issued
      auto load_a = [&](int i) -> bool {
        if (i > 0 && !mbar_wait_bounded(a_empty, (i - 1) & 1, abort_flag)) return false;
        mbar_arrive_expect_tx(a_full, kABytes);
        tma_load_2d(sA, &tmH, a_full, 0, kMBM * tile_of(i));
        tma_load_2d(sA + kAtom, &tmH, a_full, 64, kMBM * tile_of(i));
        ++na;
        return true;
      };
      // W2 panel for use g = 6 i + b (panel b) into slot g % 2, once use g - 2 is done
      auto load_p = [&](int g) -> bool {
        const int slot = g % kW2Slots;
        if (g >= kW2Slots && !mbar_wait_bounded(&p_empty[slot], ((g / kW2Slots) - 1) & 1, abort_flag)) return false;
        mbar_arrive_expect_tx(&p_full[slot], kPanel);
        tma_load_2d(sW2 + slot * kPanel, &tmW2, &p_full[slot], 64 * (g % 6), 0);
        ++np;
        return true;
      };
      bool ok = n == 0 || load_a(0);
      for (int i = 0; i < n && ok; ++i) {
        for (int b = 0; b < 3 && ok; ++b) ok = load_p(6 * i + b);
        if (ok && i + 1 < n) ok = load_a(i + 1);
        for (int b = 3; b < 6 && ok; ++b) ok = load_p(6 * i + b);
      }
      if (!ok) {
        set_device_error(err, RPP_DERR_TIMEOUT);
        *abort_flag = 1;
      }
      // copies still in flight land before the CTA can exit
      mbar_wait_bounded(w_full, 0, nullptr);
      if (na > 0) mbar_wait_bounded(a_full, (na - 1) & 1, nullptr);
      for (int g = np - kW2Slots < 0 ? 0 : np - kW2Slots; g < np; ++g)
        mbar_wait_bounded(&p_full[g % kW2Slots], (g / kW2Slots) & 1, nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait_bounded(w_full, 0, abort_flag);
      const uint64_t a0 = sw128_kmajor_desc(smem_u32(sA));
      const uint64_t a1 = sw128_kmajor_desc(smem_u32(sA + kAtom));
      // FC1 half hf of tile i: hidden columns [192 hf, 192 hf + 192), three 64-wide
      // W1 panels, K = 96 in six steps of 16 (the h tile's second atom holds K 64..95)
      auto fc1 = [&](int i, int hf) -> bool {
        if (i > 0 && !mbar_wait_bounded(&s_empty[hf], (i - 1) & 1, abort_flag)) return false;
        tc_fence_after();
#pragma unroll
        for (int jj = 0; jj < 3; ++jj) {
          const int j = 3 * hf + jj;
          const uint64_t bdesc = sw128_kmajor_desc(smem_u32(sW1 + j * kPanel));
#pragma unroll
          for (int k = 0; k < kMC / 16; ++k) {
            const uint64_t adesc = (k < 4 ? a0 : a1) + 2u * (k & 3);
            // MN-major B: 16 K rows = two 8-row swizzle atoms = +2048 bytes
            tc_mma_f16(tmem_base + 64 * j, adesc, bdesc + 128u * k, IDESC_FC1, k ? 1u : 0u);
          }
        }
        tc_commit(&s_full[hf]);
        return true;
      };
      // FC2 block b of tile i: K = hidden columns [64 b, 64 b + 64) from hidden buffer
      // (6 i + b) % 3, W2 panel b
      auto fc2 = [&](int i, int b) -> bool {
        const int g = 6 * i + b;
        const int slot = g % kW2Slots;
        if (!mbar_wait_bounded(&h_full[b], i & 1, abort_flag)) return false;
        if (!mbar_wait_bounded(&p_full[slot], (g / kW2Slots) & 1, abort_flag)) return false;
        if (b == 0 && i > 0 && !mbar_wait_bounded(o_empty, (i - 1) & 1, abort_flag)) return false;
        tc_fence_after();
        const uint64_t hdesc = sw128_kmajor_desc(smem_u32(sH + b * kHBytes));
        const uint64_t wdesc = sw128_kmajor_desc(smem_u32(sW2 + slot * kPanel));
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc_mma_f16(tmem_base + kFc2Col, hdesc + 2u * k, wdesc + 2u * k, IDESC_FC2, (b | k) ? 1u : 0u);
        tc_commit(&h_empty[b]);
        tc_commit(&p_empty[slot]);
        return true;
      };
      if (ok && n > 0) {
        ok = mbar_wait_bounded(a_full, 0, abort_flag) && fc1(0, 0) && fc1(0, 1);
        if (ok) tc_commit(a_empty);
      }
      for (int i = 0; i < n && ok; ++i) {
        for (int b = 0; b < 3 && ok; ++b) ok = fc2(i, b);
        if (ok && i + 1 < n) ok = mbar_wait_bounded(a_full, (i + 1) & 1, abort_flag) && fc1(i + 1, 0);
        for (int b = 3; b < 6 && ok; ++b) ok = fc2(i, b);
        if (ok) tc_commit(o_full);
        if (ok && i + 1 < n) {
          ok = fc1(i + 1, 1);
          if (ok) tc_commit(a_empty);
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
    // ------------------------------------------------------------ epilogue warps
    const int q = warp & 3;                  // tensor-memory lane quadrant
    const int part = (warp - 2) >> 2;        // 0 .. WPQ - 1
    const int r = q * 32 + lane;             // row of the tile
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    bool ok = true;
    // the whole warp polls (one barrier word, one answer for all lanes)
    auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, abort_flag) ? 1 : 0) != 0;
    };
    // tensor memory -> registers for hidden block b (this warp: its CW columns), not waited
    auto ld_block = [&](int b, uint32_t* v) {
      const int col = 64 * b + CW * part;
      tmem_ld_32x32b_x16(t_lane + col, v);
      if constexpr (CW == 32) tmem_ld_32x32b_x16(t_lane + col + 16, v + 16);
    };
    // G(i, b) once its accumulator values are in registers: + b1, GELU, into hidden
    // buffer b (after FC2(i - 1, b) has released it)
    auto store_block = [&](int i, int b, const uint32_t* v) -> bool {
      if (!wait_all(&h_empty[b], (i & 1) ^ 1)) return false;
      const float4* bb = reinterpret_cast<const float4*>(sB1 + 64 * b + CW * part);
      float f[CW];
#pragma unroll
      for (int k = 0; k < CW / 4; ++k) {
        const float4 bq = bb[k];
        f[4 * k + 0] = gelu_erf<5>(__uint_as_float(v[4 * k + 0]) + bq.x);
        f[4 * k + 1] = gelu_erf<5>(__uint_as_float(v[4 * k + 1]) + bq.y);
        f[4 * k + 2] = gelu_erf<5>(__uint_as_float(v[4 * k + 2]) + bq.z);
        f[4 * k + 3] = gelu_erf<5>(__uint_as_float(v[4 * k + 3]) + bq.w);
      }
      // CW columns = CW / 8 16-byte chunks of the 128-byte row, starting at chunk
      // (CW / 8) part, each at chunk ^ (r & 7) (the 128-byte swizzle)
      uint8_t* row = sH + b * kHBytes + r * 128;
#pragma unroll
      for (int c = 0; c < CW / 8; ++c)
        *reinterpret_cast<uint4*>(row + ((((CW / 8) * part + c) ^ (r & 7)) << 4)) = pack16<T>(f + 8 * c);
      fence_proxy_async_smem();   // visible to the tensor core
      __syncwarp();
      if (lane == 0) mbar_arrive(&h_full[b]);
      return true;
    };
    // this warp has read its share of FC1 half hf (its loads have completed)
    auto half_read = [&](int hf) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[hf]);
    };
    // The final epilogue works in 16-column chunks of the C = 96 outputs: chunk c of a
    // row belongs to part c % WPQ of its lane quadrant (at most NC chunks a warp).
    constexpr int NC = (kMC / 16 + WPQ - 1) / WPQ;
    // the residual rows of tile i (32 bytes a chunk), requested a few hidden blocks
    // before F(i) needs them
    auto load_resid = [&](int i, uint4* rv) {
      const long long grow = static_cast<long long>(kMBM) * tile_of(i) + r;
#pragma unroll
      for (int k = 0; k < NC; ++k) {
        const int c = part + WPQ * k;
        if (c < kMC / 16 && grow < M) {
          const uint4* rr = reinterpret_cast<const uint4*>(resid + grow * kMC + 16 * c);
          rv[2 * k] = rr[0];
          rv[2 * k + 1] = rr[1];
        }
      }
    };
    // F(i): FC2 accumulator + b2 + residual -> out
    auto final_epi = [&](int i, const uint4* rv) -> bool {
      if (!wait_all(o_full, i & 1)) return false;
      tc_fence_after();
      const long long grow = static_cast<long long>(kMBM) * tile_of(i) + r;
#pragma unroll
      for (int k = 0; k < NC; ++k) {
        const int c = part + WPQ * k;
        if (c >= kMC / 16) continue;   // uniform per warp
        uint32_t v[1][16];
        tmem_ld_32x32b_x16(t_lane + kFc2Col + 16 * c, v[0]);
        tmem_ld_wait();
        if (k + 1 >= NC || part + WPQ * (k + 1) >= kMC / 16) {   // this warp's last chunk read
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(o_empty);
        }
        if (grow < M) {
          uint4* oo = reinterpret_cast<uint4*>(out + grow * kMC + 16 * c);
          const float4* bb = reinterpret_cast<const float4*>(b2 + 16 * c);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float rf[8];
            unpack16<T>(rv[2 * k + h], rf);
            const float4 x0 = __ldg(bb + 2 * h), x1 = __ldg(bb + 2 * h + 1);
            const float bias[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            float o8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) o8[e] = __uint_as_float(v[0][8 * h + e]) + bias[e] + rf[e];
            oo[h] = pack16<T>(o8);
          }
        }
      }
      return true;
    };
    // the six hidden blocks of tile i, each block's tensor-memory load issued before the
    // previous block's arithmetic (within a half, whose accumulator is complete); F(fi)
    // (when asked) between the halves
    uint32_t va[CW], vb[CW];
    auto tile_blocks = [&](int i, bool with_f, int fi, const uint4* rv) -> bool {
      for (int hf = 0; hf < 2; ++hf) {
        const int b0 = 3 * hf;
        if (!wait_all(&s_full[hf], i & 1)) return false;
        tc_fence_after();
        ld_block(b0, va);
        tmem_ld_wait();
        ld_block(b0 + 1, vb);
        if (!store_block(i, b0, va)) return false;
        tmem_ld_wait();
        ld_block(b0 + 2, va);
        if (!store_block(i, b0 + 1, vb)) return false;
        tmem_ld_wait();
        half_read(hf);
        if (!store_block(i, b0 + 2, va)) return false;
        if (hf == 0 && with_f && !final_epi(fi, rv)) return false;
      }
      return true;
    };
    if (n > 0) ok = tile_blocks(0, false, 0, nullptr);
    for (int i = 0; i < n && ok; ++i) {
      uint4 rv[2 * NC];
      load_resid(i, rv);
      ok = i + 1 < n ? tile_blocks(i + 1, true, i, rv) : final_epi(i, rv);
    }
    if (!ok && lane == 0) {
      set_device_error(err, RPP_DERR_TIMEOUT);
      *abort_flag = 1;
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

template <typename T, int EW = kMlpEW>
cudaError_t mlp_launch(const CUtensorMap& th, const CUtensorMap& t1, const CUtensorMap& t2, const float* b1,
                       const float* b2, const void* resid, void* out, int M, int32_t* err, cudaStream_t stream) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(swin_mlp_kernel<T, EW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kMlpSmem));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const int tiles = (M + kMBM - 1) / kMBM;
  const int grid = tiles < num_sms() ? tiles : num_sms();
  return launch_pdl(swin_mlp_kernel<T, EW>, dim3(static_cast<unsigned>(grid)), dim3(mlp_threads<EW>()), kMlpSmem, stream, th, t1,
                    t2, b1, b2, static_cast<const T*>(resid), static_cast<T*>(out), M, err);
}

}  // namespace

bool swin_mlp_supported(int C, int F) { return C == kMC && F == kMF; }

cudaError_t launch_swin_mlp(const void* h, const void* w1_kn, const float* b1, const void* w2_nk, const float* b2,
                            const void* resid, void* out, int M, int C, int F, rpp_dtype dtype, int32_t* err,
                            cudaStream_t stream) {
  static_assert(kMlpSmem <= 232448, "shared memory per CTA");
  if (!swin_mlp_supported(C, F)) return cudaErrorNotSupported;
  if (dtype != RPP_F16 && dtype != RPP_BF16) return cudaErrorNotSupported;
  if (M <= 0) return cudaSuccess;
  const CUtensorMapDataType dt = dtype == RPP_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap th, t1, t2;
  // h [M, C]: boxes of 128 rows x 64 columns (columns past C read as zero)
  if (!make_tmap_2d(&th, h, dt, 2, M, C, kMBM, 64, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
  // W1 as [C = K rows, F = N columns] and W2 as [C = N rows, F = K columns]: 96 x 64 boxes
  if (!make_tmap_2d(&t1, w1_kn, dt, 2, C, F, C, 64, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
  if (!make_tmap_2d(&t2, w2_nk, dt, 2, C, F, C, 64, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
  if (dtype == RPP_F16) return mlp_launch<__half>(th, t1, t2, b1, b2, resid, out, M, err, stream);
  return mlp_launch<__nv_bfloat16>(th, t1, t2, b1, b2, resid, out, M, err, stream);
}

}  // namespace rpp
