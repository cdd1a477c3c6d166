// Persistent, warp-specialised tcgen05 GEMM for sm_103a with fused epilogues.
//
//   out[M, N] = epilogue(A[M, K] @ W[N, K]^T),   A, W fp16 or bf16 (both K-major),
//   fp32 accumulation in tensor memory.
//
// The NVIDIA Swin talk (§3) fuses the bias (and activation) into the GEMM and, when
// the op after the GEMM is LayerNorm, splits the bias off the GEMM and fuses it into
// that next op; the Kuaishou article (Fig. 6, Fig. 11) fuses the elementwise work
// into the GEMMs and tunes the GEMM tile configuration per shape.  Here the GEMM is
// written for the 5th-generation tensor cores:
//
//   warp 0      TMA producer: 2D tiled loads with 128-byte swizzle of a 128 x 64 A
//               tile and a BN x 64 W tile per pipeline stage.
//   warp 1      allocates tensor memory and issues tcgen05.mma (M = 128, N = BN,
//               K = 16 per instruction) from one thread; tcgen05.commit releases the
//               smem stage and, after the last K block, signals the accumulator.

//   warps 2..   epilogue: 8 or 16 warps, two or four per tensor-memory lane quadrant,
//               each taking every second or fourth 32-column slice: tcgen05.ld 32 lanes
//               x 32 columns (one row per thread), the epilogue arithmetic in fp32, then
//               the 32 x 32 block goes to a swizzled staging buffer in shared memory and
//               leaves with one TMA bulk-tensor store -- coalesced, asynchronous, no
//               per-row scatter.  Tiles that straddle the row count M (the ragged last
//               tile) and 16-column tails use per-row 16-byte stores instead.
//
// CTA pairs: for long-K GEMMs over many row tiles, two CTAs of a cluster compute a
// 256 x BN tile with cta_group::2 MMAs.  Each CTA loads its own 128 A rows and half of
// the W tile (BN / 2 rows), both completing on the even CTA's barrier; the even CTA
// issues M = 256 MMAs that read both CTAs' shared memory and write each CTA's 128
// accumulator rows into its own tensor memory; commits are multicast to both CTAs'
// barriers and both CTAs' epilogue warps release the accumulator on the even CTA's
// barrier.  Shared-memory operand traffic per MMA drops from (128 + BN) to
// (128 + BN / 2) rows per CTA.
//
// Epilogues: bias | bias + GELU | bias + residual (any of fp32, fp16 or the input type
// out; the encoder layer's proj / FC2 write their pre-LayerNorm sums in fp16) | raw fp32
// accumulator (calibration passes: bias and residual are added by the LayerNorm that
// reads the rows next) and the int8 variants below.
//
// The accumulator is double-buffered in tensor memory, so the epilogue of tile i
// overlaps the MMAs of tile i+1.  Work units are assigned round-robin over a
// persistent grid of at most one CTA per SM.  The row count M may live in device
// memory (the packed token count).  Every mbarrier wait is bounded; on a timeout the
// CTA records RPP_DERR_TIMEOUT, drains its in-flight copies and MMAs, frees its
// tensor memory and exits.
//
// Split-K: when a GEMM has too few output tiles to fill the SMs (narrow N, few
// tokens), each tile's K range is cut into `splits` parts; part s writes its raw fp32
// partial sum into slice s of the output and the LayerNorm that follows adds the
// slices while loading its row: no extra kernel, deterministic.
//
// int8 layers: sm_103a has no int8 kind of tcgen05.mma, so the int8 GEMM runs as an
// exact integer product on the bf16 tensor pipe.  Codes in [-127, 127] are exact in
// bf16, each product is an integer below 2^14, and K is split into chunks of at most
// 1024 so every fp32 partial sum is an integer below 2^24 and therefore exact; each
// chunk accumulates into its own tensor-memory region and the epilogue adds the
// chunks in int32.  The result equals int32 accumulation bit for bit.


#include <cstring>

#include "gemm_tc.cuh"

namespace rpp {

using namespace gemm;

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

}  // namespace

bool make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem_bytes, long long rows,
                  int cols, int box_rows, int box_cols, CUtensorMapSwizzle swz) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * elem_bytes};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

// Tile shape choice (the per-shape GEMM configuration of the Kuaishou article's
// Fig. 11): over the tile widths that divide N and the allowed K splits, minimise
// waves x (K blocks per unit x (BN + 32) + epilogue cost), using the expected number
// of rows (the caller's token-count hint, else the capacity).
struct TileChoice {
  int bn = 0;
  int splits = 1;
};

TileChoice choose_tiles(int M, int N, int K, int max_bn, int max_splits, int cl = 1, int wpq = 2) {
  static const int cands[] = {256, 192, 144, 128, 96, 64, 48, 32, 16};
  const int sms = num_sms() / cl;                       // concurrent work units (clusters)
  const int num_m = (M + kBM * cl - 1) / (kBM * cl);    // row-tile groups
  const int num_k = (K + kBK - 1) / kBK;
  TileChoice best;
  double best_cost = 1e30;
  for (int bn : cands) {
    if (N % bn || bn > max_bn) continue;
    for (int sp = 1; sp <= max_splits && sp <= num_k; ++sp) {
      const int kps = (num_k + sp - 1) / sp;
      const long long units = static_cast<long long>(num_m) * (N / bn) * sp;
      const long long waves = (units + sms - 1) / sms;
      // With a few K blocks per unit the epilogue is the bottleneck, and a tile's
      // epilogue takes as long as its busiest warp (each of the wpq warps of a lane
      // quadrant takes every wpq-th 32-column slice); with more, it overlaps the next
      // unit's MMAs and only its size counts.
      const double epi = kps <= 4 ? 6.0 * 32.0 * wpq * ((bn + 32 * wpq - 1) / (32 * wpq)) : 6.0 * bn;
      const double cost = static_cast<double>(waves) * (kps * (bn + 32.0) + epi) + (sp - 1) * 64.0;
      if (cost < best_cost - 1e-9) {
        best_cost = cost;
        best.bn = bn;
        best.splits = sp;
      }
    }
  }
  return best;
}

}  // namespace


bool gemm_tc_supported(int N, int K) {
  return K % 8 == 0 && K > 0 && N % 16 == 0 && choose_tiles(1, N, K, 256, 1).bn != 0;
}

namespace {
int g_cluster_mode = 0;   // 0 automatic, 1 never, 2 always (where the GEMM has two row tiles)
unsigned long long g_stall_next_ns = 0;   // test hook: nonzero = the next launch stalls, waits give up after this
int g_force_bn = 0;       // tuning hook: nonzero = this tile width wherever it divides N
}

void set_gemm_cluster_mode(int mode) { g_cluster_mode = mode; }
void set_gemm_force_bn(int bn) { g_force_bn = bn; }
void set_gemm_stall_next(unsigned long long limit_ns) { g_stall_next_ns = limit_ns; }

cudaError_t launch_gemm_tc(const TcGemmArgs& g, cudaStream_t stream) {
  const bool is_int = (g.epi >= EPI_I32 && g.epi <= EPI_DQ_BIAS_GELU_Q) || g.epi == EPI_DQ_BIAS_Q3;
  if (g.epi == EPI_DQ_BIAS_Q3 && (g.N % 3 || (g.N / 3) % 32)) return cudaErrorNotSupported;
  const int num_k = (g.K + kBK - 1) / kBK;
  const int nch = is_int ? (num_k + kChunkBlocks - 1) / kChunkBlocks : 1;
  if (nch > 4) return cudaErrorNotSupported;
  const int max_bn = nch > 1 ? 128 : 256;
  // splitting K is only possible for the raw fp32 accumulator output
  const bool can_split = g.max_splits > 1 && g.epi == EPI_ACC;
  const int rows_hint = (g.rows_hint > 0 && g.rows_hint < g.M_max) ? g.rows_hint : g.M_max;
  // A CTA pair (a two-CTA thread-block cluster) computes a 256-row tile with
  // cta_group::2 MMAs issued by the even CTA: each CTA holds its 128 rows of A and
  // half of the W tile, halving the shared-memory traffic per MMA.
  // Pairs pay off when the MMAs dominate (long K, many row tiles, wide N); short-K or
  // few-tile GEMMs are epilogue- or latency-bound and run unpaired, and so does a square
  // 1024 x 1024 GEMM (the BERT-large proj: 33.8 us unpaired against 35.7 paired at
  // 12 555 rows, bias epilogue, standalone; inside the step the two are within noise).
  const bool pair_auto = rows_hint >= 8192 && g.K >= 1024 && (g.N >= 2048 || g.K >= 2048);
  int cl = (!is_int && (g_cluster_mode == 2 || (g_cluster_mode == 0 && pair_auto))) ? 2 : 1;
  const int wpq = g.epi == RPP_EPI_BIAS_GELU ? epi_warps<RPP_EPI_BIAS_GELU>() / 4 : 2;
  TileChoice tc = choose_tiles(rows_hint, g.N, g.K, max_bn, can_split ? g.max_splits : 1, cl, wpq);
  if (g.force_bn) tc.bn = g.force_bn;
  else if (g_force_bn && g.N % g_force_bn == 0 && g_force_bn <= max_bn) tc.bn = g_force_bn;
  const int bn = tc.bn;
  if (!bn || g.N % bn || bn > max_bn) return cudaErrorNotSupported;
  if (g.splits_out) *g.splits_out = tc.splits;
  const CUtensorMapDataType dt =
      (is_int || g.in_dtype == RPP_BF16) ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap ta, tb;
  if (!make_tmap_2d(&ta, g.a, dt, 2, g.M_max, g.K, kBM, kBK, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
  GemmParams p{g.M_max, g.rows, g.N, g.K, g.bias, g.residual, g.out, g.a_scale, g.w_scale, g.q_scale, g.err,
               tc.splits, static_cast<long long>(g.M_max) * g.N, kWaitLimitNs, 0};
  if (g_stall_next_ns) {   // consumed by this one launch
    p.stall = 1;
    p.wait_ns = g_stall_next_ns;
    g_stall_next_ns = 0;
  }
  if (is_int) {
    if (!make_tmap_2d(&tb, g.w_t, dt, 2, g.N, g.K, bn, kBK, CU_TENSOR_MAP_SWIZZLE_128B)) return cudaErrorInvalidValue;
    return gemm_dispatch_int(nch == 1 ? 1 : 4, bn, g.epi, ta, tb, p, rows_hint, stream);
  }
  if (g.in_dtype != RPP_BF16 && g.in_dtype != RPP_F16) return cudaErrorNotSupported;
  for (;;) {
    // each CTA of a cluster loads bn / cl rows of the W tile
    if (!make_tmap_2d(&tb, g.w_t, dt, 2, g.N, g.K, bn / cl, kBK, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    cudaError_t e;
    if (g.in_dtype == RPP_BF16)
      e = cl == 2 ? gemm_dispatch_float_bf16_cl2(bn, g.epi, g.out_dtype, g.res_dtype, ta, tb, p, rows_hint, stream)
                  : gemm_dispatch_float_bf16_cl1(bn, g.epi, g.out_dtype, g.res_dtype, ta, tb, p, rows_hint, stream);
    else
      e = cl == 2 ? gemm_dispatch_float_f16_cl2(bn, g.epi, g.out_dtype, g.res_dtype, ta, tb, p, rows_hint, stream)
                  : gemm_dispatch_float_f16_cl1(bn, g.epi, g.out_dtype, g.res_dtype, ta, tb, p, rows_hint, stream);
    if (e == cudaErrorNotSupported && cl == 2) {   // no pair of SMs available: run unclustered
      cl = 1;
      continue;
    }
    return e;
  }
}

}  // namespace rpp
