// Internal launchers shared by the kernel translation units and the C ABI (api.cu).
#pragma once
#include <type_traits>

#include "common.cuh"

namespace rpp {

int num_sms();   // SM count of the current device (cached per device)

// Status of the C ABI for a CUDA runtime result; clears a sticky launch error.  Shared
// by every entry point so that the same failure maps to the same status everywhere.
inline rpp_status status_from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return RPP_OK;
  cudaGetLastError();
  if (e == cudaErrorNotSupported) return RPP_EUNSUPPORTED;
  if (e == cudaErrorInvalidValue) return RPP_EINVAL;
  return RPP_ECUDA;
}

// epilogue codes beyond the public rpp_epilogue (int8 layer)
enum InternalEpilogue {
  EPI_I32 = 3,               // raw int32 accumulators
  EPI_DQ_BIAS = 4,           // acc * s_a * s_w[n] + b
  EPI_DQ_ACC = 5,            // acc * s_a * s_w[n] (fp32; bias and residual added by the next LayerNorm)
  EPI_DQ_BIAS_GELU_Q = 6,    // int8 code of GELU(acc * s_a * s_w[n] + b), held in a bf16 container
  EPI_ACC = 7,               // raw fp32 accumulator (split-K slices; bias and residual added by LayerNorm)
  EPI_DQ_BIAS_Q3 = 8         // int8 codes of acc * s_a * s_w[n] + b with one scale per third of the columns
                             // (the Q, K and V parts of the QKV projection), held in a bf16 container
};

cudaError_t launch_build_offsets(const int32_t* lengths, int B, int L, int32_t* cu, int32_t* po, int32_t* err,
                                 cudaStream_t stream);
cudaError_t launch_remove_padding(const void* padded, const int32_t* po, const int32_t* cu, int B, int L,
                                  int row_bytes, void* packed, int32_t* err, cudaStream_t stream);
bool offsets_remove_fusable(int B);
// offset builder + padding removal in one launch (B <= 1024)
cudaError_t launch_offsets_remove(const int32_t* lengths, int B, int L, int row_bytes, const void* padded,
                                  int32_t* cu, int32_t* po, void* packed, int32_t* err, cudaStream_t stream);
cudaError_t launch_rebuild_padding(const void* packed, const int32_t* cu, int B, int L, int row_bytes, void* padded,
                                   int32_t* err, cudaStream_t stream);

bool layernorm_supported(int H, rpp_dtype dtype);
// Row LayerNorm over H columns of [rows, H]; the row normalised is x (or the sum of
// n_in fp32 split-K slices) + add_bias + residual, the last two optional.  Outputs: y
// (out_dtype), optional fp32 copy, optional bf16-held int8 codes, optional running
// max-abs.  With pad_cu set, the grid walks the padded [pad_B, pad_L] slots and writes
// y at padded rows, zeros in pad slots (the padding rebuild, fused).
struct LnArgs {
  const void* x = nullptr;
  rpp_dtype in_dtype = RPP_F32;
  int n_in = 1;
  long long in_stride = 0;
  const float* add_bias = nullptr;
  const void* residual = nullptr;
  rpp_dtype res_dtype = RPP_F32;
  int res_kind = 0;            // set by launch_layernorm
  const float* gamma = nullptr;
  const float* beta = nullptr;
  void* y = nullptr;
  rpp_dtype out_dtype = RPP_F32;
  float* y32 = nullptr;
  __half* y16 = nullptr;       // fp16 copy of y (streaming kernel only)
  void* q_codes = nullptr;
  const float* q_scale = nullptr;
  float* amax = nullptr;
  int M_max = 0;
  const int32_t* rows = nullptr;
  int H = 0;
  float eps = 0.f;
  const int32_t* pad_cu = nullptr;
  int pad_B = 0;
  int pad_L = 0;
  int32_t* err = nullptr;
};
cudaError_t launch_layernorm(const LnArgs& a, cudaStream_t stream);
cudaError_t launch_quantize(const void* x, const float* scale, int8_t* q, int M_max, const int32_t* rows, int H,
                            rpp_dtype dtype, int32_t* err, cudaStream_t stream);
cudaError_t launch_amax(const void* x, int M_max, const int32_t* rows, int H, rpp_dtype dtype, float* amax,
                        int32_t* err, cudaStream_t stream);
// per-part max |x| of [M, W] rows split into W / part_w (<= 3) column parts -> amax[part]
cudaError_t launch_amax_parts(const void* x, int M_max, const int32_t* rows, int W, int part_w, rpp_dtype dtype,
                              float* amax, int32_t* err, cudaStream_t stream);

// preprocessing and int8 code helpers (prep.cu)
cudaError_t launch_quantize_codes_bf16(const void* x, const float* scale, void* codes, int M_max, const int32_t* rows,
                                       int H, rpp_dtype dtype, int32_t* err, cudaStream_t stream);
cudaError_t launch_i8_to_bf16(const int8_t* src, void* dst, long long n, cudaStream_t stream);
cudaError_t launch_quantize_weight(const void* w, int K, int N, rpp_dtype dtype, int8_t* wq_t, void* wq_t_bf16,
                                   float* s_w, cudaStream_t stream);
cudaError_t launch_transpose_to_kmajor(const void* w, int K, int N, int elem_bytes, void* dst, int dst_ld,
                                       cudaStream_t stream);
cudaError_t launch_to_f32(const void* src, rpp_dtype dtype, long long n, float* dst, cudaStream_t stream);

struct TcGemmArgs {
  const void* a;           // [M_max, K] operand (fp16 / bf16, or bf16-held int8 codes)
  const void* w_t;         // [N, K] operand
  const float* bias;       // [N] or null (EPI_I32)
  const void* residual;    // [M_max, N] of the output type
  void* out;               // [M_max, N]
  int M_max;
  const int32_t* rows;
  int N, K;
  rpp_dtype in_dtype;      // RPP_F16 or RPP_BF16
  rpp_dtype out_dtype;     // RPP_F16 / RPP_BF16 / RPP_F32 (anything for EPI_I32)
  rpp_dtype res_dtype;     // residual type for the float path: in_dtype (default) or RPP_F32
  int epi;                 // rpp_epilogue or InternalEpilogue
  const float* a_scale;    // device scalar s_a (int8 epilogues)
  const float* w_scale;    // device [N] s_w (int8 epilogues)
  const float* q_scale;    // device scalar for the requantised output (EPI_DQ_BIAS_GELU_Q), or three
                           // (EPI_DQ_BIAS_Q3: the scales of the column thirds)
  int32_t* err;
  int force_bn;            // 0 = heuristic
  int rows_hint;           // expected rows (0 = M_max): tile shapes only, never correctness
  int max_splits;          // > 1 allows split-K (fp32 partial slices, residual epilogue only)
  int* splits_out;         // if set, receives the number of K splits used
};
bool gemm_tc_supported(int N, int K);
cudaError_t launch_gemm_tc(const TcGemmArgs& g, cudaStream_t stream);
// 0 automatic, 1 never cluster, 2 cluster whenever the GEMM is fp16/bf16
void set_gemm_cluster_mode(int mode);
// tuning hook: 0 = the tile-width heuristic, else this width wherever it divides N
void set_gemm_force_bn(int bn);
// test hook: the next tensor-core GEMM launch issues no operand loads and its pipeline
// waits give up after limit_ns (it records RPP_DERR_TIMEOUT and exits cleanly)
void set_gemm_stall_next(unsigned long long limit_ns);


cudaError_t launch_gemm_f32(const float* a, const float* w_t, const float* bias, const float* residual, float* out,
                            int M_max, const int32_t* rows, int N, int K, int epi, int32_t* err, cudaStream_t stream);

// 2D row-major [rows, cols] tensor map, box = box_cols x box_rows (defined with the GEMM)
bool make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem_bytes, long long rows,
                  int cols, int box_rows, int box_cols, CUtensorMapSwizzle swz);
// persistent longest-first tcgen05 varlen attention (S, P, O in tensor memory), head size 64
bool attention_sched_supported(int B, int max_len);
// i8_scales: device (s_q, s_k, s_v) for int8 codes held in bf16 (dtype RPP_BF16, fp16 out);
// out_scale: device s_o, the output leaves as bf16-held int8 codes of O / s_o
cudaError_t launch_attention_sched(const void* qkv, const int32_t* cu, int B, int T_max, int max_len, int nh,
                                   rpp_dtype dtype, void* out, int32_t* err, cudaStream_t stream,
                                   const float* i8_scales = nullptr, const float* out_scale = nullptr);
// tcgen05 varlen attention, head size 64, fp16 / bf16 (one CTA per 128 queries; batches
// beyond the persistent kernel's limits)
cudaError_t launch_attention_tc(const void* qkv, const int32_t* cu, int B, int T_max, int max_len, int nh,
                                rpp_dtype dtype, void* out, int32_t* err, cudaStream_t stream);
// Swin MLP fused on the tensor cores (C = 96, F = 384): out = resid + FC2(GELU(FC1(h) + b1)) + b2;
// w1_kn is W1 as [C, F] (K rows, N columns), w2_nk is W2 as [C, F] (N rows, K columns)
bool swin_mlp_supported(int C, int F);
cudaError_t launch_swin_mlp(const void* h, const void* w1_kn, const float* b1, const void* w2_nk, const float* b2,
                            const void* resid, void* out, int M, int C, int F, rpp_dtype dtype, int32_t* err,
                            cudaStream_t stream);
// Swin patch merging: the 2 x 2 gather fused into the LayerNorm over 4C channels
bool patch_merge_supported(int C, int I);
cudaError_t launch_patch_merge_ln(const void* x, int B, int I, int C, rpp_dtype dtype, const float* gamma,
                                  const float* beta, float eps, void* out, int32_t* err, cudaStream_t stream);
cudaError_t launch_attention_varlen(const void* qkv, const int32_t* cu, int B, int T_max, int max_len, int nh, int d,
                                    rpp_dtype dtype, void* out, int32_t* err, cudaStream_t stream);

bool window_attention_supported(int C, int nh, int w, int I, int s);
cudaError_t launch_window_attention(int B, const void* qkv, const float* bias, void* out, int C, int nh, int I, int w,
                                    int s, rpp_dtype dtype, int32_t* err, cudaStream_t stream);
cudaError_t launch_swin_bias(const void* table, rpp_dtype table_dtype, int w, int nh, float* bias,
                             cudaStream_t stream);

}  // namespace rpp
