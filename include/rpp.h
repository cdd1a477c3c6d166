/*
 * rpp.h -- C ABI of the padding-removed transformer encoder-layer forward pass for
 * one GB300 (sm_103a).
 *
 * Sources (by page title and figure / section):
 *  [KS] "GPU底層優化 | 如何讓Transformer在GPU上跑得更快？" (Kuaishou heterogeneous computing
 *       team): Fig. 9 padding removal through an Offset Mask, packed and padded
 *       sequences convert into each other; Fig. 10 which kernels run on packed tokens;
 *       Fig. 6 fusion of self-attention and feed-forward; Fig. 8 memory management.
 *  [SW] NVIDIA talk on Swin Transformer training / inference optimisation (Japanese
 *       transcript, m.sbmmt.com/ja/faq/533025): §1 window attention, cyclic shift,
 *       relative position bias; §3 preprocessing (bias lookup, weight reformat), fMHA,
 *       QKV GEMM + bias, GEMM + bias + activation, INT8 GEMM with int32 accumulation.
 *
 * Conventions shared by every call:
 *  - Every pointer argument named as "device" is CUDA device memory owned by the
 *    caller; the library never allocates, frees or keeps a pointer after the call
 *    returns.  Host pointers are read during the call only.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream), does no host synchronisation and no allocation, so a sequence of calls
 *    can be captured into a CUDA graph.  rpp_get_device_error is the one exception:
 *    it synchronises by design.
 *  - Matrices are row-major and contiguous.  Activation and weight pointers must be
 *    16-byte aligned; hidden sizes must keep every row a multiple of 16 bytes.
 *  - Host-detectable argument errors return a negative rpp_status and launch nothing.
 *  - Device-detectable errors (a length outside [0, L], a packed row count larger than
 *    the capacity, a kernel-internal bounded wait that gave up) write a nonzero code
 *    into the caller's `err` word (int32 in device memory, zero-initialised by the
 *    caller; may be NULL, in which case such errors are not reported).  Every kernel
 *    of this library that is given a nonzero `err` word does no work, so one check
 *    after a sequence of calls suffices.
 *  - Packed activations have a capacity T_max rows (normally B * L); the number of
 *    valid rows T = cu_seqlens[B] lives in device memory and is never read back by
 *    the library, so lengths can change between launches of a captured graph.
 */
#ifndef RPP_H_
#define RPP_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define RPP_API __attribute__((visibility("default")))
#else
#define RPP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum rpp_status {
  RPP_OK = 0,
  RPP_EINVAL = -1,        /* bad argument (null pointer, negative size, misalignment) */
  RPP_EUNSUPPORTED = -2,  /* valid but not implemented shape / dtype combination */
  RPP_ECUDA = -3,         /* a CUDA runtime call failed (launch error, bad stream) */
  RPP_EWORKSPACE = -4,    /* workspace smaller than the size query returned */
  RPP_EDEVICE = -5        /* rpp_get_device_error found a nonzero device error word */
} rpp_status;

typedef enum rpp_dtype { RPP_F32 = 0, RPP_F16 = 1, RPP_BF16 = 2, RPP_I8 = 3 } rpp_dtype;

/* codes written into the device error word */
#define RPP_DERR_LENGTH 1   /* a sequence length outside [0, L] or [0, max_len] */
#define RPP_DERR_TIMEOUT 2  /* a bounded wait inside a kernel gave up (pipeline stall) */
#define RPP_DERR_ROWS 3     /* cu_seqlens[B] larger than the packed capacity T_max */
#define RPP_DERR_TMEM 4     /* the CTAs of a paired GEMM got different tensor-memory columns */

typedef void* rpp_stream; /* cudaStream_t */

/* Human-readable name of a status code (static string). */
RPP_API const char* rpp_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
RPP_API int rpp_version(void);

/* Copy the device error word to the host (synchronises `stream`).  Returns RPP_OK
 * and *host_code = 0 when no error was recorded, RPP_EDEVICE with the code
 * otherwise; RPP_ECUDA if the copy failed. */
RPP_API rpp_status rpp_get_device_error(const int32_t* err, int32_t* host_code, rpp_stream stream);

/* Launch-event hook for profiling (the pages profile with Nsight timelines; this
 * hook lets a caller time each kernel inside the real step with CUDA events).  While
 * enabled, every kernel the path launches is followed by cudaEventRecord(events[i++])
 * on its stream, i < capacity, and its label (e.g. "gemm_fc1") is kept; on a stream
 * under capture the record is an external event node of the graph, so the times can
 * be read after each replay.  `events` is
 * a host array of cudaEvent_t owned by the caller; capacity 0 disables the hook.
 * Not thread-safe: one profiling caller at a time. */
RPP_API rpp_status rpp_set_launch_events(void* const* events, int capacity);
/* TEST / TUNING ONLY -- not part of the method's calls.  Process-wide knob of the
 * fp16 / bf16 tensor-core GEMMs (no counterpart in the pages):
 * 0 (default) pairs CTAs into two-CTA clusters running cta_group::2 MMAs on 256-row
 * tiles (each CTA holds its 128 A rows and half of the weight tile) when K >= 1024, the
 * expected row count is >= 8192 and N or K is >= 2048; 1 never pairs; 2 always pairs.  The exact int8
 * GEMM always runs unpaired (pairs measured no faster there).
 * The arithmetic per output element is the same in every mode, except that the
 * tile shape and K split are chosen per mode, and a different K split changes the
 * fp32 summation order.  Process-wide, not thread-safe; RPP_EINVAL outside 0..2. */
RPP_API rpp_status rpp_set_gemm_cluster_mode(int mode);

/* TEST / TUNING ONLY -- not part of the method's calls.  Process-wide knob of the
 * tensor-core GEMMs: 0 (default) lets the per-shape heuristic choose the tile width
 * (the number of output columns a CTA or CTA pair computes per unit); one of 16, 32, 48,
 * 64, 96, 128, 144, 192, 256 forces that width wherever it divides N (and is allowed for
 * the epilogue).  Results are the same for every width.  Process-wide, not thread-safe;
 * RPP_EINVAL for other values. */
RPP_API rpp_status rpp_set_gemm_tile_width(int bn);

/* TEST ONLY -- exercises the failure detection of the bounded waits (no counterpart in
 * the pages).  The next fp16 / bf16 / int8 tensor-core GEMM launch of this process issues
 * no operand loads, and its pipeline waits give up after `limit_us` microseconds instead
 * of the normal 4 s: the launch records RPP_DERR_TIMEOUT in the error word, drains,
 * frees its tensor memory and exits, and the context stays usable.  The setting is
 * consumed by that one launch.  Process-wide, not thread-safe; RPP_EINVAL unless
 * 1 <= limit_us <= 1000000. */
RPP_API rpp_status rpp_test_stall_next_gemm(unsigned int limit_us);

/* Restrict the hook to launches labelled `label` (NULL: every launch, the default).
 * With a filter, an event is recorded just BEFORE and just after each matching
 * launch (pairs: even index = start, odd = end), so the rest of the step keeps its
 * programmatic launch overlap.  RPP_EINVAL if the label is empty or 64+ bytes. */
RPP_API rpp_status rpp_set_launch_event_filter(const char* label);
/* Events recorded since the last rpp_set_launch_events; label of the i-th ("" if out of range). */
RPP_API int rpp_launch_event_count(void);
RPP_API const char* rpp_launch_event_label(int i);

/* ------------------------------------------------------------------------------
 * Padding removal ([KS] Fig. 9, Fig. 10)
 * ------------------------------------------------------------------------------ */

/* Offset mask of [KS] Fig. 9.
 *  lengths        device int32[B]: valid tokens of each sequence, each in [0, L].
 *  cu_seqlens     device int32[B+1] out: exclusive prefix sum, cu[0] = 0, cu[B] = T.
 *  padding_offset device int32[B*L] out: for packed row i < T, the number of pad
 *                 slots before it, so its padded flat row is i + padding_offset[i]
 *                 (= b*L - cu[b] for a token of sequence b); rows >= T are untouched.
 * A length outside [0, L] records RPP_DERR_LENGTH; the offsets are then built from
 * lengths clamped to [0, L] so that later kernels stay in bounds.  B <= 65536. */
RPP_API rpp_status rpp_build_offsets(const int32_t* lengths, int B, int L, int32_t* cu_seqlens,
                             int32_t* padding_offset, int32_t* err, rpp_stream stream);

/* Gather the valid tokens ([KS] Fig. 9): packed[i, :] = padded[i + padding_offset[i], :]
 * for i < T = cu_seqlens[B].
 *  padded  device [B*L, H] of `dtype`; pad rows are never read.
 *  packed  device [B*L, H] of `dtype` (capacity B*L rows); rows >= T untouched. */
RPP_API rpp_status rpp_remove_padding(const void* padded, const int32_t* padding_offset,
                              const int32_t* cu_seqlens, int B, int L, int H, rpp_dtype dtype,
                              void* packed, int32_t* err, rpp_stream stream);

/* Scatter back ([KS] Fig. 9): padded[b*L + p, :] = packed[cu[b] + p, :] for
 * p < len_b, and 0 for the pad slots p >= len_b.  padded: device [B*L, H]. */
RPP_API rpp_status rpp_rebuild_padding(const void* packed, const int32_t* cu_seqlens, int B, int L, int H,
                               rpp_dtype dtype, void* padded, int32_t* err, rpp_stream stream);

/* ------------------------------------------------------------------------------
 * Building blocks (each is one kernel of the layer; exposed for tests and reuse)
 * ------------------------------------------------------------------------------ */

/* Epilogues fused into the GEMM ([SW] §3: GEMM + bias, GEMM + bias + activation;
 * bias split from the GEMM and fused with the residual before LayerNorm). */
typedef enum rpp_epilogue {
  RPP_EPI_BIAS = 0,          /* out = acc + bias */
  RPP_EPI_BIAS_GELU = 1,     /* out = GELU_erf(acc + bias) */
  RPP_EPI_BIAS_RESIDUAL = 2  /* out = acc + bias + residual */
} rpp_epilogue;

/* out[M, N] = epilogue(a[M, K] @ w_t[N, K]^T).
 *  a         device [M_max, K] of dtype (row-major, K contiguous)
 *  w_t       device [N, K] of dtype: the weight transposed to K-major, as produced
 *            by the prepare calls (a PyTorch nn.Linear weight has this layout)
 *  bias      device float32[N]
 *  residual  device [M_max, N] of dtype, RPP_EPI_BIAS_RESIDUAL only (may alias out)
 *  out       device [M_max, N] of dtype
 *  rows      device int32 or NULL: if given, M = *rows (must be <= M_max), else M = M_max.
 * dtype RPP_F16 / RPP_BF16 run on the tcgen05 tensor cores (K % 8 == 0, N % 16 == 0);
 * RPP_F32 runs an fp32 CUDA-core kernel (K % 4 == 0, N % 4 == 0). */
RPP_API rpp_status rpp_linear(const void* a, const void* w_t, const float* bias, const void* residual,
                      void* out, int M_max, const int32_t* rows, int N, int K, rpp_dtype dtype,
                      rpp_epilogue epilogue, int32_t* err, rpp_stream stream);

/* Row LayerNorm, biased variance, fp32 statistics ([SW] §2-§3):
 * y = (x - mean) / sqrt(var + eps) * gamma + beta over H columns.
 *  x, y      device [M_max, H] of dtype (may alias)
 *  gamma, beta device float32[H]
 *  rows      device int32 or NULL, as for rpp_linear. */
RPP_API rpp_status rpp_layernorm(const void* x, const float* gamma, const float* beta, void* y, int M_max,
                         const int32_t* rows, int H, float eps, rpp_dtype dtype, int32_t* err,
                         rpp_stream stream);

/* Multi-head attention over packed variable-length sequences ([SW] §3 fMHA: batch GEMM,
 * softmax and batch GEMM in one kernel with the head transposes folded into its loads
 * and stores; [KS] Fig. 10: attention is the kernel that needs the sequence bounds).
 *  qkv   device [T_max, 3*nh*d] of dtype: row t holds Q | K | V, head h of each at
 *        columns h*d .. h*d+d-1 (the QKV GEMM output, token-major)
 *  out   device [T_max, nh*d] of dtype, token-major; rows >= T untouched
 * For sequence b and head h: o_i = sum_j softmax_j(q_i . k_j / sqrt(d)) v_j over the
 * keys j of the same sequence.  d must be 64.  Every len_b must be <= max_len. */
RPP_API rpp_status rpp_attention_varlen(const void* qkv, const int32_t* cu_seqlens, int B, int T_max,
                                int max_len, int nh, int d, rpp_dtype dtype, void* out, int32_t* err,
                                rpp_stream stream);

/* The same attention on int8 codes ([SW] §3 INT8 flow: every matrix product int8, with
 * quantise / dequantise around it):
 *  qkv_codes   device [T_max, 3*nh*d] int8 codes held in bf16 (each value an integer in
 *              [-127, 127], exact in bf16), laid out as for rpp_attention_varlen
 *  qkv_scales  device float32[3] = (s_q, s_k, s_v), the per-tensor scales of Q, K, V
 *  out         device [T_max, nh*d] fp16; rows >= T untouched
 * Per sequence and head: S = Qc Kc^T (exact integers), P = softmax over the sequence's
 * keys of S s_q s_k / sqrt(d) (fp32), P's codes clamp(rne(127 P), 0, 127) (P is
 * normalised before it is coded: the kernel reads S twice, first for the row maxima and
 * sums), O = (Pc Vc) s_v / 127 with Pc Vc exact.  d must be 64; B <= 2048 and
 * max_len <= 8192 (RPP_EUNSUPPORTED otherwise). */
RPP_API rpp_status rpp_attention_varlen_i8(const void* qkv_codes, const float* qkv_scales,
                                   const int32_t* cu_seqlens, int B, int T_max, int max_len, int nh,
                                   int d, void* out, int32_t* err, rpp_stream stream);

/* ------------------------------------------------------------------------------
 * Encoder layer (BERT-shaped, post-LayerNorm)
 * ------------------------------------------------------------------------------ */
typedef struct rpp_encoder_cfg {
  int hidden;    /* H */
  int heads;     /* nh */
  int head_dim;  /* d = H / nh (64) */
  int ffn;       /* F */
  float eps;     /* LayerNorm eps */
  int dtype;     /* rpp_dtype of activations and float weights: RPP_F32, RPP_F16, RPP_BF16 */
  int int8;      /* 1: the four linear GEMMs run on int8 codes (dtype must be RPP_F16);
                    2: also the attention (the QKV GEMM writes Q, K, V codes and both
                    attention products run on codes, as rpp_attention_varlen_i8) */
  int tokens_hint; /* expected valid tokens per forward call (0: unknown, the capacity T_max is
                      assumed); only tile shapes and K splits depend on it, never the result */
} rpp_encoder_cfg;

/* The caller's float weights (device, dtype of cfg, row-major [in, out] as in x @ W). */
typedef struct rpp_layer_src {
  const void *Wq, *Wk, *Wv; /* [H, H] each */
  const void *bq, *bk, *bv; /* [H] */
  const void *Wo, *bo;      /* [H, H], [H] */
  const void *W1, *b1;      /* [H, F], [F] */
  const void *W2, *b2;      /* [F, H], [H] */
  const void *gamma1, *beta1, *gamma2, *beta2; /* [H] */
} rpp_layer_src;

/* Bytes of the prepared weight block of one layer. */
RPP_API size_t rpp_layer_bytes(const rpp_encoder_cfg* cfg);

/* One-time preprocessing ([SW] §3: computed once, reused by every inference):
 * concatenates Wq|Wk|Wv into one [3H, H] K-major matrix and bq|bk|bv into one fp32
 * bias (the reformat that lets one GEMM feed the attention kernel), transposes Wo,
 * W1, W2 to K-major, widens biases and LayerNorm parameters to fp32 and, for int8
 * layers, quantises each weight matrix per output channel:
 *   s_w[n] = fp32(max_k |W[k, n]| / 127),  q = clamp(rne(fp32(W[k, n] / s_w[n])), -127, 127).
 *  dst  device, rpp_layer_bytes(cfg) bytes, 256-byte aligned; its layout is private. */
RPP_API rpp_status rpp_prepare_layer(const rpp_encoder_cfg* cfg, const rpp_layer_src* src, void* dst,
                             rpp_stream stream);

/* Workspace bytes for rpp_encoder_layer_forward / _calibrate with capacity T_max. */
RPP_API size_t rpp_encoder_workspace_bytes(const rpp_encoder_cfg* cfg, int T_max);

/* Forward pass of one post-LN encoder layer on packed tokens ([KS] Fig. 6, Fig. 10; [SW] §3):
 *   qkv = x Wqkv + bqkv;  a = MHA_varlen(qkv);  x1 = LN1(x + a Wo + bo);
 *   y = LN2(x1 + GELU(x1 W1 + b1) W2 + b2).
 *  layer       device prepared block from rpp_prepare_layer
 *  act_scales  device float32[4] for int8 layers (scales of the QKV input, attention
 *              output, FC1 input and FC2 input), float32[7] for int8 == 2 (those four,
 *              then the scales of Q, K and V), NULL otherwise
 *  x, y        device [T_max, H] of dtype; may alias
 *  cu_seqlens  device int32[B+1]; max_len >= every len_b
 *  workspace   device, >= rpp_encoder_workspace_bytes(cfg, T_max) bytes, 256-aligned */
RPP_API rpp_status rpp_encoder_layer_forward(const rpp_encoder_cfg* cfg, const void* layer,
                                     const float* act_scales, const void* x,
                                     const int32_t* cu_seqlens, int B, int T_max, int max_len,
                                     void* y, void* workspace, size_t workspace_bytes, int32_t* err,
                                     rpp_stream stream);

/* Post-training calibration for the int8 layer: runs the float layer (cfg.int8 must be
 * 0, `layer` a float prepared block) and writes amax_out[0..6] = max |.| over valid
 * rows of the QKV input, the attention output, the FC1 input, the FC2 input, Q, K and V.
 * amax_out: device float32[7], overwritten.  Scales for the int8 layer are amax / 127. */
RPP_API rpp_status rpp_encoder_layer_calibrate(const rpp_encoder_cfg* cfg, const void* layer, const void* x,
                                       const int32_t* cu_seqlens, int B, int T_max, int max_len,
                                       float* amax_out, void* workspace, size_t workspace_bytes,
                                       int32_t* err, rpp_stream stream);

/* Whole path of [KS] Fig. 9/10 in one call: offsets, remove padding, `num_layers`
 * layers in sequence, rebuild padding.
 *  lengths     device int32[B]
 *  x_padded    device [B*L, H] of dtype;  y_padded: device [B*L, H], pads written as 0
 *  layers      host array of num_layers device prepared blocks
 *  act_scales  host array of num_layers device float32[4] (int8) or NULL
 *  cu_seqlens  device int32[B+1] out; padding_offset device int32[B*L] out
 *  packed      device [B*L, H] of dtype: the packed tokens, updated in place layer by layer
 *  workspace   device, >= rpp_encoder_workspace_bytes(cfg, B*L) bytes */
RPP_API rpp_status rpp_encoder_forward(const rpp_encoder_cfg* cfg, const void* const* layers,
                               const float* const* act_scales, int num_layers,
                               const int32_t* lengths, int B, int L, const void* x_padded,
                               void* y_padded, int32_t* cu_seqlens, int32_t* padding_offset,
                               void* packed, void* workspace, size_t workspace_bytes, int32_t* err,
                               rpp_stream stream);

/* ------------------------------------------------------------------------------
 * INT8 pieces ([SW] §3 INT8 flow: quantise, int8 GEMM with int32 accumulation,
 * dequantise; the int32-output form of the GEMM)
 * ------------------------------------------------------------------------------ */

/* Per-output-channel weight quantisation of a [K, N] (in, out) matrix of dtype:
 *  wq_t  device int8[N, K] out (K-major codes), s_w device float32[N] out, with
 *  s_w[n] = fp32(max_k |W[k,n]| / 127) (1 for an all-zero column) and
 *  wq_t[n, k] = clamp(rne(fp32(W[k, n] / s_w[n])), -127, 127). */
RPP_API rpp_status rpp_quantize_weight(const void* w, int K, int N, rpp_dtype dtype, int8_t* wq_t,
                               float* s_w, rpp_stream stream);

/* Per-tensor activation quantisation: q = clamp(rne(fp32(x) * fp32(1 / *scale)), -127, 127).
 *  x device [M_max, H] of dtype, scale device float32[1], q device int8[M_max, H];
 *  rows: device int32 or NULL as for rpp_linear. */
RPP_API rpp_status rpp_quantize_activation(const void* x, const float* scale, int8_t* q, int M_max,
                                   const int32_t* rows, int H, rpp_dtype dtype, int32_t* err,
                                   rpp_stream stream);

/* Workspace bytes of rpp_gemm_i8_i32 (the operands re-encoded for the tensor cores). */
RPP_API size_t rpp_gemm_i8_workspace_bytes(int M, int N, int K);

/* acc[M, N] = aq[M, K] @ wq_t[N, K]^T exactly, int32 output (the INT32-output GEMM).
 *  aq device int8[M, K], wq_t device int8[N, K], acc device int32[M, N] (16-byte aligned).
 *  K % 16 == 0, N % 16 == 0, K <= 4096.  The product runs on the tcgen05 tensor cores:
 *  sm_103a has no int8 MMA kind, so codes are re-encoded as bf16 (exact) into the
 *  caller's workspace (>= rpp_gemm_i8_workspace_bytes) and K is split into chunks of
 *  1024 whose fp32 partial sums are integers below 2^24, hence exact; the chunks are
 *  added in int32.  The result is bit-identical to int32 accumulation. */
RPP_API rpp_status rpp_gemm_i8_i32(const int8_t* aq, const int8_t* wq_t, int32_t* acc, int M, int N, int K,
                           void* workspace, size_t workspace_bytes, int32_t* err, rpp_stream stream);

/* Allocation-free int8 GEMM (no counterpart on the pages; an addition for callers
 * that cannot allocate device memory).
 *
 * Same result as rpp_gemm_i8_i32 -- acc[M, N] = aq[M, K] @ wq_t[N, K]^T exactly, int32 --
 * but the bf16 re-encoding of the operands lives in a scratch array that is part of
 * the library (device global memory, RPP_GEMM_I8_NOALLOC_SCRATCH_BYTES on every GPU
 * that loads the library, held until the process exits) instead of a caller buffer.
 * Meant for callers that cannot allocate: plugins whose host framework owns all device
 * memory and offers no allocator, latency-critical paths that must not call cudaMalloc
 * (it may synchronise the device), or foreign-function callers that cannot manage
 * device buffer lifetimes.  The caller still passes the inputs and the output; the
 * call itself allocates nothing (no cudaMalloc / cudaFree, no allocating library).
 *  - Sizes: as rpp_gemm_i8_i32 (K % 16 == 0, N % 16 == 0, K <= 4096), and the
 *    re-encoded operands, round256(M*K*2) + round256(N*K*2) bytes, must fit the
 *    scratch; larger problems return RPP_EWORKSPACE and launch nothing.
 *  - All calls share the one scratch array, which keeps the previous call's contents;
 *    each call writes every byte it reads, so nothing needs clearing, but calls whose
 *    kernels overlap on the GPU (unordered streams) race on it.
 *  - Every call looks up the scratch array's device address on the current device
 *    (cudaGetSymbolAddress), so it stays valid across cudaDeviceReset; the first call
 *    on a device also loads the library's device code there, so make that first call
 *    before any stream capture.
 *  - Errors map to the same statuses as rpp_gemm_i8_i32. */
#define RPP_GEMM_I8_NOALLOC_SCRATCH_BYTES (8u << 20) /* 8 MiB */
RPP_API rpp_status rpp_gemm_i8_i32_noalloc(const int8_t* aq, const int8_t* wq_t, int32_t* acc, int M,
                                           int N, int K, int32_t* err, rpp_stream stream);

/* ------------------------------------------------------------------------------
 * Swin shifted-window block ([SW] §1-§3)
 * ------------------------------------------------------------------------------ */
typedef struct rpp_swin_cfg {
  int img;       /* I: image side in tokens (I % window == 0) */
  int channels;  /* C */
  int heads;     /* nh; head_dim = C / nh must be 32 */
  int window;    /* w, w * w <= 64 */
  int shift;     /* s, 0 <= s < w (0: no shift, no mask) */
  int mlp;       /* MLP hidden width (4C) */
  float eps;     /* LayerNorm eps */
  int dtype;     /* RPP_F16 or RPP_BF16 */
} rpp_swin_cfg;

/* The caller's Swin block weights (device, dtype of cfg unless noted). */
typedef struct rpp_swin_src {
  const void *gamma1, *beta1; /* [C] */
  const void *Wqkv, *bqkv;    /* [C, 3C] (columns Q | K | V, head-contiguous), [3C] */
  const void *table;          /* [(2w-1)^2, nh] relative-position bias table */
  const void *Wo, *bo;        /* [C, C], [C] */
  const void *gamma2, *beta2; /* [C] */
  const void *W1, *b1;        /* [C, mlp], [mlp] */
  const void *W2, *b2;        /* [mlp, C], [C] */
} rpp_swin_src;

/* Relative-position-bias lookup moved to preprocessing ([SW] §3):
 * bias[h, t, u] = table[(ty - uy + w - 1) * (2w - 1) + (tx - ux + w - 1), h] for in-window
 * tokens t = ty*w + tx, u = uy*w + ux.  table: device [(2w-1)^2, nh] of cfg dtype;
 * bias: device float32[nh, w*w, w*w] out. */
RPP_API rpp_status rpp_swin_prepare_bias(const rpp_swin_cfg* cfg, const void* table, float* bias,
                                 rpp_stream stream);

/* Shifted-window attention with the cyclic shift, window partition, window reverse
 * and unshift folded into the kernel's gathers and scatters ([SW] §2-§3).
 *  qkv   device [B*I*I, 3C] of dtype in raster order (the QKV GEMM output)
 *  bias  device float32[nh, w*w, w*w] from rpp_swin_prepare_bias
 *  out   device [B*I*I, C] of dtype in raster order (before the output projection)
 * Token (y, x) of the shifted frame reads raster row ((y+s) mod I, (x+s) mod I); with
 * s > 0 two tokens of a window attend only when they lie in the same region of the
 * shifted frame (per axis: c < I-w, c < I-s, else). */
RPP_API rpp_status rpp_window_attention_forward(const rpp_swin_cfg* cfg, int B, const void* qkv,
                                        const float* bias, void* out, int32_t* err,
                                        rpp_stream stream);

/* Bytes of the prepared Swin block weights, and the preparation itself (K-major
 * weights, fp32 biases / LayerNorm parameters, the relative-position bias; at C = 96
 * with mlp = 384 also W1 as given, [C, mlp], read N-major by the fused MLP). */
RPP_API size_t rpp_swin_block_bytes(const rpp_swin_cfg* cfg);
RPP_API rpp_status rpp_swin_prepare_block(const rpp_swin_cfg* cfg, const rpp_swin_src* src, void* dst,
                                  rpp_stream stream);

/* Workspace bytes for rpp_swin_block_forward on B images. */
RPP_API size_t rpp_swin_workspace_bytes(const rpp_swin_cfg* cfg, int B);

/* Pre-LN Swin block on x [B*I*I, C] (raster order), y may alias x:
 *   x' = x + proj(WindowAttention(LN1 x)),  y = x' + W2 GELU(W1 LN2(x') + b1) + b2,
 * with the QKV projection run on raster-order tokens (a row-wise GEMM commutes with
 * the window permutation) and the permutation applied inside the attention kernel.
 * At C = 96 with mlp = 384 (Swin-T stage 1) the MLP line is one kernel whose hidden
 * activation [B*I*I, mlp] stays on chip; the other widths run it as two GEMMs. */
RPP_API rpp_status rpp_swin_block_forward(const rpp_swin_cfg* cfg, const void* block, int B, const void* x,
                                  void* y, void* workspace, size_t workspace_bytes, int32_t* err,
                                  rpp_stream stream);

/* ------------------------------------------------------------------------------
 * Swin stage downsampling (the talk's downsampling between stages; standard patch
 * merging): output token (py, px) = LayerNorm over the 4C concatenation of input tokens
 * (2py, 2px), (2py+1, 2px), (2py, 2px+1), (2py+1, 2px+1), then a bias-free 4C -> 2C map.
 * ------------------------------------------------------------------------------ */
typedef struct rpp_merge_cfg {
  int img;       /* I: input image side in tokens, even */
  int channels;  /* C: input channels (multiple of 8, <= 768); the output has 2C */
  float eps;     /* LayerNorm eps */
  int dtype;     /* RPP_F16 or RPP_BF16 */
} rpp_merge_cfg;

/* Bytes of the prepared weights, and the preparation: W [4C, 2C] of cfg dtype ([in, out],
 * input blocks in the concatenation order above) stored K-major; gamma, beta [4C] of cfg
 * dtype stored fp32.  dst: device, 16-byte aligned, rpp_patch_merge_bytes bytes. */
RPP_API size_t rpp_patch_merge_bytes(const rpp_merge_cfg* cfg);
RPP_API rpp_status rpp_patch_merge_prepare(const rpp_merge_cfg* cfg, const void* gamma, const void* beta,
                                           const void* W, void* dst, rpp_stream stream);
/* Workspace bytes for B images (the normalised 4C rows). */
RPP_API size_t rpp_patch_merge_workspace_bytes(const rpp_merge_cfg* cfg, int B);
/* x: device [B*I*I, C] raster order; y: device [B*(I/2)^2, 2C] raster order of the halved
 * image.  RPP_EUNSUPPORTED for odd I or C outside the supported set; RPP_EWORKSPACE if
 * workspace_bytes is too small. */
RPP_API rpp_status rpp_patch_merge_forward(const rpp_merge_cfg* cfg, const void* prepared, int B, const void* x,
                                           void* y, void* workspace, size_t workspace_bytes, int32_t* err,
                                           rpp_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* RPP_H_ */
