// The C ABI (include/rpp.h): argument validation, prepared-weight layouts, workspace
// carving and the orchestration of the per-step kernels.  Host code here launches
// kernels only; it never allocates, synchronises (except rpp_get_device_error) or
// reads device data, so call sequences are graph-capturable.
#include <cstring>

#include "kernels.h"

namespace rpp {

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }

inline int esize(rpp_dtype dt) { return dt == RPP_F32 ? 4 : (dt == RPP_I8 ? 1 : 2); }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline rpp_status from_cuda(cudaError_t e) { return status_from_cuda(e); }

// ---------------------------------------------------------------- launch-event hook
// While enabled (rpp_set_launch_events), every kernel launch of the path is followed
// by cudaEventRecord of the next caller-provided event on the launch's stream, and its
// label is kept, so a profiler can time each kernel inside the real step (eagerly or
// on replay of a captured graph).
// With a label filter set, events are recorded only around launches of that label:
// one just before the launch and one just after, so the other launches of the step
// keep their programmatic overlap.
struct LaunchHook {
  cudaEvent_t* events = nullptr;
  int capacity = 0;
  int count = 0;
  const char* labels[4096];
  char filter[64] = {0};
};
LaunchHook g_hook;

inline bool hook_matches(const char* label) {
  return g_hook.filter[0] == 0 || std::strncmp(label, g_hook.filter, sizeof(g_hook.filter)) == 0;
}

inline cudaError_t record_next(const char* label, cudaStream_t s) {
  if (g_hook.events && g_hook.count < g_hook.capacity) {
    if (g_hook.count < 4096) g_hook.labels[g_hook.count] = label;
    // inside stream capture the record becomes an event node of the graph, so the
    // kernels can be timed on graph replay, free of host launch gaps
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return cudaErrorUnknown;
    if (cs == cudaStreamCaptureStatusActive)
      return cudaEventRecordWithFlags(g_hook.events[g_hook.count++], s, cudaEventRecordExternal);
    return cudaEventRecord(g_hook.events[g_hook.count++], s);
  }
  return cudaSuccess;
}

inline cudaError_t note_before(const char* label, cudaStream_t s) {
  if (g_hook.events && g_hook.filter[0] && hook_matches(label)) return record_next(label, s);
  return cudaSuccess;
}

inline cudaError_t note(const char* label, cudaStream_t s) {
  if (g_hook.events && hook_matches(label)) return record_next(label, s);
  return cudaSuccess;
}

#define RPP_TRY(expr)                         \
  do {                                        \
    const rpp_status st_ = from_cuda(expr);   \
    if (st_ != RPP_OK) return st_;            \
  } while (0)

// launch, then (when profiling) record the event that marks its end
#define RPP_LAUNCH(label, stream, expr)          \
  do {                                           \
    RPP_TRY(note_before(label, stream));         \
    RPP_TRY(expr);                               \
    RPP_TRY(note(label, stream));                \
  } while (0)

// ---------------------------------------------------------------- prepared encoder layer
struct LayerLayout {
  size_t wqkv, wo, w1, w2;           // K-major weights (dtype, or bf16-held int8 codes)
  size_t bqkv, bo, b1, b2;           // fp32
  size_t g1, be1, g2, be2;           // fp32
  size_t sqkv, so, s1, s2;           // fp32 per-channel weight scales (int8)
  size_t total;
};

bool encoder_cfg_ok(const rpp_encoder_cfg* c) {
  if (!c) return false;
  if (c->hidden <= 0 || c->heads <= 0 || c->ffn <= 0 || c->head_dim <= 0) return false;
  if (c->heads * c->head_dim != c->hidden) return false;
  if (c->dtype != RPP_F32 && c->dtype != RPP_F16 && c->dtype != RPP_BF16) return false;
  if (c->int8 < 0 || c->int8 > 2) return false;
  if (c->int8 && c->dtype != RPP_F16) return false;
  return true;
}

rpp_status encoder_cfg_supported(const rpp_encoder_cfg* c) {
  if (!encoder_cfg_ok(c)) return RPP_EINVAL;
  const int H = c->hidden, F = c->ffn;
  if (c->head_dim != 64) return RPP_EUNSUPPORTED;
  const rpp_dtype dt = static_cast<rpp_dtype>(c->dtype);
  if (!layernorm_supported(H, dt)) return RPP_EUNSUPPORTED;
  if (dt == RPP_F32) {
    if (H % 4 || F % 4) return RPP_EUNSUPPORTED;
  } else {
    if (!gemm_tc_supported(3 * H, H) || !gemm_tc_supported(H, H) || !gemm_tc_supported(F, H) ||
        !gemm_tc_supported(H, F))
      return RPP_EUNSUPPORTED;
    if (c->int8 && F > 4096) return RPP_EUNSUPPORTED;
  }
  return RPP_OK;
}

LayerLayout layer_layout(const rpp_encoder_cfg* c) {
  LayerLayout L{};
  const size_t H = c->hidden, F = c->ffn;
  const size_t e = c->int8 ? 2 : esize(static_cast<rpp_dtype>(c->dtype));
  size_t o = 0;
  L.wqkv = o; o = align_up(o + 3 * H * H * e);
  L.wo = o;   o = align_up(o + H * H * e);
  L.w1 = o;   o = align_up(o + F * H * e);
  L.w2 = o;   o = align_up(o + H * F * e);
  L.bqkv = o; o = align_up(o + 3 * H * 4);
  L.bo = o;   o = align_up(o + H * 4);
  L.b1 = o;   o = align_up(o + F * 4);
  L.b2 = o;   o = align_up(o + H * 4);
  L.g1 = o;   o = align_up(o + H * 4);
  L.be1 = o;  o = align_up(o + H * 4);
  L.g2 = o;   o = align_up(o + H * 4);
  L.be2 = o;  o = align_up(o + H * 4);
  if (c->int8) {
    L.sqkv = o; o = align_up(o + 3 * H * 4);
    L.so = o;   o = align_up(o + H * 4);
    L.s1 = o;   o = align_up(o + F * 4);
    L.s2 = o;   o = align_up(o + H * 4);
  }
  L.total = o;
  return L;
}

constexpr int kMaxSplits = 4;   // K splits of the proj / FC2 GEMMs (partials summed by LayerNorm)

struct EncWs {
  size_t qkv, attn, h, x1, x1f, g, cx, ca, cx1, cg, total;
};

// bf16 layers keep a finer copy of the LN1 output for the FC2 residual (fp16 in the
// forward pass, fp32 in the calibration pass): with 8 significand bits, rounding that
// residual to bf16 would add up to half a bf16 step to the final output on top of the
// output's own rounding
inline bool fp32_residual(const rpp_encoder_cfg* c) { return c->dtype == RPP_BF16 && !c->int8; }

EncWs enc_ws_layout(const rpp_encoder_cfg* c, int T_max) {
  EncWs w{};
  const size_t T = T_max, H = c->hidden, F = c->ffn;
  const size_t e = esize(static_cast<rpp_dtype>(c->dtype));
  size_t o = 0;
  w.qkv = o;  o = align_up(o + T * 3 * H * e);
  w.attn = o; o = align_up(o + T * H * e);
  w.h = o;    o = align_up(o + kMaxSplits * T * H * 4);   // fp32 pre-LayerNorm sums (split-K slices)
  w.x1 = o;   o = align_up(o + T * H * e);
  if (fp32_residual(c)) {
    w.x1f = o; o = align_up(o + T * H * 4);
  }
  w.g = o;    o = align_up(o + T * F * e);
  if (c->int8) {   // bf16-held int8 codes of the four GEMM inputs
    w.cx = o;  o = align_up(o + T * H * 2);
    w.ca = o;  o = align_up(o + T * H * 2);
    w.cx1 = o; o = align_up(o + T * H * 2);
    w.cg = o;  o = align_up(o + T * F * 2);
  }
  w.total = o;
  return w;
}

template <typename P>
inline P* at(void* base, size_t off) {
  return reinterpret_cast<P*>(static_cast<uint8_t*>(base) + off);
}
template <typename P>
inline const P* at(const void* base, size_t off) {
  return reinterpret_cast<const P*>(static_cast<const uint8_t*>(base) + off);
}

// one GEMM of the float path: tensor cores for fp16 / bf16, CUDA cores for fp32
cudaError_t linear(rpp_dtype dt, const void* a, const void* w_t, const float* bias, const void* residual, void* out,
                   int M_max, const int32_t* rows, int N, int K, int epi, int32_t* err, cudaStream_t s,
                   rpp_dtype out_dt = RPP_I8 /* = dt */, rpp_dtype res_dt = RPP_I8 /* = dt */, int rows_hint = 0,
                   int max_splits = 1, int* splits_out = nullptr) {
  if (splits_out) *splits_out = 1;
  if (out_dt == RPP_I8) out_dt = dt;
  if (res_dt == RPP_I8) res_dt = dt;
  if (dt == RPP_F32)
    return launch_gemm_f32(static_cast<const float*>(a), static_cast<const float*>(w_t), bias,
                           static_cast<const float*>(residual), static_cast<float*>(out), M_max, rows, N, K, epi, err,
                           s);
  TcGemmArgs g{};
  g.a = a; g.w_t = w_t; g.bias = bias; g.residual = residual; g.out = out;
  g.M_max = M_max; g.rows = rows; g.N = N; g.K = K;
  g.in_dtype = dt; g.out_dtype = out_dt; g.res_dtype = res_dt; g.epi = epi; g.err = err;
  g.rows_hint = rows_hint; g.max_splits = max_splits; g.splits_out = splits_out;
  return launch_gemm_tc(g, s);
}

// one GEMM of the int8 path (bf16-held codes in, fp16 / codes out)
cudaError_t linear_i8(const void* a_codes, const void* w_codes, const float* bias, const float* a_scale,
                      const float* w_scale, const float* q_scale, const void* residual, void* out, rpp_dtype out_dt,
                      int M_max, const int32_t* rows, int N, int K, int epi, int32_t* err, cudaStream_t s,
                      int rows_hint) {
  TcGemmArgs g{};
  g.rows_hint = rows_hint;
  g.a = a_codes; g.w_t = w_codes; g.bias = bias; g.residual = residual; g.out = out;
  g.M_max = M_max; g.rows = rows; g.N = N; g.K = K;
  g.in_dtype = RPP_BF16; g.out_dtype = out_dt; g.epi = epi;
  g.a_scale = a_scale; g.w_scale = w_scale; g.q_scale = q_scale; g.err = err;
  return launch_gemm_tc(g, s);
}

// Padded output of the last layer: LN2 writes y straight into the padded [B*L, H]
// layout with zero pad slots (the padding rebuild, fused into the last kernel).
struct PaddedOut {
  void* y = nullptr;
  int L = 0;
};

rpp_status encoder_layer_run(const rpp_encoder_cfg* c, const void* layer, const float* act_scales, const void* x,
                             const int32_t* cu, int B, int T_max, int max_len, void* y, void* ws, size_t ws_bytes,
                             float* amax, int32_t* err, cudaStream_t s, PaddedOut pad = PaddedOut{}) {
  rpp_status st = encoder_cfg_supported(c);
  if (st != RPP_OK) return st;
  if (!layer || !x || !cu || !y || !ws || B <= 0 || T_max <= 0 || max_len <= 0) return RPP_EINVAL;
  if (!aligned16(x) || !aligned16(y) || !aligned16(ws) || !aligned16(layer)) return RPP_EINVAL;
  if (c->int8 && !act_scales) return RPP_EINVAL;
  const EncWs W = enc_ws_layout(c, T_max);
  if (ws_bytes < W.total) return RPP_EWORKSPACE;
  const LayerLayout P = layer_layout(c);
  const rpp_dtype dt = static_cast<rpp_dtype>(c->dtype);
  const int H = c->hidden, F = c->ffn, nh = c->heads, d = c->head_dim;
  const int32_t* rows = cu + B;   // T lives in device memory
  const int hint = c->tokens_hint > 0 && c->tokens_hint < T_max ? c->tokens_hint : T_max;
  const long long hs = static_cast<long long>(T_max) * H;   // elements between split-K slices
  int sp_proj = 1, sp_fc2 = 1;
  void* qkv = at<void>(ws, W.qkv);
  void* attn = at<void>(ws, W.attn);
  void* h = at<void>(ws, W.h);
  void* x1 = at<void>(ws, W.x1);
  void* g = at<void>(ws, W.g);
  // the pre-LayerNorm residual sums stay fp32 (fp32 layers: same type)
  const rpp_dtype hdt = RPP_F32;
  const float* bqkv = at<float>(layer, P.bqkv);
  const float* bo = at<float>(layer, P.bo);
  const float* b1 = at<float>(layer, P.b1);
  const float* b2 = at<float>(layer, P.b2);
  const float* g1 = at<float>(layer, P.g1);
  const float* be1 = at<float>(layer, P.be1);
  const float* g2 = at<float>(layer, P.g2);
  const float* be2 = at<float>(layer, P.be2);

  // LayerNorm launches: LN(x_sum) with x_sum = slices of h + bias + residual
  auto ln_args = [&](const float* gamma, const float* beta) {
    LnArgs a{};
    a.x = h;
    a.in_dtype = hdt;
    a.gamma = gamma;
    a.beta = beta;
    a.out_dtype = dt;
    a.M_max = T_max;
    a.rows = rows;
    a.H = H;
    a.eps = c->eps;
    a.err = err;
    return a;
  };
  auto final_ln = [&](LnArgs a) {   // LN2: optionally straight into the padded output
    if (pad.y) {
      a.y = pad.y;
      a.pad_cu = cu;
      a.pad_B = B;
      a.pad_L = pad.L;
    }
    return a;
  };
  if (!c->int8 && dt != RPP_F32 && !amax) {
    // proj and FC2 add their bias and the residual in the GEMM epilogue and write the
    // pre-LayerNorm sum once ([SW] §3: bias split off the GEMM and fused into the op
    // before LayerNorm; [KS] Fig. 7: each kernel's precision chosen for its values).
    // fp16 layers keep the sum in fp16 (its rounding is that of the output).  bf16 layers
    // keep it in fp32, and LN1 also writes x1 in fp16 as the FC2 residual (8 times finer
    // than the bf16 x1): an fp16 sum as well put the bf16 BERT-large layer above the 2e-2
    // bound (max-abs 2.09e-2, layer 8 of 24), whose bf16 output rounding alone is 1.56e-2
    // for outputs in [4, 8); with the fp32 sum and the fp16 residual the worst layer is at
    // 1.98e-2, with an fp32 residual at 1.85e-2.
    const bool f32sum = dt == RPP_BF16;
    const rpp_dtype sdt = f32sum ? RPP_F32 : RPP_F16;
    void* hsum = h;   // [T_max, H] inside the split-K slice region
    __half* x1h = f32sum ? at<__half>(ws, W.x1f) : nullptr;   // the fp16 copy of x1 (bf16 layers)
    RPP_LAUNCH("gemm_qkv", s, linear(dt, x, at<void>(layer, P.wqkv), bqkv, nullptr, qkv, T_max, rows, 3 * H, H,
                                     RPP_EPI_BIAS, err, s, RPP_I8, RPP_I8, hint));
    RPP_LAUNCH("attention", s, launch_attention_varlen(qkv, cu, B, T_max, max_len, nh, d, dt, attn, err, s));
    RPP_LAUNCH("gemm_proj", s, linear(dt, attn, at<void>(layer, P.wo), bo, x, hsum, T_max, rows, H, H,
                                      RPP_EPI_BIAS_RESIDUAL, err, s, sdt, dt, hint));
    LnArgs l1 = ln_args(g1, be1);
    l1.x = hsum;
    l1.in_dtype = sdt;
    l1.y = x1;
    l1.y16 = x1h;
    RPP_LAUNCH("layernorm1", s, launch_layernorm(l1, s));
    RPP_LAUNCH("gemm_fc1", s, linear(dt, x1, at<void>(layer, P.w1), b1, nullptr, g, T_max, rows, F, H,
                                     RPP_EPI_BIAS_GELU, err, s, RPP_I8, RPP_I8, hint));
    RPP_LAUNCH("gemm_fc2", s, linear(dt, g, at<void>(layer, P.w2), b2, x1h ? static_cast<const void*>(x1h) : x1, hsum,
                                     T_max, rows, H, F, RPP_EPI_BIAS_RESIDUAL, err, s, sdt, x1h ? RPP_F16 : dt,
                                     hint));
    LnArgs l2 = ln_args(g2, be2);
    l2.x = hsum;
    l2.in_dtype = sdt;
    l2.y = y;
    RPP_LAUNCH(pad.y ? "layernorm2_rebuild" : "layernorm2", s, launch_layernorm(final_ln(l2), s));
    return RPP_OK;
  }
  if (!c->int8) {
    // Calibration passes of 16-bit layers: proj / FC2 write raw fp32 accumulators
    // (split-K slices); the LayerNorm after each adds the slices, the GEMM's bias and the
    // residual while it reads the row ([SW] §3: bias split off the GEMM and fused into
    // the next op), and records the max-abs of its output.  The fp32 layer runs its
    // GEMMs on CUDA cores, with bias and residual in the GEMM epilogue.
    const bool tc = dt != RPP_F32;
    float* x1f = fp32_residual(c) ? at<float>(ws, W.x1f) : nullptr;
    if (amax) RPP_LAUNCH("amax", s, launch_amax(x, T_max, rows, H, dt, amax + 0, err, s));
    RPP_LAUNCH("gemm_qkv", s, linear(dt, x, at<void>(layer, P.wqkv), bqkv, nullptr, qkv, T_max, rows, 3 * H, H,
                                     RPP_EPI_BIAS, err, s, RPP_I8, RPP_I8, hint));
    if (amax && tc) RPP_LAUNCH("amax_qkv", s, launch_amax_parts(qkv, T_max, rows, 3 * H, H, dt, amax + 4, err, s));
    RPP_LAUNCH("attention", s, launch_attention_varlen(qkv, cu, B, T_max, max_len, nh, d, dt, attn, err, s));
    if (amax) RPP_LAUNCH("amax", s, launch_amax(attn, T_max, rows, H, dt, amax + 1, err, s));
    LnArgs l1 = ln_args(g1, be1);
    l1.y = x1;
    l1.y32 = x1f;
    l1.amax = amax ? amax + 2 : nullptr;
    if (tc) {
      RPP_LAUNCH("gemm_proj", s, linear(dt, attn, at<void>(layer, P.wo), nullptr, nullptr, h, T_max, rows, H, H,
                                        EPI_ACC, err, s, hdt, RPP_I8, hint, kMaxSplits, &sp_proj));
      l1.n_in = sp_proj;
      l1.in_stride = hs;
      l1.add_bias = bo;
      l1.residual = x;
      l1.res_dtype = dt;
    } else {
      RPP_LAUNCH("gemm_proj", s, linear(dt, attn, at<void>(layer, P.wo), bo, x, h, T_max, rows, H, H,
                                        RPP_EPI_BIAS_RESIDUAL, err, s));
    }
    RPP_LAUNCH("layernorm1", s, launch_layernorm(l1, s));
    RPP_LAUNCH("gemm_fc1", s, linear(dt, x1, at<void>(layer, P.w1), b1, nullptr, g, T_max, rows, F, H,
                                     RPP_EPI_BIAS_GELU, err, s, RPP_I8, RPP_I8, hint));
    if (amax) RPP_LAUNCH("amax", s, launch_amax(g, T_max, rows, F, dt, amax + 3, err, s));
    LnArgs l2 = ln_args(g2, be2);
    l2.y = y;
    if (tc) {
      RPP_LAUNCH("gemm_fc2", s, linear(dt, g, at<void>(layer, P.w2), nullptr, nullptr, h, T_max, rows, H, F, EPI_ACC,
                                       err, s, hdt, RPP_I8, hint, kMaxSplits, &sp_fc2));
      l2.n_in = sp_fc2;
      l2.in_stride = hs;
      l2.add_bias = b2;
      l2.residual = x1f ? static_cast<const void*>(x1f) : x1;
      l2.res_dtype = x1f ? RPP_F32 : dt;
    } else {
      RPP_LAUNCH("gemm_fc2", s, linear(dt, g, at<void>(layer, P.w2), b2, x1, h, T_max, rows, H, F,
                                       RPP_EPI_BIAS_RESIDUAL, err, s));
    }
    RPP_LAUNCH(pad.y ? "layernorm2_rebuild" : "layernorm2", s, launch_layernorm(final_ln(l2), s));
    return RPP_OK;
  }
  // int8: quantise -> int8 GEMM (exact integer accumulation) -> dequantise in the epilogue
  void* cx = at<void>(ws, W.cx);
  void* ca = at<void>(ws, W.ca);
  void* cx1 = at<void>(ws, W.cx1);
  void* cg = at<void>(ws, W.cg);
  const float* s0 = act_scales + 0;
  const float* s1 = act_scales + 1;
  const float* s2 = act_scales + 2;
  const float* s3 = act_scales + 3;
  RPP_LAUNCH("quantize_x", s, launch_quantize_codes_bf16(x, s0, cx, T_max, rows, H, dt, err, s));
  if (c->int8 == 2) {
    // all-int8 flow: the QKV GEMM writes the codes of Q, K and V (scales act_scales[4..6])
    // and the attention runs both of its products on codes
    const float* sqkv = act_scales + 4;
    RPP_LAUNCH("gemm_qkv_i8", s, linear_i8(cx, at<void>(layer, P.wqkv), bqkv, s0, at<float>(layer, P.sqkv), sqkv,
                                            nullptr, qkv, RPP_BF16, T_max, rows, 3 * H, H, EPI_DQ_BIAS_Q3, err, s,
                                            hint));
    // the attention also writes the codes of its output at s1 (the proj GEMM's input)
    RPP_LAUNCH("attention_i8", s,
               launch_attention_sched(qkv, cu, B, T_max, max_len, nh, RPP_BF16, ca, err, s, sqkv, s1));
  } else {
    RPP_LAUNCH("gemm_qkv_i8", s, linear_i8(cx, at<void>(layer, P.wqkv), bqkv, s0, at<float>(layer, P.sqkv), nullptr,
                                            nullptr, qkv, dt, T_max, rows, 3 * H, H, EPI_DQ_BIAS, err, s, hint));
    if (d == 64 && attention_sched_supported(B, max_len)) {   // quantisation fused into the attention's output
      RPP_LAUNCH("attention", s,
                 launch_attention_sched(qkv, cu, B, T_max, max_len, nh, dt, ca, err, s, nullptr, s1));
    } else {
      RPP_LAUNCH("attention", s, launch_attention_varlen(qkv, cu, B, T_max, max_len, nh, d, dt, attn, err, s));
      RPP_LAUNCH("quantize_attn", s, launch_quantize_codes_bf16(attn, s1, ca, T_max, rows, H, dt, err, s));
    }
  }
  RPP_LAUNCH("gemm_proj_i8", s, linear_i8(ca, at<void>(layer, P.wo), nullptr, s1, at<float>(layer, P.so), nullptr,
                                           nullptr, h, RPP_F32, T_max, rows, H, H, EPI_DQ_ACC, err, s, hint));
  LnArgs l1 = ln_args(g1, be1);
  l1.add_bias = bo;
  l1.residual = x;
  l1.res_dtype = dt;
  l1.y = x1;
  l1.q_codes = cx1;
  l1.q_scale = s2;
  RPP_LAUNCH("layernorm1", s, launch_layernorm(l1, s));
  RPP_LAUNCH("gemm_fc1_i8", s, linear_i8(cx1, at<void>(layer, P.w1), b1, s2, at<float>(layer, P.s1), s3, nullptr, cg,
                                          RPP_BF16, T_max, rows, F, H, EPI_DQ_BIAS_GELU_Q, err, s, hint));
  RPP_LAUNCH("gemm_fc2_i8", s, linear_i8(cg, at<void>(layer, P.w2), nullptr, s3, at<float>(layer, P.s2), nullptr,
                                          nullptr, h, RPP_F32, T_max, rows, H, F, EPI_DQ_ACC, err, s, hint));
  LnArgs l2 = ln_args(g2, be2);
  l2.add_bias = b2;
  l2.residual = x1;
  l2.res_dtype = dt;
  l2.y = y;
  RPP_LAUNCH(pad.y ? "layernorm2_rebuild" : "layernorm2", s, launch_layernorm(final_ln(l2), s));
  return RPP_OK;
}

// ---------------------------------------------------------------- prepared Swin block
struct SwinLayout {
  size_t wqkv, wo, w1, w2, w1kn, bqkv, bo, b1, b2, g1, be1, g2, be2, bias, total;
};

rpp_status swin_cfg_supported(const rpp_swin_cfg* c) {
  if (!c) return RPP_EINVAL;
  if (c->img <= 0 || c->channels <= 0 || c->heads <= 0 || c->window <= 0 || c->mlp <= 0) return RPP_EINVAL;
  if (c->shift < 0 || c->shift >= c->window || c->img % c->window) return RPP_EINVAL;
  if (c->dtype != RPP_F16 && c->dtype != RPP_BF16) return RPP_EUNSUPPORTED;
  if (!window_attention_supported(c->channels, c->heads, c->window, c->img, c->shift)) return RPP_EUNSUPPORTED;
  const int C = c->channels, F = c->mlp;
  if (!layernorm_supported(C, static_cast<rpp_dtype>(c->dtype))) return RPP_EUNSUPPORTED;
  if (!gemm_tc_supported(3 * C, C) || !gemm_tc_supported(C, C) || !gemm_tc_supported(F, C) ||
      !gemm_tc_supported(C, F))
    return RPP_EUNSUPPORTED;
  return RPP_OK;
}

SwinLayout swin_layout(const rpp_swin_cfg* c) {
  SwinLayout L{};
  const size_t C = c->channels, F = c->mlp, e = 2, N = c->window * c->window;
  size_t o = 0;
  L.wqkv = o; o = align_up(o + 3 * C * C * e);
  L.wo = o;   o = align_up(o + C * C * e);
  L.w1 = o;   o = align_up(o + F * C * e);
  L.w2 = o;   o = align_up(o + C * F * e);
  L.w1kn = o; o = align_up(o + (swin_mlp_supported(c->channels, c->mlp) ? C * F * e : 0));   // fused MLP's W1
  L.bqkv = o; o = align_up(o + 3 * C * 4);
  L.bo = o;   o = align_up(o + C * 4);
  L.b1 = o;   o = align_up(o + F * 4);
  L.b2 = o;   o = align_up(o + C * 4);
  L.g1 = o;   o = align_up(o + C * 4);
  L.be1 = o;  o = align_up(o + C * 4);
  L.g2 = o;   o = align_up(o + C * 4);
  L.be2 = o;  o = align_up(o + C * 4);
  L.bias = o; o = align_up(o + c->heads * N * N * 4);
  L.total = o;
  return L;
}

struct SwinWs {
  size_t h, qkv, attn, xa, g, total;
};
SwinWs swin_ws_layout(const rpp_swin_cfg* c, int B) {
  SwinWs w{};
  const size_t T = static_cast<size_t>(B) * c->img * c->img, C = c->channels, F = c->mlp, e = 2;
  size_t o = 0;
  w.h = o;    o = align_up(o + T * C * e);
  w.qkv = o;  o = align_up(o + T * 3 * C * e);
  w.attn = o; o = align_up(o + T * C * e);
  w.xa = o;   o = align_up(o + T * C * e);
  w.g = o;    o = align_up(o + T * F * e);
  w.total = o;
  return w;
}

}  // namespace
}  // namespace rpp

using namespace rpp;

extern "C" {

const char* rpp_status_string(int status) {
  switch (status) {
    case RPP_OK: return "ok";
    case RPP_EINVAL: return "invalid argument";
    case RPP_EUNSUPPORTED: return "unsupported shape or dtype";
    case RPP_ECUDA: return "CUDA runtime error";
    case RPP_EWORKSPACE: return "workspace too small";
    case RPP_EDEVICE: return "device-side error recorded";
    default: return "unknown status";
  }
}

int rpp_version(void) { return 100; }

rpp_status rpp_set_launch_events(void* const* events, int capacity) {
  if (capacity < 0 || (capacity > 0 && !events)) return RPP_EINVAL;
  g_hook.events = capacity > 0 ? reinterpret_cast<cudaEvent_t*>(const_cast<void**>(events)) : nullptr;
  g_hook.capacity = capacity;
  g_hook.count = 0;
  return RPP_OK;
}

rpp_status rpp_set_gemm_cluster_mode(int mode) {
  if (mode < 0 || mode > 2) return RPP_EINVAL;
  set_gemm_cluster_mode(mode);
  return RPP_OK;
}

rpp_status rpp_set_gemm_tile_width(int bn) {
  static const int ok[] = {0, 16, 32, 48, 64, 96, 128, 144, 192, 256};
  for (int v : ok)
    if (bn == v) {
      set_gemm_force_bn(bn);
      return RPP_OK;
    }
  return RPP_EINVAL;
}

rpp_status rpp_test_stall_next_gemm(unsigned int limit_us) {
  if (limit_us == 0 || limit_us > 1000000u) return RPP_EINVAL;
  set_gemm_stall_next(static_cast<unsigned long long>(limit_us) * 1000ull);
  return RPP_OK;
}

rpp_status rpp_set_launch_event_filter(const char* label) {
  if (!label) {
    g_hook.filter[0] = 0;
    return RPP_OK;
  }
  const size_t n = std::strlen(label);
  if (n == 0 || n >= sizeof(g_hook.filter)) return RPP_EINVAL;
  std::memcpy(g_hook.filter, label, n + 1);
  return RPP_OK;
}

int rpp_launch_event_count(void) { return g_hook.count; }

const char* rpp_launch_event_label(int i) {
  if (i < 0 || i >= g_hook.count || i >= 4096) return "";
  return g_hook.labels[i];
}

rpp_status rpp_get_device_error(const int32_t* err, int32_t* host_code, rpp_stream stream) {
  if (!err || !host_code) return RPP_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, err, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess) return RPP_ECUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return RPP_ECUDA;
  *host_code = v;
  return v ? RPP_EDEVICE : RPP_OK;
}

rpp_status rpp_build_offsets(const int32_t* lengths, int B, int L, int32_t* cu_seqlens, int32_t* padding_offset,
                             int32_t* err, rpp_stream stream) {
  if (!lengths || !cu_seqlens || !padding_offset || B <= 0 || L <= 0 || B > 65536) return RPP_EINVAL;
  if (static_cast<long long>(B) * L > 0x7fffffffLL) return RPP_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  RPP_LAUNCH("build_offsets", s, launch_build_offsets(lengths, B, L, cu_seqlens, padding_offset, err, s));
  return RPP_OK;
}

rpp_status rpp_remove_padding(const void* padded, const int32_t* padding_offset, const int32_t* cu_seqlens, int B,
                              int L, int H, rpp_dtype dtype, void* packed, int32_t* err, rpp_stream stream) {
  if (!padded || !padding_offset || !cu_seqlens || !packed || B <= 0 || L <= 0 || H <= 0) return RPP_EINVAL;
  if (dtype < RPP_F32 || dtype > RPP_I8) return RPP_EINVAL;
  const long long row_bytes = static_cast<long long>(H) * esize(dtype);
  if (row_bytes % 16 || !aligned16(padded) || !aligned16(packed)) return RPP_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  RPP_LAUNCH("remove_padding", s, launch_remove_padding(padded, padding_offset, cu_seqlens, B, L,
                                                        static_cast<int>(row_bytes), packed, err, s));
  return RPP_OK;
}

rpp_status rpp_rebuild_padding(const void* packed, const int32_t* cu_seqlens, int B, int L, int H, rpp_dtype dtype,
                               void* padded, int32_t* err, rpp_stream stream) {
  if (!packed || !cu_seqlens || !padded || B <= 0 || L <= 0 || H <= 0) return RPP_EINVAL;
  if (dtype < RPP_F32 || dtype > RPP_I8) return RPP_EINVAL;
  const long long row_bytes = static_cast<long long>(H) * esize(dtype);
  if (row_bytes % 16 || !aligned16(padded) || !aligned16(packed)) return RPP_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  RPP_LAUNCH("rebuild_padding", s, launch_rebuild_padding(packed, cu_seqlens, B, L, static_cast<int>(row_bytes), padded,
                                                          err, s));
  return RPP_OK;
}

rpp_status rpp_linear(const void* a, const void* w_t, const float* bias, const void* residual, void* out, int M_max,
                      const int32_t* rows, int N, int K, rpp_dtype dtype, rpp_epilogue epilogue, int32_t* err,
                      rpp_stream stream) {
  if (!a || !w_t || !bias || !out || M_max <= 0 || N <= 0 || K <= 0) return RPP_EINVAL;
  if (epilogue != RPP_EPI_BIAS && epilogue != RPP_EPI_BIAS_GELU && epilogue != RPP_EPI_BIAS_RESIDUAL)
    return RPP_EINVAL;
  if (epilogue == RPP_EPI_BIAS_RESIDUAL && !residual) return RPP_EINVAL;
  if (!aligned16(a) || !aligned16(w_t) || !aligned16(out) || !aligned16(bias) || (residual && !aligned16(residual)))
    return RPP_EINVAL;
  if (dtype == RPP_F32) {
    if (K % 4 || N % 4) return RPP_EUNSUPPORTED;
  } else if (dtype == RPP_F16 || dtype == RPP_BF16) {
    if (!gemm_tc_supported(N, K)) return RPP_EUNSUPPORTED;
  } else {
    return RPP_EUNSUPPORTED;
  }
  return from_cuda(linear(dtype, a, w_t, bias, residual, out, M_max, rows, N, K, epilogue, err,
                          static_cast<cudaStream_t>(stream)));
}

rpp_status rpp_layernorm(const void* x, const float* gamma, const float* beta, void* y, int M_max, const int32_t* rows,
                         int H, float eps, rpp_dtype dtype, int32_t* err, rpp_stream stream) {
  if (!x || !gamma || !beta || !y || M_max <= 0 || H <= 0) return RPP_EINVAL;
  if (!aligned16(x) || !aligned16(y) || !aligned16(gamma) || !aligned16(beta)) return RPP_EINVAL;
  if (dtype != RPP_F32 && dtype != RPP_F16 && dtype != RPP_BF16) return RPP_EUNSUPPORTED;
  if (!layernorm_supported(H, dtype)) return RPP_EUNSUPPORTED;
  LnArgs a{};
  a.x = x;
  a.in_dtype = dtype;
  a.gamma = gamma;
  a.beta = beta;
  a.y = y;
  a.out_dtype = dtype;
  a.M_max = M_max;
  a.rows = rows;
  a.H = H;
  a.eps = eps;
  a.err = err;
  return from_cuda(launch_layernorm(a, static_cast<cudaStream_t>(stream)));
}

rpp_status rpp_attention_varlen(const void* qkv, const int32_t* cu_seqlens, int B, int T_max, int max_len, int nh,
                                int d, rpp_dtype dtype, void* out, int32_t* err, rpp_stream stream) {
  if (!qkv || !cu_seqlens || !out || B <= 0 || T_max <= 0 || max_len <= 0 || nh <= 0 || d <= 0) return RPP_EINVAL;
  if (!aligned16(qkv) || !aligned16(out)) return RPP_EINVAL;
  if (d != 64) return RPP_EUNSUPPORTED;
  if (dtype != RPP_F32 && dtype != RPP_F16 && dtype != RPP_BF16) return RPP_EUNSUPPORTED;
  if (B > 65535 || nh > 65535) return RPP_EUNSUPPORTED;
  return from_cuda(launch_attention_varlen(qkv, cu_seqlens, B, T_max, max_len, nh, d, dtype, out, err,
                                           static_cast<cudaStream_t>(stream)));
}

rpp_status rpp_attention_varlen_i8(const void* qkv_codes, const float* qkv_scales, const int32_t* cu_seqlens, int B,
                                   int T_max, int max_len, int nh, int d, void* out, int32_t* err,
                                   rpp_stream stream) {
  if (!qkv_codes || !qkv_scales || !cu_seqlens || !out || B <= 0 || T_max <= 0 || max_len <= 0 || nh <= 0 || d <= 0)
    return RPP_EINVAL;
  if (!aligned16(qkv_codes) || !aligned16(out)) return RPP_EINVAL;
  if (d != 64 || !attention_sched_supported(B, max_len) || nh > 65535) return RPP_EUNSUPPORTED;
  return from_cuda(launch_attention_sched(qkv_codes, cu_seqlens, B, T_max, max_len, nh, RPP_BF16, out, err,
                                          static_cast<cudaStream_t>(stream), qkv_scales));
}

size_t rpp_layer_bytes(const rpp_encoder_cfg* cfg) {
  if (!encoder_cfg_ok(cfg)) return 0;
  return layer_layout(cfg).total;
}

rpp_status rpp_prepare_layer(const rpp_encoder_cfg* cfg, const rpp_layer_src* src, void* dst, rpp_stream stream) {
  rpp_status st = encoder_cfg_supported(cfg);
  if (st != RPP_OK) return st;
  if (!src || !dst || !aligned16(dst)) return RPP_EINVAL;
  const void* ptrs[] = {src->Wq, src->Wk, src->Wv, src->bq, src->bk, src->bv, src->Wo, src->bo, src->W1,
                        src->b1, src->W2, src->b2, src->gamma1, src->beta1, src->gamma2, src->beta2};
  for (const void* p : ptrs)
    if (!p) return RPP_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const LayerLayout P = layer_layout(cfg);
  const rpp_dtype dt = static_cast<rpp_dtype>(cfg->dtype);
  const int H = cfg->hidden, F = cfg->ffn, e = esize(dt);
  if (!cfg->int8) {
    // Wq | Wk | Wv concatenated as rows of one [3H, H] K-major matrix
    uint8_t* wqkv = at<uint8_t>(dst, P.wqkv);
    RPP_TRY(launch_transpose_to_kmajor(src->Wq, H, H, e, wqkv, H, s));
    RPP_TRY(launch_transpose_to_kmajor(src->Wk, H, H, e, wqkv + static_cast<size_t>(H) * H * e, H, s));
    RPP_TRY(launch_transpose_to_kmajor(src->Wv, H, H, e, wqkv + 2 * static_cast<size_t>(H) * H * e, H, s));
    RPP_TRY(launch_transpose_to_kmajor(src->Wo, H, H, e, at<void>(dst, P.wo), H, s));
    RPP_TRY(launch_transpose_to_kmajor(src->W1, H, F, e, at<void>(dst, P.w1), H, s));
    RPP_TRY(launch_transpose_to_kmajor(src->W2, F, H, e, at<void>(dst, P.w2), F, s));
  } else {
    // int8: the per-channel scales of Wq, Wk, Wv are the per-column scales of the
    // concatenated [H, 3H] matrix, so each part is quantised on its own
    __nv_bfloat16* wqkv = at<__nv_bfloat16>(dst, P.wqkv);
    float* sq = at<float>(dst, P.sqkv);
    RPP_TRY(launch_quantize_weight(src->Wq, H, H, dt, nullptr, wqkv, sq, s));
    RPP_TRY(launch_quantize_weight(src->Wk, H, H, dt, nullptr, wqkv + static_cast<size_t>(H) * H, sq + H, s));
    RPP_TRY(launch_quantize_weight(src->Wv, H, H, dt, nullptr, wqkv + 2 * static_cast<size_t>(H) * H, sq + 2 * H, s));
    RPP_TRY(launch_quantize_weight(src->Wo, H, H, dt, nullptr, at<void>(dst, P.wo), at<float>(dst, P.so), s));
    RPP_TRY(launch_quantize_weight(src->W1, H, F, dt, nullptr, at<void>(dst, P.w1), at<float>(dst, P.s1), s));
    RPP_TRY(launch_quantize_weight(src->W2, F, H, dt, nullptr, at<void>(dst, P.w2), at<float>(dst, P.s2), s));
  }
  float* bqkv = at<float>(dst, P.bqkv);
  RPP_TRY(launch_to_f32(src->bq, dt, H, bqkv, s));
  RPP_TRY(launch_to_f32(src->bk, dt, H, bqkv + H, s));
  RPP_TRY(launch_to_f32(src->bv, dt, H, bqkv + 2 * H, s));
  RPP_TRY(launch_to_f32(src->bo, dt, H, at<float>(dst, P.bo), s));
  RPP_TRY(launch_to_f32(src->b1, dt, F, at<float>(dst, P.b1), s));
  RPP_TRY(launch_to_f32(src->b2, dt, H, at<float>(dst, P.b2), s));
  RPP_TRY(launch_to_f32(src->gamma1, dt, H, at<float>(dst, P.g1), s));
  RPP_TRY(launch_to_f32(src->beta1, dt, H, at<float>(dst, P.be1), s));
  RPP_TRY(launch_to_f32(src->gamma2, dt, H, at<float>(dst, P.g2), s));
  RPP_TRY(launch_to_f32(src->beta2, dt, H, at<float>(dst, P.be2), s));
  return RPP_OK;
}

size_t rpp_encoder_workspace_bytes(const rpp_encoder_cfg* cfg, int T_max) {
  if (!encoder_cfg_ok(cfg) || T_max <= 0) return 0;
  return enc_ws_layout(cfg, T_max).total;
}

rpp_status rpp_encoder_layer_forward(const rpp_encoder_cfg* cfg, const void* layer, const float* act_scales,
                                     const void* x, const int32_t* cu_seqlens, int B, int T_max, int max_len, void* y,
                                     void* workspace, size_t workspace_bytes, int32_t* err, rpp_stream stream) {
  return encoder_layer_run(cfg, layer, act_scales, x, cu_seqlens, B, T_max, max_len, y, workspace, workspace_bytes,
                           nullptr, err, static_cast<cudaStream_t>(stream));
}

rpp_status rpp_encoder_layer_calibrate(const rpp_encoder_cfg* cfg, const void* layer, const void* x,
                                       const int32_t* cu_seqlens, int B, int T_max, int max_len, float* amax_out,
                                       void* workspace, size_t workspace_bytes, int32_t* err, rpp_stream stream) {
  if (!cfg || cfg->int8 || !amax_out) return RPP_EINVAL;
  if (cfg->dtype == RPP_F32) return RPP_EUNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(amax_out, 0, 7 * sizeof(float), s) != cudaSuccess) return RPP_ECUDA;
  const size_t need = enc_ws_layout(cfg, T_max > 0 ? T_max : 1).total;
  if (workspace_bytes < need) return RPP_EWORKSPACE;
  // the output of the calibration pass is not needed: it goes to the QKV buffer, which
  // is dead once attention has run
  void* y = at<void>(workspace, enc_ws_layout(cfg, T_max).qkv);
  return encoder_layer_run(cfg, layer, nullptr, x, cu_seqlens, B, T_max, max_len, y, workspace, workspace_bytes,
                           amax_out, err, s);
}

rpp_status rpp_encoder_forward(const rpp_encoder_cfg* cfg, const void* const* layers, const float* const* act_scales,
                               int num_layers, const int32_t* lengths, int B, int L, const void* x_padded,
                               void* y_padded, int32_t* cu_seqlens, int32_t* padding_offset, void* packed,
                               void* workspace, size_t workspace_bytes, int32_t* err, rpp_stream stream) {
  rpp_status st = encoder_cfg_supported(cfg);
  if (st != RPP_OK) return st;
  if (!layers || num_layers <= 0 || !lengths || !x_padded || !y_padded || !cu_seqlens || !padding_offset || !packed)
    return RPP_EINVAL;
  for (int i = 0; i < num_layers; ++i)   // every layer is checked before any kernel is launched
    if (!layers[i] || !aligned16(layers[i])) return RPP_EINVAL;
  if (cfg->int8 && !act_scales) return RPP_EINVAL;
  const rpp_dtype dt = static_cast<rpp_dtype>(cfg->dtype);
  const int H = cfg->hidden;
  const int T_max = B * L;
  if (workspace_bytes < enc_ws_layout(cfg, T_max).total) return RPP_EWORKSPACE;
  if (offsets_remove_fusable(B) && aligned16(x_padded) && aligned16(packed) && (H * esize(dt)) % 16 == 0 &&
      static_cast<long long>(B) * L <= 0x7fffffffLL) {
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    RPP_LAUNCH("offsets_remove", cs, launch_offsets_remove(lengths, B, L, H * esize(dt), x_padded, cu_seqlens,
                                                           padding_offset, packed, err, cs));
  } else {
    st = rpp_build_offsets(lengths, B, L, cu_seqlens, padding_offset, err, stream);
    if (st != RPP_OK) return st;
    st = rpp_remove_padding(x_padded, padding_offset, cu_seqlens, B, L, H, dt, packed, err, stream);
    if (st != RPP_OK) return st;
  }
  // the last layer's LN2 writes the padded output directly (rebuild fused)
  PaddedOut pad;
  pad.y = y_padded;
  pad.L = L;
  for (int i = 0; i < num_layers; ++i) {
    st = encoder_layer_run(cfg, layers[i], cfg->int8 ? act_scales[i] : nullptr, packed, cu_seqlens, B, T_max, L,
                           packed, workspace, workspace_bytes, nullptr, err, static_cast<cudaStream_t>(stream),
                           i + 1 == num_layers ? pad : PaddedOut{});
    if (st != RPP_OK) return st;
  }
  return RPP_OK;
}

rpp_status rpp_quantize_weight(const void* w, int K, int N, rpp_dtype dtype, int8_t* wq_t, float* s_w,
                               rpp_stream stream) {
  if (!w || !wq_t || !s_w || K <= 0 || N <= 0) return RPP_EINVAL;
  if (dtype != RPP_F32 && dtype != RPP_F16 && dtype != RPP_BF16) return RPP_EUNSUPPORTED;
  return from_cuda(launch_quantize_weight(w, K, N, dtype, wq_t, nullptr, s_w, static_cast<cudaStream_t>(stream)));
}

rpp_status rpp_quantize_activation(const void* x, const float* scale, int8_t* q, int M_max, const int32_t* rows, int H,
                                   rpp_dtype dtype, int32_t* err, rpp_stream stream) {
  if (!x || !scale || !q || M_max <= 0 || H <= 0 || H % 8) return RPP_EINVAL;
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(q) & 7u)) return RPP_EINVAL;
  if (dtype != RPP_F32 && dtype != RPP_F16 && dtype != RPP_BF16) return RPP_EUNSUPPORTED;
  return from_cuda(launch_quantize(x, scale, q, M_max, rows, H, dtype, err, static_cast<cudaStream_t>(stream)));
}

size_t rpp_gemm_i8_workspace_bytes(int M, int N, int K) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  return align_up(static_cast<size_t>(M) * K * 2) + align_up(static_cast<size_t>(N) * K * 2);
}

rpp_status rpp_gemm_i8_i32(const int8_t* aq, const int8_t* wq_t, int32_t* acc, int M, int N, int K, void* workspace,
                           size_t workspace_bytes, int32_t* err, rpp_stream stream) {
  if (!aq || !wq_t || !acc || !workspace || M <= 0 || N <= 0 || K <= 0) return RPP_EINVAL;
  if (K % 16 || N % 16 || K > 4096) return RPP_EUNSUPPORTED;
  if (!aligned16(acc) || !aligned16(workspace)) return RPP_EINVAL;
  if (workspace_bytes < rpp_gemm_i8_workspace_bytes(M, N, K)) return RPP_EWORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* a_codes = workspace;
  void* w_codes = at<void>(workspace, align_up(static_cast<size_t>(M) * K * 2));
  RPP_TRY(launch_i8_to_bf16(aq, a_codes, static_cast<long long>(M) * K, s));
  RPP_TRY(launch_i8_to_bf16(wq_t, w_codes, static_cast<long long>(N) * K, s));
  TcGemmArgs g{};
  g.a = a_codes; g.w_t = w_codes; g.out = acc; g.M_max = M; g.N = N; g.K = K;
  g.in_dtype = RPP_BF16; g.out_dtype = RPP_F32; g.epi = EPI_I32; g.err = err;
  return from_cuda(launch_gemm_tc(g, s));
}

rpp_status rpp_swin_prepare_bias(const rpp_swin_cfg* cfg, const void* table, float* bias, rpp_stream stream) {
  if (!cfg || !table || !bias || cfg->window <= 0 || cfg->heads <= 0) return RPP_EINVAL;
  return from_cuda(launch_swin_bias(table, static_cast<rpp_dtype>(cfg->dtype), cfg->window, cfg->heads, bias,
                                    static_cast<cudaStream_t>(stream)));
}

rpp_status rpp_window_attention_forward(const rpp_swin_cfg* cfg, int B, const void* qkv, const float* bias, void* out,
                                        int32_t* err, rpp_stream stream) {
  rpp_status st = swin_cfg_supported(cfg);
  if (st != RPP_OK) return st;
  if (B <= 0 || !qkv || !bias || !out || !aligned16(qkv) || !aligned16(out)) return RPP_EINVAL;
  return from_cuda(launch_window_attention(B, qkv, bias, out, cfg->channels, cfg->heads, cfg->img, cfg->window,
                                           cfg->shift, static_cast<rpp_dtype>(cfg->dtype), err,
                                           static_cast<cudaStream_t>(stream)));
}

size_t rpp_swin_block_bytes(const rpp_swin_cfg* cfg) {
  if (swin_cfg_supported(cfg) == RPP_EINVAL) return 0;
  return swin_layout(cfg).total;
}

rpp_status rpp_swin_prepare_block(const rpp_swin_cfg* cfg, const rpp_swin_src* src, void* dst, rpp_stream stream) {
  rpp_status st = swin_cfg_supported(cfg);
  if (st != RPP_OK) return st;
  if (!src || !dst || !aligned16(dst)) return RPP_EINVAL;
  const void* ptrs[] = {src->gamma1, src->beta1, src->Wqkv, src->bqkv, src->table, src->Wo, src->bo,
                        src->gamma2, src->beta2, src->W1, src->b1, src->W2, src->b2};
  for (const void* p : ptrs)
    if (!p) return RPP_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const SwinLayout P = swin_layout(cfg);
  const rpp_dtype dt = static_cast<rpp_dtype>(cfg->dtype);
  const int C = cfg->channels, F = cfg->mlp;
  RPP_TRY(launch_transpose_to_kmajor(src->Wqkv, C, 3 * C, 2, at<void>(dst, P.wqkv), C, s));
  RPP_TRY(launch_transpose_to_kmajor(src->Wo, C, C, 2, at<void>(dst, P.wo), C, s));
  RPP_TRY(launch_transpose_to_kmajor(src->W1, C, F, 2, at<void>(dst, P.w1), C, s));
  RPP_TRY(launch_transpose_to_kmajor(src->W2, F, C, 2, at<void>(dst, P.w2), F, s));
  if (swin_mlp_supported(C, F))   // W1 as given ([C, F]: the fused MLP reads it N-major)
    RPP_TRY(cudaMemcpyAsync(at<void>(dst, P.w1kn), src->W1, static_cast<size_t>(C) * F * 2, cudaMemcpyDeviceToDevice, s));
  RPP_TRY(launch_to_f32(src->bqkv, dt, 3 * C, at<float>(dst, P.bqkv), s));
  RPP_TRY(launch_to_f32(src->bo, dt, C, at<float>(dst, P.bo), s));
  RPP_TRY(launch_to_f32(src->b1, dt, F, at<float>(dst, P.b1), s));
  RPP_TRY(launch_to_f32(src->b2, dt, C, at<float>(dst, P.b2), s));
  RPP_TRY(launch_to_f32(src->gamma1, dt, C, at<float>(dst, P.g1), s));
  RPP_TRY(launch_to_f32(src->beta1, dt, C, at<float>(dst, P.be1), s));
  RPP_TRY(launch_to_f32(src->gamma2, dt, C, at<float>(dst, P.g2), s));
  RPP_TRY(launch_to_f32(src->beta2, dt, C, at<float>(dst, P.be2), s));
  RPP_TRY(launch_swin_bias(src->table, dt, cfg->window, cfg->heads, at<float>(dst, P.bias), s));
  return RPP_OK;
}

size_t rpp_swin_workspace_bytes(const rpp_swin_cfg* cfg, int B) {
  if (swin_cfg_supported(cfg) == RPP_EINVAL || B <= 0) return 0;
  return swin_ws_layout(cfg, B).total;
}

rpp_status rpp_swin_block_forward(const rpp_swin_cfg* cfg, const void* block, int B, const void* x, void* y,
                                  void* workspace, size_t workspace_bytes, int32_t* err, rpp_stream stream) {
  rpp_status st = swin_cfg_supported(cfg);
  if (st != RPP_OK) return st;
  if (!block || !x || !y || !workspace || B <= 0) return RPP_EINVAL;
  if (!aligned16(x) || !aligned16(y) || !aligned16(workspace) || !aligned16(block)) return RPP_EINVAL;
  const SwinWs W = swin_ws_layout(cfg, B);
  if (workspace_bytes < W.total) return RPP_EWORKSPACE;
  const long long Tl = static_cast<long long>(B) * cfg->img * cfg->img;
  if (Tl > 0x7fffffffLL) return RPP_EUNSUPPORTED;
  const int T = static_cast<int>(Tl);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const SwinLayout P = swin_layout(cfg);
  const rpp_dtype dt = static_cast<rpp_dtype>(cfg->dtype);
  const int C = cfg->channels, F = cfg->mlp;
  void* h = at<void>(workspace, W.h);
  void* qkv = at<void>(workspace, W.qkv);
  void* attn = at<void>(workspace, W.attn);
  void* xa = at<void>(workspace, W.xa);
  void* g = at<void>(workspace, W.g);
  LnArgs l1{};
  l1.x = x;
  l1.in_dtype = dt;
  l1.gamma = at<float>(block, P.g1);
  l1.beta = at<float>(block, P.be1);
  l1.y = h;
  l1.out_dtype = dt;
  l1.M_max = T;
  l1.H = C;
  l1.eps = cfg->eps;
  l1.err = err;
  RPP_LAUNCH("layernorm1", s, launch_layernorm(l1, s));
  RPP_LAUNCH("gemm_qkv", s, linear(dt, h, at<void>(block, P.wqkv), at<float>(block, P.bqkv), nullptr, qkv, T, nullptr, 3 * C, C,
                 RPP_EPI_BIAS, err, s));
  RPP_LAUNCH("window_attention", s, launch_window_attention(B, qkv, at<float>(block, P.bias), attn, C, cfg->heads, cfg->img, cfg->window,
                                  cfg->shift, dt, err, s));
  RPP_LAUNCH("gemm_proj", s, linear(dt, attn, at<void>(block, P.wo), at<float>(block, P.bo), x, xa, T, nullptr, C, C,
                 RPP_EPI_BIAS_RESIDUAL, err, s));
  LnArgs l2 = l1;
  l2.x = xa;
  l2.gamma = at<float>(block, P.g2);
  l2.beta = at<float>(block, P.be2);
  RPP_LAUNCH("layernorm2", s, launch_layernorm(l2, s));
  if (swin_mlp_supported(C, F)) {   // FC1 + GELU + FC2 + residual in one kernel, hidden layer on chip
    RPP_LAUNCH("swin_mlp", s, launch_swin_mlp(h, at<void>(block, P.w1kn), at<float>(block, P.b1), at<void>(block, P.w2),
                                             at<float>(block, P.b2), xa, y, T, C, F, dt, err, s));
    return RPP_OK;
  }
  RPP_LAUNCH("gemm_fc1", s, linear(dt, h, at<void>(block, P.w1), at<float>(block, P.b1), nullptr, g, T, nullptr, F, C, RPP_EPI_BIAS_GELU,
                 err, s));
  RPP_LAUNCH("gemm_fc2", s, linear(dt, g, at<void>(block, P.w2), at<float>(block, P.b2), xa, y, T, nullptr, C, F, RPP_EPI_BIAS_RESIDUAL,
                 err, s));
  return RPP_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- Swin patch merging
namespace rpp {
namespace {
struct MergeLayout {
  size_t w, gamma, beta, zero_bias, total;
};
MergeLayout merge_layout(const rpp_merge_cfg* c) {
  MergeLayout L{};
  const size_t C = static_cast<size_t>(c->channels);
  size_t o = 0;
  L.w = o;         o = align_up(o + 8 * C * C * 2);   // K-major [2C, 4C]
  L.gamma = o;     o = align_up(o + 4 * C * 4);
  L.beta = o;      o = align_up(o + 4 * C * 4);
  L.zero_bias = o; o = align_up(o + 2 * C * 4);
  L.total = o;
  return L;
}
rpp_status merge_cfg_supported(const rpp_merge_cfg* c) {
  if (!c) return RPP_EINVAL;
  if (c->dtype != RPP_F16 && c->dtype != RPP_BF16) return RPP_EUNSUPPORTED;
  if (!patch_merge_supported(c->channels, c->img) || !gemm_tc_supported(2 * c->channels, 4 * c->channels))
    return RPP_EUNSUPPORTED;
  if (!(c->eps > 0.f)) return RPP_EINVAL;
  return RPP_OK;
}
}  // namespace
}  // namespace rpp

using namespace rpp;

size_t rpp_patch_merge_bytes(const rpp_merge_cfg* cfg) {
  if (merge_cfg_supported(cfg) != RPP_OK) return 0;
  return merge_layout(cfg).total;
}

rpp_status rpp_patch_merge_prepare(const rpp_merge_cfg* cfg, const void* gamma, const void* beta, const void* W,
                                   void* dst, rpp_stream stream) {
  const rpp_status st = merge_cfg_supported(cfg);
  if (st != RPP_OK) return st;
  if (!gamma || !beta || !W || !dst || !aligned16(dst)) return RPP_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const MergeLayout P = merge_layout(cfg);
  const rpp_dtype dt = static_cast<rpp_dtype>(cfg->dtype);
  const int C = cfg->channels;
  RPP_TRY(launch_transpose_to_kmajor(W, 4 * C, 2 * C, 2, at<void>(dst, P.w), 4 * C, s));
  RPP_TRY(launch_to_f32(gamma, dt, 4 * C, at<float>(dst, P.gamma), s));
  RPP_TRY(launch_to_f32(beta, dt, 4 * C, at<float>(dst, P.beta), s));
  RPP_TRY(cudaMemsetAsync(at<float>(dst, P.zero_bias), 0, 2 * static_cast<size_t>(C) * 4, s));
  return RPP_OK;
}

size_t rpp_patch_merge_workspace_bytes(const rpp_merge_cfg* cfg, int B) {
  if (merge_cfg_supported(cfg) != RPP_OK || B <= 0) return 0;
  const size_t rows = static_cast<size_t>(B) * (cfg->img / 2) * (cfg->img / 2);
  return align_up(rows * 4 * cfg->channels * 2);
}

rpp_status rpp_patch_merge_forward(const rpp_merge_cfg* cfg, const void* prepared, int B, const void* x, void* y,
                                   void* workspace, size_t workspace_bytes, int32_t* err, rpp_stream stream) {
  const rpp_status st = merge_cfg_supported(cfg);
  if (st != RPP_OK) return st;
  if (!prepared || !x || !y || !workspace || B <= 0) return RPP_EINVAL;
  if (!aligned16(prepared) || !aligned16(x) || !aligned16(y) || !aligned16(workspace)) return RPP_EINVAL;
  if (workspace_bytes < rpp_patch_merge_workspace_bytes(cfg, B)) return RPP_EWORKSPACE;
  const long long rows_l = static_cast<long long>(B) * (cfg->img / 2) * (cfg->img / 2);
  if (rows_l * 4 > 0x7fffffffLL) return RPP_EUNSUPPORTED;
  const int rows = static_cast<int>(rows_l);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const MergeLayout P = merge_layout(cfg);
  const rpp_dtype dt = static_cast<rpp_dtype>(cfg->dtype);
  const int C = cfg->channels;
  RPP_LAUNCH("patch_merge_ln", s, launch_patch_merge_ln(x, B, cfg->img, C, dt, at<float>(prepared, P.gamma),
                                                        at<float>(prepared, P.beta), cfg->eps, workspace, err, s));
  RPP_LAUNCH("gemm_reduction", s, linear(dt, workspace, at<void>(prepared, P.w), at<float>(prepared, P.zero_bias),
                                         nullptr, y, rows, nullptr, 2 * C, 4 * C, RPP_EPI_BIAS, err, s));
  return RPP_OK;
}
