// C ABI of the hybrid-head layer: argument validation, workspace planning and
// the launch sequence of prefill and decode on one stream.
//
// Prefill (paper "Hymba: A Hybrid-head Architecture for Small Language
// Models", section 2.1 eq. 3), bf16 path:
//   in_proj (tcgen05 GEMM, RoPE fused) -> proj [rows, P_in] fp16
//   attention branch: flash attention over meta + window -> att fp16
//   SSM branch: conv+SiLU -> u; x_proj (tcgen05) -> dt fp16, B/C fp32;
//               dt_proj (tcgen05, softplus fused) -> delta fp32;
//               selective scan + gate -> g fp16 (final state -> cache)
//   fuse: s = beta1 rms(att) + beta2 rms(g)  -> fp16
//   out_proj (tcgen05, residual fused) -> Y fp32
#include <algorithm>
#include <cstring>
#include <mutex>

#include "attn_tc.cuh"
#include "common.cuh"
#include "decode.cuh"
#include "gemm_tc.cuh"
#include "scan.cuh"
#include "simt.cuh"

using namespace hy;

namespace {

struct Dims {
  int B, T, M, L, d, Hq, Hkv, dh, dv, di, N, k, R, W, kv_shared, residual, dtype;
  int fusion, sw;  // sw = width of the fused rows s (and K of out_proj): di, or 2 di concatenated
  float theta, eps;
  uint64_t wait_ns;
  long long rows;
  int P_in, k_col, v_col, x_col, z_col, Rp, xo;  // xo = R + 2N
};

bool is_flag(int v) { return v == 0 || v == 1; }

hymba_status check_desc(const hymba_layer_desc* d, bool decode, Dims* o) {
  if (!d) return HYMBA_ERR_INVALID;
  if (d->reserved != 0) return HYMBA_ERR_INVALID;
  if (d->batch < 1 || d->n_tokens < 1 || d->n_meta < 0 || d->d_model < 1 || d->n_q_heads < 1 ||
      d->n_kv_heads < 1 || d->head_dim < 2 || (d->head_dim & 1) || d->v_head_dim < 1 || d->d_inner < 1 ||
      d->d_state < 1 || d->d_state > 64 || d->d_conv < 1 || d->d_conv > 8 || d->dt_rank < 1 || d->window < 0 ||
      !is_flag(d->kv_shared) || d->residual < 0 || d->residual > 2 || !(d->eps >= 0.f) || !(d->rope_theta >= 0.f) ||
      !is_flag(d->fusion) || d->reserved0 != 0)
    return HYMBA_ERR_INVALID;
  if (d->dtype != HYMBA_F32 && d->dtype != HYMBA_BF16) return HYMBA_ERR_INVALID;
  if (d->n_q_heads % d->n_kv_heads != 0) return HYMBA_ERR_INVALID;
  if (static_cast<long long>(d->n_q_heads) * d->v_head_dim != d->d_inner) return HYMBA_ERR_INVALID;
  if (decode && d->n_tokens != 1) return HYMBA_ERR_INVALID;
  if (d->v_head_dim > 256) return HYMBA_ERR_UNSUPPORTED;
  Dims& x = *o;
  x.B = d->batch;
  x.T = d->n_tokens;
  x.M = d->n_meta;
  x.L = decode ? 1 : d->n_meta + d->n_tokens;
  x.d = d->d_model;
  x.Hq = d->n_q_heads;
  x.Hkv = d->n_kv_heads;
  x.dh = d->head_dim;
  x.dv = d->v_head_dim;
  x.di = d->d_inner;
  x.N = d->d_state;
  x.k = d->d_conv;
  x.R = d->dt_rank;
  x.W = d->window;
  x.kv_shared = d->kv_shared;
  x.residual = d->residual;
  x.fusion = d->fusion;
  x.sw = d->fusion ? 2 * d->d_inner : d->d_inner;
  x.dtype = d->dtype;
  x.theta = d->rope_theta;
  x.eps = d->eps;
  x.wait_ns = static_cast<uint64_t>(d->wait_limit_us ? d->wait_limit_us : 2000000u) * 1000ull;
  x.rows = static_cast<long long>(x.B) * x.L;
  const long long kvw = x.kv_shared ? 0 : static_cast<long long>(x.Hkv) * (x.dh + x.dv);
  const long long pin = static_cast<long long>(x.Hq) * x.dh + kvw + 2LL * x.di;
  if (pin > (1 << 30) || x.rows > (1LL << 31) - 1 || x.rows * pin > (1LL << 40)) return HYMBA_ERR_INVALID;
  x.P_in = static_cast<int>(pin);
  x.k_col = x.Hq * x.dh;
  x.v_col = x.k_col + x.Hkv * x.dh;
  x.x_col = x.Hq * x.dh + static_cast<int>(kvw);
  x.z_col = x.x_col + x.di;
  x.Rp = (x.R + 7) / 8 * 8;
  x.xo = x.R + 2 * x.N;
  if (x.dtype == HYMBA_BF16) {
    // TMA / vector-store alignment of every column block (8 fp16/bf16 = 16 B)
    if (x.d % 8 || x.di % 8 || x.dh % 8 || (x.Hkv * x.dh) % 8 || (x.Hkv * x.dv) % 8 || (2 * x.N) % 4)
      return HYMBA_ERR_UNSUPPORTED;
  }
  return HYMBA_OK;
}

// Workspace plan: byte offsets of each scratch buffer (256-byte aligned).
struct Plan {
  size_t proj, u, dtr, bc, delta, att, g, s, wout, wx, wdt, part, apart, total;
  int attn_splits;
};

int num_sms();

// Key splits of the decode attention.
int decode_attn_splits(const Dims& x) {
  if (decode_attn_tc_supported(x.Hq, x.Hkv, x.dh, x.dv)) return decode_attn_tc_splits(x.B, x.Hkv, num_sms());
  const int ctas = x.B * x.Hkv;
  return std::max(1, std::min(16, (4 * 148 + ctas - 1) / ctas));
}

constexpr int kDecodeSplitsX = 25;
constexpr int kDecodeSplitsOut = 5;

Plan plan_ws(const Dims& x, bool decode) {
  Plan p{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  const size_t e = x.dtype == HYMBA_BF16 ? 2 : 4;
  const size_t r = static_cast<size_t>(x.rows);
  p.proj = take(r * x.P_in * e);
  p.u = take(r * x.di * e);
  p.dtr = take(r * (x.dtype == HYMBA_BF16 ? x.Rp : x.R) * e);
  p.bc = take(r * 2 * x.N * 4);
  // the bf16 prefill computes delta inside the scan when it can
  const bool fused = x.dtype == HYMBA_BF16 && !decode && scan_fused_supported(x.di, x.N, x.R);
  p.delta = fused ? 0 : take(r * x.di * 4);
  p.att = take(r * x.di * e);
  p.g = take(r * x.di * e);
  p.s = take(r * x.sw * e);
  if (x.dtype == HYMBA_BF16) {
    // fp16 weight copies: prefill converts W_out and W_x once per call; the
    // decode GEMMs convert their bf16 tiles in shared memory instead
    if (!decode) {
      p.wout = take(static_cast<size_t>(x.d) * x.sw * 2);
      p.wx = take(static_cast<size_t>(x.xo) * x.di * 2);
    }
    p.wdt = take(static_cast<size_t>(x.di) * x.Rp * 2);
    if (decode) {
      const size_t w1 = static_cast<size_t>(kDecodeSplitsX) * r * ((x.xo + 15) / 16 * 16);
      const size_t w2 = static_cast<size_t>(kDecodeSplitsOut) * r * x.d;
      p.part = take(std::max(w1, w2) * 4);
      p.attn_splits = decode_attn_splits(x);
      p.apart = take(decode_attn_split_scratch(x.B, x.Hq, x.dv, p.attn_splits));
    }
  }
  p.total = off;
  return p;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

hymba_status check_weights(const hymba_layer_weights* w, const Dims& x) {
  if (!w || !w->W_in || !w->W_out || !w->W_x || !w->W_dt || !w->dt_bias || !w->A_log || !w->D || !w->conv_w ||
      !w->conv_b || !w->beta1 || !w->beta2)
    return HYMBA_ERR_INVALID;
  const size_t a = x.dtype == HYMBA_BF16 ? 16 : 4;
  if (!aligned(w->W_in, a) || !aligned(w->W_out, a) || !aligned(w->W_x, a) || !aligned(w->W_dt, 2) ||
      !aligned(w->dt_bias, 4) || !aligned(w->A_log, 4) || !aligned(w->D, 4) || !aligned(w->conv_w, 4) ||
      !aligned(w->conv_b, 4) || !aligned(w->beta1, 4) || !aligned(w->beta2, 4))
    return HYMBA_ERR_INVALID;
  return HYMBA_OK;
}

int num_sms() {
  int dev = 0, n = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 148;
}

#define TRY(...)                           \
  do {                                     \
    hymba_status s_ = (__VA_ARGS__);       \
    if (s_ != HYMBA_OK) return s_;         \
  } while (0)

// Optional per-stage CUDA events (hymba_layer_fwd_events): events[0] before
// the first launch, events[k] after stage k.
struct Marks {
  void* const* ev = nullptr;
  int n = 0;
  int i = 0;
  cudaStream_t st = nullptr;
  void mark() {
    if (ev && i < n) cudaEventRecord(static_cast<cudaEvent_t>(ev[i]), st);
    ++i;
  }
};

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

// ---------------------------------------------------------------------------
// fp32 path (SIMT)
// ---------------------------------------------------------------------------
hymba_status fwd_f32(const Dims& x, const Plan& pl, const hymba_layer_weights* w, const float* X, float* Y,
                     const hymba_cache* cache_out, const hymba_kv* kv_in, const hymba_kv* kv_out, void* ws,
                     Marks& mk, cudaStream_t st) {
  float* proj = at<float>(ws, pl.proj);
  float* u = at<float>(ws, pl.u);
  float* dtr = at<float>(ws, pl.dtr);
  float* bc = at<float>(ws, pl.bc);
  float* delta = at<float>(ws, pl.delta);
  float* att = at<float>(ws, pl.att);
  float* g = at<float>(ws, pl.g);
  float* s = at<float>(ws, pl.s);
  const int rows = static_cast<int>(x.rows);
  const float* Win = static_cast<const float*>(w->W_in);
  mk.mark();
  mk.mark();  // no weight conversion on this path
  TRY(gemm_simt<float>(rows, x.P_in, x.d, X, x.d, Win, x.d, SE_STORE, proj, x.P_in, nullptr, 0, 0, nullptr,
                       nullptr, 0, st));
  if (x.theta > 0) {
    TRY(rope_simt<float>(proj, x.P_in, rows, 0, x.Hq, x.dh, x.theta, x.L, nullptr, 0, st));
    if (!x.kv_shared) TRY(rope_simt<float>(proj, x.P_in, rows, x.k_col, x.Hkv, x.dh, x.theta, x.L, nullptr, 0, st));
  }
  mk.mark();
  const float* Kp = x.kv_shared ? static_cast<const float*>(kv_in->k) : proj + x.k_col;
  const float* Vp = x.kv_shared ? static_cast<const float*>(kv_in->v) : proj + x.v_col;
  const long long ldk = x.kv_shared ? static_cast<long long>(x.Hkv) * x.dh : x.P_in;
  const long long ldv = x.kv_shared ? static_cast<long long>(x.Hkv) * x.dv : x.P_in;
  if (kv_out) {
    TRY(copy2d<float, float>(Kp, ldk, static_cast<float*>(kv_out->k), static_cast<long long>(x.Hkv) * x.dh, x.rows,
                             x.Hkv * x.dh, st));
    TRY(copy2d<float, float>(Vp, ldv, static_cast<float*>(kv_out->v), static_cast<long long>(x.Hkv) * x.dv, x.rows,
                             x.Hkv * x.dv, st));
  }
  mk.mark();
  TRY(attention_simt<float>(x.B, x.L, x.M, x.Hq, x.Hkv, x.dh, x.dv, x.W, proj, x.P_in, Kp, ldk, Vp, ldv, att,
                            x.di, st));
  mk.mark();
  TRY(conv_silu<float, float>(proj + x.x_col, x.P_in, u, x.di, x.B, x.L, x.di, x.k, w->conv_w, w->conv_b, st));
  mk.mark();
  TRY(gemm_simt<float>(rows, x.xo, x.di, u, x.di, static_cast<const float*>(w->W_x), x.di, SE_XPROJ, bc, 2 * x.N,
                       dtr, x.R, x.R, nullptr, nullptr, 0, st));
  mk.mark();
  TRY(gemm_simt<float>(rows, x.di, x.R, dtr, x.R, static_cast<const float*>(w->W_dt), x.R, SE_SOFTPLUS, delta,
                       x.di, nullptr, 0, 0, w->dt_bias, nullptr, 0, st));
  mk.mark();
  float* h_out = cache_out ? cache_out->ssm_state : nullptr;
  TRY(scan_simt<float>(x.B, x.L, x.di, x.N, u, x.di, proj + x.z_col, x.P_in, delta, x.di, bc, bc + x.N, 2 * x.N,
                       w->A_log, w->D, g, x.di, nullptr, h_out, st));
  mk.mark();
  TRY(fuse_norm<float>(rows, x.di, att, g, w->beta1, w->beta2, x.eps, s, st, x.fusion != 0));
  mk.mark();
  TRY(gemm_simt<float>(rows, x.d, x.sw, s, x.sw, static_cast<const float*>(w->W_out), x.sw, SE_RESID, Y, x.d,
                       nullptr, 0, 0, nullptr, x.residual == 1 ? X : x.residual == 2 ? Y : nullptr, x.d, st));
  mk.mark();
  if (cache_out) {
    TRY(emit_cache<float, float>(x.B, x.L, x.M, x.T, cache_out->cap, x.Hkv, x.dh, x.dv, x.di, x.k,
                                 x.kv_shared ? nullptr : Kp, ldk, Vp, ldv, proj + x.x_col, x.P_in,
                                 static_cast<float*>(cache_out->k_ring), static_cast<float*>(cache_out->v_ring),
                                 static_cast<float*>(cache_out->k_meta), static_cast<float*>(cache_out->v_meta),
                                 cache_out->conv_state, cache_out->pos, st));
  }
  mk.mark();
  return HYMBA_OK;
}

// ---------------------------------------------------------------------------
// bf16 path (tensor cores)
// ---------------------------------------------------------------------------
GemmParams gp(int M, int N, int K, int32_t* status, uint64_t wait_ns) {
  GemmParams p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.rows_per_seq = 1;
  p.status = status;
  p.wait_ns = wait_ns;
  return p;
}

hymba_status convert_weights(const Dims& x, const Plan& pl, const hymba_layer_weights* w, void* ws,
                             cudaStream_t st) {
  TRY(copy2d<__nv_bfloat16, __half>(static_cast<const __nv_bfloat16*>(w->W_out), x.sw, at<__half>(ws, pl.wout),
                                    x.sw, x.d, x.sw, st));
  TRY(copy2d<__nv_bfloat16, __half>(static_cast<const __nv_bfloat16*>(w->W_x), x.di, at<__half>(ws, pl.wx), x.di,
                                    x.xo, x.di, st));
  TRY(copy2d<__nv_bfloat16, __half>(static_cast<const __nv_bfloat16*>(w->W_dt), x.R, at<__half>(ws, pl.wdt), x.Rp,
                                    x.di, x.R, st));
  return HYMBA_OK;
}

// X is bf16 against the bf16 W_in, or fp16 against an fp16 copy of W_in
// (w_in_f16 set: a residual stack's later layers).
hymba_status in_proj_bf16(const Dims& x, const void* X, const hymba_layer_weights* w, __half* proj, int rows,
                          const int32_t* pos, int pos_base, int rows_per_seq, int32_t* status, int sms,
                          cudaStream_t st, const __half* w_in_f16 = nullptr, bool pdl = false) {
  GemmParams p = gp(rows, x.P_in, x.d, status, x.wait_ns);
  p.pdl = pdl;
  p.C = proj;
  p.ldc = x.P_in;
  const bool fused_rope = x.theta > 0 && x.dh == 64;
  if (fused_rope) {
    p.rope_cols = x.Hq * x.dh + (x.kv_shared ? 0 : x.Hkv * x.dh);
    p.rope_log2_step = -2.0f / x.dh * log2f(x.theta);
  }
  p.rows_per_seq = rows_per_seq;
  p.pos = pos;
  p.pos_base = pos_base;
  if (w_in_f16)
    TRY(gemm_tc(0, X, x.d, w_in_f16, x.d, EPI_F16, p, 0, 1, sms, st));
  else
    TRY(gemm_tc(1, X, x.d, w->W_in, x.d, EPI_F16, p, 0, 1, sms, st));
  if (x.theta > 0 && !fused_rope) {
    TRY(rope_simt<__half>(proj, x.P_in, rows, 0, x.Hq, x.dh, x.theta, rows_per_seq, pos, pos_base, st));
    if (!x.kv_shared)
      TRY(rope_simt<__half>(proj, x.P_in, rows, x.k_col, x.Hkv, x.dh, x.theta, rows_per_seq, pos, pos_base, st));
  }
  return HYMBA_OK;
}

// Meta-prefix precompute: `out` set = produce (x holds the M meta rows of one
// sequence: B = 1, T = 0, L = M); `in` set = consume (x holds only the T real
// rows of each sequence: L = T, while x.M keeps the logical meta count).
struct MetaCtx {
  const hymba_meta* in = nullptr;
  const hymba_meta* out = nullptr;
};

// A residual stack's plumbing: the layer reads X in fp16 against an fp16
// copy of W_in (w_in_f16), and out_proj also writes the updated stream
// rounded to fp16 (y_f16), the next layer's input.
struct StackIO {
  const __half* w_in_f16 = nullptr;
  __half* y_f16 = nullptr;
};

hymba_status fwd_bf16(const Dims& x, const Plan& pl, const hymba_layer_weights* w, const void* X, float* Y,
                      const hymba_cache* cache_out, const hymba_kv* kv_in, const hymba_kv* kv_out, void* ws,
                      int32_t* status, Marks& mk, cudaStream_t st, const MetaCtx& mc = MetaCtx{},
                      const StackIO& sio = StackIO{}) {
  const int sms = num_sms();
  const hymba_meta* mi = mc.in;
  const int rows = static_cast<int>(x.rows);
  __half* proj = at<__half>(ws, pl.proj);
  __half* u = at<__half>(ws, pl.u);
  __half* dtr = at<__half>(ws, pl.dtr);
  float* bc = at<float>(ws, pl.bc);
  float* delta = at<float>(ws, pl.delta);
  __half* att = at<__half>(ws, pl.att);
  __half* g = at<__half>(ws, pl.g);
  __half* s = at<__half>(ws, pl.s);
  mk.mark();
  TRY(convert_weights(x, pl, w, ws, st));
  mk.mark();
  // positions: logical (meta rows first), so real rows start at M when the meta rows are cached
  TRY(in_proj_bf16(x, X, w, proj, rows, nullptr, mi ? x.M : 0, x.L, status, sms, st, sio.w_in_f16));
  mk.mark();

  const __half* Kp = x.kv_shared ? static_cast<const __half*>(kv_in->k) : proj + x.k_col;
  const __half* Vp = x.kv_shared ? static_cast<const __half*>(kv_in->v) : proj + x.v_col;
  const long long ldk = x.kv_shared ? static_cast<long long>(x.Hkv) * x.dh : x.P_in;
  const long long ldv = x.kv_shared ? static_cast<long long>(x.Hkv) * x.dv : x.P_in;
  if (kv_out) {
    TRY(copy2d<__half, __half>(Kp, ldk, static_cast<__half*>(kv_out->k), static_cast<long long>(x.Hkv) * x.dh,
                               x.rows, x.Hkv * x.dh, st));
    TRY(copy2d<__half, __half>(Vp, ldv, static_cast<__half*>(kv_out->v), static_cast<long long>(x.Hkv) * x.dv,
                               x.rows, x.Hkv * x.dv, st));
  }
  mk.mark();
  // attention branch
  if (mi) {
    TRY(attn_tc_meta(x.B, x.T, x.M, static_cast<const __half*>(mi->k), static_cast<const __half*>(mi->v), x.Hq,
                     x.Hkv, x.dh, x.dv, x.W, proj, x.P_in, Kp, ldk, Vp, ldv, att, x.di, status, x.wait_ns, sms, st));
  } else if (attn_tc_supported(x.dh, x.dv)) {
    TRY(attn_tc(x.B, x.L, x.M, x.Hq, x.Hkv, x.dh, x.dv, x.W, proj, x.P_in, Kp, ldk, Vp, ldv, att, x.di, status,
                x.wait_ns, sms, st));
  } else {
    TRY(attention_simt<__half>(x.B, x.L, x.M, x.Hq, x.Hkv, x.dh, x.dv, x.W, proj, x.P_in, Kp, ldk, Vp, ldv, att,
                               x.di, st));
  }
  mk.mark();
  // SSM branch
  if (conv_tma_supported(x.di, x.k, x.P_in, x.di, proj + x.x_col, u))
    TRY(conv_silu_tma(proj + x.x_col, x.P_in, u, x.di, x.B, x.L, x.di, x.k, w->conv_w, w->conv_b, status, x.wait_ns,
                      sms, st, mi ? mi->conv_tail : nullptr));
  else
    TRY(conv_silu<__half, __half>(proj + x.x_col, x.P_in, u, x.di, x.B, x.L, x.di, x.k, w->conv_w, w->conv_b, st));
  mk.mark();
  {
    GemmParams p = gp(rows, x.xo, x.di, status, x.wait_ns);
    p.C = bc;
    p.ldc = 2 * x.N;
    p.C2 = dtr;
    p.ldc2 = x.Rp;
    p.xproj_R = x.R;
    TRY(gemm_tc(0, u, x.di, at<__half>(ws, pl.wx), x.di, EPI_XPROJ, p, 0, 1, sms, st));
  }
  mk.mark();
  float* h_out = cache_out ? cache_out->ssm_state : (mc.out ? mc.out->ssm_state : nullptr);
  if (scan_fused_supported(x.di, x.N, x.R)) {
    // dt projection + softplus run inside the scan (no delta in HBM)
    mk.mark();
    TRY(scan_fused_f16(x.B, x.L, x.di, x.N, x.R, u, x.di, proj + x.z_col, x.P_in, dtr, x.Rp,
                       static_cast<const __nv_bfloat16*>(w->W_dt), w->dt_bias, bc, w->A_log, w->D, g,
                       mi ? mi->ssm_state : nullptr, h_out, status, x.wait_ns, 0, 0, st, mi != nullptr));
  } else {
    GemmParams p = gp(rows, x.di, x.R, status, x.wait_ns);
    p.C = delta;
    p.ldc = x.di;
    p.bias = w->dt_bias;
    TRY(gemm_tc(0, dtr, x.Rp, at<__half>(ws, pl.wdt), x.Rp, EPI_SOFTPLUS, p, 0, 1, sms, st));
    mk.mark();
    TRY(scan_f16(x.B, x.L, x.di, x.N, u, x.di, proj + x.z_col, x.P_in, delta, bc, w->A_log, w->D, g, nullptr, h_out,
                 status, x.wait_ns, 0, 0, st));
  }
  mk.mark();
  // fuse + out_proj
  TRY(fuse_norm<__half>(rows, x.di, att, g, w->beta1, w->beta2, x.eps, s, st, x.fusion != 0));
  mk.mark();
  {
    GemmParams p = gp(rows, x.d, x.sw, status, x.wait_ns);
    p.C = Y;
    p.ldc = x.d;
    p.resid = x.residual == 1 ? static_cast<const __nv_bfloat16*>(X) : nullptr;
    p.resid_f32 = x.residual == 2 ? Y : nullptr;
    p.ld_resid = x.d;
    p.C2 = sio.y_f16;  // a stack's next layer input: the stream rounded to fp16
    p.ldc2 = x.d;
    TRY(gemm_tc(0, s, x.sw, at<__half>(ws, pl.wout), x.sw, EPI_F32, p, 0, 1, sms, st));
  }
  mk.mark();
  if (cache_out && mi) {
    // ring and conv tail from the real rows (the tail falls back on the meta
    // rows' tail), the meta K/V from the cached meta state
    TRY(emit_cache<__half, __nv_bfloat16>(
        x.B, x.L, 0, x.T, cache_out->cap, x.Hkv, x.dh, x.dv, x.di, x.k, x.kv_shared ? nullptr : Kp, ldk, Vp, ldv,
        proj + x.x_col, x.P_in, static_cast<__nv_bfloat16*>(cache_out->k_ring),
        static_cast<__nv_bfloat16*>(cache_out->v_ring), nullptr, nullptr, cache_out->conv_state, cache_out->pos, st,
        mi->conv_tail));
    if (!x.kv_shared) {
      TRY(copy2d<__half, __nv_bfloat16>(static_cast<const __half*>(mi->k), static_cast<long long>(x.Hkv) * x.dh,
                                        static_cast<__nv_bfloat16*>(cache_out->k_meta),
                                        static_cast<long long>(x.Hkv) * x.dh, x.M, x.Hkv * x.dh, st));
      TRY(copy2d<__half, __nv_bfloat16>(static_cast<const __half*>(mi->v), static_cast<long long>(x.Hkv) * x.dv,
                                        static_cast<__nv_bfloat16*>(cache_out->v_meta),
                                        static_cast<long long>(x.Hkv) * x.dv, x.M, x.Hkv * x.dv, st));
    }
  } else if (cache_out) {
    TRY(emit_cache<__half, __nv_bfloat16>(
        x.B, x.L, x.M, x.T, cache_out->cap, x.Hkv, x.dh, x.dv, x.di, x.k, x.kv_shared ? nullptr : Kp, ldk, Vp, ldv,
        proj + x.x_col, x.P_in, static_cast<__nv_bfloat16*>(cache_out->k_ring),
        static_cast<__nv_bfloat16*>(cache_out->v_ring), static_cast<__nv_bfloat16*>(cache_out->k_meta),
        static_cast<__nv_bfloat16*>(cache_out->v_meta), cache_out->conv_state, cache_out->pos, st));
  }
  if (mc.out) {
    // what the real tokens need from the meta rows: K/V (fp16) and the conv tail
    if (!x.kv_shared) {
      TRY(copy2d<__half, __half>(Kp, ldk, static_cast<__half*>(mc.out->k), static_cast<long long>(x.Hkv) * x.dh, x.M,
                                 x.Hkv * x.dh, st));
      TRY(copy2d<__half, __half>(Vp, ldv, static_cast<__half*>(mc.out->v), static_cast<long long>(x.Hkv) * x.dv, x.M,
                                 x.Hkv * x.dv, st));
    }
    TRY(emit_cache<__half, __nv_bfloat16>(1, x.L, x.M, 0, 1, x.Hkv, x.dh, x.dv, x.di, x.k, nullptr, ldk, nullptr, ldv,
                                          proj + x.x_col, x.P_in, nullptr, nullptr, nullptr, nullptr,
                                          mc.out->conv_tail, nullptr, st));
  }
  mk.mark();
  return HYMBA_OK;
}

// ---------------------------------------------------------------------------
// decode
// ---------------------------------------------------------------------------
hymba_status decode_f32(const Dims& x, const Plan& pl, const hymba_layer_weights* w, const float* Xn, float* Y,
                        const hymba_cache* c, const hymba_cache* kvc, void* ws, cudaStream_t st) {
  float* proj = at<float>(ws, pl.proj);
  float* u = at<float>(ws, pl.u);
  float* dtr = at<float>(ws, pl.dtr);
  float* bc = at<float>(ws, pl.bc);
  float* delta = at<float>(ws, pl.delta);
  float* att = at<float>(ws, pl.att);
  float* g = at<float>(ws, pl.g);
  float* s = at<float>(ws, pl.s);
  const int B = x.B;
  TRY(gemm_simt<float>(B, x.P_in, x.d, Xn, x.d, static_cast<const float*>(w->W_in), x.d, SE_STORE, proj, x.P_in,
                       nullptr, 0, 0, nullptr, nullptr, 0, st));
  if (x.theta > 0) {
    TRY(rope_simt<float>(proj, x.P_in, B, 0, x.Hq, x.dh, x.theta, 1, c->pos, x.M, st));
    if (!x.kv_shared) TRY(rope_simt<float>(proj, x.P_in, B, x.k_col, x.Hkv, x.dh, x.theta, 1, c->pos, x.M, st));
  }
  if (!x.kv_shared)
    TRY(kv_append<float, float>(B, x.Hkv, x.dh, x.dv, x.W, c->cap, proj, x.P_in, x.k_col, x.v_col, c->pos,
                                static_cast<float*>(c->k_ring), static_cast<float*>(c->v_ring), st));
  TRY(decode_attention<float, float>(B, x.M, x.Hq, x.Hkv, x.dh, x.dv, x.W, kvc->cap, proj, x.P_in,
                                     static_cast<const float*>(kvc->k_meta), static_cast<const float*>(kvc->v_meta),
                                     static_cast<const float*>(kvc->k_ring), static_cast<const float*>(kvc->v_ring),
                                     c->pos, att, x.di, st));
  TRY(conv_step<float>(B, x.di, x.k, proj + x.x_col, x.P_in, w->conv_w, w->conv_b, c->conv_state, u, x.di, st));
  TRY(gemm_simt<float>(B, x.xo, x.di, u, x.di, static_cast<const float*>(w->W_x), x.di, SE_XPROJ, bc, 2 * x.N, dtr,
                       x.R, x.R, nullptr, nullptr, 0, st));
  TRY(gemm_simt<float>(B, x.di, x.R, dtr, x.R, static_cast<const float*>(w->W_dt), x.R, SE_SOFTPLUS, delta, x.di,
                       nullptr, 0, 0, w->dt_bias, nullptr, 0, st));
  TRY(scan_simt<float>(B, 1, x.di, x.N, u, x.di, proj + x.z_col, x.P_in, delta, x.di, bc, bc + x.N, 2 * x.N,
                       w->A_log, w->D, g, x.di, c->ssm_state, c->ssm_state, st));
  TRY(fuse_norm<float>(B, x.di, att, g, w->beta1, w->beta2, x.eps, s, st, x.fusion != 0));
  TRY(gemm_simt<float>(B, x.d, x.sw, s, x.sw, static_cast<const float*>(w->W_out), x.sw, SE_RESID, Y, x.d, nullptr,
                       0, 0, nullptr, x.residual == 1 ? Xn : x.residual == 2 ? Y : nullptr, x.d, st));
  return pos_increment(B, c->pos, st);
}

hymba_status decode_bf16(const Dims& x, const Plan& pl, const hymba_layer_weights* w, const void* Xn, float* Y,
                         const hymba_cache* c, const hymba_cache* kvc, void* ws, int32_t* status, Marks& mk,
                         cudaStream_t st) {
  const int sms = num_sms();
  const int B = x.B;
  __half* proj = at<__half>(ws, pl.proj);
  __half* u = at<__half>(ws, pl.u);
  __half* dtr = at<__half>(ws, pl.dtr);
  float* bc = at<float>(ws, pl.bc);
  float* delta = at<float>(ws, pl.delta);
  __half* att = at<__half>(ws, pl.att);
  __half* g = at<__half>(ws, pl.g);
  __half* s = at<__half>(ws, pl.s);
  float* part = at<float>(ws, pl.part);
  const bool ssm_fused = decode_ssm_step_supported(x.N, x.R);
  const int ldp_x = (x.xo + 15) / 16 * 16;
  // the buffers the split-K GEMMs add into are cleared first, so that the
  // step's kernels follow one another with nothing in between (each may
  // start while the one before it finishes)
  if (ssm_fused && cudaMemsetAsync(part, 0, static_cast<size_t>(B) * ldp_x * sizeof(float), st) != cudaSuccess)
    return HYMBA_ERR_CUDA;
  if (x.residual == 0 && cudaMemsetAsync(Y, 0, static_cast<size_t>(B) * x.d * sizeof(float), st) != cudaSuccess)
    return HYMBA_ERR_CUDA;
  mk.mark();
  // W_x and W_out are converted to fp16 inside the GEMMs (cvt_b); only the
  // unfused dt projection needs a converted W_dt
  if (!ssm_fused)
    TRY(copy2d<__nv_bfloat16, __half>(static_cast<const __nv_bfloat16*>(w->W_dt), x.R, at<__half>(ws, pl.wdt),
                                      x.Rp, x.di, x.R, st));
  mk.mark();
  TRY(in_proj_bf16(x, Xn, w, proj, B, c->pos, x.M, 1, status, sms, st, nullptr, true));
  mk.mark();
  // the new token's K/V into the ring and the conv step, one launch
  TRY(decode_prep(B, x.di, x.k, proj, x.P_in, x.x_col, x.k_col, x.v_col, x.Hkv, x.dh, x.dv, x.W, c->cap, c->pos,
                  static_cast<__nv_bfloat16*>(c->k_ring), static_cast<__nv_bfloat16*>(c->v_ring), w->conv_w,
                  w->conv_b, c->conv_state, u, x.di, !x.kv_shared, st));
  mk.mark();
  if (decode_attn_tc_supported(x.Hq, x.Hkv, x.dh, x.dv)) {
    TRY(decode_attention_tc(B, x.M, x.Hq, x.Hkv, x.dh, x.dv, x.W, kvc->cap, pl.attn_splits, proj, x.P_in,
                            static_cast<const __nv_bfloat16*>(kvc->k_meta),
                            static_cast<const __nv_bfloat16*>(kvc->v_meta),
                            static_cast<const __nv_bfloat16*>(kvc->k_ring),
                            static_cast<const __nv_bfloat16*>(kvc->v_ring), c->pos, at<float>(ws, pl.apart), att,
                            x.di, sms, status, x.wait_ns, st));
  } else if (decode_attn_split_supported(x.Hq, x.Hkv, x.dh, x.dv)) {
    const int max_keys = x.M + (x.W > 0 ? std::min(x.W, kvc->cap) : kvc->cap);
    TRY(decode_attention_split(B, x.M, x.Hq, x.Hkv, x.dh, x.dv, x.W, kvc->cap, pl.attn_splits, proj, x.P_in,
                               static_cast<const __nv_bfloat16*>(kvc->k_meta),
                               static_cast<const __nv_bfloat16*>(kvc->v_meta),
                               static_cast<const __nv_bfloat16*>(kvc->k_ring),
                               static_cast<const __nv_bfloat16*>(kvc->v_ring), c->pos, at<float>(ws, pl.apart), att,
                               x.di, max_keys, st));
  } else {
    TRY(decode_attention<__half, __nv_bfloat16>(
        B, x.M, x.Hq, x.Hkv, x.dh, x.dv, x.W, kvc->cap, proj, x.P_in, static_cast<const __nv_bfloat16*>(kvc->k_meta),
        static_cast<const __nv_bfloat16*>(kvc->v_meta), static_cast<const __nv_bfloat16*>(kvc->k_ring),
        static_cast<const __nv_bfloat16*>(kvc->v_ring), c->pos, att, x.di, st));
  }
  mk.mark();  // (conv step ran with the ring append)
  mk.mark();
  {
    const int ldp = (x.xo + 15) / 16 * 16;
    GemmParams p = gp(B, x.xo, x.di, status, x.wait_ns);
    p.pdl = 1;
    p.C = part;
    p.ldc = ldp;
    p.cvt_b = 1;
    if (ssm_fused) {
      // split-K partials added straight into the [B, ldp] fp32 buffer cleared
      // at the start, which the SSM step reads as [dt | B | C]
      TRY(gemm_tc(0, u, x.di, w->W_x, x.di, EPI_ATOMIC, p, 0, kDecodeSplitsX, sms, st));
    } else {
      TRY(gemm_tc(0, u, x.di, w->W_x, x.di, EPI_PARTIAL, p, 0, kDecodeSplitsX, sms, st));
      const int n_kb = (x.di + 63) / 64;
      const int kbs = (n_kb + std::min(kDecodeSplitsX, n_kb) - 1) / std::min(kDecodeSplitsX, n_kb);
      const int splits = (n_kb + kbs - 1) / kbs;
      TRY(splitk_reduce(splits, B, x.xo, part, ldp, RE_XPROJ, x.R, dtr, x.Rp, bc, 2 * x.N, nullptr, 0, false, st));
    }
  }
  mk.mark();
  if (ssm_fused) {
    mk.mark();  // dt projection is fused into the step below
    TRY(decode_ssm_step(B, x.di, x.N, x.R, u, x.di, proj + x.z_col, x.P_in, part, (x.xo + 15) / 16 * 16,
                        static_cast<const __nv_bfloat16*>(w->W_dt), w->dt_bias, w->A_log, w->D, c->ssm_state, g, x.di,
                        c->pos, st));  // also advances pos
  } else {
    GemmParams p = gp(B, x.di, x.R, status, x.wait_ns);
    p.pdl = 1;
    p.C = delta;
    p.ldc = x.di;
    p.bias = w->dt_bias;
    TRY(gemm_tc(0, dtr, x.Rp, at<__half>(ws, pl.wdt), x.Rp, EPI_SOFTPLUS, p, 0, 1, sms, st));
    mk.mark();
    TRY(scan_simt<__half>(B, 1, x.di, x.N, u, x.di, proj + x.z_col, x.P_in, delta, x.di, bc, bc + x.N, 2 * x.N,
                          w->A_log, w->D, g, x.di, c->ssm_state, c->ssm_state, st));
  }
  mk.mark();
  TRY(fuse_norm<__half>(B, x.di, att, g, w->beta1, w->beta2, x.eps, s, st, x.fusion != 0));
  mk.mark();
  {
    GemmParams p = gp(B, x.d, x.sw, status, x.wait_ns);
    p.pdl = 1;
    p.cvt_b = 1;
    if (x.residual != 1) {
      // split-K partials added straight into Y, which holds the fp32 residual
      // already (residual = 2) or was cleared at the start of the step
      p.C = Y;
      p.ldc = x.d;
      TRY(gemm_tc(0, s, x.sw, w->W_out, x.sw, EPI_ATOMIC, p, 0, kDecodeSplitsOut, sms, st));
    } else {
      p.C = part;
      p.ldc = x.d;
      TRY(gemm_tc(0, s, x.sw, w->W_out, x.sw, EPI_PARTIAL, p, 0, kDecodeSplitsOut, sms, st));
      const int n_kb = (x.sw + 63) / 64;
      const int sp = std::min(kDecodeSplitsOut, n_kb);
      const int kbs = (n_kb + sp - 1) / sp;
      const int splits = (n_kb + kbs - 1) / kbs;
      TRY(splitk_reduce(splits, B, x.d, part, x.d, RE_F32, 0, nullptr, 0, Y, x.d,
                        static_cast<const __nv_bfloat16*>(Xn), x.d, false, st));
    }
  }
  mk.mark();
  if (!ssm_fused) TRY(pos_increment(B, c->pos, st));
  mk.mark();
  return HYMBA_OK;
}

// Dims of a meta-prefix call: produce = the M meta rows of one sequence
// (B = 1, T = 0, L = M); otherwise the T real rows of each sequence (L = T).
hymba_status meta_dims(const hymba_layer_desc* d, bool produce, Dims* x) {
  if (!d) return HYMBA_ERR_INVALID;
  hymba_layer_desc dd = *d;
  if (produce) {
    dd.batch = 1;
    dd.n_tokens = 1;  // validated as one token; the call processes none
  }
  TRY(check_desc(&dd, false, x));
  if (x->dtype != HYMBA_BF16 || !attn_tc_supported(x->dh, x->dv) || x->M < 64 || x->M % 64 != 0 ||
      !scan_fused_supported(x->di, x->N, x->R) || (x->theta > 0 && x->dh != 64))
    return HYMBA_ERR_UNSUPPORTED;
  if (produce) {
    x->B = 1;
    x->T = 0;
    x->L = x->M;
    x->rows = x->M;
  } else {
    x->L = x->T;
    x->rows = static_cast<long long>(x->B) * x->T;
  }
  return HYMBA_OK;
}

}  // namespace

extern "C" {

int32_t hymba_abi_version(void) { return HYMBA_ABI_VERSION; }

const char* hymba_status_str(hymba_status s) {
  switch (s) {
    case HYMBA_OK: return "HYMBA_OK";
    case HYMBA_ERR_INVALID: return "HYMBA_ERR_INVALID: invalid argument";
    case HYMBA_ERR_UNSUPPORTED: return "HYMBA_ERR_UNSUPPORTED: shape or option not implemented";
    case HYMBA_ERR_WORKSPACE: return "HYMBA_ERR_WORKSPACE: workspace too small";
    case HYMBA_ERR_CUDA: return "HYMBA_ERR_CUDA: CUDA runtime error";
    case HYMBA_ERR_TIMEOUT: return "HYMBA_ERR_TIMEOUT: a bounded in-kernel wait gave up";
    case HYMBA_ERR_RANGE: return "HYMBA_ERR_RANGE: fp16 intermediate overflow";
    default: return "unknown hymba_status";
  }
}

size_t hymba_layer_fwd_workspace(const hymba_layer_desc* d) {
  Dims x;
  if (check_desc(d, false, &x) != HYMBA_OK) return 0;
  return plan_ws(x, false).total;
}

size_t hymba_layer_decode_workspace(const hymba_layer_desc* d) {
  Dims x;
  if (check_desc(d, true, &x) != HYMBA_OK) return 0;
  return plan_ws(x, true).total;
}

static hymba_status layer_fwd_impl(const hymba_layer_desc* d, const hymba_layer_weights* w, const void* x_in,
                                   float* y, const hymba_cache* cache_out, const hymba_kv* kv_in,
                                   const hymba_kv* kv_out, void* ws, size_t ws_bytes, int32_t* dev_status,
                                   void* const* events, int32_t n_events, void* stream) {
  Dims x;
  TRY(check_desc(d, false, &x));
  TRY(check_weights(w, x));
  if (!x_in || !y || !ws) return HYMBA_ERR_INVALID;
  if ((x.kv_shared != 0) != (kv_in != nullptr)) return HYMBA_ERR_INVALID;
  if (kv_in && (!kv_in->k || !kv_in->v)) return HYMBA_ERR_INVALID;
  if (kv_out && (!kv_out->k || !kv_out->v)) return HYMBA_ERR_INVALID;
  const size_t a = x.dtype == HYMBA_BF16 ? 16 : 4;
  if (!aligned(x_in, a) || !aligned(y, 16) || !aligned(ws, 256)) return HYMBA_ERR_INVALID;
  if (kv_in && (!aligned(kv_in->k, a) || !aligned(kv_in->v, a))) return HYMBA_ERR_INVALID;
  if (cache_out) {
    if (!cache_out->ssm_state || !cache_out->conv_state || cache_out->reserved != 0) return HYMBA_ERR_INVALID;
    if (!x.kv_shared) {
      if (!cache_out->k_ring || !cache_out->v_ring || !cache_out->k_meta || !cache_out->v_meta)
        return HYMBA_ERR_INVALID;
      if (cache_out->cap < 1) return HYMBA_ERR_INVALID;
      if (x.W > 0 ? cache_out->cap < x.W : cache_out->cap < x.T) return HYMBA_ERR_INVALID;
    }
  }
  if (n_events < 0 || (n_events > 0 && !events)) return HYMBA_ERR_INVALID;
  const Plan pl = plan_ws(x, false);
  if (ws_bytes < pl.total) return HYMBA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaGetLastError();  // clear a stale error so launch checks below are ours
  Marks mk;
  mk.ev = events;
  mk.n = n_events;
  mk.st = st;
  if (x.dtype == HYMBA_F32)
    return fwd_f32(x, pl, w, static_cast<const float*>(x_in), y, cache_out, kv_in, kv_out, ws, mk, st);
  return fwd_bf16(x, pl, w, x_in, y, cache_out, kv_in, kv_out, ws, dev_status, mk, st);
}

hymba_status hymba_layer_fwd(const hymba_layer_desc* d, const hymba_layer_weights* w, const void* x_in, float* y,
                             const hymba_cache* cache_out, const hymba_kv* kv_in, const hymba_kv* kv_out, void* ws,
                             size_t ws_bytes, int32_t* dev_status, void* stream) {
  return layer_fwd_impl(d, w, x_in, y, cache_out, kv_in, kv_out, ws, ws_bytes, dev_status, nullptr, 0, stream);
}

hymba_status hymba_layer_fwd_events(const hymba_layer_desc* d, const hymba_layer_weights* w, const void* x_in,
                                    float* y, const hymba_cache* cache_out, const hymba_kv* kv_in,
                                    const hymba_kv* kv_out, void* ws, size_t ws_bytes, int32_t* dev_status,
                                    void* const* events, int32_t n_events, void* stream) {
  return layer_fwd_impl(d, w, x_in, y, cache_out, kv_in, kv_out, ws, ws_bytes, dev_status, events, n_events, stream);
}

size_t hymba_meta_prefill_workspace(const hymba_layer_desc* d) {
  Dims x;
  if (meta_dims(d, true, &x) != HYMBA_OK) return 0;
  return plan_ws(x, false).total;
}

hymba_status hymba_meta_prefill(const hymba_layer_desc* d, const hymba_layer_weights* w, const void* x_meta,
                                const hymba_meta* meta, const hymba_kv* kv_in, void* ws, size_t ws_bytes,
                                int32_t* dev_status, void* stream) {
  Dims x;
  TRY(meta_dims(d, true, &x));
  TRY(check_weights(w, x));
  if (!x_meta || !meta || !meta->ssm_state || !meta->conv_tail || !meta->y || !ws) return HYMBA_ERR_INVALID;
  if (!x.kv_shared && (!meta->k || !meta->v)) return HYMBA_ERR_INVALID;
  if ((x.kv_shared != 0) != (kv_in != nullptr)) return HYMBA_ERR_INVALID;
  if (kv_in && (!kv_in->k || !kv_in->v || !aligned(kv_in->k, 16) || !aligned(kv_in->v, 16))) return HYMBA_ERR_INVALID;
  if (!aligned(x_meta, 16) || !aligned(meta->y, 16) || !aligned(ws, 256) || !aligned(meta->ssm_state, 4) ||
      !aligned(meta->conv_tail, 4) || (meta->k && !aligned(meta->k, 16)) || (meta->v && !aligned(meta->v, 16)))
    return HYMBA_ERR_INVALID;
  const Plan pl = plan_ws(x, false);
  if (ws_bytes < pl.total) return HYMBA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  Marks mk;
  mk.st = st;
  MetaCtx mc;
  mc.out = meta;
  return fwd_bf16(x, pl, w, x_meta, meta->y, nullptr, kv_in, nullptr, ws, dev_status, mk, st, mc);
}

size_t hymba_layer_fwd_meta_workspace(const hymba_layer_desc* d) {
  Dims x;
  if (meta_dims(d, false, &x) != HYMBA_OK) return 0;
  return plan_ws(x, false).total;
}

hymba_status hymba_layer_fwd_meta(const hymba_layer_desc* d, const hymba_layer_weights* w, const hymba_meta* meta,
                                  const void* x_in, float* y, const hymba_cache* cache_out, const hymba_kv* kv_in,
                                  const hymba_kv* kv_out, void* ws, size_t ws_bytes, int32_t* dev_status,
                                  void* stream) {
  Dims x;
  TRY(meta_dims(d, false, &x));
  TRY(check_weights(w, x));
  if (!meta || !meta->k || !meta->v || !meta->ssm_state || !meta->conv_tail || !x_in || !y || !ws)
    return HYMBA_ERR_INVALID;
  if (!aligned(meta->k, 16) || !aligned(meta->v, 16) || !aligned(meta->ssm_state, 4) || !aligned(meta->conv_tail, 4))
    return HYMBA_ERR_INVALID;
  if ((x.kv_shared != 0) != (kv_in != nullptr)) return HYMBA_ERR_INVALID;
  if (kv_in && (!kv_in->k || !kv_in->v || !aligned(kv_in->k, 16) || !aligned(kv_in->v, 16))) return HYMBA_ERR_INVALID;
  if (kv_out && (!kv_out->k || !kv_out->v)) return HYMBA_ERR_INVALID;
  if (!aligned(x_in, 16) || !aligned(y, 16) || !aligned(ws, 256)) return HYMBA_ERR_INVALID;
  if (cache_out) {
    if (!cache_out->ssm_state || !cache_out->conv_state || cache_out->reserved != 0) return HYMBA_ERR_INVALID;
    if (!x.kv_shared) {
      if (!cache_out->k_ring || !cache_out->v_ring || !cache_out->k_meta || !cache_out->v_meta)
        return HYMBA_ERR_INVALID;
      if (cache_out->cap < 1) return HYMBA_ERR_INVALID;
      if (x.W > 0 ? cache_out->cap < x.W : cache_out->cap < x.T) return HYMBA_ERR_INVALID;
    }
  }
  const Plan pl = plan_ws(x, false);
  if (ws_bytes < pl.total) return HYMBA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  Marks mk;
  mk.st = st;
  MetaCtx mc;
  mc.in = meta;
  return fwd_bf16(x, pl, w, x_in, y, cache_out, kv_in, kv_out, ws, dev_status, mk, st, mc);
}

// ---- full residual block ---------------------------------------------------

namespace {

struct BlockPlan {
  Plan layer;
  size_t xn, h, wdown, total;
};

hymba_status block_dims(const hymba_layer_desc* d, int32_t d_ff, Dims* x) {
  if (!d) return HYMBA_ERR_INVALID;
  TRY(check_desc(d, false, x));
  if (x->dtype != HYMBA_BF16 || x->residual != 0) return d->residual != 0 ? HYMBA_ERR_INVALID : HYMBA_ERR_UNSUPPORTED;
  if (d_ff < 8 || d_ff % 8 || x->d % 8) return HYMBA_ERR_UNSUPPORTED;
  x->residual = 2;  // the layer adds its output into the stream
  return HYMBA_OK;
}

BlockPlan plan_block(const Dims& x, int d_ff) {
  BlockPlan b{};
  b.layer = plan_ws(x, false);
  size_t off = align_up(b.layer.total, 256);
  const size_t r = static_cast<size_t>(x.rows);
  b.xn = off;
  off = align_up(off + r * x.d * 2, 256);
  b.h = off;
  off = align_up(off + r * static_cast<size_t>(d_ff) * 2, 256);
  b.wdown = off;
  off = align_up(off + static_cast<size_t>(x.d) * d_ff * 2, 256);
  b.total = off;
  return b;
}

}  // namespace

size_t hymba_block_fwd_workspace(const hymba_layer_desc* d, int32_t d_ff) {
  Dims x;
  if (block_dims(d, d_ff, &x) != HYMBA_OK) return 0;
  return plan_block(x, d_ff).total;
}

hymba_status hymba_block_fwd(const hymba_layer_desc* d, const hymba_block_weights* w, int32_t d_ff, float* xs,
                             void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
  Dims x;
  TRY(block_dims(d, d_ff, &x));
  if (!w || !xs || !ws) return HYMBA_ERR_INVALID;
  TRY(check_weights(&w->mix, x));
  if (!w->norm1 || !w->norm2 || !w->W_gu || !w->W_down) return HYMBA_ERR_INVALID;
  if (!aligned(xs, 16) || !aligned(ws, 256) || !aligned(w->norm1, 16) || !aligned(w->norm2, 16) ||
      !aligned(w->W_gu, 16) || !aligned(w->W_down, 16))
    return HYMBA_ERR_INVALID;
  const BlockPlan bp = plan_block(x, d_ff);
  if (ws_bytes < bp.total) return HYMBA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  const int sms = num_sms();
  const int rows = static_cast<int>(x.rows);
  __nv_bfloat16* xn = at<__nv_bfloat16>(ws, bp.xn);
  __half* h = at<__half>(ws, bp.h);
  __half* wdown = at<__half>(ws, bp.wdown);
  // x += Layer(RMSNorm(x; norm1))
  TRY(rmsnorm_bf16(rows, x.d, xs, x.d, w->norm1, x.eps, xn, x.d, st));
  Marks mk;
  mk.st = st;
  TRY(fwd_bf16(x, bp.layer, &w->mix, xn, xs, nullptr, nullptr, nullptr, ws, dev_status, mk, st));
  // x += W_down (GeLU(W_gate h) * (W_up h)),  h = RMSNorm(x; norm2)
  TRY(rmsnorm_bf16(rows, x.d, xs, x.d, w->norm2, x.eps, xn, x.d, st));
  TRY(copy2d<__nv_bfloat16, __half>(static_cast<const __nv_bfloat16*>(w->W_down), d_ff, wdown, d_ff, x.d, d_ff, st));
  {
    GemmParams p = gp(rows, 2 * d_ff, x.d, dev_status, x.wait_ns);
    p.C = h;
    p.ldc = d_ff;
    TRY(gemm_tc(1, xn, x.d, w->W_gu, x.d, EPI_GEGLU, p, 0, 1, sms, st));
  }
  {
    GemmParams p = gp(rows, x.d, d_ff, dev_status, x.wait_ns);
    p.C = xs;
    p.ldc = x.d;
    p.resid_f32 = xs;
    p.ld_resid = x.d;
    TRY(gemm_tc(0, h, d_ff, wdown, d_ff, EPI_F32, p, 0, 1, sms, st));
  }
  return HYMBA_OK;
}

// ---- residual stack ---------------------------------------------------------

namespace {

constexpr int kMaxStackLayers = 256;

struct StackPlan {
  size_t layer_ws, xs, w16, kv_k, kv_v, total;
};

// Every layer on the bf16 path, one batch shape, residual 0 (the stack adds
// the stream), no K/V sharing into layer 0.  dims[l] get residual 1 for layer
// 0 (Y = X~ + layer) and 2 after (Y += layer, in place).
hymba_status stack_dims(int32_t n, const hymba_layer_desc* d, Dims* dims, StackPlan* sp) {
  if (n < 1 || n > kMaxStackLayers || !d) return HYMBA_ERR_INVALID;
  StackPlan p{};
  size_t kv_k = 0, kv_v = 0;
  for (int l = 0; l < n; ++l) {
    TRY(check_desc(&d[l], false, &dims[l]));
    const Dims& x = dims[l];
    if (d[l].residual != 0) return HYMBA_ERR_INVALID;
    if (x.dtype != HYMBA_BF16) return HYMBA_ERR_UNSUPPORTED;
    if (x.B != dims[0].B || x.L != dims[0].L || x.M != dims[0].M || x.d != dims[0].d) return HYMBA_ERR_INVALID;
    if (x.kv_shared) {
      if (l == 0) return HYMBA_ERR_INVALID;
      const Dims& pr = dims[l - 1];
      if (pr.Hkv != x.Hkv || pr.dh != x.dh || pr.dv != x.dv) return HYMBA_ERR_INVALID;
      kv_k = std::max(kv_k, static_cast<size_t>(x.rows) * x.Hkv * x.dh * 2);
      kv_v = std::max(kv_v, static_cast<size_t>(x.rows) * x.Hkv * x.dv * 2);
    }
    dims[l].residual = l == 0 ? 1 : 2;
    p.layer_ws = std::max(p.layer_ws, plan_ws(dims[l], false).total);
  }
  size_t w16 = 0;
  for (int l = 1; l < n; ++l) w16 = std::max(w16, static_cast<size_t>(dims[l].P_in) * dims[l].d * 2);
  size_t off = align_up(p.layer_ws, 256);
  p.xs = off;
  off = align_up(off + static_cast<size_t>(dims[0].rows) * dims[0].d * 2, 256);
  p.w16 = off;
  off = align_up(off + w16, 256);
  p.kv_k = off;
  off = align_up(off + kv_k, 256);
  p.kv_v = off;
  off = align_up(off + kv_v, 256);
  p.total = off;
  *sp = p;
  return HYMBA_OK;
}

}  // namespace

size_t hymba_stack_fwd_workspace(int32_t n_layers, const hymba_layer_desc* descs) {
  if (n_layers < 1 || n_layers > kMaxStackLayers) return 0;
  Dims dims[kMaxStackLayers];
  StackPlan sp;
  if (stack_dims(n_layers, descs, dims, &sp) != HYMBA_OK) return 0;
  return sp.total;
}

hymba_status hymba_stack_fwd(int32_t n_layers, const hymba_layer_desc* descs, const hymba_layer_weights* weights,
                             const void* x_in, float* y, void* ws, size_t ws_bytes, int32_t* dev_status,
                             void* stream) {
  if (n_layers < 1 || n_layers > kMaxStackLayers) return HYMBA_ERR_INVALID;
  Dims dims[kMaxStackLayers];
  StackPlan sp;
  TRY(stack_dims(n_layers, descs, dims, &sp));
  if (!weights || !x_in || !y || !ws) return HYMBA_ERR_INVALID;
  for (int l = 0; l < n_layers; ++l) TRY(check_weights(&weights[l], dims[l]));
  if (!aligned(x_in, 16) || !aligned(y, 16) || !aligned(ws, 256)) return HYMBA_ERR_INVALID;
  if (ws_bytes < sp.total) return HYMBA_ERR_WORKSPACE;
  const size_t stream_bytes = static_cast<size_t>(dims[0].rows) * dims[0].d;
  const char* xb0 = static_cast<const char*>(x_in);
  const char* yb0 = reinterpret_cast<const char*>(y);
  if (xb0 < yb0 + stream_bytes * 4 && yb0 < xb0 + stream_bytes * 2) return HYMBA_ERR_INVALID;  // y may not overlap x
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  __half* xs = at<__half>(ws, sp.xs);     // the stream rounded to fp16: layers 1.. read it
  __half* w16 = at<__half>(ws, sp.w16);   // fp16 copy of the current layer's W_in
  hymba_kv kv{at<void>(ws, sp.kv_k), at<void>(ws, sp.kv_v)};
  for (int l = 0; l < n_layers; ++l) {
    const Dims& x = dims[l];
    const bool last = l + 1 == n_layers;
    // export K/V when the next layer shares them (a shared layer's K/V are
    // already in the buffer)
    const bool export_kv = !last && dims[l + 1].kv_shared && !x.kv_shared;
    StackIO sio;
    sio.y_f16 = last ? nullptr : xs;
    if (l > 0) {
      TRY(copy2d<__nv_bfloat16, __half>(static_cast<const __nv_bfloat16*>(weights[l].W_in), x.d, w16, x.d, x.P_in,
                                        x.d, st));
      sio.w_in_f16 = w16;
    }
    Marks mk;
    mk.st = st;
    TRY(fwd_bf16(x, plan_ws(x, false), &weights[l], l == 0 ? x_in : xs, y, nullptr, x.kv_shared ? &kv : nullptr,
                 export_kv ? &kv : nullptr, ws, dev_status, mk, st, MetaCtx{}, sio));
  }
  return HYMBA_OK;
}

static hymba_status layer_decode_impl(const hymba_layer_desc* d, const hymba_layer_weights* w, const void* x_new,
                                      float* y, const hymba_cache* cache, const hymba_cache* shared_cache, void* ws,
                                      size_t ws_bytes, int32_t* dev_status, void* const* events, int32_t n_events,
                                      void* stream) {
  Dims x;
  TRY(check_desc(d, true, &x));
  TRY(check_weights(w, x));
  if (!x_new || !y || !ws || !cache) return HYMBA_ERR_INVALID;
  if ((x.kv_shared != 0) != (shared_cache != nullptr)) return HYMBA_ERR_INVALID;
  const hymba_cache* kvc = x.kv_shared ? shared_cache : cache;
  if (!cache->ssm_state || !cache->conv_state || !cache->pos || cache->reserved != 0) return HYMBA_ERR_INVALID;
  if (!kvc->k_ring || !kvc->v_ring || (x.M > 0 && (!kvc->k_meta || !kvc->v_meta)) || kvc->cap < 1)
    return HYMBA_ERR_INVALID;
  if (x.W > 0 && kvc->cap < x.W) return HYMBA_ERR_INVALID;
  const size_t a = x.dtype == HYMBA_BF16 ? 16 : 4;
  if (!aligned(x_new, a) || !aligned(y, 16) || !aligned(ws, 256)) return HYMBA_ERR_INVALID;
  if (n_events < 0 || (n_events > 0 && !events)) return HYMBA_ERR_INVALID;
  const Plan pl = plan_ws(x, true);
  if (ws_bytes < pl.total) return HYMBA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaGetLastError();
  if (x.dtype == HYMBA_F32)
    return decode_f32(x, pl, w, static_cast<const float*>(x_new), y, cache, kvc, ws, st);
  Marks mk;
  mk.ev = events;
  mk.n = n_events;
  mk.st = st;
  return decode_bf16(x, pl, w, x_new, y, cache, kvc, ws, dev_status, mk, st);
}

hymba_status hymba_layer_decode(const hymba_layer_desc* d, const hymba_layer_weights* w, const void* x_new,
                                float* y, const hymba_cache* cache, const hymba_cache* shared_cache, void* ws,
                                size_t ws_bytes, int32_t* dev_status, void* stream) {
  return layer_decode_impl(d, w, x_new, y, cache, shared_cache, ws, ws_bytes, dev_status, nullptr, 0, stream);
}

hymba_status hymba_layer_decode_events(const hymba_layer_desc* d, const hymba_layer_weights* w, const void* x_new,
                                       float* y, const hymba_cache* cache, const hymba_cache* shared_cache,
                                       void* ws, size_t ws_bytes, int32_t* dev_status, void* const* events,
                                       int32_t n_events, void* stream) {
  return layer_decode_impl(d, w, x_new, y, cache, shared_cache, ws, ws_bytes, dev_status, events, n_events,
                           stream);
}

// --------------------------------------------------------------------------- tests

hymba_status hymba_test_gemm(int32_t M, int32_t N, int32_t K, int32_t ab_dtype, const void* A, int32_t lda,
                             const void* B, int32_t ldb, float* C, int32_t ldc, int32_t* dev_status, void* stream) {
  if (M < 1 || N < 1 || K < 1 || !A || !B || !C || ab_dtype < 1 || ab_dtype > 3 || ldc < N)
    return HYMBA_ERR_INVALID;
  GemmParams p{};
  p.cvt_b = ab_dtype == 3 ? 1 : 0;
  p.M = M;
  p.N = N;
  p.K = K;
  p.C = C;
  p.ldc = ldc;
  p.rows_per_seq = 1;
  p.status = dev_status;
  p.wait_ns = 2000000000ull;
  cudaGetLastError();
  return gemm_tc(ab_dtype == 1 ? 1 : 0, A, lda, B, ldb, EPI_F32, p, 0, 1, num_sms(),
                 static_cast<cudaStream_t>(stream));
}

hymba_status hymba_test_conv(int32_t B, int32_t L, int32_t di, int32_t k, const void* x, int32_t ld_x, void* u,
                             const float* conv_w, const float* conv_b, int32_t* dev_status, void* stream) {
  if (B < 1 || L < 1 || di < 1 || !x || !u || !conv_w || !conv_b || ld_x < di) return HYMBA_ERR_INVALID;
  if (!conv_tma_supported(di, k, ld_x, di, x, u)) return HYMBA_ERR_UNSUPPORTED;
  cudaGetLastError();
  return conv_silu_tma(static_cast<const __half*>(x), ld_x, static_cast<__half*>(u), di, B, L, di, k, conv_w, conv_b,
                       dev_status, 2000000000ull, num_sms(), static_cast<cudaStream_t>(stream));
}

static bool scan_layout_ok(int32_t tpc, int32_t cpt) {
  if (tpc == 0) return cpt == 0;
  if (tpc != 1 && tpc != 2 && tpc != 4) return false;
  return cpt == 0 || cpt == 1 || (cpt == 2 && tpc != 1);
}

hymba_status hymba_test_scan(int32_t B, int32_t L, int32_t di, int32_t N, const void* u, int32_t ld_u, const void* z,
                             int32_t ld_z, const float* delta, const float* BC, const float* A_log, const float* D,
                             void* g, float* h_out, int32_t threads_per_channel, int32_t channels_per_thread,
                             void* stream) {
  if (B < 1 || L < 1 || di < 1 || N < 1 || N > 64 || !u || !z || !delta || !BC || !A_log || !D || !g ||
      !scan_layout_ok(threads_per_channel, channels_per_thread))
    return HYMBA_ERR_INVALID;
  cudaGetLastError();
  return scan_f16(B, L, di, N, static_cast<const __half*>(u), ld_u, static_cast<const __half*>(z), ld_z, delta, BC,
                  A_log, D, static_cast<__half*>(g), nullptr, h_out, nullptr, 2000000000ull, threads_per_channel,
                  channels_per_thread, static_cast<cudaStream_t>(stream));
}

hymba_status hymba_test_scan_fused(int32_t B, int32_t L, int32_t di, int32_t N, int32_t R, const void* u,
                                   int32_t ld_u, const void* z, int32_t ld_z, const void* dtr, int32_t ld_dtr,
                                   const void* W_dt, const float* dt_bias, const float* BC, const float* A_log,
                                   const float* D, void* g, float* h_out, int32_t threads_per_channel,
                                   int32_t channels_per_thread, void* stream) {
  if (B < 1 || L < 1 || di < 1 || N < 1 || R < 1 || !u || !z || !dtr || !W_dt || !dt_bias || !BC || !A_log || !D ||
      !g || !scan_layout_ok(threads_per_channel, channels_per_thread))
    return HYMBA_ERR_INVALID;
  cudaGetLastError();
  return scan_fused_f16(B, L, di, N, R, static_cast<const __half*>(u), ld_u, static_cast<const __half*>(z), ld_z,
                        static_cast<const __half*>(dtr), ld_dtr, static_cast<const __nv_bfloat16*>(W_dt), dt_bias, BC,
                        A_log, D, static_cast<__half*>(g), nullptr, h_out, nullptr, 2000000000ull, threads_per_channel,
                        channels_per_thread, static_cast<cudaStream_t>(stream));
}

hymba_status hymba_test_attention(int32_t B, int32_t L, int32_t M, int32_t Hq, int32_t Hkv, int32_t dh, int32_t dv,
                                  int32_t window, int32_t use_tc, const void* Q, const void* K, const void* V,
                                  void* O, int32_t* dev_status, void* stream) {
  if (B < 1 || L < 1 || M < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv || dh < 1 || dv < 1 || window < 0 || !Q || !K ||
      !V || !O)
    return HYMBA_ERR_INVALID;
  cudaGetLastError();
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const __half* q = static_cast<const __half*>(Q);
  const __half* k = static_cast<const __half*>(K);
  const __half* v = static_cast<const __half*>(V);
  __half* o = static_cast<__half*>(O);
  if (use_tc) {
    if (!attn_tc_supported(dh, dv)) return HYMBA_ERR_UNSUPPORTED;
    return attn_tc(B, L, M, Hq, Hkv, dh, dv, window, q, static_cast<long long>(Hq) * dh, k,
                   static_cast<long long>(Hkv) * dh, v, static_cast<long long>(Hkv) * dv, o,
                   static_cast<long long>(Hq) * dv, dev_status, 2000000000ull, num_sms(), st);
  }
  return attention_simt<__half>(B, L, M, Hq, Hkv, dh, dv, window, q, static_cast<long long>(Hq) * dh, k,
                                static_cast<long long>(Hkv) * dh, v, static_cast<long long>(Hkv) * dv, o,
                                static_cast<long long>(Hq) * dv, st);
}

hymba_status hymba_test_wait_timeout(uint32_t limit_us, int32_t* dev_status, void* stream) {
  if (!dev_status || limit_us == 0 || limit_us > 10000000u) return HYMBA_ERR_INVALID;
  cudaGetLastError();
  return wait_timeout_probe(limit_us, dev_status, static_cast<cudaStream_t>(stream));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Decode without caller-supplied workspace (hymba_layer_decode_static).
//
// For callers that cannot allocate device memory when they run a decode step
// (a plugin whose host framework owns all device memory, a serving loop whose
// memory is fully reserved by its cache pool): the scratch is this file-scope
// device buffer.  Host code must not use the symbol itself as a device
// address; it fetches the per-device address once with cudaGetSymbolAddress.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_decode_scratch[HYMBA_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device (looked up on the
// first call per device, with that device current).
hymba_status static_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return HYMBA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return HYMBA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return HYMBA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return HYMBA_OK;
}

}  // namespace

extern "C" hymba_status hymba_layer_decode_static(const hymba_layer_desc* d, const hymba_layer_weights* w,
                                                  const void* x_new, float* y, const hymba_cache* cache,
                                                  const hymba_cache* shared_cache, int32_t* dev_status,
                                                  void* stream) {
  const size_t need = hymba_layer_decode_workspace(d);
  if (need == 0)  // invalid descriptor: report its error without touching the device
    return hymba_layer_decode(d, w, x_new, y, cache, shared_cache, nullptr, 0, dev_status, stream);
  if (need > HYMBA_STATIC_SCRATCH_BYTES) return HYMBA_ERR_WORKSPACE;
  void* ws = nullptr;
  const hymba_status s = static_scratch(&ws);
  if (s != HYMBA_OK) return s;
  return hymba_layer_decode(d, w, x_new, y, cache, shared_cache, ws, HYMBA_STATIC_SCRATCH_BYTES, dev_status, stream);
}
