// Decode-step kernels: ring-buffer K/V append, attention over meta + ring,
// conv step from the carried tail, split-K reduction, position advance.
#include <algorithm>

#include "decode.cuh"

namespace hy {
namespace {

HY_DEV float to_f(float v) { return v; }
HY_DEV float to_f(__half v) { return __half2float(v); }
HY_DEV float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T>
HY_DEV T from_f(float v);
template <>
HY_DEV float from_f<float>(float v) { return v; }
template <>
HY_DEV __half from_f<__half>(float v) { return __float2half_rn(v); }
template <>
HY_DEV __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

inline hymba_status last_err() { return cudaGetLastError() == cudaSuccess ? HYMBA_OK : HYMBA_ERR_CUDA; }

HY_DEV int ring_slot(int p, int window, int cap) { return window > 0 ? p % cap : p; }

template <typename TS, typename TC>
__global__ void kv_append_kernel(int B, int Hkv, int dh, int dv, int window, int cap, const TS* proj,
                                 long long ldp, int k_col, int v_col, const int32_t* pos, TC* k_ring,
                                 TC* v_ring) {
  const int wk = Hkv * dh, wv = Hkv * dv;
  const int n = B * (wk + wv);
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += gridDim.x * blockDim.x) {
    const int b = idx / (wk + wv);
    const int c = idx % (wk + wv);
    const int slot = ring_slot(pos[b], window, cap);
    if (c < wk)
      k_ring[(static_cast<long long>(b) * cap + slot) * wk + c] = from_f<TC>(to_f(proj[b * ldp + k_col + c]));
    else
      v_ring[(static_cast<long long>(b) * cap + slot) * wv + (c - wk)] =
          from_f<TC>(to_f(proj[b * ldp + v_col + (c - wk)]));
  }
}

// one warp per (b, query head); keys 0..M-1 are meta, M.. are ring entries
// newest first.
template <typename TQ, typename TC>
__global__ void __launch_bounds__(128) decode_attention_kernel(int B, int M, int Hq, int Hkv, int dh, int dv,
                                                               int window, int cap, const TQ* q, long long ldq,
                                                               const TC* k_meta, const TC* v_meta,
                                                               const TC* k_ring, const TC* v_ring,
                                                               const int32_t* pos, TQ* out, long long ldo) {
  extern __shared__ float qs[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wid = blockIdx.x * 4 + warp;
  const bool active = wid < B * Hq;
  const int b = active ? wid / Hq : 0;
  const int h = active ? wid % Hq : 0;
  const int gidx = (h * Hkv) / Hq;
  float* qv = qs + warp * dh;
  const float scale = rsqrtf(static_cast<float>(dh));
  for (int e = lane; e < dh; e += 32) qv[e] = active ? to_f(q[b * ldq + h * dh + e]) * scale : 0.f;
  __syncwarp();
  if (!active) return;
  const int p = pos[b];
  int n_vis = window > 0 ? min(p + 1, window) : p + 1;
  n_vis = min(n_vis, cap);
  const int n_keys = M + n_vis;
  constexpr int MAXR = 8;
  float o[MAXR];
#pragma unroll
  for (int r = 0; r < MAXR; ++r) o[r] = 0.f;
  float m = -INFINITY, lsum = 0.f;
  const long long wk = static_cast<long long>(Hkv) * dh, wv = static_cast<long long>(Hkv) * dv;
  for (int j0 = 0; j0 < n_keys; j0 += 32) {
    const int j = j0 + lane;
    float sc = -INFINITY;
    if (j < n_keys) {
      const TC* kr;
      if (j < M) {
        kr = k_meta + j * wk + gidx * dh;
      } else {
        const int rel = j - M;  // 0 = this token; p - rel >= 0 since rel < n_vis <= p + 1
        const int slot = window > 0 ? (p - rel) % cap : p - rel;
        kr = k_ring + (static_cast<long long>(b) * cap + slot) * wk + gidx * dh;
      }
      float acc = 0.f;
      for (int e = 0; e < dh; ++e) acc = fmaf(qv[e], to_f(kr[e]), acc);
      sc = acc;
    }
    float mx = sc;
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float m_new = fmaxf(m, mx);
    const float alpha = (m == -INFINITY) ? 0.f : expf(m - m_new);
    const float pj_own = (sc == -INFINITY) ? 0.f : expf(sc - m_new);
    float ps = pj_own;
    for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
    lsum = lsum * alpha + ps;
#pragma unroll
    for (int r = 0; r < MAXR; ++r) o[r] *= alpha;
    const int nk = min(32, n_keys - j0);
    for (int jj = 0; jj < nk; ++jj) {
      const float pj = __shfl_sync(0xffffffffu, pj_own, jj);
      const int jk = j0 + jj;
      const TC* vr;
      if (jk < M) {
        vr = v_meta + jk * wv + gidx * dv;
      } else {
        const int rel = jk - M;
        const int slot = window > 0 ? (p - rel) % cap : p - rel;
        vr = v_ring + (static_cast<long long>(b) * cap + slot) * wv + gidx * dv;
      }
#pragma unroll
      for (int r = 0; r < MAXR; ++r) {
        const int e = lane + 32 * r;
        if (e < dv) o[r] = fmaf(pj, to_f(vr[e]), o[r]);
      }
    }
    m = m_new;
  }
  const float inv = 1.0f / lsum;
#pragma unroll
  for (int r = 0; r < MAXR; ++r) {
    const int e = lane + 32 * r;
    if (e < dv) out[b * ldo + h * dv + e] = from_f<TQ>(o[r] * inv);
  }
}

template <typename T>
__global__ void conv_step_kernel(int B, int di, int k, const T* x, long long ldx, const float* w,
                                 const float* bias, float* conv_state, T* u, long long ldu) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= B * di) return;
  const int b = idx / di, c = idx % di;
  float* st = conv_state + static_cast<long long>(idx) * (k - 1);
  const float xv = to_f(x[b * ldx + c]);
  float acc = bias[c];
  for (int j = 0; j < k - 1; ++j) acc = fmaf(w[c * k + j], st[j], acc);
  acc = fmaf(w[c * k + k - 1], xv, acc);
  for (int j = 0; j + 1 < k - 1; ++j) st[j] = st[j + 1];
  if (k > 1) st[k - 2] = xv;
  u[b * ldu + c] = from_f<T>(acc / (1.0f + expf(-acc)));
}

__global__ void splitk_reduce_kernel(int splits, int rows, int N, const float* part, long long ldp, int epi,
                                     int R, __half* dtr, long long ldd, float* C, long long ldc,
                                     const __nv_bfloat16* resid, long long ld_resid, int accumulate) {
  const long long n = static_cast<long long>(rows) * N;
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < n;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int row = static_cast<int>(idx / N), col = static_cast<int>(idx % N);
    float acc = 0.f;
    for (int s = 0; s < splits; ++s) acc += part[(static_cast<long long>(s) * rows + row) * ldp + col];
    if (epi == RE_XPROJ) {
      if (col < R)
        dtr[row * ldd + col] = __float2half_rn(acc);
      else
        C[row * ldc + col - R] = acc;
    } else {
      if (resid) acc += __bfloat162float(resid[row * ld_resid + col]);
      if (accumulate) acc += C[row * ldc + col];
      C[row * ldc + col] = acc;
    }
  }
}

__global__ void pos_increment_kernel(int B, int32_t* pos) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) pos[b] += 1;
}

}  // namespace

template <typename TS, typename TC>
hymba_status kv_append(int B, int Hkv, int dh, int dv, int window, int cap, const TS* proj, long long ldp,
                       int k_col, int v_col, const int32_t* pos, TC* k_ring, TC* v_ring, cudaStream_t st) {
  const int n = B * Hkv * (dh + dv);
  kv_append_kernel<TS, TC><<<std::min((n + 255) / 256, 148 * 8), 256, 0, st>>>(
      B, Hkv, dh, dv, window, cap, proj, ldp, k_col, v_col, pos, k_ring, v_ring);
  return last_err();
}

template <typename TQ, typename TC>
hymba_status decode_attention(int B, int M, int Hq, int Hkv, int dh, int dv, int window, int cap, const TQ* q,
                              long long ldq, const TC* k_meta, const TC* v_meta, const TC* k_ring,
                              const TC* v_ring, const int32_t* pos, TQ* out, long long ldo, cudaStream_t st) {
  if (dv > 256) return HYMBA_ERR_UNSUPPORTED;
  const int warps = B * Hq;
  decode_attention_kernel<TQ, TC><<<(warps + 3) / 4, 128, 4 * dh * sizeof(float), st>>>(
      B, M, Hq, Hkv, dh, dv, window, cap, q, ldq, k_meta, v_meta, k_ring, v_ring, pos, out, ldo);
  return last_err();
}

template <typename T>
hymba_status conv_step(int B, int di, int k, const T* x, long long ldx, const float* w, const float* bias,
                       float* conv_state, T* u, long long ldu, cudaStream_t st) {
  const int n = B * di;
  conv_step_kernel<T><<<(n + 255) / 256, 256, 0, st>>>(B, di, k, x, ldx, w, bias, conv_state, u, ldu);
  return last_err();
}

hymba_status splitk_reduce(int splits, int rows, int N, const float* part, long long ldp, int epi, int R,
                           __half* dtr, long long ldd, float* C, long long ldc, const __nv_bfloat16* resid,
                           long long ld_resid, bool accumulate, cudaStream_t st) {
  const long long n = static_cast<long long>(rows) * N;
  splitk_reduce_kernel<<<static_cast<unsigned>(std::min<long long>((n + 255) / 256, 148 * 8)), 256, 0, st>>>(
      splits, rows, N, part, ldp, epi, R, dtr, ldd, C, ldc, resid, ld_resid, accumulate ? 1 : 0);
  return last_err();
}

hymba_status pos_increment(int B, int32_t* pos, cudaStream_t st) {
  pos_increment_kernel<<<(B + 255) / 256, 256, 0, st>>>(B, pos);
  return last_err();
}

template hymba_status kv_append<float, float>(int, int, int, int, int, int, const float*, long long, int, int,
                                              const int32_t*, float*, float*, cudaStream_t);
template hymba_status kv_append<__half, __nv_bfloat16>(int, int, int, int, int, int, const __half*, long long,
                                                       int, int, const int32_t*, __nv_bfloat16*,
                                                       __nv_bfloat16*, cudaStream_t);
template hymba_status decode_attention<float, float>(int, int, int, int, int, int, int, int, const float*,
                                                     long long, const float*, const float*, const float*,
                                                     const float*, const int32_t*, float*, long long,
                                                     cudaStream_t);
template hymba_status decode_attention<__half, __nv_bfloat16>(int, int, int, int, int, int, int, int,
                                                              const __half*, long long, const __nv_bfloat16*,
                                                              const __nv_bfloat16*, const __nv_bfloat16*,
                                                              const __nv_bfloat16*, const int32_t*, __half*,
                                                              long long, cudaStream_t);
template hymba_status conv_step<float>(int, int, int, const float*, long long, const float*, const float*,
                                       float*, float*, long long, cudaStream_t);
template hymba_status conv_step<__half>(int, int, int, const __half*, long long, const float*, const float*,
                                        float*, __half*, long long, cudaStream_t);

}  // namespace hy
