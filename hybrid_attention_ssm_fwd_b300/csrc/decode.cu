// Decode-step kernels: ring-buffer K/V append, attention over meta + ring,
// conv step from the carried tail, split-K reduction, position advance.
// One new token per sequence through the layer of eq. 3 ("Hymba: A Hybrid-head Architecture for Small Language Models",
// section 2.1), with the sliding-window cache and the meta K/V that every
// later token sees (sections 2.2 and 2.3).
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
    if (slot < 0 || slot >= cap) continue;  // a full global cache (or pos < 0): write nothing
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

// Split-KV decode attention for bf16 caches.  One CTA per (sequence b, KV
// group g, key split sp) serves all G = Hq/Hkv query heads of the group, so
// each K/V row of the cache is read once per step.  Keys 0..M-1 are the meta
// prefix, keys M.. the visible ring entries (newest first).  Each thread
// scores whole keys (16-byte K loads); P.V walks the keys with the threads
// spread over the value dims.  Output: per (b, head, split) the partial
// max m (log2 units), sum l and unnormalised o[dv], all fp32.
constexpr int DA_THREADS = 128;
constexpr int DA_MAXG = 8;

__global__ void __launch_bounds__(DA_THREADS)
    decode_attn_split_kernel(int M, int Hq, int Hkv, int dh, int dv, int window, int cap, int nsplit,
                             const __half* __restrict__ q, long long ldq, const __nv_bfloat16* __restrict__ k_meta,
                             const __nv_bfloat16* __restrict__ v_meta, const __nv_bfloat16* __restrict__ k_ring,
                             const __nv_bfloat16* __restrict__ v_ring, const int32_t* __restrict__ pos,
                             float* __restrict__ part) {
  extern __shared__ float sm[];
  const int G = Hq / Hkv;
  const int sp = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;
  const int p = pos[b];
  const int n_vis = min(window > 0 ? min(p + 1, window) : p + 1, cap);
  const int n_keys = M + n_vis;
  const int per = (n_keys + nsplit - 1) / nsplit;
  const int k_lo = sp * per, k_hi = min(n_keys, k_lo + per);
  const int nk = max(0, k_hi - k_lo);
  float* qs = sm;                       // [G][dh], pre-scaled by log2(e)/sqrt(dh)
  float* sc = sm + DA_MAXG * 128;       // [G][per]
  float* red = sc + G * per;            // [2][G][4]
  const float qscale = 1.4426950408889634f * rsqrtf(static_cast<float>(dh));
  for (int idx = tid; idx < G * dh; idx += DA_THREADS) {
    const int hh = idx / dh, e = idx % dh;
    qs[idx] = __half2float(q[b * ldq + (g * G + hh) * dh + e]) * qscale;
  }
  __syncthreads();
  const long long wk = static_cast<long long>(Hkv) * dh, wv = static_cast<long long>(Hkv) * dv;
  auto krow = [&](int j) -> const __nv_bfloat16* {
    if (j < M) return k_meta + j * wk + g * dh;
    const int rel = j - M;  // 0 = this token
    const int slot = window > 0 ? (p - rel) % cap : p - rel;
    return k_ring + (static_cast<long long>(b) * cap + slot) * wk + g * dh;
  };
  auto vrow = [&](int j) -> const __nv_bfloat16* {
    if (j < M) return v_meta + j * wv + g * dv;
    const int rel = j - M;
    const int slot = window > 0 ? (p - rel) % cap : p - rel;
    return v_ring + (static_cast<long long>(b) * cap + slot) * wv + g * dv;
  };
  // scores
  float lmax[DA_MAXG];
#pragma unroll
  for (int hh = 0; hh < DA_MAXG; ++hh) lmax[hh] = -INFINITY;
  for (int kk = tid; kk < nk; kk += DA_THREADS) {
    const uint4* kr = reinterpret_cast<const uint4*>(krow(k_lo + kk));
    float acc[DA_MAXG];
#pragma unroll
    for (int hh = 0; hh < DA_MAXG; ++hh) acc[hh] = 0.f;
    for (int c = 0; c < dh / 8; ++c) {
      const uint4 v = kr[c];
      const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int e2 = 0; e2 < 4; ++e2) {
        const float2 f = __bfloat1622float2(h2[e2]);
#pragma unroll
        for (int hh = 0; hh < DA_MAXG; ++hh)
          if (hh < G) acc[hh] = fmaf(qs[hh * dh + c * 8 + 2 * e2 + 1], f.y, fmaf(qs[hh * dh + c * 8 + 2 * e2], f.x, acc[hh]));
      }
    }
#pragma unroll
    for (int hh = 0; hh < DA_MAXG; ++hh)
      if (hh < G) {
        sc[hh * per + kk] = acc[hh];
        lmax[hh] = fmaxf(lmax[hh], acc[hh]);
      }
  }
  // block max per head
  const int w = tid >> 5, l = tid & 31;
#pragma unroll
  for (int hh = 0; hh < DA_MAXG; ++hh) {
    if (hh >= G) break;
    float v = lmax[hh];
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (l == 0) red[hh * 4 + w] = v;
  }
  __syncthreads();
  // probabilities and sums
  float lsum[DA_MAXG];
  float mh[DA_MAXG];
#pragma unroll
  for (int hh = 0; hh < DA_MAXG; ++hh) {
    lsum[hh] = 0.f;
    mh[hh] = hh < G ? fmaxf(fmaxf(red[hh * 4], red[hh * 4 + 1]), fmaxf(red[hh * 4 + 2], red[hh * 4 + 3])) : 0.f;
  }
  for (int kk = tid; kk < nk; kk += DA_THREADS) {
#pragma unroll
    for (int hh = 0; hh < DA_MAXG; ++hh)
      if (hh < G) {
        const float e = ex2_approx(sc[hh * per + kk] - mh[hh]);
        sc[hh * per + kk] = e;
        lsum[hh] += e;
      }
  }
  float* red2 = red + G * 4;
#pragma unroll
  for (int hh = 0; hh < DA_MAXG; ++hh) {
    if (hh >= G) break;
    float v = lsum[hh];
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (l == 0) red2[hh * 4 + w] = v;
  }
  __syncthreads();
  // P.V: a thread owns a pair of value dims for one key phase; with dv/2 < 128
  // pairs the threads split the keys into nkh phases merged through smem
  const int npairs = dv / 2;
  const int nkh = max(1, DA_THREADS / npairs);
  float* ored = red2 + G * 4;  // [nkh][G][dv]
  for (int pr0 = 0; pr0 < npairs; pr0 += DA_THREADS) {
    const int pr = pr0 + tid % npairs;
    const int kh = (npairs >= DA_THREADS) ? 0 : tid / npairs;
    const bool act = pr < npairs && kh < nkh;
    const int e = 2 * pr;
    float o0[DA_MAXG], o1[DA_MAXG];
#pragma unroll
    for (int hh = 0; hh < DA_MAXG; ++hh) o0[hh] = o1[hh] = 0.f;
    if (act) {
      for (int kk = kh; kk < nk; kk += nkh) {
        const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(vrow(k_lo + kk) + e));
#pragma unroll
        for (int hh = 0; hh < DA_MAXG; ++hh)
          if (hh < G) {
            const float pp = sc[hh * per + kk];
            o0[hh] = fmaf(pp, v.x, o0[hh]);
            o1[hh] = fmaf(pp, v.y, o1[hh]);
          }
      }
      if (nkh > 1) {
#pragma unroll
        for (int hh = 0; hh < DA_MAXG; ++hh)
          if (hh < G) {
            ored[(kh * G + hh) * dv + e] = o0[hh];
            ored[(kh * G + hh) * dv + e + 1] = o1[hh];
          }
      }
    }
    if (nkh > 1) {
      __syncthreads();
      for (int idx = tid; idx < G * dv; idx += DA_THREADS) {
        const int hh = idx / dv, ee = idx % dv;
        float acc = 0.f;
        for (int q2 = 0; q2 < nkh; ++q2) acc += ored[(q2 * G + hh) * dv + ee];
        part[((static_cast<long long>(b) * Hq + g * G + hh) * nsplit + sp) * (dv + 2) + 2 + ee] = acc;
      }
    } else if (act) {
#pragma unroll
      for (int hh = 0; hh < DA_MAXG; ++hh)
        if (hh < G) {
          float* dst = part + ((static_cast<long long>(b) * Hq + g * G + hh) * nsplit + sp) * (dv + 2);
          dst[2 + e] = o0[hh];
          dst[3 + e] = o1[hh];
        }
    }
  }
  if (tid < G) {
    const int hh = tid;
    float* dst = part + ((static_cast<long long>(b) * Hq + g * G + hh) * nsplit + sp) * (dv + 2);
    dst[0] = nk > 0 ? mh[hh] : -INFINITY;
    dst[1] = red2[hh * 4] + red2[hh * 4 + 1] + red2[hh * 4 + 2] + red2[hh * 4 + 3];
  }
}

// Merges the splits of each (b, head): o = sum_s 2^(m_s - m) o_s / sum_s 2^(m_s - m) l_s.
__global__ void decode_attn_combine_kernel(int Hq, int dv, int nsplit, const float* __restrict__ part,
                                           __half* __restrict__ out, long long ldo) {
  pdl_wait();
  pdl_trigger();
  const int h = blockIdx.x, b = blockIdx.y;
  const float* pp = part + (static_cast<long long>(b) * Hq + h) * nsplit * (dv + 2);
  float m = -INFINITY;
  for (int s = 0; s < nsplit; ++s) m = fmaxf(m, pp[s * (dv + 2)]);
  float den = 0.f;
  for (int s = 0; s < nsplit; ++s) {
    const float ms = pp[s * (dv + 2)];
    if (ms != -INFINITY) den += ex2_approx(ms - m) * pp[s * (dv + 2) + 1];
  }
  const float inv = 1.0f / den;
  for (int e = threadIdx.x; e < dv; e += blockDim.x) {
    float num = 0.f;
    for (int s = 0; s < nsplit; ++s) {
      const float ms = pp[s * (dv + 2)];
      if (ms != -INFINITY) num += ex2_approx(ms - m) * pp[s * (dv + 2) + 2 + e];
    }
    out[b * ldo + h * dv + e] = __float2half_rn(num * inv);
  }
}

// One decode step of the SSM branch with the dt projection fused:
//   delta = softplus(dt[b] . W_dt[c] + bias[c]),  h = exp(delta A) h + delta u B[b],
//   y = C[b] . h + D u,  g = y silu(z);  the state is updated in place.
// A block owns DS_CH channels x DS_SEQ sequences:
//   0. every thread issues its loads of the state rows first, before waiting
//      for the preceding kernel (their HBM latency overlaps the rest and that
//      kernel's tail), then dt (fp16) and W_dt (bf16 -> fp16,
//      the same rounding as the prefill's weight conversion) are staged in
//      shared memory with 8-byte vector loads, zero-padded to 16 columns;
//   1. warps 0-3 compute delta for the block (16 sequences x 32 channels) on
//      the tensor cores, m16n8k16 (one 8-channel n-tile per warp), then leave
//      (delta, delta * u) in shared memory;
//   2. four threads per (sequence, channel), one float4 of the 16 states
//      each, so a warp reads and writes 8 consecutive channels' state rows
//      (512 contiguous bytes); the four partial C.h are summed with shuffles.
constexpr int DS_CH = 32;
constexpr int DS_SEQ = 16;         // = the m16 MMA tile
constexpr int DS_THREADS = 256;
constexpr int DS_RMAX = 128;
constexpr int DS_KSTR = DS_RMAX + 8;  // fp16 row stride of the staged tiles: conflict-free ldmatrix

HY_DEV void ldsm_x4_dec(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
HY_DEV void ldsm_x2_dec(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

// Four blocks per SM (64 registers, no spills): the 800 blocks of the
// batch-128 step run in 1.35 waves instead of 1.8 (graph step 109.9 ->
// 109.0 us; five or six blocks spill and were slower).
template <int N>
__global__ void __launch_bounds__(DS_THREADS, 4)
    decode_ssm_step_kernel(int B, int di, int R, const __half* __restrict__ u, long long ldu,
                           const __half* __restrict__ z, long long ldz, const float* __restrict__ xp,
                           long long ld_xp, const __nv_bfloat16* __restrict__ W_dt,
                           const float* __restrict__ dt_bias, const float* __restrict__ A_log,
                           const float* __restrict__ D, float* __restrict__ state, __half* __restrict__ g,
                           long long ldg, int32_t* __restrict__ pos) {
  static_assert(N == 16, "four threads x float4 per state row");
  __shared__ __align__(16) __half sW[DS_CH][DS_KSTR];     // W_dt rows of the block's channels (fp16)
  __shared__ __align__(16) __half sdt[DS_SEQ][DS_KSTR];   // dt rows of the block's sequences
  __shared__ __align__(16) float sbc[DS_SEQ][2 * N];      // [B | C] of each sequence
  __shared__ __align__(16) float sA2[DS_CH][N];
  __shared__ __align__(8) float2 sdu[DS_SEQ][DS_CH];      // (delta, delta * u)
  __shared__ float sbias[DS_CH], sD[DS_CH];                // dt_bias and D of the block's channels
  __shared__ __align__(16) __half su[DS_SEQ][DS_CH];      // u and z of the block's (sequence, channel) tile
  __shared__ __align__(16) __half sz[DS_SEQ][DS_CH];
  const int c0 = blockIdx.x * DS_CH, b0 = blockIdx.y * DS_SEQ;
  const int tid = threadIdx.x;
  const int KP = (R + 15) / 16 * 16;  // padded dt rank
  // ---- 0. state loads (phase-2 thread: quarter q of the rows j = tid/4 + 64 i)
  constexpr int NJ = DS_SEQ * DS_CH / (DS_THREADS / 4);
  const int q = tid & 3;
  float4 hv[NJ];
#pragma unroll
  for (int i = 0; i < NJ; ++i) {
    const int j = (tid >> 2) + i * (DS_THREADS / 4);
    const int b = b0 + j / DS_CH, c = c0 + j % DS_CH;
    hv[i] = (b < B && c < di)
                ? reinterpret_cast<const float4*>(state + (static_cast<long long>(b) * di + c) * N)[q]
                : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // W_dt rows: 8 threads per row, 4 values per 8-byte load; every load of a
  // thread is issued before the first is used (one round trip, not four)
  {
    constexpr int NK = DS_RMAX / 4 / 8;
    const int row = tid >> 3, l8 = tid & 7;  // 32 rows
    const int c = c0 + row;
    const bool vec = (reinterpret_cast<uintptr_t>(W_dt) & 7) == 0 && (R & 3) == 0;
    uint2 raw[NK];
#pragma unroll
    for (int i = 0; i < NK; ++i) {
      const int k = 4 * (l8 + 8 * i);
      raw[i] = make_uint2(0u, 0u);
      if (c < di && k < KP) {
        const __nv_bfloat16* src = W_dt + static_cast<long long>(c) * R + k;
        if (vec && k + 4 <= R) {
          raw[i] = *reinterpret_cast<const uint2*>(src);
        } else {
          __nv_bfloat16 e4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) e4[e] = k + e < R ? src[e] : __float2bfloat16_rn(0.f);
          raw[i] = make_uint2(*reinterpret_cast<const uint32_t*>(&e4[0]), *reinterpret_cast<const uint32_t*>(&e4[2]));
        }
      }
    }
#pragma unroll
    for (int i = 0; i < NK; ++i) {
      const int k = 4 * (l8 + 8 * i);
      if (k < KP) {
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw[i].x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw[i].y));
        *reinterpret_cast<uint2*>(&sW[row][k]) = make_uint2(pack_half2(a.x, a.y), pack_half2(b.x, b.y));
      }
    }
  }
  for (int idx = tid; idx < DS_CH * N; idx += DS_THREADS) {
    const int cc = idx / N;
    sA2[cc][idx % N] = (c0 + cc < di) ? -__expf(A_log[static_cast<long long>(c0) * N + idx]) * 1.4426950408889634f
                                      : 0.f;
  }
  if (tid < DS_CH) {
    sbias[tid] = c0 + tid < di ? dt_bias[c0 + tid] : 0.f;
    sD[tid] = c0 + tid < di ? D[c0 + tid] : 0.f;
  }
  // everything above reads weights and the state only (no kernel of the
  // step before this one writes the state, and all but the immediately
  // preceding kernel have completed); the rest reads what they wrote
  pdl_wait();
  pdl_trigger();
  // dt rows: 16 threads per row, all loads issued first (the padding columns
  // past R are zeroed, never read); dt rounds to fp16 as in prefill
  {
    constexpr int NK = DS_RMAX / 4 / 16;
    const int row = tid >> 4, l16 = tid & 15;
    const int b = b0 + row;
    const bool vec = ((reinterpret_cast<uintptr_t>(xp) | static_cast<uintptr_t>(ld_xp * 4)) & 15) == 0;
    float4 raw[NK];
#pragma unroll
    for (int i = 0; i < NK; ++i) {
      const int k = 4 * (l16 + 16 * i);
      raw[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (b < B && k < KP) {
        const float* src = xp + b * ld_xp + k;
        if (vec && k + 4 <= R) {
          raw[i] = *reinterpret_cast<const float4*>(src);
        } else {
          raw[i].x = k < R ? src[0] : 0.f;
          raw[i].y = k + 1 < R ? src[1] : 0.f;
          raw[i].z = k + 2 < R ? src[2] : 0.f;
          raw[i].w = k + 3 < R ? src[3] : 0.f;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < NK; ++i) {
      const int k = 4 * (l16 + 16 * i);
      if (k < KP)
        *reinterpret_cast<uint2*>(&sdt[row][k]) =
            make_uint2(pack_half2(raw[i].x, raw[i].y), pack_half2(raw[i].z, raw[i].w));
    }
  }
  for (int idx = tid; idx < DS_SEQ * 2 * N; idx += DS_THREADS) {
    const int s = idx / (2 * N);
    sbc[s][idx % (2 * N)] = (b0 + s < B) ? xp[(b0 + s) * ld_xp + R + idx % (2 * N)] : 0.f;
  }
  // u and z tiles: threads 0..63 load u, 64..127 z, 8 channels (16 bytes) each
  if (tid < 2 * DS_SEQ * (DS_CH / 8)) {
    const bool is_z = tid >= DS_SEQ * (DS_CH / 8);
    const int t = is_z ? tid - DS_SEQ * (DS_CH / 8) : tid;
    const int s = t / (DS_CH / 8), c8 = (t % (DS_CH / 8)) * 8;
    const int b = b0 + s, c = c0 + c8;
    const __half* src = is_z ? z + b * ldz + c : u + b * ldu + c;
    const long long ld = is_z ? ldz : ldu;
    __half* dst = is_z ? &sz[s][c8] : &su[s][c8];
    if (b < B && c + 8 <= di && ((reinterpret_cast<uintptr_t>(src) | static_cast<uintptr_t>(ld * 2)) & 15) == 0) {
      *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) dst[e] = (b < B && c + e < di) ? src[e] : __float2half_rn(0.f);
    }
  }
  __syncthreads();
  // every kernel of the step that reads pos ran before this one: advance it
  if (pos != nullptr && blockIdx.x == 0 && tid < DS_SEQ && b0 + tid < B) pos[b0 + tid] += 1;
  // ---- 1. delta = softplus(dt . W_dt^T + bias) on the tensor cores
  const int warp = tid >> 5, lane = tid & 31;
  if (warp < DS_CH / 8) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t a_base = smem_u32(&sdt[lane & 15][(lane >> 4) * 8]);
    const uint32_t b_base = smem_u32(&sW[warp * 8 + (lane & 7)][((lane >> 3) & 1) * 8]);
    for (int kk = 0; kk < KP / 16; ++kk) {
      uint32_t af[4], b0f, b1f;
      ldsm_x4_dec(a_base + kk * 32, af);
      ldsm_x2_dec(b_base + kk * 32, b0f, b1f);
      mma_16816_f16(acc, af, b0f, b1f);
    }
    // acc: rows (sequences) lane/4 and lane/4 + 8, columns (channels) 2(lane%4), +1
    const int grp = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int s = grp + (e >> 1) * 8, cl = warp * 8 + 2 * tig + (e & 1);
      const int b = b0 + s, c = c0 + cl;
      float dt = 0.f, uu = 0.f;
      if (b < B && c < di) {
        dt = softplus_fast(acc[e] + sbias[cl]);
        uu = __half2float(su[s][cl]);
      }
      sdu[s][cl] = make_float2(dt, dt * uu);
    }
  }
  __syncthreads();
  // ---- 2. state update, 4 threads per (sequence, channel): rows j = tid/4 + 64 i
  //      are channel cl = (tid/4) % 32 of sequences s = (tid/4)/32 + 2 i
  const int cl = (tid >> 2) % DS_CH, c = c0 + cl;
  const int s_first = (tid >> 2) / DS_CH;
  float4* hp = reinterpret_cast<float4*>(state + (static_cast<long long>(b0 + s_first) * di + c) * N) + q;
  const long long hstep = static_cast<long long>(DS_THREADS / 4 / DS_CH) * di * N / 4;  // float4 per step of i
  const float4 a = *reinterpret_cast<const float4*>(&sA2[cl][4 * q]);
  const float Dc = sD[cl];
#pragma unroll
  for (int i = 0; i < NJ; ++i, hp += hstep) {
    const int s = s_first + i * (DS_THREADS / 4 / DS_CH);
    const int b = b0 + s;
    const bool ok = b < B && c < di;
    float4 h = hv[i];
    const float2 du = sdu[s][cl];
    const float4 bb = *reinterpret_cast<const float4*>(&sbc[s][4 * q]);
    const float4 cc = *reinterpret_cast<const float4*>(&sbc[s][N + 4 * q]);
    h.x = fmaf(ex2_approx(du.x * a.x), h.x, du.y * bb.x);
    h.y = fmaf(ex2_approx(du.x * a.y), h.y, du.y * bb.y);
    h.z = fmaf(ex2_approx(du.x * a.z), h.z, du.y * bb.z);
    h.w = fmaf(ex2_approx(du.x * a.w), h.w, du.y * bb.w);
    float y = fmaf(cc.x, h.x, fmaf(cc.y, h.y, fmaf(cc.z, h.z, cc.w * h.w)));
    y += __shfl_xor_sync(0xffffffffu, y, 1);
    y += __shfl_xor_sync(0xffffffffu, y, 2);
    if (ok) {
      *hp = h;
      if (q == 0) {
        const float uu = __half2float(su[s][cl]);
        const float zz = __half2float(sz[s][cl]);
        y = fmaf(Dc, uu, y);
        // y * silu(z) = y * z / (1 + 2^(-z log2 e))
        g[b * ldg + c] = __float2half_rn(y * zz * rcp_approx(1.0f + ex2_approx(-1.4426950408889634f * zz)));
      }
    }
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

bool decode_attn_split_supported(int Hq, int Hkv, int dh, int dv) {
  return Hq / Hkv <= DA_MAXG && dh <= 128 && dh % 8 == 0 && dv % 2 == 0 && dv <= 512;
}

size_t decode_attn_split_scratch(int B, int Hq, int dv, int nsplit) {
  return static_cast<size_t>(B) * Hq * nsplit * (dv + 2) * sizeof(float);
}

hymba_status decode_attention_split(int B, int M, int Hq, int Hkv, int dh, int dv, int window, int cap, int nsplit,
                                    const __half* q, long long ldq, const __nv_bfloat16* k_meta,
                                    const __nv_bfloat16* v_meta, const __nv_bfloat16* k_ring,
                                    const __nv_bfloat16* v_ring, const int32_t* pos, float* part, __half* out,
                                    long long ldo, int max_keys, cudaStream_t st) {
  if (!decode_attn_split_supported(Hq, Hkv, dh, dv)) return HYMBA_ERR_UNSUPPORTED;
  const int G = Hq / Hkv;
  const int per = (max_keys + nsplit - 1) / nsplit;
  const int nkh = std::max(1, DA_THREADS / (dv / 2));
  const size_t smem =
      (DA_MAXG * 128 + static_cast<size_t>(G) * per + 2 * G * 4 + static_cast<size_t>(nkh) * G * dv) * sizeof(float);
  if (smem > 200 * 1024) return HYMBA_ERR_UNSUPPORTED;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(decode_attn_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return HYMBA_ERR_CUDA;
  decode_attn_split_kernel<<<dim3(nsplit, Hkv, B), DA_THREADS, smem, st>>>(
      M, Hq, Hkv, dh, dv, window, cap, nsplit, q, ldq, k_meta, v_meta, k_ring, v_ring, pos, part);
  decode_attn_combine_kernel<<<dim3(Hq, B), 128, 0, st>>>(Hq, dv, nsplit, part, out, ldo);
  return last_err();
}

hymba_status decode_attn_combine(int B, int Hq, int dv, int nsplit, const float* part, __half* out, long long ldo,
                                 cudaStream_t st) {
  if (launch_pdl(decode_attn_combine_kernel, dim3(Hq, B), dim3(128), 0, st, Hq, dv, nsplit, part, out, ldo) !=
      cudaSuccess)
    return HYMBA_ERR_CUDA;
  return last_err();
}

bool decode_ssm_step_supported(int N, int R) { return N == 16 && R >= 1 && R <= DS_RMAX; }

hymba_status decode_ssm_step(int B, int di, int N, int R, const __half* u, long long ldu, const __half* z,
                             long long ldz, const float* xp, long long ld_xp, const __nv_bfloat16* W_dt, const float* dt_bias, const float* A_log, const float* D,
                             float* state, __half* g, long long ldg, int32_t* pos, cudaStream_t st) {
  if (!decode_ssm_step_supported(N, R)) return HYMBA_ERR_UNSUPPORTED;
  if (B < 1 || di < 1) return HYMBA_OK;
  dim3 grid((di + DS_CH - 1) / DS_CH, (B + DS_SEQ - 1) / DS_SEQ);
  if (launch_pdl(decode_ssm_step_kernel<16>, grid, dim3(DS_THREADS), 0, st, B, di, R, u, ldu, z, ldz, xp, ld_xp, W_dt,
                 dt_bias, A_log, D, state, g, ldg, pos) != cudaSuccess)
    return HYMBA_ERR_CUDA;
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

namespace hy {
namespace {

// The decode step's K/V ring append and conv step in one launch (same
// arithmetic as kv_append_kernel and conv_step_kernel): elements
// [0, B*di) are conv channels, the rest ring entries of the new token.
// One decode step's conv step and ring append, one launch.  Conv: a thread
// per (sequence, 4 adjacent channels) -- the 4 x (k-1) carried rows of the
// group are contiguous in conv_state, so k = 4 moves them in three 16-byte
// loads and stores (`vec`: k = 4 and 16-byte aligned conv_state / conv_w);
// otherwise the scalar loop.  Append: a thread per
// 8 consecutive K or V values of one sequence (16-byte loads and stores).
__global__ void decode_prep_kernel(int B, int di, int k, const __half* __restrict__ proj, long long ldp, int x_col,
                                   int k_col, int v_col, int Hkv, int dh, int dv, int window, int cap,
                                   const int32_t* __restrict__ pos, __nv_bfloat16* __restrict__ k_ring,
                                   __nv_bfloat16* __restrict__ v_ring, const float* __restrict__ w,
                                   const float* __restrict__ bias, float* __restrict__ conv_state,
                                   __half* __restrict__ u, long long ldu, int append, int vec) {
  pdl_wait();
  pdl_trigger();
  const int g4 = di / 4;                       // channel groups per sequence
  const int n_conv = B * g4;
  const int wk = Hkv * dh, wv = Hkv * dv;
  const int kv8 = (wk + wv) / 8;               // 8-value groups per sequence
  const int n = n_conv + (append ? B * kv8 : 0);
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += gridDim.x * blockDim.x) {
    if (idx < n_conv) {
      const int b = idx / g4, c = (idx - b * g4) * 4;
      const long long bc = static_cast<long long>(b) * di + c;
      float* st = conv_state + bc * (k - 1);
      const uint2 xr = *reinterpret_cast<const uint2*>(proj + b * ldp + x_col + c);
      const float2 x01 = __half22float2(*reinterpret_cast<const __half2*>(&xr.x));
      const float2 x23 = __half22float2(*reinterpret_cast<const __half2*>(&xr.y));
      const float xv[4] = {x01.x, x01.y, x23.x, x23.y};
      float acc[4] = {bias[c], bias[c + 1], bias[c + 2], bias[c + 3]};
      if (vec) {
        float4 s4[3];
#pragma unroll
        for (int i = 0; i < 3; ++i) s4[i] = reinterpret_cast<const float4*>(st)[i];
        const float* sv = reinterpret_cast<const float*>(s4);  // channel e: sv[3e..3e+2], oldest first
        float nv[12];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float4 we = *reinterpret_cast<const float4*>(w + (c + e) * 4);
          acc[e] = fmaf(we.x, sv[3 * e], fmaf(we.y, sv[3 * e + 1], fmaf(we.z, sv[3 * e + 2], fmaf(we.w, xv[e], acc[e]))));
          nv[3 * e] = sv[3 * e + 1];
          nv[3 * e + 1] = sv[3 * e + 2];
          nv[3 * e + 2] = xv[e];
        }
#pragma unroll
        for (int i = 0; i < 3; ++i)
          reinterpret_cast<float4*>(st)[i] = make_float4(nv[4 * i], nv[4 * i + 1], nv[4 * i + 2], nv[4 * i + 3]);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float* se = st + e * (k - 1);
          for (int j = 0; j < k - 1; ++j) acc[e] = fmaf(w[(c + e) * k + j], se[j], acc[e]);
          acc[e] = fmaf(w[(c + e) * k + k - 1], xv[e], acc[e]);
          for (int j = 0; j + 1 < k - 1; ++j) se[j] = se[j + 1];
          if (k > 1) se[k - 2] = xv[e];
        }
      }
      // silu(a) = a / (1 + 2^(-a log2 e))
      uint2 o;
      o.x = pack_half2(acc[0] * rcp_approx(1.0f + ex2_approx(-1.4426950408889634f * acc[0])),
                       acc[1] * rcp_approx(1.0f + ex2_approx(-1.4426950408889634f * acc[1])));
      o.y = pack_half2(acc[2] * rcp_approx(1.0f + ex2_approx(-1.4426950408889634f * acc[2])),
                       acc[3] * rcp_approx(1.0f + ex2_approx(-1.4426950408889634f * acc[3])));
      *reinterpret_cast<uint2*>(u + b * ldu + c) = o;
    } else {
      const int r = idx - n_conv;
      const int b = r / kv8, c = (r - b * kv8) * 8;
      const int p = pos[b];
      const int slot = window > 0 ? p % cap : p;
      if (slot < 0 || slot >= cap) continue;  // a full global cache: the token is not stored
      const bool is_k = c < wk;
      const uint4 src = *reinterpret_cast<const uint4*>(proj + b * ldp + (is_k ? k_col + c : v_col + c - wk));
      const __half2* sh = reinterpret_cast<const __half2*>(&src);
      uint4 dst;
      uint32_t* d32 = reinterpret_cast<uint32_t*>(&dst);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(sh[e]);
        __nv_bfloat162 h = __floats2bfloat162_rn(f.x, f.y);
        d32[e] = *reinterpret_cast<uint32_t*>(&h);
      }
      __nv_bfloat16* drow = is_k ? k_ring + (static_cast<long long>(b) * cap + slot) * wk + c
                                 : v_ring + (static_cast<long long>(b) * cap + slot) * wv + (c - wk);
      *reinterpret_cast<uint4*>(drow) = dst;
    }
  }
}

}  // namespace

hymba_status decode_prep(int B, int di, int k, const __half* proj, long long ldp, int x_col, int k_col, int v_col,
                         int Hkv, int dh, int dv, int window, int cap, const int32_t* pos, __nv_bfloat16* k_ring,
                         __nv_bfloat16* v_ring, const float* conv_w, const float* conv_b, float* conv_state,
                         __half* u, long long ldu, bool append, cudaStream_t st) {
  // whole 4-channel / 8-value groups on 16-byte boundaries (the bf16 path's
  // shape rules give them; the ring rows must be 16-byte aligned, as the
  // decode attention's TMA maps need anyway)
  if (di % 4 || (Hkv * dh) % 8 || (Hkv * dv) % 8 || ldp % 8 || ldu % 4 || x_col % 4 || k_col % 8 || v_col % 8)
    return HYMBA_ERR_UNSUPPORTED;
  if (append && ((reinterpret_cast<uintptr_t>(k_ring) & 15) || (reinterpret_cast<uintptr_t>(v_ring) & 15)))
    return HYMBA_ERR_INVALID;
  const int vec = k == 4 && !(reinterpret_cast<uintptr_t>(conv_state) & 15) && !(reinterpret_cast<uintptr_t>(conv_w) & 15);
  const long long n = static_cast<long long>(B) * (di / 4) + (append ? static_cast<long long>(B) * Hkv * (dh + dv) / 8 : 0);
  if (n <= 0) return HYMBA_OK;
  if (n > (1LL << 30)) return HYMBA_ERR_INVALID;
  if (launch_pdl(decode_prep_kernel, dim3(static_cast<unsigned>(std::min<long long>((n + 255) / 256, 148 * 8))),
                 dim3(256), 0, st, B, di, k, proj, ldp, x_col, k_col, v_col, Hkv, dh, dv, window, cap, pos, k_ring,
                 v_ring, conv_w, conv_b, conv_state, u, ldu, append ? 1 : 0, vec) != cudaSuccess)
    return HYMBA_ERR_CUDA;
  return last_err();
}

}  // namespace hy
