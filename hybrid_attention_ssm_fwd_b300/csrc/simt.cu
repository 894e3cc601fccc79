// SIMT kernels of the hybrid-head layer (fp32 path and generic pieces): every
// stage of eq. 3 ("Hymba: A Hybrid-head Architecture for Small Language Models",
// section 2.1) in fp32, and on the bf16 path the fused norm / beta / sum
// that feeds W_out, the cache emission and the block's RMSNorm.
#include <algorithm>
#include <type_traits>

#include "simt.cuh"

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

inline unsigned grid1d(long long n, int block) {
  return static_cast<unsigned>((n + block - 1) / block);
}

// ---------------------------------------------------------------------------
// fp32 GEMM (64x64 tile, 16-deep K slices, 4x4 outputs per thread)
// ---------------------------------------------------------------------------
template <typename TA>
__global__ void __launch_bounds__(256) gemm_simt_kernel(int M, int N, int K, const TA* __restrict__ A,
                                                        long long lda, const TA* __restrict__ B,
                                                        long long ldb, int epi, float* C, long long ldc,
                                                        float* C2, long long ldc2, int R,
                                                        const float* bias, const TA* resid,
                                                        long long ld_resid) {
  __shared__ float As[16][68];
  __shared__ float Bs[16][68];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += 16) {
    for (int i = threadIdx.x; i < 1024; i += 256) {
      const int r = i >> 4, kk = i & 15;
      const int gk = k0 + kk;
      const int gm = m0 + r, gn = n0 + r;
      As[kk][r] = (gm < M && gk < K) ? to_f(A[static_cast<long long>(gm) * lda + gk]) : 0.f;
      Bs[kk][r] = (gn < N && gk < K) ? to_f(B[static_cast<long long>(gn) * ldb + gk]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[kk][ty * 4 + i];
        b[i] = Bs[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = m0 + ty * 4 + i;
    if (row >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = n0 + tx * 4 + j;
      if (col >= N) continue;
      float v = acc[i][j];
      if (epi == SE_XPROJ) {
        if (col < R)
          C2[static_cast<long long>(row) * ldc2 + col] = v;
        else
          C[static_cast<long long>(row) * ldc + col - R] = v;
        continue;
      }
      if (epi == SE_SOFTPLUS) {
        const float x = v + bias[col];
        v = x > 20.f ? x : log1pf(expf(x));
      } else if (epi == SE_RESID && resid) {
        v += to_f(resid[static_cast<long long>(row) * ld_resid + col]);
      }
      C[static_cast<long long>(row) * ldc + col] = v;
    }
  }
}

// ---------------------------------------------------------------------------
// RoPE (rotate-half), generic head dim
// ---------------------------------------------------------------------------
template <typename T>
__global__ void rope_kernel(T* X, long long ld, int rows, int col0, int n_heads, int dh, float theta,
                            int rows_per_seq, const int32_t* pos, int pos_base) {
  const int half = dh / 2;
  const long long n = static_cast<long long>(rows) * n_heads * half;
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < n;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int i = static_cast<int>(idx % half);
    const int h = static_cast<int>((idx / half) % n_heads);
    const int row = static_cast<int>(idx / (static_cast<long long>(half) * n_heads));
    const int p = pos ? pos_base + pos[row] : row % rows_per_seq;
    T* base = X + static_cast<long long>(row) * ld + col0 + h * dh;
    const float x1 = to_f(base[i]), x2 = to_f(base[i + half]);
    float c, s;
    if (std::is_same<T, float>::value) {
      const double ang = static_cast<double>(p) * pow(static_cast<double>(theta), -2.0 * i / dh);
      double sd, cd;
      sincos(ang, &sd, &cd);
      c = static_cast<float>(cd);
      s = static_cast<float>(sd);
    } else {
      const float ang = static_cast<float>(p) * exp2f(-2.0f * i / dh * log2f(theta));
      sincosf(ang, &s, &c);
    }
    base[i] = from_f<T>(x1 * c - x2 * s);
    base[i + half] = from_f<T>(x2 * c + x1 * s);
  }
}

// ---------------------------------------------------------------------------
// causal depthwise conv + SiLU
// ---------------------------------------------------------------------------
template <typename TI, typename TO>
__global__ void conv_silu_kernel(const TI* __restrict__ x, long long ld_x, TO* __restrict__ u,
                                 long long ld_u, int B, int L, int di, int k, const float* __restrict__ w,
                                 const float* __restrict__ bias) {
  const long long n = static_cast<long long>(B) * L * di;
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < n;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(idx % di);
    const long long row = idx / di;
    const int t = static_cast<int>(row % L);
    float acc = bias[c];
    for (int j = 0; j < k; ++j) {
      const int src = t - (k - 1) + j;
      if (src >= 0) acc = fmaf(w[c * k + j], to_f(x[(row - (t - src)) * ld_x + c]), acc);
    }
    const float sv = acc / (1.0f + expf(-acc));
    u[row * ld_u + c] = from_f<TO>(sv);
  }
}

// fp16 conv: one thread owns 8 consecutive channels (one 16-byte vector) for
// a tile of CONV_TT consecutive rows and keeps the last K-1 inputs in
// registers, so x is read once and u written once, both fully coalesced.
constexpr int CONV_TT = 64;

template <int K>
__global__ void __launch_bounds__(128) conv_silu_vec_kernel(const __half* __restrict__ x, long long ld_x,
                                                            __half* __restrict__ u, long long ld_u, int L, int di,
                                                            const float* __restrict__ w,
                                                            const float* __restrict__ bias) {
  const int cg = blockIdx.x * blockDim.x + threadIdx.x;  // channel group of 8
  if (cg * 8 >= di) return;
  const int t0 = blockIdx.y * CONV_TT;
  const int b = blockIdx.z;
  const int c0 = cg * 8;
  float wt[8][K], bs[8], win[K][8];  // win[j] = row t - (K-1) + j for the next row t (j < K-1)
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    bs[e] = bias[c0 + e];
#pragma unroll
    for (int j = 0; j < K; ++j) wt[e][j] = w[(c0 + e) * K + j];
  }
  const long long rb = static_cast<long long>(b) * L;
#pragma unroll
  for (int j = 0; j < K - 1; ++j) {
    const int src = t0 - (K - 1) + j;
    if (src >= 0) {
      const uint4 q = *reinterpret_cast<const uint4*>(x + (rb + src) * ld_x + c0);
      const __half* hq = reinterpret_cast<const __half*>(&q);
#pragma unroll
      for (int e = 0; e < 8; ++e) win[j][e] = __half2float(hq[e]);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) win[j][e] = 0.f;
    }
  }
  const int t1 = min(t0 + CONV_TT, L);
  constexpr int RB = 8;  // rows loaded per batch: 8 independent 16-byte loads in flight
  for (int tb = t0; tb < t1; tb += RB) {
    uint4 qv[RB];
#pragma unroll
    for (int r = 0; r < RB; ++r)
      if (tb + r < t1) qv[r] = *reinterpret_cast<const uint4*>(x + (rb + tb + r) * ld_x + c0);
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      if (tb + r >= t1) break;
      const __half* hq = reinterpret_cast<const __half*>(&qv[r]);
#pragma unroll
      for (int e = 0; e < 8; ++e) win[K - 1][e] = __half2float(hq[e]);
      float out[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float acc = bs[e];
#pragma unroll
        for (int j = 0; j < K; ++j) acc = fmaf(wt[e][j], win[j][e], acc);
        out[e] = acc / (1.0f + __expf(-acc));
      }
#pragma unroll
      for (int j = 0; j + 1 < K; ++j)
#pragma unroll
        for (int e = 0; e < 8; ++e) win[j][e] = win[j + 1][e];
      uint4 o;
      o.x = pack_half2(out[0], out[1]);
      o.y = pack_half2(out[2], out[3]);
      o.z = pack_half2(out[4], out[5]);
      o.w = pack_half2(out[6], out[7]);
      *reinterpret_cast<uint4*>(u + (rb + tb + r) * ld_u + c0) = o;
    }
  }
}

// ---------------------------------------------------------------------------
// generic selective scan + gate (one thread per (b, channel))
// ---------------------------------------------------------------------------
template <typename T>
__global__ void scan_simt_kernel(int B, int L, int di, int N, const T* __restrict__ u, long long ld_u,
                                 const T* __restrict__ z, long long ld_z, const float* __restrict__ delta,
                                 long long ld_delta, const float* __restrict__ Bm,
                                 const float* __restrict__ Cm, long long ld_bc,
                                 const float* __restrict__ A_log, const float* __restrict__ D, T* g,
                                 long long ld_g, const float* h0, float* h_out) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= B * di) return;
  const int b = idx / di, c = idx % di;
  float h[64], A[64];
  for (int n = 0; n < N; ++n) {
    A[n] = -expf(A_log[c * N + n]);
    h[n] = h0 ? h0[(static_cast<long long>(b) * di + c) * N + n] : 0.f;
  }
  const float Dc = D[c];
  for (int t = 0; t < L; ++t) {
    const long long row = static_cast<long long>(b) * L + t;
    const float dt = delta[row * ld_delta + c];
    const float uu = to_f(u[row * ld_u + c]);
    const float du = dt * uu;
    float y = 0.f;
    for (int n = 0; n < N; ++n) {
      h[n] = expf(dt * A[n]) * h[n] + du * Bm[row * ld_bc + n];
      y = fmaf(Cm[row * ld_bc + n], h[n], y);
    }
    y = fmaf(Dc, uu, y);
    const float zz = to_f(z[row * ld_z + c]);
    g[row * ld_g + c] = from_f<T>(y * (zz / (1.0f + expf(-zz))));
  }
  if (h_out)
    for (int n = 0; n < N; ++n) h_out[(static_cast<long long>(b) * di + c) * N + n] = h[n];
}

// ---------------------------------------------------------------------------
// fused RMSNorm x2, beta scaling and sum (one block per row)
// ---------------------------------------------------------------------------
// concatenation fusion: 8 channels of beta1 * att * ra to `da` and of
// beta2 * g * rg to `dg` (the two halves of a 2 di wide row)
__device__ __forceinline__ void fuse_norm_concat8(const uint4& av, const uint4& gv, const float* b1, const float* b2,
                                                  float ra, float rg, uint4* da, uint4* dg) {
  const __half2* ah = reinterpret_cast<const __half2*>(&av);
  const __half2* gh = reinterpret_cast<const __half2*>(&gv);
  uint32_t oa[4], og[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 fa = __half22float2(ah[e]), fg = __half22float2(gh[e]);
    oa[e] = pack_half2(__ldg(b1 + 2 * e) * fa.x * ra, __ldg(b1 + 2 * e + 1) * fa.y * ra);
    og[e] = pack_half2(__ldg(b2 + 2 * e) * fg.x * rg, __ldg(b2 + 2 * e + 1) * fg.y * rg);
  }
  *da = make_uint4(oa[0], oa[1], oa[2], oa[3]);
  *dg = make_uint4(og[0], og[1], og[2], og[3]);
}

template <typename T>
__global__ void __launch_bounds__(256) fuse_norm_kernel(int di, const T* __restrict__ att,
                                                        const T* __restrict__ g,
                                                        const float* __restrict__ beta1,
                                                        const float* __restrict__ beta2, float eps,
                                                        T* __restrict__ s, int concat) {
  pdl_wait();
  pdl_trigger();
  const long long row = blockIdx.x;
  const T* a = att + row * di;
  const T* gg = g + row * di;
  float sa = 0.f, sg = 0.f;
  for (int c = threadIdx.x; c < di; c += blockDim.x) {
    const float va = to_f(a[c]), vg = to_f(gg[c]);
    sa = fmaf(va, va, sa);
    sg = fmaf(vg, vg, sg);
  }
  __shared__ float red[2][32];
  for (int o = 16; o > 0; o >>= 1) {
    sa += __shfl_xor_sync(0xffffffffu, sa, o);
    sg += __shfl_xor_sync(0xffffffffu, sg, o);
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) {
    red[0][w] = sa;
    red[1][w] = sg;
  }
  __syncthreads();
  if (w == 0) {
    const int nw = blockDim.x >> 5;
    sa = l < nw ? red[0][l] : 0.f;
    sg = l < nw ? red[1][l] : 0.f;
    for (int o = 16; o > 0; o >>= 1) {
      sa += __shfl_xor_sync(0xffffffffu, sa, o);
      sg += __shfl_xor_sync(0xffffffffu, sg, o);
    }
    if (l == 0) {
      red[0][0] = rsqrtf(sa / di + eps);
      red[1][0] = rsqrtf(sg / di + eps);
    }
  }
  __syncthreads();
  const float ra = red[0][0], rg = red[1][0];
  if (concat) {
    for (int c = threadIdx.x; c < di; c += blockDim.x) {
      s[row * 2 * di + c] = from_f<T>(beta1[c] * to_f(a[c]) * ra);
      s[row * 2 * di + di + c] = from_f<T>(beta2[c] * to_f(gg[c]) * rg);
    }
  } else {
    for (int c = threadIdx.x; c < di; c += blockDim.x)
      s[row * di + c] = from_f<T>(beta1[c] * to_f(a[c]) * ra + beta2[c] * to_f(gg[c]) * rg);
  }
}

// fp16 fused norm: 16-byte vectors kept in registers (one HBM read of att
// and g), up to FN_MAXC vectors of each per thread.
constexpr int FN_MAXC = 4;

template <bool CONCAT>
__global__ void __launch_bounds__(256) fuse_norm_vec_kernel(int di, const __half* __restrict__ att,
                                                            const __half* __restrict__ g,
                                                            const float* __restrict__ beta1,
                                                            const float* __restrict__ beta2, float eps,
                                                            __half* __restrict__ s) {
  const long long row = blockIdx.x;
  const int nch = di / 8;
  // the weights do not depend on the preceding kernel: load them before
  // waiting for it
  float4 b1v[FN_MAXC][2], b2v[FN_MAXC][2];
  if (!CONCAT) {
#pragma unroll
    for (int q = 0; q < FN_MAXC; ++q) {
      const int ch = threadIdx.x + q * 256;
      if (ch < nch) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          b1v[q][h] = *reinterpret_cast<const float4*>(beta1 + ch * 8 + 4 * h);
          b2v[q][h] = *reinterpret_cast<const float4*>(beta2 + ch * 8 + 4 * h);
        }
      }
    }
  }
  pdl_wait();
  pdl_trigger();
  const uint4* a4 = reinterpret_cast<const uint4*>(att + row * di);
  const uint4* g4 = reinterpret_cast<const uint4*>(g + row * di);
  uint4 av[FN_MAXC], gv[FN_MAXC];
  float sa = 0.f, sg = 0.f;
#pragma unroll
  for (int q = 0; q < FN_MAXC; ++q) {
    const int ch = threadIdx.x + q * 256;
    if (ch < nch) {
      av[q] = a4[ch];
      gv[q] = g4[ch];
      const __half2* ah = reinterpret_cast<const __half2*>(&av[q]);
      const __half2* gh = reinterpret_cast<const __half2*>(&gv[q]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fa = __half22float2(ah[e]), fg = __half22float2(gh[e]);
        sa = fmaf(fa.x, fa.x, fmaf(fa.y, fa.y, sa));
        sg = fmaf(fg.x, fg.x, fmaf(fg.y, fg.y, sg));
      }
    }
  }
  __shared__ float red[2][8];
  for (int o = 16; o > 0; o >>= 1) {
    sa += __shfl_xor_sync(0xffffffffu, sa, o);
    sg += __shfl_xor_sync(0xffffffffu, sg, o);
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) {
    red[0][w] = sa;
    red[1][w] = sg;
  }
  __syncthreads();
  float ta = 0.f, tg = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    ta += red[0][i];
    tg += red[1][i];
  }
  const float ra = rsqrtf(ta / di + eps), rg = rsqrtf(tg / di + eps);
  uint4* s4 = reinterpret_cast<uint4*>(s + row * di * (CONCAT ? 2 : 1));
#pragma unroll
  for (int q = 0; q < FN_MAXC; ++q) {
    const int ch = threadIdx.x + q * 256;
    if (CONCAT && ch < nch) {
      fuse_norm_concat8(av[q], gv[q], beta1 + ch * 8, beta2 + ch * 8, ra, rg, s4 + ch, s4 + nch + ch);
    } else if (!CONCAT && ch < nch) {
      const __half2* ah = reinterpret_cast<const __half2*>(&av[q]);
      const __half2* gh = reinterpret_cast<const __half2*>(&gv[q]);
      const float4 b1a = b1v[q][0], b1b = b1v[q][1], b2a = b2v[q][0], b2b = b2v[q][1];
      const float bb1[8] = {b1a.x, b1a.y, b1a.z, b1a.w, b1b.x, b1b.y, b1b.z, b1b.w};
      const float bb2[8] = {b2a.x, b2a.y, b2a.z, b2a.w, b2b.x, b2b.y, b2b.z, b2b.w};
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fa = __half22float2(ah[e]), fg = __half22float2(gh[e]);
        o[e] = pack_half2(bb1[2 * e] * fa.x * ra + bb2[2 * e] * fg.x * rg,
                          bb1[2 * e + 1] * fa.y * ra + bb2[2 * e + 1] * fg.y * rg);
      }
      s4[ch] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// fp16 fused norm, one warp per row: a lane holds up to FW_V 16-byte vectors
// of att and of g, all loaded before the first use (one HBM read, many loads
// in flight), and the two sums of squares are reduced with shuffles only.
constexpr int FW_V = 16;  // di <= 32 * 8 * FW_V = 4096

template <bool CONCAT>
__global__ void __launch_bounds__(128) fuse_norm_warp_kernel(int rows, int di, const __half* __restrict__ att,
                                                             const __half* __restrict__ g,
                                                             const float* __restrict__ beta1,
                                                             const float* __restrict__ beta2, float eps,
                                                             __half* __restrict__ s) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int nch = di / 8;
  const uint4* a4 = reinterpret_cast<const uint4*>(att + row * di);
  const uint4* g4 = reinterpret_cast<const uint4*>(g + row * di);
  uint4 av[FW_V], gv[FW_V];
#pragma unroll
  for (int q = 0; q < FW_V; ++q) {
    const int ch = lane + q * 32;
    if (ch < nch) {
      av[q] = __ldcs(a4 + ch);  // read once: do not keep in L2
      gv[q] = __ldcs(g4 + ch);
    }
  }
  float sa = 0.f, sg = 0.f;
#pragma unroll
  for (int q = 0; q < FW_V; ++q) {
    if (lane + q * 32 < nch) {
      const __half2* ah = reinterpret_cast<const __half2*>(&av[q]);
      const __half2* gh = reinterpret_cast<const __half2*>(&gv[q]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fa = __half22float2(ah[e]), fg = __half22float2(gh[e]);
        sa = fmaf(fa.x, fa.x, fmaf(fa.y, fa.y, sa));
        sg = fmaf(fg.x, fg.x, fmaf(fg.y, fg.y, sg));
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    sa += __shfl_xor_sync(0xffffffffu, sa, o);
    sg += __shfl_xor_sync(0xffffffffu, sg, o);
  }
  const float ra = rsqrtf(sa / di + eps), rg = rsqrtf(sg / di + eps);
  uint4* s4 = reinterpret_cast<uint4*>(s + row * di * (CONCAT ? 2 : 1));
#pragma unroll
  for (int q = 0; q < FW_V; ++q) {
    const int ch = lane + q * 32;
    if (CONCAT && ch < nch) {
      fuse_norm_concat8(av[q], gv[q], beta1 + ch * 8, beta2 + ch * 8, ra, rg, s4 + ch, s4 + nch + ch);
    } else if (!CONCAT && ch < nch) {
      const __half2* ah = reinterpret_cast<const __half2*>(&av[q]);
      const __half2* gh = reinterpret_cast<const __half2*>(&gv[q]);
      const float4 b1a = __ldg(reinterpret_cast<const float4*>(beta1 + ch * 8));
      const float4 b1b = __ldg(reinterpret_cast<const float4*>(beta1 + ch * 8 + 4));
      const float4 b2a = __ldg(reinterpret_cast<const float4*>(beta2 + ch * 8));
      const float4 b2b = __ldg(reinterpret_cast<const float4*>(beta2 + ch * 8 + 4));
      const float bb1[8] = {b1a.x * ra, b1a.y * ra, b1a.z * ra, b1a.w * ra, b1b.x * ra, b1b.y * ra, b1b.z * ra,
                            b1b.w * ra};
      const float bb2[8] = {b2a.x * rg, b2a.y * rg, b2a.z * rg, b2a.w * rg, b2b.x * rg, b2b.y * rg, b2b.z * rg,
                            b2b.w * rg};
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fa = __half22float2(ah[e]), fg = __half22float2(gh[e]);
        o[e] = pack_half2(fmaf(bb1[2 * e], fa.x, bb2[2 * e] * fg.x), fmaf(bb1[2 * e + 1], fa.y, bb2[2 * e + 1] * fg.y));
      }
      s4[ch] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// ---------------------------------------------------------------------------
// SIMT attention: one warp per (b, row i, query head)
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(128) attention_simt_kernel(int B, int L, int M, int Hq, int Hkv, int dh,
                                                             int dv, int window, const T* __restrict__ Q,
                                                             long long ldq, const T* __restrict__ K,
                                                             long long ldk, const T* __restrict__ V,
                                                             long long ldv, T* __restrict__ O,
                                                             long long ldo) {
  extern __shared__ float qs[];  // [4][dh]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long wid = static_cast<long long>(blockIdx.x) * 4 + warp;
  const bool active = wid < static_cast<long long>(B) * L * Hq;
  const int h = active ? static_cast<int>(wid % Hq) : 0;
  const long long rowg = active ? wid / Hq : 0;  // b*L + i
  const int i = static_cast<int>(rowg % L);
  const long long brow0 = rowg - i;                // b*L
  const int gidx = (h * Hkv) / Hq;
  float* q = qs + warp * dh;
  const float scale = rsqrtf(static_cast<float>(dh));
  for (int e = lane; e < dh; e += 32) q[e] = active ? to_f(Q[rowg * ldq + h * dh + e]) * scale : 0.f;
  __syncwarp();
  if (!active) return;
  constexpr int MAXR = 8;  // dv <= 256
  float o[MAXR];
#pragma unroll
  for (int r = 0; r < MAXR; ++r) o[r] = 0.f;
  float m = -INFINITY, lsum = 0.f;
  // visible keys: one range [0, i] or the two ranges [0, M) and [i-W+1, i]
  int r0a = 0, r0b = i, r1a = 1, r1b = 0;
  if (window > 0 && i - window + 1 > M) {
    r0b = M - 1;
    r1a = i - window + 1;
    r1b = i;
  }
  for (int part = 0; part < 2; ++part) {
    const int ja = part == 0 ? r0a : r1a;
    const int jb = part == 0 ? r0b : r1b;
    for (int j0 = ja; j0 <= jb; j0 += 32) {
      const int j = j0 + lane;
      float sc = -INFINITY;
      if (j <= jb) {
        const T* kr = K + (brow0 + j) * ldk + gidx * dh;
        float acc = 0.f;
        for (int e = 0; e < dh; ++e) acc = fmaf(q[e], to_f(kr[e]), acc);
        sc = acc;
      }
      float mx = sc;
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_new = fmaxf(m, mx);
      const float alpha = (m == -INFINITY) ? 0.f : expf(m - m_new);
      const float p = (sc == -INFINITY) ? 0.f : expf(sc - m_new);
      float ps = p;
      for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
      lsum = lsum * alpha + ps;
#pragma unroll
      for (int r = 0; r < MAXR; ++r) o[r] *= alpha;
      const int nk = min(32, jb - j0 + 1);
      for (int jj = 0; jj < nk; ++jj) {
        const float pj = __shfl_sync(0xffffffffu, p, jj);
        const T* vr = V + (brow0 + j0 + jj) * ldv + gidx * dv;
#pragma unroll
        for (int r = 0; r < MAXR; ++r) {
          const int e = lane + 32 * r;
          if (e < dv) o[r] = fmaf(pj, to_f(vr[e]), o[r]);
        }
      }
      m = m_new;
    }
  }
  const float inv = 1.0f / lsum;
#pragma unroll
  for (int r = 0; r < MAXR; ++r) {
    const int e = lane + 32 * r;
    if (e < dv) O[rowg * ldo + h * dv + e] = from_f<T>(o[r] * inv);
  }
}

template <typename TS, typename TD>
__global__ void copy2d_kernel(const TS* __restrict__ src, long long lds, TD* __restrict__ dst, long long ldd,
                              long long rows, int cols) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= cols) return;
  for (long long r = blockIdx.y; r < rows; r += gridDim.y) dst[r * ldd + c] = from_f<TD>(to_f(src[r * lds + c]));
}

// RMSNorm of fp32 rows with a learned weight, stored as bf16: one warp per
// row, two passes over the row (the second hits L1/L2).
__global__ void __launch_bounds__(256) rmsnorm_bf16_kernel(int rows, int d, const float* __restrict__ x,
                                                           long long ldx, const float* __restrict__ w, float eps,
                                                           __nv_bfloat16* __restrict__ y, long long ldy) {
  const int lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const float4* xr = reinterpret_cast<const float4*>(x + row * ldx);
  const float4* w4 = reinterpret_cast<const float4*>(w);
  const int n4 = d / 4;
  float ss = 0.f;
  for (int i = lane; i < n4; i += 32) {
    const float4 v = xr[i];
    ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float r = rsqrtf(ss / d + eps);
  uint2* yr = reinterpret_cast<uint2*>(y + row * ldy);
  for (int i = lane; i < n4; i += 32) {
    const float4 v = xr[i], g = __ldg(w4 + i);
    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x * r * g.x, v.y * r * g.y);
    const __nv_bfloat162 b = __floats2bfloat162_rn(v.z * r * g.z, v.w * r * g.w);
    yr[i] = make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
  }
}

__global__ void bf16_to_f16_vec_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, long long n8) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const uint4 v = src[i];
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&v);
    uint4 o;
    uint32_t* o32 = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(b2[e]);
      o32[e] = pack_half2(f.x, f.y);
    }
    dst[i] = o;
  }
}

template <typename TS, typename TC>
__global__ void emit_ring_kernel(int B, int L, int M, int T, int cap, int n_keep, int width,
                                 const TS* __restrict__ src, long long lds, TC* __restrict__ ring) {
  const long long n = static_cast<long long>(B) * n_keep * width;
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < n;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(idx % width);
    const int tr = static_cast<int>((idx / width) % n_keep);
    const int b = static_cast<int>(idx / (static_cast<long long>(width) * n_keep));
    const int t = T - n_keep + tr;
    const int slot = t % cap;
    ring[(static_cast<long long>(b) * cap + slot) * width + c] =
        from_f<TC>(to_f(src[(static_cast<long long>(b) * L + M + t) * lds + c]));
  }
}

template <typename TS>
__global__ void emit_conv_tail_kernel(int B, int L, int di, int k, const TS* __restrict__ x, long long ldx,
                                      float* __restrict__ conv_state, const float* __restrict__ prev) {
  const long long n = static_cast<long long>(B) * di * (k - 1);
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < n;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int j = static_cast<int>(idx % (k - 1));
    const int c = static_cast<int>((idx / (k - 1)) % di);
    const int b = static_cast<int>(idx / (static_cast<long long>(k - 1) * di));
    const int row = L - (k - 1) + j;
    // rows before the first come from `prev` ([di, k-1], oldest first), else zero
    conv_state[idx] = row >= 0 ? to_f(x[(static_cast<long long>(b) * L + row) * ldx + c])
                               : (prev ? prev[static_cast<long long>(c) * (k - 1) + (k - 1) + row] : 0.f);
  }
}

__global__ void fill_i32_kernel(int n, int32_t* dst, int32_t v) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) dst[i] = v;
}

inline hymba_status last_err() {
  return cudaGetLastError() == cudaSuccess ? HYMBA_OK : HYMBA_ERR_CUDA;
}

}  // namespace

template <typename TA>
hymba_status gemm_simt(int M, int N, int K, const TA* A, long long lda, const TA* B, long long ldb, int epi,
                       float* C, long long ldc, float* C2, long long ldc2, int R, const float* bias,
                       const TA* resid, long long ld_resid, cudaStream_t st) {
  if (M <= 0 || N <= 0) return HYMBA_OK;
  dim3 grid((N + 63) / 64, (M + 63) / 64);
  gemm_simt_kernel<TA><<<grid, 256, 0, st>>>(M, N, K, A, lda, B, ldb, epi, C, ldc, C2, ldc2, R, bias, resid,
                                            ld_resid);
  return last_err();
}

template <typename T>
hymba_status rope_simt(T* X, long long ld, int rows, int col0, int n_heads, int dh, float theta,
                       int rows_per_seq, const int32_t* pos, int pos_base, cudaStream_t st) {
  const long long n = static_cast<long long>(rows) * n_heads * (dh / 2);
  if (n <= 0) return HYMBA_OK;
  rope_kernel<T><<<std::min<long long>(grid1d(n, 256), 148 * 16), 256, 0, st>>>(
      X, ld, rows, col0, n_heads, dh, theta, rows_per_seq, pos, pos_base);
  return last_err();
}

template <typename TI, typename TO>
hymba_status conv_silu(const TI* x, long long ld_x, TO* u, long long ld_u, int B, int L, int di, int k,
                       const float* w, const float* bias, cudaStream_t st) {
  if (std::is_same<TI, __half>::value && std::is_same<TO, __half>::value && di % 8 == 0 && ld_x % 8 == 0 &&
      ld_u % 8 == 0 && (k == 2 || k == 3 || k == 4) && (reinterpret_cast<uintptr_t>(x) & 15) == 0 &&
      (reinterpret_cast<uintptr_t>(u) & 15) == 0) {
    const int groups = di / 8;
    dim3 grid((groups + 127) / 128, (L + CONV_TT - 1) / CONV_TT, B);
    const __half* xh = reinterpret_cast<const __half*>(x);
    __half* uh = reinterpret_cast<__half*>(u);
    if (k == 4) conv_silu_vec_kernel<4><<<grid, 128, 0, st>>>(xh, ld_x, uh, ld_u, L, di, w, bias);
    else if (k == 3) conv_silu_vec_kernel<3><<<grid, 128, 0, st>>>(xh, ld_x, uh, ld_u, L, di, w, bias);
    else conv_silu_vec_kernel<2><<<grid, 128, 0, st>>>(xh, ld_x, uh, ld_u, L, di, w, bias);
    return last_err();
  }
  const long long n = static_cast<long long>(B) * L * di;
  conv_silu_kernel<TI, TO><<<std::min<long long>(grid1d(n, 256), 148 * 32), 256, 0, st>>>(
      x, ld_x, u, ld_u, B, L, di, k, w, bias);
  return last_err();
}

template <typename T>
hymba_status scan_simt(int B, int L, int di, int N, const T* u, long long ld_u, const T* z, long long ld_z,
                       const float* delta, long long ld_delta, const float* Bm, const float* Cm,
                       long long ld_bc, const float* A_log, const float* D, T* g, long long ld_g,
                       const float* h0, float* h_out, cudaStream_t st) {
  if (N > 64) return HYMBA_ERR_UNSUPPORTED;
  const int n = B * di;
  scan_simt_kernel<T><<<(n + 127) / 128, 128, 0, st>>>(B, L, di, N, u, ld_u, z, ld_z, delta, ld_delta, Bm, Cm,
                                                      ld_bc, A_log, D, g, ld_g, h0, h_out);
  return last_err();
}

template <typename T>
hymba_status fuse_norm(int rows, int di, const T* att, const T* g, const float* beta1, const float* beta2,
                       float eps, T* s, cudaStream_t st, bool concat) {
  const int cc = concat ? 1 : 0;
  if (rows <= 0) return HYMBA_OK;
  const bool vec_ok = std::is_same<T, __half>::value && di % 8 == 0 && (reinterpret_cast<uintptr_t>(beta1) & 15) == 0 &&
                      (reinterpret_cast<uintptr_t>(beta2) & 15) == 0 && (reinterpret_cast<uintptr_t>(att) & 15) == 0 &&
                      (reinterpret_cast<uintptr_t>(g) & 15) == 0 && (reinterpret_cast<uintptr_t>(s) & 15) == 0;
  // one warp per row wants many rows (a decode step's 128 rows would fill
  // 32 SMs): below that, one block per row
  if (vec_ok && di <= 32 * 8 * FW_V && rows >= 4 * 148 * 4) {
    if (launch_kernel(false, cc ? fuse_norm_warp_kernel<true> : fuse_norm_warp_kernel<false>, dim3((rows + 3) / 4),
                   dim3(128), 0, st, rows, di, reinterpret_cast<const __half*>(att),
                   reinterpret_cast<const __half*>(g), beta1, beta2, eps, reinterpret_cast<__half*>(s)) !=
        cudaSuccess)
      return HYMBA_ERR_CUDA;
    return last_err();
  }
  if (vec_ok && di <= 8 * 256 * FN_MAXC) {
    if (launch_pdl(cc ? fuse_norm_vec_kernel<true> : fuse_norm_vec_kernel<false>, dim3(rows), dim3(256), 0, st, di,
                   reinterpret_cast<const __half*>(att), reinterpret_cast<const __half*>(g), beta1, beta2, eps,
                   reinterpret_cast<__half*>(s)) != cudaSuccess)
      return HYMBA_ERR_CUDA;
    return last_err();
  }
  if (launch_pdl(fuse_norm_kernel<T>, dim3(rows), dim3(256), 0, st, di, att, g, beta1, beta2, eps, s, cc) !=
      cudaSuccess)
    return HYMBA_ERR_CUDA;
  return last_err();
}

hymba_status rmsnorm_bf16(int rows, int d, const float* x, long long ldx, const float* w, float eps,
                          __nv_bfloat16* y, long long ldy, cudaStream_t st) {
  if (rows <= 0) return HYMBA_OK;
  if (d % 4 || ldx % 4 || ldy % 4 || (reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(w) & 15) ||
      (reinterpret_cast<uintptr_t>(y) & 7))
    return HYMBA_ERR_INVALID;
  rmsnorm_bf16_kernel<<<(rows + 7) / 8, 256, 0, st>>>(rows, d, x, ldx, w, eps, y, ldy);
  return last_err();
}

template <typename T>
hymba_status attention_simt(int B, int L, int M, int Hq, int Hkv, int dh, int dv, int window, const T* Q,
                            long long ldq, const T* K, long long ldk, const T* V, long long ldv, T* O,
                            long long ldo, cudaStream_t st) {
  if (dv > 256) return HYMBA_ERR_UNSUPPORTED;
  const long long warps = static_cast<long long>(B) * L * Hq;
  attention_simt_kernel<T><<<grid1d(warps, 4), 128, 4 * dh * sizeof(float), st>>>(
      B, L, M, Hq, Hkv, dh, dv, window, Q, ldq, K, ldk, V, ldv, O, ldo);
  return last_err();
}

template <typename TS, typename TD>
hymba_status copy2d(const TS* src, long long lds, TD* dst, long long ldd, long long rows, int cols,
                    cudaStream_t st) {
  if (std::is_same<TS, __nv_bfloat16>::value && std::is_same<TD, __half>::value && lds == cols && ldd == cols &&
      (static_cast<long long>(rows) * cols) % 8 == 0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0 &&
      (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
    const long long n8 = rows * cols / 8;
    bf16_to_f16_vec_kernel<<<static_cast<unsigned>(std::min<long long>((n8 + 255) / 256, 148 * 8)), 256, 0, st>>>(
        reinterpret_cast<const uint4*>(src), reinterpret_cast<uint4*>(dst), n8);
    return last_err();
  }
  if (rows <= 0 || cols <= 0) return HYMBA_OK;
  const unsigned gx = grid1d(cols, 256);
  const unsigned gy = static_cast<unsigned>(std::min<long long>(rows, std::max<long long>(1, 148 * 64 / gx)));
  copy2d_kernel<TS, TD><<<dim3(gx, std::min(gy, 65535u)), 256, 0, st>>>(src, lds, dst, ldd, rows, cols);
  return last_err();
}

template <typename TS, typename TC>
hymba_status emit_cache(int B, int L, int M, int T, int cap, int Hkv, int dh, int dv, int di, int k,
                        const TS* Kp, long long ldk, const TS* Vp, long long ldv, const TS* xp, long long ldx,
                        TC* k_ring, TC* v_ring, TC* k_meta, TC* v_meta, float* conv_state, int32_t* pos,
                        cudaStream_t st, const float* prev_tail) {
  if (pos) fill_i32_kernel<<<(B + 255) / 256, 256, 0, st>>>(B, pos, T);
  const int n_keep = std::min(T, cap);
  if (Kp && k_ring && n_keep > 0) {
    long long n = static_cast<long long>(B) * n_keep * Hkv * dh;
    emit_ring_kernel<TS, TC><<<std::min<long long>(grid1d(n, 256), 148 * 32), 256, 0, st>>>(
        B, L, M, T, cap, n_keep, Hkv * dh, Kp, ldk, k_ring);
    n = static_cast<long long>(B) * n_keep * Hkv * dv;
    emit_ring_kernel<TS, TC><<<std::min<long long>(grid1d(n, 256), 148 * 32), 256, 0, st>>>(
        B, L, M, T, cap, n_keep, Hkv * dv, Vp, ldv, v_ring);
  }
  if (Kp && k_meta && M > 0) {
    hymba_status s = copy2d<TS, TC>(Kp, ldk, k_meta, static_cast<long long>(Hkv) * dh, M, Hkv * dh, st);
    if (s != HYMBA_OK) return s;
    s = copy2d<TS, TC>(Vp, ldv, v_meta, static_cast<long long>(Hkv) * dv, M, Hkv * dv, st);
    if (s != HYMBA_OK) return s;
  }
  if (conv_state && k > 1) {
    const long long n = static_cast<long long>(B) * di * (k - 1);
    emit_conv_tail_kernel<TS><<<std::min<long long>(grid1d(n, 256), 148 * 32), 256, 0, st>>>(B, L, di, k, xp,
                                                                                          ldx, conv_state, prev_tail);
  }
  return last_err();
}

// explicit instantiations ----------------------------------------------------
template hymba_status gemm_simt<float>(int, int, int, const float*, long long, const float*, long long, int,
                                       float*, long long, float*, long long, int, const float*, const float*,
                                       long long, cudaStream_t);
template hymba_status rope_simt<float>(float*, long long, int, int, int, int, float, int, const int32_t*, int,
                                       cudaStream_t);
template hymba_status rope_simt<__half>(__half*, long long, int, int, int, int, float, int, const int32_t*,
                                        int, cudaStream_t);
template hymba_status conv_silu<float, float>(const float*, long long, float*, long long, int, int, int, int,
                                              const float*, const float*, cudaStream_t);
template hymba_status conv_silu<__half, __half>(const __half*, long long, __half*, long long, int, int, int,
                                                int, const float*, const float*, cudaStream_t);
template hymba_status scan_simt<float>(int, int, int, int, const float*, long long, const float*, long long,
                                       const float*, long long, const float*, const float*, long long,
                                       const float*, const float*, float*, long long, const float*, float*,
                                       cudaStream_t);
template hymba_status scan_simt<__half>(int, int, int, int, const __half*, long long, const __half*, long long,
                                        const float*, long long, const float*, const float*, long long,
                                        const float*, const float*, __half*, long long, const float*, float*,
                                        cudaStream_t);
template hymba_status fuse_norm<float>(int, int, const float*, const float*, const float*, const float*, float,
                                       float*, cudaStream_t, bool);
template hymba_status fuse_norm<__half>(int, int, const __half*, const __half*, const float*, const float*,
                                        float, __half*, cudaStream_t, bool);
template hymba_status attention_simt<float>(int, int, int, int, int, int, int, int, const float*, long long,
                                            const float*, long long, const float*, long long, float*,
                                            long long, cudaStream_t);
template hymba_status attention_simt<__half>(int, int, int, int, int, int, int, int, const __half*, long long,
                                             const __half*, long long, const __half*, long long, __half*,
                                             long long, cudaStream_t);
template hymba_status copy2d<float, float>(const float*, long long, float*, long long, long long, int,
                                           cudaStream_t);
template hymba_status copy2d<__half, __half>(const __half*, long long, __half*, long long, long long, int,
                                             cudaStream_t);
template hymba_status copy2d<__nv_bfloat16, __half>(const __nv_bfloat16*, long long, __half*, long long,
                                                    long long, int, cudaStream_t);
template hymba_status copy2d<__half, __nv_bfloat16>(const __half*, long long, __nv_bfloat16*, long long,
                                                    long long, int, cudaStream_t);
template hymba_status emit_cache<float, float>(int, int, int, int, int, int, int, int, int, int, const float*,
                                               long long, const float*, long long, const float*, long long,
                                               float*, float*, float*, float*, float*, int32_t*, cudaStream_t, const float*);
template hymba_status emit_cache<__half, __nv_bfloat16>(int, int, int, int, int, int, int, int, int, int,
                                                        const __half*, long long, const __half*, long long,
                                                        const __half*, long long, __nv_bfloat16*,
                                                        __nv_bfloat16*, __nv_bfloat16*, __nv_bfloat16*, float*,
                                                        int32_t*, cudaStream_t, const float*);

}  // namespace hy
