// Causal depthwise conv1d + SiLU of the SSM branch on the fp16 path
// ("Hymba: A Hybrid-head Architecture for Small Language Models", section 2.1:
// the SSM heads' input goes through a short causal convolution before the
// selective scan):
//     u[b, t, c] = silu(bias[c] + sum_{j<K} w[c, j] * x[b, t - K + 1 + j, c]),
// with x = 0 before the first row of each sequence.
//
// The step reads x once and writes u once, so it is bound by HBM.  Persistent
// blocks own one channel tile (its weights stay in registers) and walk row
// tiles of TT rows x CW channels of one sequence; thread 0 streams
// each tile, together with its K-1 rows of causal history, into a ring of
// shared-memory stages with one 3-D TMA load (sequence, row, channel).  The
// load of a tile that starts at row 0 begins at row -(K-1), which TMA fills
// with zeros: that is the causal zero padding, and no row of the previous
// sequence is ever read.  When a history `tail` is given (the meta rows
// processed once for the whole batch), its K-1 rows replace that zero
// padding in shared memory.  Each thread then computes 8 rows x 4 channels
// from shared memory and writes 8-byte vectors of u (a warp covers 256
// contiguous bytes of a row); at 64 registers a thread, four blocks fit on an
// SM.  Every wait is bounded.
#include "simt.cuh"

namespace hy {
namespace {

constexpr int CV_TT = 64;       // rows per tile
constexpr int CV_CW = 128;      // channels per tile (256-byte rows)
constexpr int CV_S = 3;         // ring stages
constexpr int CV_VEC = 4;       // channels per thread (one 8-byte vector)
constexpr int CV_THREADS = 256; // 32 channel groups x 8 row groups
constexpr int CV_RPT = CV_TT / (CV_THREADS / (CV_CW / CV_VEC));  // rows per thread = 8
constexpr float kCvLog2e = 1.4426950408889634f;

template <int K>
struct ConvCfg {
  static constexpr int ROWS = CV_TT + K - 1;         // rows per stage, history included
  static constexpr int STAGE = ROWS * CV_CW * 2;     // bytes per stage
  static constexpr int SMEM = 128 + CV_S * STAGE;    // + mbarriers
};

template <int K>
__global__ void __launch_bounds__(CV_THREADS, 4)
    conv_tma_kernel(const __grid_constant__ CUtensorMap tmX, __half* __restrict__ u, long long ld_u, int B, int L,
                    int di, const float* __restrict__ w, const float* __restrict__ bias,
                    const float* __restrict__ tail, int32_t* status, uint64_t wait_ns) {
  using Cfg = ConvCfg<K>;
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + CV_S * Cfg::STAGE);
  __shared__ int abort_flag;
  const int tid = threadIdx.x;
  const int cg = tid % (CV_CW / CV_VEC), rg = tid / (CV_CW / CV_VEC);
  // block -> (channel tile ct, slot j); slot j walks row tiles j, j + per_ct, ...
  const int n_ct = (di + CV_CW - 1) / CV_CW, n_tt = (L + CV_TT - 1) / CV_TT;
  const int per_ct = gridDim.x / n_ct;
  const int ct = blockIdx.x % n_ct, slot = blockIdx.x / n_ct;
  const int n_rt = B * n_tt;  // row tiles
  if (tid == 0) {
    for (int s = 0; s < CV_S; ++s) mbar_init(smem_u32(&bars[s]), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtl wc{&abort_flag, status, wait_ns};
  auto issue = [&](int rt, int s) {
    const int tt = rt % n_tt, b = rt / n_tt;
    const uint32_t bar = smem_u32(&bars[s]);
    mbar_arrive_expect_tx(bar, Cfg::STAGE);
    tma_load_3d(smem_u32(smem + s * Cfg::STAGE), &tmX, bar, ct * CV_CW, tt * CV_TT - (K - 1), b);
  };
  int issued = 0;  // tiles issued by this block (thread 0's count)
  if (tid == 0) {
    tma_prefetch_desc(&tmX);
    for (int j = 0; j < CV_S; ++j) {
      const int rt = slot + j * per_ct;
      if (rt < n_rt) {
        issue(rt, j);
        ++issued;
      }
    }
  }
  const int c0 = ct * CV_CW + cg * CV_VEC;
  float wt[CV_VEC][K], bs[CV_VEC];
#pragma unroll
  for (int e = 0; e < CV_VEC; ++e) {
    bs[e] = c0 < di ? __ldg(bias + c0 + e) : 0.f;
#pragma unroll
    for (int j = 0; j < K; ++j) wt[e][j] = c0 < di ? __ldg(w + (c0 + e) * K + j) : 0.f;
  }
  int it = 0;
  for (int rt = slot; rt < n_rt; rt += per_ct, ++it) {
    const int s = it % CV_S;
    bool ok = mbar_wait(smem_u32(&bars[s]), (it / CV_S) & 1, wc);
    if (!__syncthreads_and(ok)) break;
    const int tt = rt % n_tt, b = rt / n_tt;
    if (tail != nullptr && tt == 0) {
      // history rows of the first tile: the tail [di, K-1] (oldest first), not zeros
      __half* hist = reinterpret_cast<__half*>(smem + s * Cfg::STAGE);
      for (int i = tid; i < (K - 1) * CV_CW; i += CV_THREADS) {
        const int j = i / CV_CW, cc = i % CV_CW, c = ct * CV_CW + cc;
        hist[j * CV_CW + cc] = __float2half_rn(c < di ? tail[static_cast<long long>(c) * (K - 1) + j] : 0.f);
      }
      fence_proxy_async_smem();  // these stores come before the stage's next TMA write
      __syncthreads();
    }
    if (c0 < di) {
      const uint8_t* st = smem + s * Cfg::STAGE + cg * (CV_VEC * 2);
      const int r0 = rg * CV_RPT;  // first output row of this thread within the tile
      float win[K][CV_VEC];        // win[j] = x row (output row - K + 1 + j)
#pragma unroll
      for (int j = 0; j < K - 1; ++j) {
        const uint2 q = *reinterpret_cast<const uint2*>(st + (r0 + j) * (CV_CW * 2));
        const __half2* hq = reinterpret_cast<const __half2*>(&q);
#pragma unroll
        for (int e = 0; e < CV_VEC / 2; ++e) {
          const float2 f = __half22float2(hq[e]);
          win[j][2 * e] = f.x;
          win[j][2 * e + 1] = f.y;
        }
      }
      const long long row_base = static_cast<long long>(b) * L + tt * CV_TT;
#pragma unroll
      for (int r = 0; r < CV_RPT; ++r) {
        const uint2 q = *reinterpret_cast<const uint2*>(st + (r0 + r + K - 1) * (CV_CW * 2));
        const __half2* hq = reinterpret_cast<const __half2*>(&q);
#pragma unroll
        for (int e = 0; e < CV_VEC / 2; ++e) {
          const float2 f = __half22float2(hq[e]);
          win[K - 1][2 * e] = f.x;
          win[K - 1][2 * e + 1] = f.y;
        }
        float o[CV_VEC];
#pragma unroll
        for (int e = 0; e < CV_VEC; ++e) {
          float acc = bs[e];
#pragma unroll
          for (int j = 0; j < K; ++j) acc = fmaf(wt[e][j], win[j][e], acc);
          o[e] = acc * rcp_approx(1.0f + ex2_approx(-kCvLog2e * acc));  // silu
        }
#pragma unroll
        for (int j = 0; j + 1 < K; ++j)
#pragma unroll
          for (int e = 0; e < CV_VEC; ++e) win[j][e] = win[j + 1][e];
        const int t = tt * CV_TT + r0 + r;
        if (t < L)
          *reinterpret_cast<uint2*>(u + (row_base + r0 + r) * ld_u + c0) =
              make_uint2(pack_half2(o[0], o[1]), pack_half2(o[2], o[3]));
      }
    }
    __syncthreads();  // every thread is done with stage s
    if (tid == 0) {
      const int next = rt + CV_S * per_ct;
      if (next < n_rt) {
        issue(next, s);
        ++issued;
      }
    }
  }
  // after a wait gave up, let this block's loads in flight land before exit
  if (tid == 0 && abort_flag)
    for (int j = max(0, issued - CV_S); j < issued; ++j)
      mbar_wait_drain(smem_u32(&bars[j % CV_S]), (j / CV_S) & 1, 1000000);
}

template <int K>
hymba_status launch_conv(const CUtensorMap& m, __half* u, long long ld_u, int B, int L, int di, const float* w,
                         const float* bias, const float* tail, int32_t* status, uint64_t wait_ns, int num_sms,
                         cudaStream_t st) {
  using Cfg = ConvCfg<K>;
  auto kern = conv_tma_kernel<K>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM) != cudaSuccess)
    return HYMBA_ERR_CUDA;
  // every channel tile gets the same number of blocks (about four per SM in all)
  const int n_ct = (di + CV_CW - 1) / CV_CW;
  const long long n_rt = static_cast<long long>(B) * ((L + CV_TT - 1) / CV_TT);
  const int per_ct = static_cast<int>(std::max(1LL, std::min(n_rt, (4LL * num_sms + n_ct - 1) / n_ct)));
  const int grid = n_ct * per_ct;
  if (launch_kernel(false, kern, dim3(grid), dim3(CV_THREADS), Cfg::SMEM, st, m, u, ld_u, B, L, di, w, bias, tail, status,
                 wait_ns) != cudaSuccess)
    return HYMBA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? HYMBA_OK : HYMBA_ERR_CUDA;
}

}  // namespace

bool conv_tma_supported(int di, int k, long long ld_x, long long ld_u, const void* x, const void* u) {
  return di % 8 == 0 && k >= 2 && k <= 4 && ld_x % 8 == 0 && ld_u % 8 == 0 &&
         (reinterpret_cast<uintptr_t>(x) & 15) == 0 && (reinterpret_cast<uintptr_t>(u) & 15) == 0;
}

hymba_status conv_silu_tma(const __half* x, long long ld_x, __half* u, long long ld_u, int B, int L, int di, int k,
                           const float* w, const float* bias, int32_t* status, uint64_t wait_ns, int num_sms,
                           cudaStream_t st, const float* tail) {
  if (!conv_tma_supported(di, k, ld_x, ld_u, x, u)) return HYMBA_ERR_UNSUPPORTED;
  if (B < 1 || L < 1) return HYMBA_OK;
  CUtensorMap m;
  const uint64_t dims[3] = {static_cast<uint64_t>(di), static_cast<uint64_t>(L), static_cast<uint64_t>(B)};
  const uint64_t str[2] = {static_cast<uint64_t>(ld_x) * 2, static_cast<uint64_t>(ld_x) * 2 * L};
  const uint32_t box[3] = {static_cast<uint32_t>(CV_CW), static_cast<uint32_t>(CV_TT + k - 1), 1};
  if (!encode_tmap(&m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, x, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE))
    return HYMBA_ERR_CUDA;
  switch (k) {
    case 2: return launch_conv<2>(m, u, ld_u, B, L, di, w, bias, tail, status, wait_ns, num_sms, st);
    case 3: return launch_conv<3>(m, u, ld_u, B, L, di, w, bias, tail, status, wait_ns, num_sms, st);
    default: return launch_conv<4>(m, u, ld_u, B, L, di, w, bias, tail, status, wait_ns, num_sms, st);
  }
}

}  // namespace hy
