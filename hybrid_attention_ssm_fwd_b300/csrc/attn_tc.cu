// Flash attention on tcgen05 for the hybrid head's attention branch
// ("Hymba: A Hybrid-head Architecture for Small Language Models", section 2.2
// sliding-window / global attention, section 2.3 meta tokens): query row i
// sees key j iff j <= i and (window == 0 or i - j < window or j < M).
//
// One persistent CTA per SM walks work units (batch, 128-row query tile,
// query head), heaviest query tiles first.  Per unit only the key tiles that
// can hold a visible key are visited: the meta tiles and the tiles of the
// window (all tiles up to the diagonal for a global layer).
//
//   warp 0      TMA: Q tile once per unit; K tiles and V tiles through two
//               2-stage rings (128-byte swizzle).
//   warp 1      TMEM owner; one thread issues S = Q K^T (M=128, N=128, K=16
//               x4) into one of two TMEM S buffers and O += P V (N = dv, K=16
//               x8, V read MN-major) into the TMEM O accumulator, in the order
//               S0 S1 PV0 S2 PV1 ... so softmax of tile j overlaps S_{j+1} and
//               PV_{j-1}.
//   warps 2..5  softmax, one query row per thread (TMEM lane = row): masked
//               row max, exp2, row sum, P (fp16) written to shared memory in
//               the swizzled K-major layout the MMA reads.  The running max is
//               only raised when a tile's max exceeds it by more than 2^8
//               (then O is rescaled in TMEM after the previous PV completes);
//               otherwise P stays <= 2^8, which fp16 and fp32 hold exactly
//               enough.  At the end of a unit O / l is stored as fp16.
// Every wait is bounded (see WaitCtl).
#include "attn_tc.cuh"

namespace hy {
namespace {

constexpr int BQ = 128;        // query rows per unit
constexpr int BKV = 128;       // keys per tile
constexpr int DH = 64;         // Q/K head dim handled here
constexpr float kRescaleLog2 = 8.0f;

struct AttnParams {
  int B, L, M, Hq, Hkv, dv, window, n_qt, n_units;
  float scale_log2;  // log2(e) / sqrt(dh)
  __half* O;
  long long ldo;
  int32_t* status;
  uint64_t wait_ns;
};

struct Unit {
  int b, h, g, q0, qv1;  // qv1 = min(q0 + BQ, L)
  int n_tiles, meta_last, win_first, split;  // split: tiles [0, split) are 0.., rest start at win_first
};

HY_DEV Unit make_unit(const AttnParams& p, int u) {
  Unit U;
  U.h = u % p.Hq;
  const int r = u / p.Hq;
  const int qt = p.n_qt - 1 - (r % p.n_qt);
  U.b = r / p.n_qt;
  U.g = (U.h * p.Hkv) / p.Hq;
  U.q0 = qt * BQ;
  U.qv1 = min(U.q0 + BQ, p.L);
  const int diag = (U.qv1 - 1) / BKV;
  U.meta_last = p.M > 0 ? (p.M - 1) / BKV : -1;
  U.win_first = p.window > 0 ? max(0, U.q0 - p.window + 1) / BKV : 0;
  if (U.win_first <= U.meta_last + 1) {
    U.n_tiles = diag + 1;
    U.split = U.n_tiles;
  } else {
    U.split = U.meta_last + 1;
    U.n_tiles = U.split + diag - U.win_first + 1;
  }
  return U;
}

HY_DEV int tile_kt(const Unit& U, int t) { return t < U.split ? t : U.win_first + (t - U.split); }

template <int DV>
struct AttnCfg {
  static constexpr int Q_BYTES = BQ * DH * 2;            // 16 KB
  static constexpr int K_BYTES = BKV * DH * 2;           // 16 KB
  static constexpr int V_BYTES = BKV * DV * 2;           // 16/32 KB
  static constexpr int P_BYTES = BQ * BKV * 2;           // 32 KB
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + 2 * K_BYTES;
  static constexpr int OFF_P = OFF_V + 2 * V_BYTES;
  static constexpr int OFF_BAR = OFF_P + 2 * P_BYTES;
  static constexpr int SMEM = 1024 + OFF_BAR + 256;
  static constexpr uint32_t TMEM_COLS = 512;             // S0, S1 (128 each), O (DV)
  static constexpr uint32_t O_COL = 256;
};

// barrier indices
enum {
  B_QFULL = 0, B_QEMPTY, B_KFULL0, B_KFULL1, B_KEMPTY0, B_KEMPTY1, B_VFULL0, B_VFULL1, B_VEMPTY0, B_VEMPTY1,
  B_SFULL0, B_SFULL1, B_SEMPTY0, B_SEMPTY1, B_PFULL0, B_PFULL1, B_PVDONE0, B_PVDONE1, B_OEMPTY, B_COUNT
};

template <int DV>
__global__ void __launch_bounds__(192, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  using Cfg = AttnCfg<DV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + B_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t sQ = smem_u32(smem + Cfg::OFF_Q);
  const uint32_t sK = smem_u32(smem + Cfg::OFF_K);
  const uint32_t sV = smem_u32(smem + Cfg::OFF_V);
  const uint32_t sP = smem_u32(smem + Cfg::OFF_P);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < B_COUNT; ++i) {
      const bool four = (i == B_SEMPTY0 || i == B_SEMPTY1 || i == B_PFULL0 || i == B_PFULL1 || i == B_OEMPTY);
      mbar_init(bar(i), four ? 4 : 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), Cfg::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{abort_flag, p.status, p.wait_ns};

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      uint32_t kc = 0, uc = 0;
      uint32_t issued = 0, par = 0;  // bits: Q, K0, K1, V0, V1 outstanding + their parities
      bool ok = true;
      for (int u = blockIdx.x; u < p.n_units && ok; u += gridDim.x, ++uc) {
        const Unit U = make_unit(p, u);
        if (!mbar_wait(bar(B_QEMPTY), (uc & 1) ^ 1, wc)) { ok = false; break; }
        mbar_arrive_expect_tx(bar(B_QFULL), Cfg::Q_BYTES);
        tma_load_3d(sQ, &tmQ, bar(B_QFULL), U.h * DH, U.q0, U.b);
        issued |= 1u;
        par = (par & ~1u) | (uc & 1);
        for (int t = 0; t < U.n_tiles; ++t, ++kc) {
          const int s = kc & 1;
          const uint32_t ph = (kc >> 1) & 1;
          const int k0 = tile_kt(U, t) * BKV;
          if (!mbar_wait(bar(B_KEMPTY0 + s), ph ^ 1, wc)) { ok = false; break; }
          mbar_arrive_expect_tx(bar(B_KFULL0 + s), Cfg::K_BYTES);
          tma_load_3d(sK + s * Cfg::K_BYTES, &tmK, bar(B_KFULL0 + s), U.g * DH, k0, U.b);
          issued |= 2u << s;
          par = (par & ~(2u << s)) | (ph << (1 + s));
          if (!mbar_wait(bar(B_VEMPTY0 + s), ph ^ 1, wc)) { ok = false; break; }
          mbar_arrive_expect_tx(bar(B_VFULL0 + s), Cfg::V_BYTES);
#pragma unroll
          for (int c = 0; c < DV / 64; ++c)
            tma_load_3d(sV + s * Cfg::V_BYTES + c * (BKV * 128), &tmV, bar(B_VFULL0 + s), U.g * DV + c * 64, k0, U.b);
          issued |= 8u << s;
          par = (par & ~(8u << s)) | (ph << (3 + s));
        }
      }
      if (!ok) {
        if (issued & 1u) mbar_wait_drain(bar(B_QFULL), par & 1, 1000000);
        for (int s = 0; s < 2; ++s) {
          if (issued & (2u << s)) mbar_wait_drain(bar(B_KFULL0 + s), (par >> (1 + s)) & 1, 1000000);
          if (issued & (8u << s)) mbar_wait_drain(bar(B_VFULL0 + s), (par >> (3 + s)) & 1, 1000000);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_f16(128, BKV, 0, false, false);
      constexpr uint32_t idPV = idesc_f16(128, DV, 0, false, true);
      uint32_t kc = 0, jt = 0, uc = 0;
      uint32_t last_commit_bar = 0xffffffffu, last_commit_par = 0;
      bool ok = true;
      auto issue_S = [&](uint32_t j_global, uint32_t kcl) -> bool {
        const int s = kcl & 1;
        const int sb = j_global & 1;
        if (!mbar_wait(bar(B_KFULL0 + s), (kcl >> 1) & 1, wc)) return false;
        if (!mbar_wait(bar(B_SEMPTY0 + sb), ((j_global >> 1) & 1) ^ 1, wc)) return false;
        tc_fence_after();
        const uint64_t dq = sdesc_sw128(sQ, 16, 1024);
        const uint64_t dk = sdesc_sw128(sK + s * Cfg::K_BYTES, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) tc_mma_f16(tmem + sb * BKV, dq + 2 * kk, dk + 2 * kk, idS, kk > 0);
        tc_commit(bar(B_SFULL0 + sb));
        tc_commit(bar(B_KEMPTY0 + s));
        last_commit_bar = B_SFULL0 + sb;
        last_commit_par = (j_global >> 1) & 1;
        return true;
      };
      auto issue_PV = [&](uint32_t j_global, uint32_t kcl, bool first) -> bool {
        const int s = kcl & 1;
        const int pb = j_global & 1;
        if (!mbar_wait(bar(B_PFULL0 + pb), (j_global >> 1) & 1, wc)) return false;
        if (!mbar_wait(bar(B_VFULL0 + s), (kcl >> 1) & 1, wc)) return false;
        tc_fence_after();
        const uint32_t pbase = sP + pb * Cfg::P_BYTES;
        const uint32_t vbase = sV + s * Cfg::V_BYTES;
#pragma unroll
        for (int kk = 0; kk < BKV / 16; ++kk) {
          const uint64_t da = sdesc_sw128(pbase + (kk >> 2) * (BQ * 128) + (kk & 3) * 32, 16, 1024);
          const uint64_t db = sdesc_sw128(vbase + kk * 16 * 128, BKV * 128, 1024);
          tc_mma_f16(tmem + Cfg::O_COL, da, db, idPV, (first && kk == 0) ? 0u : 1u);
        }
        tc_commit(bar(B_PVDONE0 + pb));
        tc_commit(bar(B_VEMPTY0 + s));
        last_commit_bar = B_PVDONE0 + pb;
        last_commit_par = (j_global >> 1) & 1;
        return true;
      };
      for (int u = blockIdx.x; u < p.n_units && ok; u += gridDim.x, ++uc) {
        const Unit U = make_unit(p, u);
        if (!mbar_wait(bar(B_QFULL), uc & 1, wc)) { ok = false; break; }
        const uint32_t j0 = jt, k0c = kc;
        if (!issue_S(j0, k0c)) { ok = false; break; }
        for (int t = 0; t < U.n_tiles; ++t) {
          if (t + 1 < U.n_tiles) {
            if (!issue_S(j0 + t + 1, k0c + t + 1)) { ok = false; break; }
          } else {
            tc_commit(bar(B_QEMPTY));  // every S MMA of the unit is issued: Q may be replaced
          }
          if (t == 0 && !mbar_wait(bar(B_OEMPTY), (uc & 1) ^ 1, wc)) { ok = false; break; }
          if (!issue_PV(j0 + t, k0c + t, t == 0)) { ok = false; break; }
        }
        jt = j0 + U.n_tiles;
        kc = k0c + U.n_tiles;
      }
      if (!ok && last_commit_bar != 0xffffffffu) mbar_wait_drain(bar(last_commit_bar), last_commit_par, 1000000);
    }
  } else {
    // ---------------------------------------------------------------- softmax warps
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
    uint32_t jt = 0, uc = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < p.n_units && ok; u += gridDim.x, ++uc) {
      const Unit U = make_unit(p, u);
      const int i = U.q0 + r;  // query row (may be >= L on the last tile)
      float m_run = -INFINITY, l_run = 0.f;
      for (int t = 0; t < U.n_tiles; ++t, ++jt) {
        const int sb = jt & 1;
        const bool got = mbar_wait(bar(B_SFULL0 + sb), (jt >> 1) & 1, wc);
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        tc_fence_after();
        float s[BKV];
        {
          uint32_t rr[4][32];
#pragma unroll
          for (int c = 0; c < BKV / 32; ++c) tmem_ld32(lane_base + sb * BKV + c * 32, rr[c]);
          tc_wait_ld();
#pragma unroll
          for (int c = 0; c < BKV / 32; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(rr[c][e]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_SEMPTY0 + sb));
        // mask (raw scores; the positive scale is applied inside the exp2 below)
        const int k0 = tile_kt(U, t) * BKV;
        const bool full_vis = (k0 + BKV - 1 <= U.q0) && (k0 + BKV <= p.L) &&
                              (p.window == 0 || k0 + BKV <= p.M || (U.qv1 - 1) - max(k0, p.M) < p.window);
        if (!full_vis) {
          // key e of this tile (j = k0 + e) is visible iff e <= hi and (e >= lo or e < ml)
          const int hi = min(i, p.L - 1) - k0;
          const int lo = p.window > 0 ? i - p.window + 1 - k0 : -BKV;
          const int ml = p.M - k0;
#pragma unroll
          for (int e = 0; e < BKV; ++e) {
            const bool vis = (e <= hi) && (e >= lo || e < ml);
            s[e] = vis ? s[e] : -INFINITY;
          }
        }
        float mp[8];
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) mp[q8] = s[q8];
#pragma unroll
        for (int e = 8; e < BKV; ++e) mp[e & 7] = fmaxf(mp[e & 7], s[e]);
        const float mt = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                               fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7]))) * p.scale_log2;
        // running max (log2 units): set on the first tile; raised only when a tile exceeds it by > 2^8
        bool need = (t == 0) ? true : (mt > m_run + kRescaleLog2);
        if (t > 0 && __any_sync(0xffffffffu, need)) {
          const float m_new = fmaxf(m_run, mt);
          const float alpha = (m_run == -INFINITY) ? 0.f : ex2_approx(m_run - m_new);
          // O holds PV of earlier tiles: wait for the last one, then scale O in TMEM
          const uint32_t jp = jt - 1;
          const bool g2 = mbar_wait(bar(B_PVDONE0 + (jp & 1)), (jp >> 1) & 1, wc);
          if (!__all_sync(0xffffffffu, g2)) { ok = false; break; }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < DV / 32; ++c) {
            uint32_t rr[32];
            tmem_ld32(lane_base + Cfg::O_COL + c * 32, rr);
            tc_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * alpha);
            tmem_st32(lane_base + Cfg::O_COL + c * 32, rr);
          }
          tc_wait_st();
          l_run *= alpha;
          m_run = m_new;
        } else if (t == 0) {
          m_run = mt;
        }
        const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
        // P buffer sb is free once PV of tile jt-2 completed
        const bool g3 = mbar_wait(bar(B_PVDONE0 + sb), ((jt >> 1) & 1) ^ 1, wc);
        if (!__all_sync(0xffffffffu, g3)) { ok = false; break; }
        const uint32_t prow = sP + sb * Cfg::P_BYTES + r * 128;
        float ls[8];
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) ls[q8] = 0.f;
#pragma unroll
        for (int c = 0; c < BKV / 8; ++c) {  // 16 chunks of 8 keys (16 bytes)
          float pv[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            pv[e] = ex2_approx(fmaf(s[c * 8 + e], p.scale_log2, neg_m));
            ls[e] += pv[e];
          }
          const uint32_t w0 = pack_half2(pv[0], pv[1]), w1 = pack_half2(pv[2], pv[3]);
          const uint32_t w2 = pack_half2(pv[4], pv[5]), w3 = pack_half2(pv[6], pv[7]);
          const int sub = c >> 3, cc = c & 7;
          const uint32_t addr = prow + sub * (BQ * 128) + ((cc ^ (r & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w0), "r"(w1), "r"(w2), "r"(w3)
                       : "memory");
        }
        const float lsum = ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
        l_run += lsum;
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_PFULL0 + sb));
      }
      if (!ok) break;
      // epilogue: O / l -> fp16
      const uint32_t jl = jt - 1;
      const bool g4 = mbar_wait(bar(B_PVDONE0 + (jl & 1)), (jl >> 1) & 1, wc);
      if (!__all_sync(0xffffffffu, g4)) { ok = false; break; }
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.0f / l_run : 0.f;
      __half* orow = p.O + (static_cast<long long>(U.b) * p.L + i) * p.ldo + U.h * DV;
#pragma unroll 1
      for (int c = 0; c < DV / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(lane_base + Cfg::O_COL + c * 32, rr);
        tc_wait_ld();
        if (i < p.L) {
#pragma unroll
          for (int g8 = 0; g8 < 4; ++g8) {
            uint4 v;
            v.x = pack_half2(__uint_as_float(rr[g8 * 8 + 0]) * inv, __uint_as_float(rr[g8 * 8 + 1]) * inv);
            v.y = pack_half2(__uint_as_float(rr[g8 * 8 + 2]) * inv, __uint_as_float(rr[g8 * 8 + 3]) * inv);
            v.z = pack_half2(__uint_as_float(rr[g8 * 8 + 4]) * inv, __uint_as_float(rr[g8 * 8 + 5]) * inv);
            v.w = pack_half2(__uint_as_float(rr[g8 * 8 + 6]) * inv, __uint_as_float(rr[g8 * 8 + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + c * 32 + g8 * 8) = v;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_OEMPTY));
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, Cfg::TMEM_COLS);
}

template <int DV>
hymba_status launch(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const AttnParams& p,
                    int grid, cudaStream_t st) {
  auto kern = attn_tc_kernel<DV>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, AttnCfg<DV>::SMEM) != cudaSuccess)
    return HYMBA_ERR_CUDA;
  kern<<<grid, 192, AttnCfg<DV>::SMEM, st>>>(q, k, v, p);
  return cudaGetLastError() == cudaSuccess ? HYMBA_OK : HYMBA_ERR_CUDA;
}

bool make_map3(CUtensorMap* m, const __half* base, int cols, int L, int B, long long ld) {
  const uint64_t dims[3] = {static_cast<uint64_t>(cols), static_cast<uint64_t>(L), static_cast<uint64_t>(B)};
  const uint64_t str[2] = {static_cast<uint64_t>(ld) * 2, static_cast<uint64_t>(ld) * 2 * L};
  const uint32_t box[3] = {64, 128, 1};
  return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, base, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

bool attn_tc_supported(int dh, int dv) { return dh == DH && (dv == 64 || dv == 128); }

hymba_status attn_tc(int B, int L, int M, int Hq, int Hkv, int dh, int dv, int window, const __half* Q, long long ldq,
                     const __half* K, long long ldk, const __half* V, long long ldv, __half* O, long long ldo,
                     int32_t* status, uint64_t wait_ns, int num_sms, cudaStream_t st) {
  if (!attn_tc_supported(dh, dv)) return HYMBA_ERR_UNSUPPORTED;
  auto al = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; };
  if (!al(Q) || !al(K) || !al(V) || !al(O) || ldq % 8 || ldk % 8 || ldv % 8 || ldo % 8) return HYMBA_ERR_INVALID;
  CUtensorMap tq, tk, tv;
  if (!make_map3(&tq, Q, Hq * dh, L, B, ldq) || !make_map3(&tk, K, Hkv * dh, L, B, ldk) ||
      !make_map3(&tv, V, Hkv * dv, L, B, ldv))
    return HYMBA_ERR_CUDA;
  AttnParams p{};
  p.B = B;
  p.L = L;
  p.M = M;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.dv = dv;
  p.window = window;
  p.n_qt = (L + BQ - 1) / BQ;
  p.n_units = B * p.n_qt * Hq;
  p.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(dh));
  p.O = O;
  p.ldo = ldo;
  p.status = status;
  p.wait_ns = wait_ns;
  const int grid = std::min(p.n_units, std::max(1, num_sms));
  return dv == 128 ? launch<128>(tq, tk, tv, p, grid, st) : launch<64>(tq, tk, tv, p, grid, st);
}

}  // namespace hy
