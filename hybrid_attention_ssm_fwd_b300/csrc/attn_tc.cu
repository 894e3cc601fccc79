// Flash attention on tcgen05 for the hybrid head's attention branch
// ("Hymba: A Hybrid-head Architecture for Small Language Models", section 2.2
// sliding-window / global attention, section 2.3 meta tokens): query row i
// sees key j iff j <= i and (window == 0 or i - j < window or j < M).
//
// One persistent CTA per SM walks work units (batch b, 128-row query tile,
// pair of query heads A and B of one KV group), heaviest query tiles first.
// Both heads of a unit read the same K/V tiles, so each tile is loaded once
// for two heads.  Per unit only the 64-key tiles that can hold a visible key
// are visited: the meta tiles and the tiles of the window (all tiles up to the
// diagonal for a global layer).
//
//   warps 0-3  softmax of head A, warps 4-7 softmax of head B: one query row
//              per thread (TMEM lane = row).  Masked row max, exp2, row sum;
//              P (fp16) is written back into TMEM over the first half of the
//              S buffer it came from.  The running max is only raised when a
//              tile's max exceeds it by more than 2^8 (then O is rescaled in
//              TMEM), so P stays <= 2^8.  At the end of a unit O / l is stored.
//   warp 8     TMA: Q of both heads once per unit; K and V tiles through two
//              6-stage rings (128-byte swizzle).
//   warps 9-12 one thread each issues the MMAs of one kind for one head:
//              S of head A, S of head B, P V of head A, P V of head B (warp
//              9 also owns TMEM).  S is double-buffered per head, so S of
//              tile t+1 is computed while the softmax works on tile t; S of
//              tile t+2 reuses the buffer of tile t once P V of tile t has
//              completed.  Four issuing threads keep the tensor core fed with
//              these small MMAs (N = 64 / dv, K = 16).
//              S = Q K^T reads Q and K from shared memory; O += P V reads P
//              from TMEM and V from shared memory.
// TMEM columns: S_A buffers [0,64) [64,128), S_B buffers [128,192) [192,256),
// O_A [256, 256+dv), O_B after it.  Every wait is bounded (see WaitCtl).
#include "attn_tc.cuh"

namespace hy {
namespace {

constexpr int BQ = 128;        // query rows per unit
constexpr int BKV = 64;        // keys per tile
constexpr int DH = 64;         // Q/K head dim handled here
constexpr int KV_STAGES = 6;   // K and V ring depth
constexpr int MAX_HU = 128;    // head units (pairs or single heads)
constexpr float kRescaleLog2 = 8.0f;
constexpr int NTHREADS = 416;  // 13 warps
constexpr int W_TMA = 8, W_MMA = 9;  // MMA issuers: warps 9-12

struct AttnParams {
  int B, L, M, Hq, Hkv, dv, window, n_qt, n_hu, n_units;
  // L and M are logical (meta rows first).  Normally the Q/K/V/O tensors
  // hold all L rows of a sequence (q_off = 0, Lq = L).  With meta_sep the
  // meta keys come from their own [M, ...] tensors, shared by the batch, and
  // Q/K/V/O hold only the Lq = L - M real rows (q_off = M).
  int meta_sep, q_off, Lq;
  float scale_log2;  // log2(e) / sqrt(dh)
  __half* O;
  long long ldo;
  int32_t* status;
  uint64_t wait_ns;
  int16_t hA[MAX_HU], hB[MAX_HU];  // head unit -> heads (hB = -1: single head)
};

struct Unit {
  int b, hA, hB, g, q0, qv1;  // qv1 = min(q0 + BQ, L)
  int n_tiles, win_first, split;  // split: tiles [0, split) are 0.., rest start at win_first
};

HY_DEV Unit make_unit(const AttnParams& p, int u) {
  Unit U;
  const int hu = u % p.n_hu;
  const int r = u / p.n_hu;
  const int qt = p.n_qt - 1 - (r % p.n_qt);
  U.b = r / p.n_qt;
  U.hA = p.hA[hu];
  U.hB = p.hB[hu];
  U.g = (U.hA * p.Hkv) / p.Hq;
  U.q0 = p.q_off + qt * BQ;  // logical position of the tile's first row
  U.qv1 = min(U.q0 + BQ, p.L);
  const int diag = (U.qv1 - 1) / BKV;
  const int meta_last = p.M > 0 ? (p.M - 1) / BKV : -1;
  U.win_first = p.window > 0 ? max(0, U.q0 - p.window + 1) / BKV : 0;
  if (U.win_first <= meta_last + 1) {
    U.n_tiles = diag + 1;
    U.split = U.n_tiles;
  } else {
    U.split = meta_last + 1;
    U.n_tiles = U.split + diag - U.win_first + 1;
  }
  return U;
}

HY_DEV int tile_kt(const Unit& U, int t) { return t < U.split ? t : U.win_first + (t - U.split); }

template <int DV>
struct AttnCfg {
  static constexpr int Q_BYTES = BQ * DH * 2;            // 16 KB per head
  static constexpr int K_BYTES = BKV * DH * 2;           // 8 KB
  static constexpr int V_BYTES = BKV * DV * 2;           // 8/16 KB
  static constexpr int OFF_Q = 0;                        // Q_A | Q_B
  static constexpr int OFF_K = OFF_Q + 2 * Q_BYTES;
  static constexpr int OFF_V = OFF_K + KV_STAGES * K_BYTES;
  static constexpr int OFF_BAR = OFF_V + KV_STAGES * V_BYTES;
  static constexpr int SMEM = 1024 + OFF_BAR + 512;
  static constexpr uint32_t TMEM_COLS = 512;
  // S buffer `buf` of head x, O of head x
  static HY_DEV uint32_t s_col(int x, uint32_t buf) { return static_cast<uint32_t>(x) * 128u + (buf & 1u) * 64u; }
  static HY_DEV uint32_t o_col(int x) { return x == 0 ? 256u : 256u + DV; }
};

// barrier indices
enum {
  B_QFULL = 0, B_QEMPTY,
  B_KFULL = 2,                        // [KV_STAGES]
  B_KEMPTY = B_KFULL + KV_STAGES,     // [KV_STAGES]
  B_VFULL = B_KEMPTY + KV_STAGES,     // [KV_STAGES]
  B_VEMPTY = B_VFULL + KV_STAGES,     // [KV_STAGES]
  B_SFULL = B_VEMPTY + KV_STAGES,     // [head][buffer]
  B_PFULL = B_SFULL + 4,              // [head][buffer], 4 arrivals (softmax warps)
  B_PVDONE = B_PFULL + 4,             // [head]
  B_OEMPTY = B_PVDONE + 2,            // [head], 4 arrivals
  B_PVFREE = B_OEMPTY + 2,            // [head][buffer]: P V of the buffer's tile completed
  B_COUNT = B_PVFREE + 4
};

HY_DEV void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

HY_DEV float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// O += P V with A (P, fp16, 128 x 16 per MMA) read from TMEM.
HY_DEV void tc_mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

template <int DV>
__global__ void __launch_bounds__(NTHREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmKm,
                   const __grid_constant__ CUtensorMap tmVm, const __grid_constant__ AttnParams p) {
  using Cfg = AttnCfg<DV>;
  pdl_wait();  // nothing before: the preceding kernel may still hold this SM's tensor memory
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem<1024>(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + B_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t sQ = smem_u32(smem + Cfg::OFF_Q);
  const uint32_t sK = smem_u32(smem + Cfg::OFF_K);
  const uint32_t sV = smem_u32(smem + Cfg::OFF_V);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < B_COUNT; ++i) {
      const bool four = (i >= B_PFULL && i < B_PFULL + 4) || i == B_OEMPTY || i == B_OEMPTY + 1;
      // ring slots and Q are released by both MMA issuers
      const bool two = i == B_QEMPTY || (i >= B_KEMPTY && i < B_KEMPTY + KV_STAGES) ||
                       (i >= B_VEMPTY && i < B_VEMPTY + KV_STAGES);
      mbar_init(bar(i), four ? 4 : two ? 2 : 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == W_MMA) tmem_alloc(smem_u32(tmem_slot), Cfg::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{abort_flag, p.status, p.wait_ns};

  if (warp == W_TMA) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      uint32_t kc = 0, uc = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.n_units && ok; u += gridDim.x, ++uc) {
        const Unit U = make_unit(p, u);
        if (!mbar_wait(bar(B_QEMPTY), (uc & 1) ^ 1, wc)) { ok = false; break; }
        mbar_arrive_expect_tx(bar(B_QFULL), (U.hB >= 0 ? 2 : 1) * Cfg::Q_BYTES);
        tma_load_3d(sQ, &tmQ, bar(B_QFULL), U.hA * DH, U.q0 - p.q_off, U.b);
        if (U.hB >= 0) tma_load_3d(sQ + Cfg::Q_BYTES, &tmQ, bar(B_QFULL), U.hB * DH, U.q0 - p.q_off, U.b);
        for (int t = 0; t < U.n_tiles; ++t, ++kc) {
          const int s = kc % KV_STAGES;
          const uint32_t ph = (kc / KV_STAGES) & 1;
          const int k0 = tile_kt(U, t) * BKV;
          // key source: the shared meta tensors, or this sequence's rows
          const bool from_meta = p.meta_sep && k0 < p.M;
          const CUtensorMap* mk = from_meta ? &tmKm : &tmK;
          const CUtensorMap* mv = from_meta ? &tmVm : &tmV;
          const int kr = from_meta ? k0 : k0 - p.q_off;
          const int kb = from_meta ? 0 : U.b;
          if (!mbar_wait(bar(B_KEMPTY + s), ph ^ 1, wc)) { ok = false; break; }
          mbar_arrive_expect_tx(bar(B_KFULL + s), Cfg::K_BYTES);
          tma_load_3d(sK + s * Cfg::K_BYTES, mk, bar(B_KFULL + s), U.g * DH, kr, kb);
          if (!mbar_wait(bar(B_VEMPTY + s), ph ^ 1, wc)) { ok = false; break; }
          mbar_arrive_expect_tx(bar(B_VFULL + s), Cfg::V_BYTES);
#pragma unroll
          for (int c = 0; c < DV / 64; ++c)
            tma_load_3d(sV + s * Cfg::V_BYTES + c * (BKV * 128), mv, bar(B_VFULL + s), U.g * DV + c * 64, kr, kb);
        }
      }
      // after a wait gave up, let the loads this thread issued land before
      // the CTA exits (each ring slot's recent loads and the last Q load)
      if (!ok) {
        for (uint32_t j = (kc >= KV_STAGES ? kc - KV_STAGES : 0); j <= kc; ++j) {
          mbar_wait_drain(bar(B_KFULL + j % KV_STAGES), (j / KV_STAGES) & 1, 1000000);
          mbar_wait_drain(bar(B_VFULL + j % KV_STAGES), (j / KV_STAGES) & 1, 1000000);
        }
        mbar_wait_drain(bar(B_QFULL), uc & 1, 1000000);
      }
    }
  } else if (warp >= W_MMA && warp < W_MMA + 4) {
    // ---------------------------------------------------------------- MMA issuers
    // four issuing threads: warp W_MMA + x issues S = Q K^T of head x, warp
    // W_MMA + 2 + x issues O += P V of head x.  Each walks all units; the
    // ring barriers take one arrival from each thread of the pair that
    // releases them (a thread whose head is absent in a unit only waits and
    // arrives).  S of tile J reuses the buffer of tile J-2, so it waits until
    // P V of tile J-2 has completed (PVFREE of that buffer).
    if (lane == 0) {
      const int role = warp - W_MMA;  // 0, 1: S of head A, B;  2, 3: P V of head A, B
      const int x = role & 1;
      const bool is_s = role < 2;
      constexpr uint32_t idS = idesc_f16(128, BKV, 0, false, false);
      constexpr uint32_t idPV = idesc_f16(128, DV, 0, false, true);
      uint32_t J = 0;           // global tile counter of head x (S buffer = J & 1)
      uint32_t ju = 0;          // units of head x (OEMPTY phase)
      uint32_t kc = 0, uc = 0;  // K/V ring position of the unit's first tile; unit count (QFULL phase)
      bool ok = true;
      bool any_commit = false;
      uint32_t last_bar = 0, last_par = 0;
      const uint64_t dq = sdesc_sw128(sQ + x * Cfg::Q_BYTES, 16, 1024);
      auto commit = [&](int b, uint32_t par) {
        tc_commit(bar(b));
        any_commit = true;
        last_bar = b;
        last_par = par;
      };
      for (int u = blockIdx.x; u < p.n_units && ok; u += gridDim.x, ++uc) {
        const Unit U = make_unit(p, u);
        const bool mine = x == 0 || U.hB >= 0;
        if (is_s && !mbar_wait(bar(B_QFULL), uc & 1, wc)) { ok = false; break; }
        for (int t = 0; t < U.n_tiles; ++t) {
          const uint32_t kct = kc + t;
          const int slot = kct % KV_STAGES;
          const uint32_t ph = (kct / KV_STAGES) & 1;
          if (is_s) {
            if (!mbar_wait(bar(B_KFULL + slot), ph, wc)) { ok = false; break; }
            if (mine) {
              if (J >= 2 && !mbar_wait(bar(B_PVFREE + 2 * x + (J & 1)), ((J >> 1) - 1) & 1, wc)) { ok = false; break; }
              tc_fence_after();
              const uint64_t dk = sdesc_sw128(sK + slot * Cfg::K_BYTES, 16, 1024);
              const uint32_t d = tmem + Cfg::s_col(x, J);
#pragma unroll
              for (int kk = 0; kk < DH / 16; ++kk) tc_mma_f16(d, dq + 2 * kk, dk + 2 * kk, idS, kk > 0);
              commit(B_SFULL + 2 * x + (J & 1), (J >> 1) & 1);
              ++J;
            }
            commit(B_KEMPTY + slot, ph);
            if (t + 1 == U.n_tiles) commit(B_QEMPTY, uc & 1);  // every S of the unit is issued
          } else {
            if (!mbar_wait(bar(B_VFULL + slot), ph, wc)) { ok = false; break; }
            if (mine) {
              if (t == 0 && !mbar_wait(bar(B_OEMPTY + x), (ju & 1) ^ 1, wc)) { ok = false; break; }
              if (!mbar_wait(bar(B_PFULL + 2 * x + (J & 1)), (J >> 1) & 1, wc)) { ok = false; break; }
              tc_fence_after();
              const uint32_t vbase = sV + slot * Cfg::V_BYTES;
              const uint32_t a = tmem + Cfg::s_col(x, J);
#pragma unroll
              for (int kk = 0; kk < BKV / 16; ++kk) {
                const uint64_t db = sdesc_sw128(vbase + kk * 16 * 128, BKV * 128, 1024);
                tc_mma_f16_ts(tmem + Cfg::o_col(x), a + kk * 8, db, idPV, (t == 0 && kk == 0) ? 0u : 1u);
              }
              commit(B_PVDONE + x, J & 1);
              commit(B_PVFREE + 2 * x + (J & 1), (J >> 1) & 1);
              ++J;
            }
            commit(B_VEMPTY + slot, ph);
          }
        }
        if (!ok) break;
        if (!is_s && mine) ++ju;
        kc += U.n_tiles;
      }
      if (!ok && any_commit) mbar_wait_drain(bar(last_bar), last_par, 1000000);
    }
  } else {
    // ---------------------------------------------------------------- softmax warps
    const int x = warp >> 2;  // 0 = head A, 1 = head B
    const int q = warp & 3;   // TMEM lane quarter of this warp
    const int r = q * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t o_col = Cfg::o_col(x);
    uint32_t J = 0;  // global tile counter of this head
    bool ok = true;
    for (int u = blockIdx.x; u < p.n_units && ok; u += gridDim.x) {
      const Unit U = make_unit(p, u);
      const int h = x == 0 ? U.hA : U.hB;
      if (h < 0) continue;  // single-head unit: nothing for head B
      const int i = U.q0 + r;  // query row (may be >= L on the last tile)
      float m_run = -INFINITY, l_run = 0.f;
      for (int t = 0; t < U.n_tiles; ++t, ++J) {
        const uint32_t s_col = Cfg::s_col(x, J);
        const bool got = mbar_wait(bar(B_SFULL + 2 * x + (J & 1)), (J >> 1) & 1, wc);
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        tc_fence_after();
        uint32_t sr[BKV / 32][32];  // raw scores (fp32 bits)
#pragma unroll
        for (int c = 0; c < BKV / 32; ++c) tmem_ld32(lane_base + s_col + c * 32, sr[c]);
        tc_wait_ld();
        // mask (raw scores; the positive scale is applied inside the exp2 below).
        // Decided for this warp's 32 rows: the causal bound (and the sequence
        // end) cuts the tile unless every key precedes the warp's first row;
        // the window cuts it unless the warp's last row still sees the
        // tile's first non-meta key.  Most cut tiles are cut by one bound
        // only, and take a one-comparison loop.
        const int k0 = tile_kt(U, t) * BKV;
        const int w_lo = U.q0 + q * 32, w_hi = min(w_lo + 31, p.L - 1);
        const bool causal_ok = (k0 + BKV - 1 <= w_lo) && (k0 + BKV <= p.L);
        const bool window_ok = p.window == 0 || k0 + BKV <= p.M || w_hi - max(k0, p.M) < p.window;
        if (!(causal_ok && window_ok)) {
          // key e of this tile (j = k0 + e) is visible iff e <= hi and (e >= lo or e < ml)
          const int hi = min(i, p.L - 1) - k0;
          const int lo = p.window > 0 ? i - p.window + 1 - k0 : -BKV;
          const int ml = p.M - k0;
          if (window_ok) {
#pragma unroll
            for (int e = 0; e < BKV; ++e) sr[e >> 5][e & 31] = e <= hi ? sr[e >> 5][e & 31] : 0xff800000u;  // -inf
          } else if (causal_ok && ml <= 0) {
#pragma unroll
            for (int e = 0; e < BKV; ++e) sr[e >> 5][e & 31] = e >= lo ? sr[e >> 5][e & 31] : 0xff800000u;
          } else {
#pragma unroll
            for (int e = 0; e < BKV; ++e) {
              const bool vis = (e <= hi) && (e >= lo || e < ml);
              sr[e >> 5][e & 31] = vis ? sr[e >> 5][e & 31] : 0xff800000u;
            }
          }
        }
        auto sv = [&](int e) { return __uint_as_float(sr[e >> 5][e & 31]); };
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int e = 0; e < BKV; e += 8)
#pragma unroll
          for (int j = 0; j < 4; ++j) m4[j] = max3f(m4[j], sv(e + 2 * j), sv(e + 2 * j + 1));
        const float mt = max3f(m4[0], m4[1], fmaxf(m4[2], m4[3])) * p.scale_log2;
        // running max (log2 units): set on the first tile; raised only when a tile exceeds it by > 2^8
        const bool need = (t == 0) ? true : (mt > m_run + kRescaleLog2);
        if (t > 0 && __any_sync(0xffffffffu, need)) {
          const float m_new = fmaxf(m_run, mt);
          const float alpha = (m_run == -INFINITY) ? 0.f : ex2_approx(m_run - m_new);
          // O must hold every earlier tile: wait for P V of tile J-1 (tile
          // J-2 is complete, as S of this tile was issued after it)
          const bool g2 = mbar_wait(bar(B_PVDONE + x), (J - 1) & 1, wc);
          if (!__all_sync(0xffffffffu, g2)) { ok = false; break; }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < DV / 16; ++c) {
            uint32_t rr[16];
            tmem_ld16(lane_base + o_col + c * 16, rr);
            tc_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * alpha);
            tmem_st16(lane_base + o_col + c * 16, rr);
          }
          l_run *= alpha;
          m_run = m_new;
        } else if (t == 0) {
          m_run = mt;
        }
        const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
        // P = 2^(s * scale - m) as fp16 pairs over the first 32 columns of the
        // buffer; pairs of scores go through one f32x2 FMA and one f32x2 add
        const uint64_t scale2 = pk2(p.scale_log2, p.scale_log2), negm2 = pk2(neg_m, neg_m);
        uint64_t ls2[4] = {pk2(0.f, 0.f), pk2(0.f, 0.f), pk2(0.f, 0.f), pk2(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < BKV / 32; ++c) {  // 32 keys -> 16 packed columns
          uint32_t pk[16];
#pragma unroll
          for (int e2 = 0; e2 < 16; ++e2) {
            const int e = c * 32 + 2 * e2;
            const float2 y = up2(fma2(pk2(sv(e), sv(e + 1)), scale2, negm2));
            const float p0 = ex2_approx(y.x), p1 = ex2_approx(y.y);
            ls2[e2 & 3] = add2(ls2[e2 & 3], pk2(p0, p1));
            pk[e2] = pack_half2(p0, p1);
          }
          tmem_st16(lane_base + s_col + c * 16, pk);
        }
        {
          const float2 a = up2(add2(add2(ls2[0], ls2[1]), add2(ls2[2], ls2[3])));
          l_run += a.x + a.y;
        }
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_PFULL + 2 * x + (J & 1)));
      }
      if (!ok) break;
      // epilogue: O / l -> fp16, once the last two P V of this head completed
      // (waited in order, so that each parity wait is unambiguous)
      bool g4 = true;
      if (U.n_tiles >= 2) g4 = mbar_wait(bar(B_PVDONE + x), (J - 2) & 1, wc);
      g4 = g4 && mbar_wait(bar(B_PVDONE + x), (J - 1) & 1, wc);
      if (!__all_sync(0xffffffffu, g4)) { ok = false; break; }
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.0f / l_run : 0.f;
      __half* orow = p.O + (static_cast<long long>(U.b) * p.Lq + (i - p.q_off)) * p.ldo + h * DV;
#pragma unroll 1
      for (int c = 0; c < DV / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(lane_base + o_col + c * 32, rr);
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
      if (lane == 0) mbar_arrive(bar(B_OEMPTY + x));
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == W_MMA) tmem_dealloc(tmem, Cfg::TMEM_COLS);
}

template <int DV>
hymba_status launch(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& km,
                    const CUtensorMap& vm, const AttnParams& p, int grid, cudaStream_t st) {
  auto kern = attn_tc_kernel<DV>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, AttnCfg<DV>::SMEM) != cudaSuccess)
    return HYMBA_ERR_CUDA;
  if (launch_kernel(false, kern, dim3(grid), dim3(NTHREADS), AttnCfg<DV>::SMEM, st, q, k, v, km, vm, p) != cudaSuccess)
    return HYMBA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? HYMBA_OK : HYMBA_ERR_CUDA;
}

bool make_map3(CUtensorMap* m, const __half* base, int cols, int L, int B, long long ld, int box_rows) {
  const uint64_t dims[3] = {static_cast<uint64_t>(cols), static_cast<uint64_t>(L), static_cast<uint64_t>(B)};
  const uint64_t str[2] = {static_cast<uint64_t>(ld) * 2, static_cast<uint64_t>(ld) * 2 * L};
  const uint32_t box[3] = {64, static_cast<uint32_t>(box_rows), 1};
  return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, base, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

bool attn_tc_supported(int dh, int dv) { return dh == DH && (dv == 64 || dv == 128); }

namespace {

hymba_status attn_tc_impl(int B, int L, int M, int Lq, const __half* Km, const __half* Vm, int Hq, int Hkv, int dh,
                          int dv, int window, const __half* Q, long long ldq, const __half* K, long long ldk,
                          const __half* V, long long ldv, __half* O, long long ldo, int32_t* status, uint64_t wait_ns,
                          int num_sms, cudaStream_t st) {
  if (!attn_tc_supported(dh, dv) || Hq > MAX_HU || Hkv < 1 || Hkv > Hq) return HYMBA_ERR_UNSUPPORTED;
  const bool sep = Km != nullptr;
  if (sep && (M < 1 || M % BKV != 0 || !Vm)) return HYMBA_ERR_UNSUPPORTED;
  auto al = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; };
  if (!al(Q) || !al(K) || !al(V) || !al(O) || ldq % 8 || ldk % 8 || ldv % 8 || ldo % 8) return HYMBA_ERR_INVALID;
  if (sep && (!al(Km) || !al(Vm))) return HYMBA_ERR_INVALID;
  if (Lq < 1) return HYMBA_OK;
  CUtensorMap tq, tk, tv, tkm, tvm;
  if (!make_map3(&tq, Q, Hq * dh, Lq, B, ldq, BQ) || !make_map3(&tk, K, Hkv * dh, Lq, B, ldk, BKV) ||
      !make_map3(&tv, V, Hkv * dv, Lq, B, ldv, BKV))
    return HYMBA_ERR_CUDA;
  if (sep) {
    if (!make_map3(&tkm, Km, Hkv * dh, M, 1, static_cast<long long>(Hkv) * dh, BKV) ||
        !make_map3(&tvm, Vm, Hkv * dv, M, 1, static_cast<long long>(Hkv) * dv, BKV))
      return HYMBA_ERR_CUDA;
  } else {
    tkm = tk;  // never read
    tvm = tv;
  }
  AttnParams p{};
  p.B = B;
  p.L = L;
  p.M = M;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.dv = dv;
  p.window = window;
  p.meta_sep = sep ? 1 : 0;
  p.q_off = L - Lq;
  p.Lq = Lq;
  p.n_qt = (Lq + BQ - 1) / BQ;
  // head units: consecutive heads of one KV group in pairs, a group's odd head alone
  int n_hu = 0;
  for (int h = 0; h < Hq;) {
    const int g = (h * Hkv) / Hq;
    const bool pair = h + 1 < Hq && ((h + 1) * Hkv) / Hq == g;
    p.hA[n_hu] = static_cast<int16_t>(h);
    p.hB[n_hu] = static_cast<int16_t>(pair ? h + 1 : -1);
    ++n_hu;
    h += pair ? 2 : 1;
  }
  p.n_hu = n_hu;
  p.n_units = B * p.n_qt * n_hu;
  p.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(dh));
  p.O = O;
  p.ldo = ldo;
  p.status = status;
  p.wait_ns = wait_ns;
  const int grid = std::min(p.n_units, std::max(1, num_sms));
  return dv == 128 ? launch<128>(tq, tk, tv, tkm, tvm, p, grid, st) : launch<64>(tq, tk, tv, tkm, tvm, p, grid, st);
}

}  // namespace

hymba_status attn_tc(int B, int L, int M, int Hq, int Hkv, int dh, int dv, int window, const __half* Q, long long ldq,
                     const __half* K, long long ldk, const __half* V, long long ldv, __half* O, long long ldo,
                     int32_t* status, uint64_t wait_ns, int num_sms, cudaStream_t st) {
  return attn_tc_impl(B, L, M, L, nullptr, nullptr, Hq, Hkv, dh, dv, window, Q, ldq, K, ldk, V, ldv, O, ldo, status,
                      wait_ns, num_sms, st);
}

hymba_status attn_tc_meta(int B, int T, int M, const __half* Km, const __half* Vm, int Hq, int Hkv, int dh, int dv,
                          int window, const __half* Q, long long ldq, const __half* K, long long ldk, const __half* V,
                          long long ldv, __half* O, long long ldo, int32_t* status, uint64_t wait_ns, int num_sms,
                          cudaStream_t st) {
  return attn_tc_impl(B, M + T, M, T, Km, Vm, Hq, Hkv, dh, dv, window, Q, ldq, K, ldk, V, ldv, O, ldo, status,
                      wait_ns, num_sms, st);
}

}  // namespace hy
