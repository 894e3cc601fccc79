// Selective scan + gate of the SSM branch on the bf16 path, and the
// bounded-wait probe.  The SSM heads are M_ssm of the hybrid-head layer
// ("Hymba: A Hybrid-head Architecture for Small Language Models",
// section 2.1, eq. 3), running in parallel with the attention heads on the
// same input projection.
//
// Recurrence (per batch b, channel c, state n), run literally in time:
//     h_t = exp(delta_t * A) * h_{t-1} + (delta_t * u_t) * B_t
//     y_t = C_t . h_t + D * u_t,   g_t = y_t * silu(z_t),   A = -exp(A_log)
// with delta = softplus(dt W_dt^T + dt_bias) computed here (dt projection
// fused in) or read from a delta buffer (component-test mode).
//
// Work split.  A block owns CH channels of one sequence and walks the whole
// sequence in chunks of SC_T rows.  The warps of a block specialise, like
// the stages of a pipeline, so that the short dependent steps of one role
// overlap the work of the others:
//   delta warps (ND)  per chunk: delta for the block's channels x SC_T rows
//                     (fused mode: mma.sync of the dt tile against W_dt
//                     fragments held in registers or shared memory, then
//                     softplus;
//                     otherwise the delta tile itself) and delta*u, as
//                     (d, d*u) pairs; rows past the end of the sequence get
//                     d = 0, which leaves the state unchanged;
//   scan warps        the recurrence, fully unrolled over the chunk.  TPC
//                     threads share one channel, each holding 16/TPC of its
//                     states in registers for the whole sequence; their
//                     partial C.h are stored per row (two threads and two
//                     channels per thread) or first summed with shuffles;
//   gate warp (1)     y = C.h + D*u (adding the stored partials), g =
//                     y*silu(z) on packed float pairs, eight channels of one row
//                     per lane and one 16-byte store to global memory; its
//                     lane 0 also issues the TMA loads of the chunk's dt (or
//                     delta), u, z and [B|C] tiles into an SC_S-stage ring,
//                     refilling a stage as soon as the gate is done with it
//                     (the gate is the last reader of every stage).
// (delta, delta*u) and C.h pass from role to role through double-buffered
// shared-memory tiles guarded by mbarriers.  TPC is picked on the host from
// the channels per SM.  Every wait is bounded.
#include <type_traits>

#include "scan.cuh"
#include "simt.cuh"

namespace hy {
namespace {

constexpr int SC_N = 16;  // states per channel on this path
constexpr int SC_T = 16;  // time rows per chunk
constexpr int SC_H = 8;   // rows per partial-sum reduction of C.h
constexpr int SC_S = 3;   // TMA pipeline stages
constexpr float kLog2e = 1.4426950408889634f;

// KS = 16-wide k steps of the fused dt projection (0: delta is an input);
// TPC threads share a channel's states; each scan thread runs CPT adjacent
// channels over the same states, so one read of B_t / C_t serves CPT channels.
template <int KS, int TPC, int CH, int CPT>
struct ScanCfg {
  static constexpr int NWS = CH * TPC / (32 * CPT);   // scan warps
  static constexpr int ND = CH >= 64 ? CH / 32 : 1;   // delta warps
  static constexpr int NW = NWS + ND + 1;             // + gate warp
  static constexpr int NT = NW * 32;
  static constexpr int W_DELTA = NWS;                 // first delta warp
  static constexpr int W_GATE = NWS + ND;
  static constexpr int CHW = 32 * CPT / TPC;          // channels per scan warp
  static constexpr int NS = SC_N / TPC;               // states per scan thread
  static constexpr int CHD = CH / ND;                 // channels per delta warp
  static constexpr int NTD = CHD / 8;                 // mma n-tiles per delta warp
  static constexpr int KP = KS * 16;                  // padded dt rank
  static constexpr int X_BYTES = KS > 0 ? SC_T * KP * 2 : SC_T * CH * 4;
  static constexpr int U_BYTES = SC_T * CH * 2;
  static constexpr int BC_BYTES = SC_T * 2 * SC_N * 4;
  // The u tile lands first in its stage.  With 128-byte rows it is loaded
  // with the 128-byte swizzle (16-byte chunk c of row r stored at chunk
  // c ^ (r % 8)), so that the delta warps' column reads, eight rows at a
  // time, fall in different banks; that needs 1024-byte aligned stages.
  static constexpr bool SWZ_U = CH * 2 == 128;
  static constexpr int STAGE_ALIGN = SWZ_U ? 1024 : 128;
  static constexpr int OFF_U = 0;
  static constexpr int OFF_X = U_BYTES;
  static constexpr int OFF_Z = OFF_X + X_BYTES;
  static constexpr int OFF_BC = OFF_Z + U_BYTES;
  static constexpr int TX_BYTES = OFF_BC + BC_BYTES;  // bytes landing per stage
  static constexpr int STAGE = (TX_BYTES + STAGE_ALIGN - 1) / STAGE_ALIGN * STAGE_ALIGN;
  // row strides of the (d, d*u) and C.h tiles, padded so that the delta
  // warps' stores (eight rows x four column pairs) and the scan warps' row
  // stores (rows SC_H / TPC apart) hit distinct banks
  static constexpr int DU_STR = CH + 8;               // float2 per row of a (d, d*u) tile
  static constexpr int DU_BYTES = SC_T * DU_STR * 8;
  // C.h leaves the scan warps either as TPC partials per row, added by the
  // gate warp (two threads and two channels per thread), or summed across
  // the TPC threads by shuffles (the other layouts, where the gate warp's
  // share of the work is larger); measured both ways
  static constexpr bool PARTIALS = TPC == 2 && CPT == 2;
  static constexpr int NP = PARTIALS ? TPC : 1;        // partials stored per row
  static constexpr int RPL = SC_H / TPC;              // rows a thread stores per SC_H rows (shuffled sums)
  static constexpr int Y_STR = CH + 4;                // floats per (row, partial) of a C.h tile
  static constexpr int Y_BYTES = SC_T * NP * Y_STR * 4;  // C.h [SC_T][NP][Y_STR] fp32
  // W_dt mma fragments: in registers when three blocks of NT threads leave
  // 128 registers a thread, otherwise in shared memory
  static constexpr bool W_REG = NT <= 160;
  static constexpr int W_BYTES = KS > 0 && !W_REG ? (CH / 8) * KS * 32 * 8 : 0;
  static constexpr int OFF_DU = SC_S * STAGE;
  static constexpr int OFF_Y = OFF_DU + 2 * DU_BYTES;
  static constexpr int OFF_W = OFF_Y + 2 * Y_BYTES;
  static constexpr int OFF_BAR = OFF_W + W_BYTES;
  static constexpr int N_BAR = SC_S + 8;
  static constexpr int SMEM = STAGE_ALIGN + OFF_BAR + N_BAR * 8;
  static_assert(NWS >= 1 && CHD % 8 == 0 && CH % 8 == 0 && SC_H % TPC == 0 && SC_T % SC_H == 0 && (CPT == 1 || CPT == 2) &&
                    CH % CHW == 0,
                "scan block shape");
};

struct ScanArgs {
  int L, di, R;
  const __nv_bfloat16* W_dt;  // [di, R] (fused mode)
  const float* dt_bias;       // [di]    (fused mode)
  const float* A_log;
  const float* D;
  __half* g;
  const float* h0;
  long long h0_bs;  // elements between the initial states of two sequences (0: one shared state)
  float* h_out;
  int32_t* status;
  uint64_t wait_ns;
};

HY_DEV void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// softplus(v) = max(v, 0) + log1p(e) with e = e^-|v| in (0, 1], and
// log1p(e) = e q(e), q a degree-7 polynomial fitted to log1p(e)/e on [0, 1]
// (least squares on Chebyshev nodes, reweighted toward equal relative error):
// relative error of e q(e) below 4e-7 in float32 arithmetic.  One SFU
// operation and no branch.
HY_DEV float softplus_scan(float v) {
  const float e = ex2_approx(-fabsf(v) * kLog2e);
  float q = -0.008539227768778801f;
  q = fmaf(q, e, 0.044089701026678085f);
  q = fmaf(q, e, -0.10768181085586548f);
  q = fmaf(q, e, 0.1774524748325348f);
  q = fmaf(q, e, -0.2449546456336975f);
  q = fmaf(q, e, 0.33275479078292847f);
  q = fmaf(q, e, -0.4999740421772003f);
  q = fmaf(q, e, 0.9999998211860657f);
  return fmaxf(v, 0.f) + e * q;
}

// (y0 + D0 u0, y1 + D1 u1) gated by (z0, z1) on packed float pairs:
// y * silu(z) = y * z / (1 + 2^(-z log2 e))
HY_DEV uint32_t gate2(uint64_t y, uint64_t Dp, uint64_t u, uint64_t z) {
  const uint64_t yv = fma2(Dp, u, y);
  const float2 t = up2(mul2(z, pk2(-kLog2e, -kLog2e)));
  const float2 dd = up2(add2(pk2(ex2_approx(t.x), ex2_approx(t.y)), pk2(1.0f, 1.0f)));
  const float2 o = up2(mul2(mul2(yv, z), pk2(rcp_approx(dd.x), rcp_approx(dd.y))));
  return pack_half2(o.x, o.y);
}

template <int KS, int TPC, int CH, int CPT>
__global__ void __launch_bounds__(ScanCfg<KS, TPC, CH, CPT>::NT, 3)
    scan_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmU,
                const __grid_constant__ CUtensorMap tmZ, const __grid_constant__ CUtensorMap tmBC,
                const ScanArgs a) {
  using Cfg = ScanCfg<KS, TPC, CH, CPT>;
  constexpr int N = SC_N;
  pdl_wait();
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem<Cfg::STAGE_ALIGN>(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
  // full[SC_S] | du_full[2] | du_empty[2] | y_full[2] | y_empty[2]
  auto full = [&](int s) { return smem_u32(&bars[s]); };
  auto du_full = [&](int i) { return smem_u32(&bars[SC_S + i]); };
  auto du_empty = [&](int i) { return smem_u32(&bars[SC_S + 2 + i]); };
  auto y_full = [&](int i) { return smem_u32(&bars[SC_S + 4 + i]); };
  auto y_empty = [&](int i) { return smem_u32(&bars[SC_S + 6 + i]); };
  __shared__ int abort_flag;
  __shared__ int n_issued;  // TMA chunks issued (read after the final barrier)

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int c0 = blockIdx.x * CH;
  const int b = blockIdx.y;
  const int L = a.L, di = a.di;
  const long long row0 = static_cast<long long>(b) * L;
  const int n_chunks = (L + SC_T - 1) / SC_T;

  if (tid == 0) {
    for (int s = 0; s < SC_S; ++s) mbar_init(full(s), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(du_full(i), Cfg::ND * 32);
      mbar_init(du_empty(i), Cfg::NWS * 32);
      mbar_init(y_full(i), Cfg::NWS * 32);
      mbar_init(y_empty(i), 32);
    }
    abort_flag = 0;
    n_issued = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtl wc{&abort_flag, a.status, a.wait_ns};
  auto stage = [&](int k) { return smem + (k % SC_S) * Cfg::STAGE; };
  auto du_tile = [&](int k) { return reinterpret_cast<float2*>(smem + Cfg::OFF_DU + (k & 1) * Cfg::DU_BYTES); };
  auto y_tile = [&](int k) { return reinterpret_cast<float*>(smem + Cfg::OFF_Y + (k & 1) * Cfg::Y_BYTES); };
  // element index of u[row][col] in a stage's u tile
  auto u_at = [](int row, int col) {
    return Cfg::SWZ_U ? row * CH + ((((col >> 3) ^ (row & 7)) << 3) | (col & 7)) : row * CH + col;
  };

  if (warp < Cfg::NWS) {
    // ------------------------------------------------------------ scan warps
    constexpr int NS = Cfg::NS;
    const int sub = lane % TPC;
    const int chl = warp * Cfg::CHW + (lane / TPC) * CPT;  // first of this thread's CPT channels
    const int c = c0 + chl;
    uint64_t A2[CPT][NS / 2], h2[CPT][NS / 2];
#pragma unroll
    for (int j = 0; j < CPT; ++j)
#pragma unroll
      for (int p = 0; p < NS / 2; ++p) {
        const int s0 = (c + j) * N + sub * NS + 2 * p;
        A2[j][p] = pk2(-__expf(a.A_log[s0]) * kLog2e, -__expf(a.A_log[s0 + 1]) * kLog2e);
        const long long hb = static_cast<long long>(b) * a.h0_bs + static_cast<long long>(c + j) * N + sub * NS + 2 * p;
        h2[j][p] = a.h0 ? pk2(a.h0[hb], a.h0[hb + 1]) : pk2(0.f, 0.f);
      }
    bool ok = true;
    for (int k = 0; k < n_chunks; ++k) {
      const int i = k & 1;
      ok = mbar_wait(du_full(i), (k >> 1) & 1, wc) && mbar_wait(y_empty(i), ((k >> 1) & 1) ^ 1, wc);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      const float2* du_p = du_tile(k) + chl;
      const float* sBC = reinterpret_cast<const float*>(stage(k) + Cfg::OFF_BC);
      float* y_p = y_tile(k) + chl;
      // C.h of SC_H rows stays in registers and is stored after them (no
      // store inside the row loop, so the loads of later rows can be issued
      // early): one partial per thread, or the TPC partials summed by a
      // transposing butterfly of shuffles
#pragma unroll
      for (int hh = 0; hh < SC_T / SC_H; ++hh) {
        float yr[CPT][SC_H];
#pragma unroll
        for (int tr = 0; tr < SC_H; ++tr) {
          const int t = hh * SC_H + tr;
          // (delta, delta*u) of the thread's channels: one 8- or 16-byte load
          float dl[CPT], dul[CPT];
          if constexpr (CPT == 2) {
            const float4 q = *reinterpret_cast<const float4*>(du_p + t * Cfg::DU_STR);
            dl[0] = q.x;
            dul[0] = q.y;
            dl[1] = q.z;
            dul[1] = q.w;
          } else {
            const float2 q = du_p[t * Cfg::DU_STR];
            dl[0] = q.x;
            dul[0] = q.y;
          }
          const float4* Bp = reinterpret_cast<const float4*>(sBC + t * 2 * N + sub * NS);
          const float4* Cp = reinterpret_cast<const float4*>(sBC + t * 2 * N + N + sub * NS);
          // one packed accumulator per channel: a single fma2 per state pair
          // (two accumulators cost an extra add2 per channel and row)
          uint64_t y0[CPT];
#pragma unroll
          for (int j = 0; j < CPT; ++j) y0[j] = pk2(0.f, 0.f);
#pragma unroll
          for (int qq = 0; qq < NS / 4; ++qq) {
            const float4 bb = Bp[qq], cc = Cp[qq];
#pragma unroll
            for (int p2 = 0; p2 < 2; ++p2) {
              const int p = qq * 2 + p2;
              const uint64_t bp = p2 == 0 ? pk2(bb.x, bb.y) : pk2(bb.z, bb.w);
              const uint64_t cp = p2 == 0 ? pk2(cc.x, cc.y) : pk2(cc.z, cc.w);
#pragma unroll
              for (int j = 0; j < CPT; ++j) {
                const float2 ea = up2(mul2(pk2(dl[j], dl[j]), A2[j][p]));
                const uint64_t av = pk2(ex2_approx(ea.x), ex2_approx(ea.y));
                h2[j][p] = fma2(av, h2[j][p], mul2(pk2(dul[j], dul[j]), bp));
                y0[j] = fma2(cp, h2[j][p], y0[j]);
              }
            }
          }
#pragma unroll
          for (int j = 0; j < CPT; ++j) {
            const float2 ys = up2(y0[j]);
            yr[j][tr] = ys.x + ys.y;
          }
        }
        if constexpr (Cfg::PARTIALS) {
#pragma unroll
          for (int r = 0; r < SC_H; ++r)
            *reinterpret_cast<float2*>(y_p + ((hh * SC_H + r) * TPC + sub) * Cfg::Y_STR) =
                make_float2(yr[0][r], yr[1][r]);
        } else {
          // lane `sub` ends with the totals of rows sub*RPL .. sub*RPL + RPL - 1
          // of these SC_H rows
#pragma unroll
          for (int o = TPC / 2, m = SC_H; o >= 1; o >>= 1, m >>= 1) {
            const bool upper = (sub & o) != 0;
#pragma unroll
            for (int j = 0; j < CPT; ++j)
#pragma unroll
              for (int r = 0; r < m / 2; ++r) {
                const float keep = upper ? yr[j][m / 2 + r] : yr[j][r];
                const float send = upper ? yr[j][r] : yr[j][m / 2 + r];
                yr[j][r] = keep + __shfl_xor_sync(0xffffffffu, send, o);
              }
          }
#pragma unroll
          for (int r = 0; r < Cfg::RPL; ++r) {
            const int row = hh * SC_H + sub * Cfg::RPL + r;
            if constexpr (CPT == 2)
              *reinterpret_cast<float2*>(y_p + row * Cfg::Y_STR) = make_float2(yr[0][r], yr[1][r]);
            else
              y_p[row * Cfg::Y_STR] = yr[0][r];
          }
        }
      }
      mbar_arrive(du_empty(i));
      mbar_arrive(y_full(i));
    }
    if (ok && a.h_out) {
#pragma unroll
      for (int j = 0; j < CPT; ++j)
#pragma unroll
        for (int p = 0; p < NS / 2; ++p) {
          const float2 hv = up2(h2[j][p]);
          const long long hb = (static_cast<long long>(b) * di + c + j) * N + sub * NS + 2 * p;
          a.h_out[hb] = hv.x;
          a.h_out[hb + 1] = hv.y;
        }
    }
  } else if (warp < Cfg::W_GATE) {
    // ------------------------------------------------------------ delta warps
    const int dw = warp - Cfg::W_DELTA;
    const int grp = lane >> 2, tig = lane & 3;
    const int dc0 = dw * Cfg::CHD;  // first channel of this warp within the block
    constexpr int NTD = Cfg::NTD;
    // W_dt as mma B fragments for the whole sequence: wreg[n-tile][k-step],
    // or [n-tile][k-step][lane] in shared memory
    constexpr bool WR = Cfg::W_REG;
    uint2 wreg[WR ? NTD : 1][WR && KS > 0 ? KS : 1];
    uint2* sW = reinterpret_cast<uint2*>(smem + Cfg::OFF_W) + dw * NTD * KS * 32 + lane;
    float bias_c[NTD][2];
    if constexpr (KS > 0) {
#pragma unroll
      for (int nt = 0; nt < NTD; ++nt) {
        const int ch = c0 + dc0 + nt * 8 + grp;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          uint32_t f[2];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int r0 = kk * 16 + hh * 8 + tig * 2;
            const float v0 = r0 < a.R ? __bfloat162float(a.W_dt[static_cast<long long>(ch) * a.R + r0]) : 0.f;
            const float v1 =
                r0 + 1 < a.R ? __bfloat162float(a.W_dt[static_cast<long long>(ch) * a.R + r0 + 1]) : 0.f;
            f[hh] = pack_half2(v0, v1);
          }
          if constexpr (WR)
            wreg[nt][kk] = make_uint2(f[0], f[1]);
          else
            sW[(nt * KS + kk) * 32] = make_uint2(f[0], f[1]);
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) bias_c[nt][e] = a.dt_bias[c0 + dc0 + nt * 8 + tig * 2 + e];
      }
      __syncwarp();
    }
    for (int k = 0; k < n_chunks; ++k) {
      const int i = k & 1;
      bool ok = mbar_wait(full(k % SC_S), (k / SC_S) & 1, wc) && mbar_wait(du_empty(i), ((k >> 1) & 1) ^ 1, wc);
      if (!__all_sync(0xffffffffu, ok)) break;
      const uint8_t* st = stage(k);
      const __half* sU = reinterpret_cast<const __half*>(st + Cfg::OFF_U);
      float2* du = du_tile(k);
      const int nt_rows = min(SC_T, L - k * SC_T);
      if constexpr (KS > 0) {
        float acc[NTD][4];
#pragma unroll
        for (int nt = 0; nt < NTD; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
        const uint32_t abase = smem_u32(st + Cfg::OFF_X) + ((lane & 15) * Cfg::KP + (lane >> 4) * 8) * 2;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          uint32_t af[4];
          ldsm_x4(abase + kk * 32, af);
#pragma unroll
          for (int nt = 0; nt < NTD; ++nt) {
            const uint2 bw = WR ? wreg[WR ? nt : 0][WR ? kk : 0] : sW[(nt * KS + kk) * 32];
            mma_16816_f16(acc[nt], af, bw.x, bw.y);
          }
        }
#pragma unroll
        for (int nt = 0; nt < NTD; ++nt) {
          const int col = dc0 + nt * 8 + tig * 2;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int row = grp + hh * 8;
            const float2 uv = __half22float2(*reinterpret_cast<const __half2*>(sU + u_at(row, col)));
            float d0 = softplus_scan(acc[nt][2 * hh] + bias_c[nt][0]);
            float d1 = softplus_scan(acc[nt][2 * hh + 1] + bias_c[nt][1]);
            if (row >= nt_rows) d0 = d1 = 0.f;
            *reinterpret_cast<float4*>(du + row * Cfg::DU_STR + col) = make_float4(d0, d0 * uv.x, d1, d1 * uv.y);
          }
        }
      } else {
        const float* sDl = reinterpret_cast<const float*>(st + Cfg::OFF_X);
        for (int idx = lane; idx < SC_T * Cfg::CHD; idx += 32) {
          const int row = idx / Cfg::CHD, col = dc0 + idx % Cfg::CHD;
          const float d = row < nt_rows ? sDl[row * CH + col] : 0.f;
          du[row * Cfg::DU_STR + col] = make_float2(d, d * __half2float(sU[u_at(row, col)]));
        }
      }
      mbar_arrive(du_full(i));
    }
  } else {
    // ------------------------------------------------------------ gate warp (+ TMA)
    constexpr int GPR = CH / 8;             // 8-channel groups per row
    constexpr int ITEMS = SC_T * GPR;       // (row, group) items per chunk
    const int gq = lane % GPR;
    uint64_t Dg[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) Dg[e] = pk2(a.D[c0 + gq * 8 + 2 * e], a.D[c0 + gq * 8 + 2 * e + 1]);
    auto issue = [&](int k) {
      uint8_t* st = stage(k);
      const uint32_t bar = full(k % SC_S);
      const int r = static_cast<int>(row0) + k * SC_T;
      mbar_arrive_expect_tx(bar, Cfg::TX_BYTES);
      tma_load_2d(smem_u32(st + Cfg::OFF_X), &tmX, bar, KS > 0 ? 0 : c0, r);
      tma_load_2d(smem_u32(st + Cfg::OFF_U), &tmU, bar, c0, r);
      tma_load_2d(smem_u32(st + Cfg::OFF_Z), &tmZ, bar, c0, r);
      tma_load_2d(smem_u32(st + Cfg::OFF_BC), &tmBC, bar, 0, r);
    };
    int issued = 0;
    if (lane == 0)
      for (; issued < min(SC_S, n_chunks); ++issued) issue(issued);
    for (int k = 0; k < n_chunks; ++k) {
      const int i = k & 1;
      const bool ok = mbar_wait(y_full(i), (k >> 1) & 1, wc);
      if (!__all_sync(0xffffffffu, ok)) break;
      const uint8_t* st = stage(k);
      const __half* sU = reinterpret_cast<const __half*>(st + Cfg::OFF_U);
      const __half* sZ = reinterpret_cast<const __half*>(st + Cfg::OFF_Z);
      const float* yt = y_tile(k);
      const int nt_rows = min(SC_T, L - k * SC_T);
      for (int it = lane; it < ITEMS; it += 32) {
        const int row = it / GPR;
        if (row >= nt_rows) break;
        const float* yrow = yt + row * Cfg::NP * Cfg::Y_STR + gq * 8;
        float4 ya = *reinterpret_cast<const float4*>(yrow);
        float4 yb = *reinterpret_cast<const float4*>(yrow + 4);
        if constexpr (Cfg::PARTIALS) {  // C.h = partial 0 + partial 1
          const float4 pa = *reinterpret_cast<const float4*>(yrow + Cfg::Y_STR);
          const float4 pb = *reinterpret_cast<const float4*>(yrow + Cfg::Y_STR + 4);
          ya = make_float4(ya.x + pa.x, ya.y + pa.y, ya.z + pa.z, ya.w + pa.w);
          yb = make_float4(yb.x + pb.x, yb.y + pb.y, yb.z + pb.z, yb.w + pb.w);
        }
        const uint64_t y[4] = {pk2(ya.x, ya.y), pk2(ya.z, ya.w), pk2(yb.x, yb.y), pk2(yb.z, yb.w)};
        const uint4 uv = *reinterpret_cast<const uint4*>(sU + u_at(row, gq * 8));
        const uint4 zv = *reinterpret_cast<const uint4*>(sZ + row * CH + gq * 8);
        const __half2* uh = reinterpret_cast<const __half2*>(&uv);
        const __half2* zh = reinterpret_cast<const __half2*>(&zv);
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 uf = __half22float2(uh[e]), zf = __half22float2(zh[e]);
          o[e] = gate2(y[e], Dg[e], pk2(uf.x, uf.y), pk2(zf.x, zf.y));
        }
        *reinterpret_cast<uint4*>(a.g + (row0 + k * SC_T + row) * di + c0 + gq * 8) =
            make_uint4(o[0], o[1], o[2], o[3]);
      }
      __syncwarp();
      mbar_arrive(y_empty(i));
      // the gate is the last reader of stage k: refill it with chunk k + SC_S
      if (lane == 0 && issued < n_chunks) issue(issued++);
    }
    if (lane == 0) n_issued = issued;
  }
  // After a bounded wait gave up, loads may still be in flight: let the last
  // stages land before the block exits (no-ops otherwise).
  __syncthreads();
  if (warp == Cfg::W_GATE && lane == 0) {
    const int last = n_issued;
    for (int j = max(0, last - SC_S); j < last; ++j) mbar_wait_drain(full(j % SC_S), (j / SC_S) & 1, 1000000);
  }
}

__global__ void wait_probe_kernel(uint64_t limit_ns, int32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtl wc{&abort_flag, status, limit_ns};
    mbar_wait(smem_u32(&bar), 0, wc);  // nothing arrives: gives up after limit_ns
  }
  __syncthreads();
}

bool map2(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, long long cols, long long rows,
          long long ld, int box_c, int box_r, bool swizzle128 = false) {
  const uint64_t dims[2] = {static_cast<uint64_t>(cols), static_cast<uint64_t>(rows)};
  const uint64_t str[1] = {static_cast<uint64_t>(ld) * esize};
  const uint32_t box[2] = {static_cast<uint32_t>(box_c), static_cast<uint32_t>(box_r)};
  return encode_tmap(m, dt, 2, base, dims, str, box, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
}

template <int KS, int TPC, int CH, int CPT>
hymba_status launch_scan(int B, int L, int di, const CUtensorMap& mX, const __half* u, long long ld_u,
                         const __half* z, long long ld_z, const float* BC, const ScanArgs& args, cudaStream_t st) {
  using Cfg = ScanCfg<KS, TPC, CH, CPT>;
  const long long rows = static_cast<long long>(B) * L;
  CUtensorMap mU, mZ, mBC;
  if (!map2(&mU, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, u, di, rows, ld_u, CH, SC_T, Cfg::SWZ_U) ||
      !map2(&mZ, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, z, di, rows, ld_z, CH, SC_T) ||
      !map2(&mBC, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, BC, 2 * SC_N, rows, 2 * SC_N, 2 * SC_N, SC_T))
    return HYMBA_ERR_CUDA;
  auto kern = scan_kernel<KS, TPC, CH, CPT>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM) != cudaSuccess)
    return HYMBA_ERR_CUDA;
  dim3 grid(di / CH, B);
  if (launch_kernel(false, kern, grid, dim3(Cfg::NT), Cfg::SMEM, st, mX, mU, mZ, mBC, args) != cudaSuccess)
    return HYMBA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? HYMBA_OK : HYMBA_ERR_CUDA;
}

// Threads per channel and channels per thread, from the channels each SM
// gets.  Each thread walks its chains (states x channels) through the whole
// sequence; fewer chains per thread mean more warps to hide the latency of
// each step, while two channels per thread halve the shared-memory reads of
// B_t / C_t.  Measured on B300 at d_inner 3200, L 8320 (scan alone):
//   ~43 channels/SM:  (4,1) 0.49 ms, (2,1) 0.59, (4,2) 0.62, (1,1) 0.69, (2,2) 0.72
//   ~86 channels/SM:  (2,1) 0.89 ms, (4,2) 0.92, (4,1) 1.05, (1,1) 1.12, (2,2) 1.14
//   ~173 channels/SM: (2,2) 1.28 ms, (1,1) 1.28, (2,1) 1.30, (4,2) 1.33, (4,1) 1.80
struct ScanLayout {
  int tpc, cpt;
};

ScanLayout pick_layout(int B, int di, int num_sms) {
  const long long per_sm = static_cast<long long>(B) * di / num_sms;
  if (per_sm >= 128) return {2, 2};
  if (per_sm >= 64) return {2, 1};
  return {4, 1};
}

// Channels per block: 64 (one wave of 2-3 blocks per SM at the 1.5B
// shapes), 16 at four threads per channel so that a small batch still
// spreads over the SMs.
int block_channels(ScanLayout lo) { return lo.tpc == 4 && lo.cpt == 1 ? 16 : 64; }

template <int KS>
hymba_status launch_layout(ScanLayout lo, int B, int L, int di, const CUtensorMap& mX, const __half* u,
                           long long ld_u, const __half* z, long long ld_z, const float* BC, const ScanArgs& args,
                           cudaStream_t st) {
  if (lo.tpc == 1 && lo.cpt == 1) return launch_scan<KS, 1, 64, 1>(B, L, di, mX, u, ld_u, z, ld_z, BC, args, st);
  if (lo.tpc == 2 && lo.cpt == 1) return launch_scan<KS, 2, 64, 1>(B, L, di, mX, u, ld_u, z, ld_z, BC, args, st);
  if (lo.tpc == 2 && lo.cpt == 2) return launch_scan<KS, 2, 64, 2>(B, L, di, mX, u, ld_u, z, ld_z, BC, args, st);
  if (lo.tpc == 4 && lo.cpt == 1) return launch_scan<KS, 4, 16, 1>(B, L, di, mX, u, ld_u, z, ld_z, BC, args, st);
  if (lo.tpc == 4 && lo.cpt == 2) return launch_scan<KS, 4, 64, 2>(B, L, di, mX, u, ld_u, z, ld_z, BC, args, st);
  return HYMBA_ERR_UNSUPPORTED;
}

hymba_status launch_fused(int KS, ScanLayout lo, int B, int L, int di, const CUtensorMap& mX, const __half* u,
                          long long ld_u, const __half* z, long long ld_z, const float* BC, const ScanArgs& args,
                          cudaStream_t st) {
  switch (KS) {
    case 1: return launch_layout<1>(lo, B, L, di, mX, u, ld_u, z, ld_z, BC, args, st);
    case 2: return launch_layout<2>(lo, B, L, di, mX, u, ld_u, z, ld_z, BC, args, st);
    case 3: return launch_layout<3>(lo, B, L, di, mX, u, ld_u, z, ld_z, BC, args, st);
    case 4: return launch_layout<4>(lo, B, L, di, mX, u, ld_u, z, ld_z, BC, args, st);
    case 5: return launch_layout<5>(lo, B, L, di, mX, u, ld_u, z, ld_z, BC, args, st);
    case 6: return launch_layout<6>(lo, B, L, di, mX, u, ld_u, z, ld_z, BC, args, st);
    case 7: return launch_layout<7>(lo, B, L, di, mX, u, ld_u, z, ld_z, BC, args, st);
    case 8: return launch_layout<8>(lo, B, L, di, mX, u, ld_u, z, ld_z, BC, args, st);
    default: return HYMBA_ERR_UNSUPPORTED;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// tpc == 0: both chosen here; otherwise cpt 0 means one channel per thread.
// {-1, -1} for a combination that has no kernel.
ScanLayout resolve_layout(int tpc, int cpt, int B, int di) {
  ScanLayout lo{tpc, cpt == 0 ? 1 : cpt};
  if (tpc == 0) {
    int dev = 0, n = kNumSMsHint;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    lo = pick_layout(B, di, n > 0 ? n : kNumSMsHint);
  }
  const bool known = lo.tpc == 1 ? lo.cpt == 1 : (lo.tpc == 2 || lo.tpc == 4) && (lo.cpt == 1 || lo.cpt == 2);
  if (!known) return {-1, -1};
  if (di % block_channels(lo) != 0) lo = {4, 1};  // 16-channel blocks fit any di % 16 == 0
  return lo;
}

}  // namespace

bool scan_fused_supported(int di, int N, int R) { return di % 16 == 0 && N == SC_N && R >= 1 && R <= 128; }

hymba_status scan_f16(int B, int L, int di, int N, const __half* u, long long ld_u, const __half* z,
                      long long ld_z, const float* delta, const float* BC, const float* A_log, const float* D,
                      __half* g, const float* h0, float* h_out, int32_t* status, uint64_t wait_ns, int tpc,
                      int cpt, cudaStream_t st) {
  const bool tma_ok = di % 16 == 0 && ld_u % 8 == 0 && ld_z % 8 == 0 && aligned16(u) && aligned16(z) &&
                      aligned16(delta) && aligned16(BC) && aligned16(g);
  if (tma_ok && N == SC_N) {
    const ScanLayout lo = resolve_layout(tpc, cpt, B, di);
    if (lo.tpc < 0) return HYMBA_ERR_INVALID;
    CUtensorMap mX;
    if (!map2(&mX, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, delta, di, static_cast<long long>(B) * L, di,
              block_channels(lo), SC_T))
      return HYMBA_ERR_CUDA;
    ScanArgs args{L, di, 0, nullptr, nullptr, A_log, D, g, h0, static_cast<long long>(di) * N, h_out, status, wait_ns};
    return launch_layout<0>(lo, B, L, di, mX, u, ld_u, z, ld_z, BC, args, st);
  }
  return scan_simt<__half>(B, L, di, N, u, ld_u, z, ld_z, delta, di, BC, BC + N, 2 * N, A_log, D, g, di, h0, h_out,
                           st);
}

hymba_status scan_fused_f16(int B, int L, int di, int N, int R, const __half* u, long long ld_u, const __half* z,
                            long long ld_z, const __half* dtr, long long ld_dtr, const __nv_bfloat16* W_dt,
                            const float* dt_bias, const float* BC, const float* A_log, const float* D, __half* g,
                            const float* h0, float* h_out, int32_t* status, uint64_t wait_ns, int tpc,
                            int cpt, cudaStream_t st, bool h0_shared) {
  if (!scan_fused_supported(di, N, R)) return HYMBA_ERR_UNSUPPORTED;
  if (ld_u % 8 || ld_z % 8 || ld_dtr % 8 || !aligned16(u) || !aligned16(z) || !aligned16(dtr) || !aligned16(BC) ||
      !aligned16(g))
    return HYMBA_ERR_INVALID;
  const ScanLayout lo = resolve_layout(tpc, cpt, B, di);
  if (lo.tpc < 0) return HYMBA_ERR_INVALID;
  const int KS = (R + 15) / 16;
  CUtensorMap mX;
  if (!map2(&mX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, dtr, R, static_cast<long long>(B) * L, ld_dtr, KS * 16, SC_T))
    return HYMBA_ERR_CUDA;
  ScanArgs args{L, di, R, W_dt, dt_bias, A_log, D, g, h0, h0_shared ? 0LL : static_cast<long long>(di) * N, h_out,
                status, wait_ns};
  return launch_fused(KS, lo, B, L, di, mX, u, ld_u, z, ld_z, BC, args, st);
}

hymba_status wait_timeout_probe(uint32_t limit_us, int32_t* status, cudaStream_t st) {
  wait_probe_kernel<<<1, 32, 0, st>>>(static_cast<uint64_t>(limit_us) * 1000ull, status);
  return cudaGetLastError() == cudaSuccess ? HYMBA_OK : HYMBA_ERR_CUDA;
}

}  // namespace hy
