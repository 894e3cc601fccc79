// Persistent warp-specialised tcgen05 GEMM for sm_103a: the layer's dense
// projections -- the shared input projection and W_out of eq. 3
// ("Hymba: A Hybrid-head Architecture for Small Language Models",
// section 2.1) and the SSM branch's x_proj -- plus the residual block's MLP.
//
//   warp 0      TMA producer: 128x64 A tile + BNx64 B tile per stage (128-byte
//               swizzle), completion counted on the stage's "full" mbarrier.
//   warp 1      allocates TMEM; one thread issues tcgen05.mma (M=128, N=BN,
//               K=16, fp32 accumulate) into one of two TMEM accumulators and
//               commits stage releases / accumulator-ready arrivals.
//   warps 2..5  epilogue: tcgen05.ld of the accumulator rows they own (TMEM
//               lanes 32*(warp%4) ..), fused epilogue, direct global stores;
//               then release the accumulator so the next tile's MMAs, which
//               overlap this epilogue, can reuse it.  With cvt_b (a bf16
//               weight matrix against fp16 activations) these warps first
//               convert each B stage of the tile to fp16 in place, in shared
//               memory, and the MMA waits for that instead of the TMA: the
//               weights are read from HBM once and never copied.
//
// Tiles are visited in row-major tile order (N fastest) by a static
// round-robin over CTAs, so the CTAs resident at one time share a few A
// row-blocks and the weight matrix stays in L2.  Every wait is bounded.
//
// CTA pairs (PAIR, many row blocks): a 2-CTA cluster computes a 256 x BN
// tile with tcgen05.mma.cta_group::2, issued by the even CTA.  Each CTA
// loads its own 128-row A block and its own half (BN/2 rows) of the B block
// with plain TMA loads into its own shared memory, so a CTA pulls 128 + BN/2
// operand rows per k-step from L2 instead of 128 + BN: at the large tiles the
// single-CTA kernel is bound by L2-to-SM bandwidth (about 135 GB/s per SM
// measured), which this halves for B.  The odd CTA's loads count their bytes
// directly on the even CTA's stage barrier (.cta_group::2 tensor loads), whose
// producer expects both CTAs' bytes; the even CTA's commits release the stage
// and signal the accumulator in both CTAs; both CTAs' epilogues release the
// accumulator on the even CTA's barrier.  No load is multicast.
#include "gemm_tc.cuh"

#include <atomic>

namespace hy {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
// widest tile run as CTA pairs (each CTA holds a 128 x BN accumulator pair in
// its tensor memory, 2 BN columns)
constexpr int kPairMaxBN = 256;
constexpr int A_BYTES = BM * BK * 2;

// KC 64-column chunks of K per pipeline stage: with KC = 2 one 3-D tensor
// load ([chunk][row][64]) brings both chunks of A and one both of B, halving
// the copies a stage needs (one issuing thread sustains about one tensor copy
// per 170-220 ns, longer than the MMAs of a 64-wide k-step at BN <= 160).
// STG: bytes of the epilogue warps' store-staging tiles (see store_rows_*).
template <int BN, bool PAIR = false, int KC = 1, int STG = 0>
struct GemmCfg {
  static constexpr int B_CHUNK = (PAIR ? BN / 2 : BN) * BK * 2;  // this CTA's B rows, one chunk
  static constexpr int A_STAGE = KC * A_BYTES;
  static constexpr int B_BYTES = KC * B_CHUNK;                    // this CTA's B rows, one stage
  static constexpr int STAGE = A_STAGE + B_BYTES;
  static constexpr int BUDGET = 220 * 1024 - 2048 - STG;
  static constexpr int S0 = BUDGET / STAGE;
  static constexpr int STAGES = S0 > 8 ? 8 : S0;
  static constexpr uint32_t TMEM_COLS = (2 * BN <= 32) ? 32 : (2 * BN <= 64) ? 64 : (2 * BN <= 128) ? 128
                                        : (2 * BN <= 256) ? 256 : 512;
  static constexpr int OFF_STG = STAGES * STAGE + 512;
  static constexpr int SMEM = 1024 + OFF_STG + STG;
};

// Row-per-thread results stored through a per-warp shared-memory tile: each
// lane writes its row's 32 values, then the warp stores whole 64- or 128-byte
// row pieces, several rows per instruction, instead of 32 rows' 16-byte
// pieces per instruction.  Row strides padded by 16 bytes against bank
// conflicts.
constexpr int STG_F16_STR = 32 * 2 + 16, STG_F32_STR = 32 * 4 + 16;
template <int EPI>
constexpr int epi_stg_bytes() {
  return EPI == 0 || EPI == 6 ? 4 * 32 * STG_F16_STR : EPI == 3 ? 4 * 32 * STG_F32_STR : 0;  // EPI_F16, EPI_GEGLU, EPI_F32
}

// fp16 [32 rows][32 columns]: lane l holds row row0 + l; `valid` (a multiple
// of 8) leading columns are inside N; rows at or past M are not stored
HY_DEV void store_rows_f16(uint8_t* stg, __half* C, long long ldc, int row0, int M, int col, int valid,
                           const float (&v)[32], int lane) {
  uint8_t* my = stg + lane * STG_F16_STR;
#pragma unroll
  for (int g = 0; g < 4; ++g)
    *reinterpret_cast<uint4*>(my + 16 * g) =
        make_uint4(pack_half2(v[8 * g], v[8 * g + 1]), pack_half2(v[8 * g + 2], v[8 * g + 3]),
                   pack_half2(v[8 * g + 4], v[8 * g + 5]), pack_half2(v[8 * g + 6], v[8 * g + 7]));
  __syncwarp();
  const int ch = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = (lane >> 2) + 8 * i;
    const uint4 q = *reinterpret_cast<const uint4*>(stg + r * STG_F16_STR + 16 * ch);
    if (row0 + r < M && 8 * ch < valid)
      *reinterpret_cast<uint4*>(C + static_cast<long long>(row0 + r) * ldc + col + 8 * ch) = q;
  }
  __syncwarp();
}

// fp16 [32 rows][16 columns], as store_rows_f16 (`valid` a multiple of 8)
HY_DEV void store_rows_f16x16(uint8_t* stg, __half* C, long long ldc, int row0, int M, int col, int valid,
                              const float (&v)[16], int lane) {
  uint8_t* my = stg + lane * STG_F16_STR;
#pragma unroll
  for (int g = 0; g < 2; ++g)
    *reinterpret_cast<uint4*>(my + 16 * g) =
        make_uint4(pack_half2(v[8 * g], v[8 * g + 1]), pack_half2(v[8 * g + 2], v[8 * g + 3]),
                   pack_half2(v[8 * g + 4], v[8 * g + 5]), pack_half2(v[8 * g + 6], v[8 * g + 7]));
  __syncwarp();
  const int ch = lane & 1;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = (lane >> 1) + 16 * i;
    const uint4 q = *reinterpret_cast<const uint4*>(stg + r * STG_F16_STR + 16 * ch);
    if (row0 + r < M && 8 * ch < valid)
      *reinterpret_cast<uint4*>(C + static_cast<long long>(row0 + r) * ldc + col + 8 * ch) = q;
  }
  __syncwarp();
}

// fp32 [32 rows][32 columns], as store_rows_f16 (any `valid`), plus at most
// one residual (bf16 rb or fp32 rf, may alias C) read and an optional fp16
// copy C2 written in the same row pieces.  All eight residual pieces of a
// lane are loaded before its first store (a residual aliasing C would
// otherwise order each load behind the previous store).  C, ldc and rf on
// 16-byte boundaries, rb and C2 on 8-byte ones.  Returns whether a value of
// the fp16 copy is out of fp16 range.
HY_DEV bool store_rows_f32(uint8_t* stg, float* C, long long ldc, int row0, int M, int col, int valid,
                           const float (&v)[32], int lane, const __nv_bfloat16* rb, const float* rf, long long ldr,
                           __half* C2, long long ldc2) {
  uint8_t* my = stg + lane * STG_F32_STR;
#pragma unroll
  for (int g = 0; g < 8; ++g)
    *reinterpret_cast<float4*>(my + 16 * g) = make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
  __syncwarp();
  const int ch = lane & 7;
  const int c = col + 4 * ch;
  const bool full = 4 * ch + 4 <= valid;  // this lane's piece lies inside N
  float4 a[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const long long row = row0 + (lane >> 3) + 4 * i;
    a[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (row < M && full) {
      if (rf) {
        a[i] = *reinterpret_cast<const float4*>(rf + row * ldr + c);
      } else if (rb) {
        const uint2 w = *reinterpret_cast<const uint2*>(rb + row * ldr + c);
        const float2 a0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
        const float2 a1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
        a[i] = make_float4(a0.x, a0.y, a1.x, a1.y);
      }
    }
  }
  bool over = false;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = (lane >> 3) + 4 * i;
    const long long row = row0 + r;
    if (row >= M || 4 * ch >= valid) continue;
    float4 q = *reinterpret_cast<const float4*>(stg + r * STG_F32_STR + 16 * ch);
    if (full) {
      q = make_float4(q.x + a[i].x, q.y + a[i].y, q.z + a[i].z, q.w + a[i].w);
      *reinterpret_cast<float4*>(C + row * ldc + c) = q;
      if (C2) {
        over |= !(fabsf(q.x) <= kHalfMax) | !(fabsf(q.y) <= kHalfMax) | !(fabsf(q.z) <= kHalfMax) |
                !(fabsf(q.w) <= kHalfMax);
        *reinterpret_cast<uint2*>(C2 + row * ldc2 + c) = make_uint2(pack_half2(q.x, q.y), pack_half2(q.z, q.w));
      }
    } else {
      const float e4[4] = {q.x, q.y, q.z, q.w};
      for (int e = 0; e < valid - 4 * ch; ++e) {
        float t = e4[e];
        if (rf) t += rf[row * ldr + c + e];
        else if (rb) t += __bfloat162float(rb[row * ldr + c + e]);
        C[row * ldc + c + e] = t;
        if (C2) {
          over |= !(fabsf(t) <= kHalfMax);
          C2[row * ldc2 + c + e] = __float2half_rn(t);
        }
      }
    }
  }
  __syncwarp();
  return over;
}

struct TileCoord {
  int m, n, kb0, kb1, split;
};

// tile pair t of a pair launch, for the CTA of cluster rank r: row block 2 mp + r
HY_DEV TileCoord pair_coord(const GemmParams& p, int t, int r) {
  TileCoord c;
  const int mp = t / p.tiles_n;
  c.n = t - mp * p.tiles_n;
  c.m = 2 * mp + r;  // may be tiles_m (odd tiles_m): its rows load as zeros and are not stored
  c.split = 0;
  c.kb0 = 0;
  c.kb1 = p.n_kb;
  return c;
}

HY_DEV TileCoord tile_coord(const GemmParams& p, int t) {
  TileCoord c;
  const int mn = p.tiles_m * p.tiles_n;
  c.split = t / mn;
  const int r = t - c.split * mn;
  c.m = r / p.tiles_n;
  c.n = r - c.m * p.tiles_n;
  c.kb0 = c.split * p.kb_per_split;
  c.kb1 = min(p.n_kb, c.kb0 + p.kb_per_split);
  return c;
}

// ---- epilogue helpers --------------------------------------------------------

HY_DEV void store_f16x32(__half* dst, const float (&v)[32], int valid) {
  // valid = number of leading columns inside N (multiple of 8 or >= 32)
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    if (g * 8 < valid) {
      uint4 q;
      q.x = pack_half2(v[g * 8 + 0], v[g * 8 + 1]);
      q.y = pack_half2(v[g * 8 + 2], v[g * 8 + 3]);
      q.z = pack_half2(v[g * 8 + 4], v[g * 8 + 5]);
      q.w = pack_half2(v[g * 8 + 6], v[g * 8 + 7]);
      *reinterpret_cast<uint4*>(dst + g * 8) = q;
    }
  }
}

// 32 fp32 values; `valid` leading columns are inside N.  Compile-time
// indices only, so v stays in registers.
HY_DEV void store_f32x32(float* dst, const float (&v)[32], int valid) {
  if (valid >= 32 && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
#pragma unroll
    for (int g = 0; g < 32; g += 4)
      *reinterpret_cast<float4*>(dst + g) = make_float4(v[g], v[g + 1], v[g + 2], v[g + 3]);
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < valid) dst[j] = v[j];
  }
}

HY_DEV bool any_over_half(const float (&v)[32]) {
  bool o = false;
#pragma unroll
  for (int j = 0; j < 32; ++j) o |= !(fabsf(v[j]) <= kHalfMax);
  return o;
}

template <int BN, int EPI, bool PAIR, int KC>
__global__ void __launch_bounds__(192, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmParams p, const uint32_t idesc) {
  using Cfg = GemmCfg<BN, PAIR, KC, epi_stg_bytes<EPI>()>;
  constexpr int S = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem<1024>(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = smem + S * Cfg::A_STAGE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * Cfg::STAGE);
  // bars: full[S], empty[S], tfull[2], tempty[2], cvt[S]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * S + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* rope_tab = reinterpret_cast<float*>(tmem_slot + 4);  // 32 floats

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  auto full = [&](int s) { return smem_u32(&bars[s]); };
  auto empty = [&](int s) { return smem_u32(&bars[S + s]); };
  auto tfull = [&](int a) { return smem_u32(&bars[2 * S + a]); };
  auto tempty = [&](int a) { return smem_u32(&bars[2 * S + 2 + a]); };
  auto cvt = [&](int s) { return smem_u32(&bars[2 * S + 4 + s]); };

  // tile walk: a static round-robin over the CTAs, or over the CTA pairs
  const int rank = PAIR ? static_cast<int>(cluster_rank()) : 0;
  const bool leader = rank == 0;
  const int t_first = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int t_step = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  const int t_count = PAIR ? p.total_pairs : p.total_tiles;
  auto coord = [&](int t) { return PAIR ? pair_coord(p, t, rank) : tile_coord(p, t); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull(a), 1);
      mbar_init(tempty(a), PAIR ? 8 : 4);  // pair: both CTAs' epilogue warps
    }
    for (int s = 0; s < S; ++s) mbar_init(cvt(s), 4);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (EPI == EPI_F16 && threadIdx.x < 32) rope_tab[threadIdx.x] = exp2f(threadIdx.x * p.rope_log2_step);
  if (warp == 1) {
    if constexpr (PAIR)
      tmem_alloc_pair(smem_u32(tmem_slot), Cfg::TMEM_COLS);
    else
      tmem_alloc(smem_u32(tmem_slot), Cfg::TMEM_COLS);
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // the peer's barriers exist before any remote arrive
  tc_fence_after();
  // In a programmatic launch (the decode step's GEMMs) the B operand is a
  // weight no kernel of the step writes: the producer issues B of the first
  // tile's first stages before waiting for the preceding kernel, so that
  // the weight stream starts during that kernel's tail; A follows the wait.
  int pre_b = 0;
  if constexpr (!PAIR) {
    if (p.pdl && warp == 0 && lane == 0 && t_first < t_count) {
      const TileCoord c = coord(t_first);
      pre_b = min(S, c.kb1 - c.kb0);
      for (int j = 0; j < pre_b; ++j) {
        const int kb = c.kb0 + j;
        mbar_arrive_expect_tx(full(j), Cfg::STAGE);
        if constexpr (KC == 1)
          tma_load_2d(smem_u32(sB + j * Cfg::B_BYTES), &tmB, full(j), kb * BK, c.n * BN);
        else
          tma_load_3d(smem_u32(sB + j * Cfg::B_BYTES), &tmB, full(j), 0, c.n * BN, kb * KC);
      }
    }
  }
  pdl_wait();  // only the setup above may overlap the preceding kernel
  pdl_trigger();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtl wc{abort_flag, p.status, p.wait_ns};

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      uint32_t it = 0, issued = 0;
      uint32_t last_par = 0;  // bit s: parity of the last load issued into stage s
      bool ok = true;
      for (int t = t_first; t < t_count && ok; t += t_step) {
        const TileCoord c = coord(t);
        for (int kb = c.kb0; kb < c.kb1; ++kb, ++it) {
          const int s = it % S;
          const uint32_t ph = (it / S) & 1;
          if (static_cast<int>(it) < pre_b) {
            // B of this stage is on its way (issued before the wait): A only
            if constexpr (KC == 1)
              tma_load_2d(smem_u32(sA + s * Cfg::A_STAGE), &tmA, full(s), kb * BK, c.m * BM);
            else
              tma_load_3d(smem_u32(sA + s * Cfg::A_STAGE), &tmA, full(s), 0, c.m * BM, kb * KC);
            issued |= 1u << s;
            last_par = (last_par & ~(1u << s)) | (ph << s);
            continue;
          }
          if (!mbar_wait(empty(s), ph ^ 1, wc)) { ok = false; break; }
          if (!PAIR || leader) {
            // a pair's even CTA expects both CTAs' bytes on its own barrier
            mbar_arrive_expect_tx(full(s), PAIR ? 2 * Cfg::STAGE : Cfg::STAGE);
            if constexpr (KC == 1) {
              tma_load_2d(smem_u32(sA + s * Cfg::A_STAGE), &tmA, full(s), kb * BK, c.m * BM);
              tma_load_2d(smem_u32(sB + s * Cfg::B_BYTES), &tmB, full(s), kb * BK, c.n * BN + rank * (BN / 2));
            } else {
              tma_load_3d(smem_u32(sA + s * Cfg::A_STAGE), &tmA, full(s), 0, c.m * BM, kb * KC);
              tma_load_3d(smem_u32(sB + s * Cfg::B_BYTES), &tmB, full(s), 0, c.n * BN + rank * (BN / 2), kb * KC);
            }
          } else {
            const uint32_t bar0 = mapa_shared(full(s), 0);
            if constexpr (KC == 1) {
              tma_load_2d_pair(smem_u32(sA + s * Cfg::A_STAGE), &tmA, bar0, kb * BK, c.m * BM);
              tma_load_2d_pair(smem_u32(sB + s * Cfg::B_BYTES), &tmB, bar0, kb * BK, c.n * BN + rank * (BN / 2));
            } else {
              tma_load_3d_pair(smem_u32(sA + s * Cfg::A_STAGE), &tmA, bar0, 0, c.m * BM, kb * KC);
              tma_load_3d_pair(smem_u32(sB + s * Cfg::B_BYTES), &tmB, bar0, 0, c.n * BN + rank * (BN / 2), kb * KC);
            }
          }
          issued |= 1u << s;
          last_par = (last_par & ~(1u << s)) | (ph << s);
        }
      }
      // let the copies already in flight land before the CTA exits (a pair's
      // odd CTA counts on the even CTA's barriers, whose drain covers them;
      // the final cluster barrier keeps the odd CTA until then)
      if (!ok && (!PAIR || leader)) {
        for (int s = 0; s < S; ++s)
          if (issued & (1u << s)) mbar_wait_drain(full(s), (last_par >> s) & 1, 1000000);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (PAIR && !leader) {
      // the odd CTA issues no MMA: its tiles are loaded by its producer and
      // consumed by the even CTA's MMAs
    } else if (lane == 0) {
      uint32_t it = 0, committed = 0, last_par = 0, tcommitted = 0, tlast = 0;
      bool ok = true;
      int local = 0;
      for (int t = t_first; t < t_count && ok; t += t_step, ++local) {
        const TileCoord c = coord(t);
        const int a = local & 1;
        const uint32_t u = (local >> 1) & 1;
        if (!(PAIR ? mbar_wait_cluster(tempty(a), u ^ 1, wc) : mbar_wait(tempty(a), u ^ 1, wc))) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem_base + a * BN;
        for (int kb = c.kb0; kb < c.kb1; ++kb, ++it) {
          const int s = it % S;
          const uint32_t ph = (it / S) & 1;
          const bool got = PAIR ? mbar_wait_cluster(full(s), ph, wc) : mbar_wait(p.cvt_b ? cvt(s) : full(s), ph, wc);
          if (!got) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < KC * BK / 16; ++kk) {
            // chunk kk / 4 of the stage, 16-wide step kk % 4 within it
            const uint64_t da = sdesc_sw128(smem_u32(sA + s * Cfg::A_STAGE + (kk / 4) * A_BYTES), 16, 1024) +
                                2 * (kk % 4);
            const uint64_t db = sdesc_sw128(smem_u32(sB + s * Cfg::B_BYTES + (kk / 4) * Cfg::B_CHUNK), 16, 1024) +
                                2 * (kk % 4);
            if constexpr (PAIR)
              tc_mma_f16_pair(d, da, db, idesc, (kb > c.kb0 || kk > 0) ? 1u : 0u);
            else
              tc_mma_f16(d, da, db, idesc, (kb > c.kb0 || kk > 0) ? 1u : 0u);
          }
          if constexpr (PAIR)
            tc_commit_pair(empty(s), 0x3);  // the stage is free in both CTAs
          else
            tc_commit(empty(s));
          committed |= 1u << s;
          last_par = (last_par & ~(1u << s)) | (ph << s);
        }
        if (!ok) break;
        if constexpr (PAIR)
          tc_commit_pair(tfull(a), 0x3);  // the accumulator is ready in both CTAs
        else
          tc_commit(tfull(a));
        tcommitted |= 1u << a;
        tlast = (tlast & ~(1u << a)) | (u << a);
      }
      if (!ok) {  // wait for issued MMAs before TMEM is released
        for (int s = 0; s < S; ++s)
          if (committed & (1u << s)) mbar_wait_drain(empty(s), (last_par >> s) & 1, 1000000);
        for (int a = 0; a < 2; ++a)
          if (tcommitted & (1u << a)) mbar_wait_drain(tfull(a), (tlast >> a) & 1, 1000000);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int row_in_tile = q * 32 + lane;
    const int ct = threadIdx.x - 64;  // 0..127 over the four epilogue warps
    // fp32 results, residual and fp16 copy in whole row pieces when every
    // pointer and leading dimension allows the vector accesses
    const bool f32_staged =
        EPI == EPI_F32 && ((reinterpret_cast<uintptr_t>(p.C) | static_cast<uintptr_t>(p.ldc * 4)) & 15) == 0 &&
        ((reinterpret_cast<uintptr_t>(p.resid_f32) | static_cast<uintptr_t>(p.resid_f32 ? p.ld_resid * 4 : 0)) & 15) ==
            0 &&
        ((reinterpret_cast<uintptr_t>(p.resid) | static_cast<uintptr_t>(p.resid ? p.ld_resid * 2 : 0)) & 7) == 0 &&
        ((reinterpret_cast<uintptr_t>(p.C2) | static_cast<uintptr_t>(p.C2 ? p.ldc2 * 2 : 0)) & 7) == 0 &&
        !(p.resid && p.resid_f32);
    int local = 0;
    uint32_t cit = 0;  // k-block counter of the conversion (follows the producer's)
    bool cok = true;
    for (int t = t_first; t < t_count; t += t_step, ++local) {
      const TileCoord c = coord(t);
      const int a = local & 1;
      const uint32_t u = (local >> 1) & 1;
      if (p.cvt_b) {
        // bf16 -> fp16 of every B stage of this tile, in place (elementwise:
        // the swizzled layout is unchanged)
        for (int kb = c.kb0; kb < c.kb1 && cok; ++kb, ++cit) {
          const int s = cit % S;
          const bool gotb = mbar_wait(full(s), (cit / S) & 1, wc);
          if (!__all_sync(0xffffffffu, gotb)) { cok = false; break; }
          uint4* b16 = reinterpret_cast<uint4*>(sB + s * Cfg::B_BYTES);
#pragma unroll
          for (int i = ct; i < Cfg::B_BYTES / 16; i += 128) {
            const uint4 v = b16[i];
            const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&v);
            uint4 o;
            uint32_t* o32 = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = __bfloat1622float2(b2[e]);
              o32[e] = pack_half2(f.x, f.y);
            }
            b16[i] = o;
          }
          fence_proxy_async_smem();  // generic stores -> tensor-core reads
          __syncwarp();
          if (lane == 0) mbar_arrive(cvt(s));
        }
        if (!cok) break;
      }
      const bool got = mbar_wait(tfull(a), u, wc);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      const int row = c.m * BM + row_in_tile;
      const bool row_ok = row < p.M;
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + a * BN;
      const int col_tile = c.n * BN;
      bool over = false;

      if (EPI == EPI_F16 && p.rope_cols > 0 && col_tile < p.rope_cols) {
        // RoPE: 64-column heads, pair (i, i+32) rotated by pos * inv_freq[i].
        // The angles depend on the row and i only, so each (sin, cos) is made
        // once per row and tile, 16 frequencies at a time, and applied to
        // every head of the tile.
        const int posn = p.pos_base + (p.pos ? p.pos[min(row, p.M - 1)] : (row % p.rows_per_seq));
#pragma unroll 1
        for (int jg = 0; jg < 2; ++jg) {
          float sn[16], cs[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) sincosf(static_cast<float>(posn) * rope_tab[jg * 16 + j], &sn[j], &cs[j]);
#pragma unroll 1
          for (int c0 = 0; c0 < BN; c0 += 64) {
            const int col = col_tile + c0;
            if (col >= p.N) break;
            uint32_t r0[16], r1[16];
            tmem_ld16(tbase + c0 + jg * 16, r0);
            tmem_ld16(tbase + c0 + 32 + jg * 16, r1);
            tc_wait_ld();
            float v0[16], v1[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              v0[j] = __uint_as_float(r0[j]);
              v1[j] = __uint_as_float(r1[j]);
            }
            if (col < p.rope_cols) {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float x1 = v0[j], x2 = v1[j];
                v0[j] = x1 * cs[j] - x2 * sn[j];
                v1[j] = x2 * cs[j] + x1 * sn[j];
              }
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) over |= !(fabsf(v0[j]) <= kHalfMax) | !(fabsf(v1[j]) <= kHalfMax);
            // all lanes: the stores go through the warp's staging tile
            uint8_t* stg = smem + Cfg::OFF_STG + q * 32 * STG_F16_STR;
            __half* out = reinterpret_cast<__half*>(p.C);
            store_rows_f16x16(stg, out, p.ldc, c.m * BM + q * 32, p.M, col + jg * 16, p.N - col - jg * 16, v0, lane);
            store_rows_f16x16(stg, out, p.ldc, c.m * BM + q * 32, p.M, col + 32 + jg * 16, p.N - col - 32 - jg * 16,
                              v1, lane);
          }
        }
      } else {
        for (int c0 = 0; c0 < BN; c0 += 32) {
          const int col = col_tile + c0;
          if (col >= p.N) break;
          const int nv = (c0 + 32 <= BN) ? 32 : 16;
          float v[32];
          if (nv == 32) {
            uint32_t r[32];
            tmem_ld32(tbase + c0, r);
            tc_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
          } else {
            uint32_t r[16];
            tmem_ld16(tbase + c0, r);
            tc_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
#pragma unroll
            for (int j = 16; j < 32; ++j) v[j] = 0.f;
          }
          const int valid = min(nv, p.N - col);
          if (EPI == EPI_F16) {  // all lanes: the store goes through the warp's staging tile
            if (row_ok) over |= any_over_half(v);
            store_rows_f16(smem + Cfg::OFF_STG + q * 32 * STG_F16_STR, reinterpret_cast<__half*>(p.C), p.ldc,
                           c.m * BM + q * 32, p.M, col, valid, v, lane);
            continue;
          }
          if (EPI == EPI_F32 && f32_staged) {
            over |= store_rows_f32(smem + Cfg::OFF_STG + q * 32 * STG_F32_STR, reinterpret_cast<float*>(p.C), p.ldc,
                                   c.m * BM + q * 32, p.M, col, valid, v, lane, p.resid, p.resid_f32, p.ld_resid,
                                   reinterpret_cast<__half*>(p.C2), p.ldc2);
            continue;
          }
          if (EPI == EPI_GEGLU) {
            // exact GeLU, x Phi(x) with Phi from erff; 16 outputs per 32
            // columns, stored through the staging tile
            float o[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float gt = v[2 * e], up = v[2 * e + 1];
              o[e] = 0.5f * gt * (1.0f + erff(gt * 0.7071067811865476f)) * up;
              if (row_ok) over |= !(fabsf(o[e]) <= kHalfMax);
            }
            store_rows_f16x16(smem + Cfg::OFF_STG + q * 32 * STG_F16_STR, reinterpret_cast<__half*>(p.C), p.ldc,
                              c.m * BM + q * 32, p.M, col / 2, valid / 2, o, lane);
            continue;
          }
          if (!row_ok) continue;
          if (EPI == EPI_F16) {
          } else if (EPI == EPI_XPROJ) {
            // groups of 8 columns: a whole dt group is one 16-byte fp16
            // store, a whole [B | C] group two 16-byte fp32 stores; the group
            // that straddles R and the ragged end go element by element
            __half* drow = reinterpret_cast<__half*>(p.C2) + static_cast<long long>(row) * p.ldc2;
            float* brow = reinterpret_cast<float*>(p.C) + static_cast<long long>(row) * p.ldc;  // column R
            const bool vec_d = ((reinterpret_cast<uintptr_t>(p.C2) | static_cast<uintptr_t>(p.ldc2 * 2)) & 15) == 0;
            const bool vec_b = ((reinterpret_cast<uintptr_t>(p.C) | static_cast<uintptr_t>(p.ldc * 4)) & 15) == 0 &&
                               (p.xproj_R & 3) == 0;
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) {
              const int j0 = 8 * g8, c = col + j0;
              if (j0 >= valid) break;
              if (vec_d && c + 8 <= p.xproj_R) {
                uint4 o;
                o.x = pack_half2(v[j0], v[j0 + 1]);
                o.y = pack_half2(v[j0 + 2], v[j0 + 3]);
                o.z = pack_half2(v[j0 + 4], v[j0 + 5]);
                o.w = pack_half2(v[j0 + 6], v[j0 + 7]);
#pragma unroll
                for (int e = 0; e < 8; ++e) over |= !(fabsf(v[j0 + e]) <= kHalfMax);
                *reinterpret_cast<uint4*>(drow + c) = o;
              } else if (vec_b && c >= p.xproj_R && j0 + 8 <= valid) {
                float* bp = brow + (c - p.xproj_R);
                *reinterpret_cast<float4*>(bp) = make_float4(v[j0], v[j0 + 1], v[j0 + 2], v[j0 + 3]);
                *reinterpret_cast<float4*>(bp + 4) = make_float4(v[j0 + 4], v[j0 + 5], v[j0 + 6], v[j0 + 7]);
              } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  const int j = j0 + e, cj = c + e;
                  if (j < valid) {
                    if (cj < p.xproj_R) {
                      over |= !(fabsf(v[j]) <= kHalfMax);
                      drow[cj] = __float2half_rn(v[j]);
                    } else {
                      brow[cj - p.xproj_R] = v[j];
                    }
                  }
                }
              }
            }
          } else if (EPI == EPI_SOFTPLUS) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < valid) v[j] = softplus_f(v[j] + p.bias[col + j]);
            store_f32x32(reinterpret_cast<float*>(p.C) + static_cast<long long>(row) * p.ldc + col, v, valid);
          } else if (EPI == EPI_F32) {
            if (p.resid) {
              const __nv_bfloat16* rr = p.resid + static_cast<long long>(row) * p.ld_resid + col;
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j < valid) v[j] += __bfloat162float(rr[j]);
            } else if (p.resid_f32) {
              const float* rr = p.resid_f32 + static_cast<long long>(row) * p.ld_resid + col;
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j < valid) v[j] += rr[j];
            }
            store_f32x32(reinterpret_cast<float*>(p.C) + static_cast<long long>(row) * p.ldc + col, v, valid);
            if (p.C2) {  // the updated stream rounded to fp16: the next layer's input
              over |= any_over_half(v);
              store_f16x32(reinterpret_cast<__half*>(p.C2) + static_cast<long long>(row) * p.ldc2 + col, v, valid);
            }
          } else if (EPI == EPI_ATOMIC) {
            float* dst = reinterpret_cast<float*>(p.C) + static_cast<long long>(row) * p.ldc + col;
            if (valid == 32 && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
#pragma unroll
              for (int g = 0; g < 32; g += 4)
                asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + g), "f"(v[g]),
                             "f"(v[g + 1]), "f"(v[g + 2]), "f"(v[g + 3])
                             : "memory");
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j < valid) atomicAdd(dst + j, v[j]);
            }
          } else {  // EPI_PARTIAL
            float* dst = reinterpret_cast<float*>(p.C) +
                         (static_cast<long long>(c.split) * p.M + row) * p.ldc + col;
            store_f32x32(dst, v, valid);
          }
        }
      }
      if (over) set_status(p.status, HYMBA_ERR_RANGE);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR && !leader)
          mbar_arrive_remote(mapa_shared(tempty(a), 0));  // the even CTA reuses this CTA's accumulator too
        else
          mbar_arrive(tempty(a));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // no CTA leaves while its peer may still reach its memory
  tc_fence_after();
  if (warp == 1) {
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
    else
      tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

// Kernel attributes and occupancy figures belong to one device: the
// launchers cache them per device ordinal (devices past the table's end are
// set up on every call).
constexpr int kMaxDevices = 64;

template <int BN, int EPI, bool PAIR, int KC>
hymba_status launch_bn(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p, uint32_t idesc, int grid,
                       cudaStream_t st) {
  using Cfg = GemmCfg<BN, PAIR, KC, epi_stg_bytes<EPI>()>;
  auto kern = gemm_tc_kernel<BN, EPI, PAIR, KC>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return HYMBA_ERR_CUDA;
  const bool cached = dev < kMaxDevices;
  // setting the attribute twice is harmless, so two threads may race here
  static std::atomic<bool> attr_done[kMaxDevices];
  if (!cached || !attr_done[dev].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM) != cudaSuccess)
      return HYMBA_ERR_CUDA;
    if (cached) attr_done[dev].store(true, std::memory_order_release);
  }
  if constexpr (!PAIR) {
    if (launch_kernel(p.pdl != 0, kern, dim3(grid), dim3(192), Cfg::SMEM, st, ta, tb, p, idesc) != cudaSuccess)
      return HYMBA_ERR_CUDA;
  } else {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(192, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;  // the occupancy query takes the cluster shape only
    // persistent: no more pairs than can be resident at once, so no tile
    // waits for a second wave
    static std::atomic<int> max_clusters_dev[kMaxDevices];
    int max_clusters = cached ? max_clusters_dev[dev].load(std::memory_order_relaxed) : 0;
    if (max_clusters == 0) {
      cfg.gridDim = dim3(2 * std::max(1, grid / 2), 1, 1);
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) return HYMBA_ERR_CUDA;
      max_clusters = n;
      if (cached) max_clusters_dev[dev].store(n, std::memory_order_relaxed);
    }
    const int clusters = std::max(1, std::min(std::min(grid / 2, max_clusters), p.total_pairs));
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.numAttrs = p.pdl ? 2 : 1;
    if (cudaLaunchKernelEx(&cfg, kern, ta, tb, p, idesc) != cudaSuccess) return HYMBA_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? HYMBA_OK : HYMBA_ERR_CUDA;
}

template <int EPI, bool PAIR = false>
hymba_status launch_epi(int bn, int kc, const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p,
                        uint32_t ab_fmt, int grid, cudaStream_t st) {
  const uint32_t id = idesc_f16(PAIR ? 2 * BM : BM, bn, ab_fmt, false, false);
  if (kc == 2) {
    switch (bn) {
      case 64: return launch_bn<64, EPI, PAIR, 2>(ta, tb, p, id, grid, st);
      case 128: return launch_bn<128, EPI, PAIR, 2>(ta, tb, p, id, grid, st);
      case 144: return launch_bn<144, EPI, PAIR, 2>(ta, tb, p, id, grid, st);
      case 160: return launch_bn<160, EPI, PAIR, 2>(ta, tb, p, id, grid, st);
      default: return HYMBA_ERR_UNSUPPORTED;
    }
  }
  switch (bn) {
    case 64: return launch_bn<64, EPI, PAIR, 1>(ta, tb, p, id, grid, st);
    case 128: return launch_bn<128, EPI, PAIR, 1>(ta, tb, p, id, grid, st);
    case 144: return launch_bn<144, EPI, PAIR, 1>(ta, tb, p, id, grid, st);
    case 160: return launch_bn<160, EPI, PAIR, 1>(ta, tb, p, id, grid, st);
    case 256: return launch_bn<256, EPI, PAIR, 1>(ta, tb, p, id, grid, st);
    default: return HYMBA_ERR_UNSUPPORTED;
  }
}

}  // namespace

// Tile width: least padded N, each width weighted by its measured cost per
// column relative to 256-wide tiles (narrower tiles read more of A from L2
// per FLOP and issue more MMAs and epilogues: in_proj at 256 reaches 0.93 of
// the bf16 peak; out_proj, N = 1600, ran 0.474 ms at 160 against 0.465 ms at
// 256 with 12% of the columns padding), so a wide tile wins unless it pads N
// by more than about 15%.
int gemm_pick_bn(int N, bool small_m) {
  if (small_m) return 64;
  static const int cand[] = {256, 160, 144, 128, 64};
  static const int cost[] = {100, 118, 120, 122, 135};
  int best = 256;
  long long best_cost = 1LL << 60;
  for (int i = 0; i < 5; ++i) {
    const int bn = cand[i];
    const long long c = static_cast<long long>((N + bn - 1) / bn) * bn * cost[i];
    if (c < best_cost) {
      best_cost = c;
      best = bn;
    }
  }
  return best;
}

hymba_status gemm_tc(int ab_fmt, const void* A, long long lda, const void* B, long long ldb, int epi,
                     GemmParams p, int bn, int splits, int num_sms, cudaStream_t st) {
  if (p.M <= 0 || p.N <= 0 || p.K <= 0) return HYMBA_OK;
  if (p.cvt_b && ab_fmt != 0) return HYMBA_ERR_INVALID;  // converted B meets fp16 A
  if ((reinterpret_cast<uintptr_t>(A) & 15) || (reinterpret_cast<uintptr_t>(B) & 15) || (lda % 8) ||
      (ldb % 8) || lda < p.K || ldb < p.K)
    return HYMBA_ERR_INVALID;
  if (bn == 0) bn = gemm_pick_bn(p.N, p.M <= BM);
  const CUtensorMapDataType dt = ab_fmt == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  // two 64-column chunks of K per stage (one 3-D copy of each operand) when
  // the MMAs of one chunk are shorter than two copies: BN <= 160; the chunks
  // must not run past K, so K % 64 == 0
  // (split partial sums that a separate pass reduces keep one chunk per stage:
  // their callers count the splits over 64-wide chunks)
  const int kc = (p.K % BK == 0 && bn <= 160 && epi != EPI_PARTIAL) ? 2 : 1;
  const int n_chunks = (p.K + BK - 1) / BK;
  CUtensorMap ta, tb;
  if (kc == 2) {
    const uint64_t dims[3] = {static_cast<uint64_t>(BK), static_cast<uint64_t>(p.M), static_cast<uint64_t>(n_chunks)};
    const uint64_t str[2] = {static_cast<uint64_t>(lda) * 2, BK * 2};
    const uint32_t box[3] = {BK, BM, 2};
    if (!encode_tmap(&ta, dt, 3, A, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return HYMBA_ERR_CUDA;
  } else {
    const uint64_t dims[2] = {static_cast<uint64_t>(p.K), static_cast<uint64_t>(p.M)};
    const uint64_t str[1] = {static_cast<uint64_t>(lda) * 2};
    const uint32_t box[2] = {BK, BM};
    if (!encode_tmap(&ta, dt, 2, A, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return HYMBA_ERR_CUDA;
  }
  p.tiles_m = (p.M + BM - 1) / BM;
  // CTA pairs (256-row tiles, each CTA loading half of B) once there are
  // several row blocks; not for split-K or converted-B launches
  const bool pair = splits <= 1 && !p.cvt_b && p.tiles_m >= 4 && num_sms >= 2 && bn <= kPairMaxBN;
  {
    const CUtensorMapDataType dtb = p.cvt_b ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : dt;
    const uint32_t rows_b = static_cast<uint32_t>(pair ? bn / 2 : bn);
    if (kc == 2) {
      const uint64_t dims[3] = {static_cast<uint64_t>(BK), static_cast<uint64_t>(p.N),
                                static_cast<uint64_t>(n_chunks)};
      const uint64_t str[2] = {static_cast<uint64_t>(ldb) * 2, BK * 2};
      const uint32_t box[3] = {BK, rows_b, 2};
      if (!encode_tmap(&tb, dtb, 3, B, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return HYMBA_ERR_CUDA;
    } else {
      const uint64_t dims[2] = {static_cast<uint64_t>(p.K), static_cast<uint64_t>(p.N)};
      const uint64_t str[1] = {static_cast<uint64_t>(ldb) * 2};
      const uint32_t box[2] = {BK, rows_b};
      if (!encode_tmap(&tb, dtb, 2, B, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return HYMBA_ERR_CUDA;
    }
  }
  p.tiles_n = (p.N + bn - 1) / bn;
  p.n_kb = (n_chunks + kc - 1) / kc;  // pipeline stages of K (kc chunks each)
  splits = std::max(1, std::min(splits, p.n_kb));
  p.kb_per_split = (p.n_kb + splits - 1) / splits;
  p.splits = (p.n_kb + p.kb_per_split - 1) / p.kb_per_split;
  p.total_tiles = p.tiles_m * p.tiles_n * p.splits;
  p.total_pairs = (p.tiles_m + 1) / 2 * p.tiles_n;
  if (p.splits > 1 && epi != EPI_PARTIAL && epi != EPI_ATOMIC) return HYMBA_ERR_INVALID;
  if (epi == EPI_GEGLU && (p.N % 16 || p.ldc % 8 || (reinterpret_cast<uintptr_t>(p.C) & 15))) return HYMBA_ERR_INVALID;
  const int grid = std::min(p.total_tiles, std::max(1, num_sms));
  const uint32_t fmt = ab_fmt == 1 ? 1u : 0u;
  if (pair) {
    switch (epi) {
      case EPI_F16: return launch_epi<EPI_F16, true>(bn, kc, ta, tb, p, fmt, num_sms, st);
      case EPI_XPROJ: return launch_epi<EPI_XPROJ, true>(bn, kc, ta, tb, p, fmt, num_sms, st);
      case EPI_SOFTPLUS: return launch_epi<EPI_SOFTPLUS, true>(bn, kc, ta, tb, p, fmt, num_sms, st);
      case EPI_F32: return launch_epi<EPI_F32, true>(bn, kc, ta, tb, p, fmt, num_sms, st);
      case EPI_GEGLU: return launch_epi<EPI_GEGLU, true>(bn, kc, ta, tb, p, fmt, num_sms, st);
      default: return HYMBA_ERR_INVALID;
    }
  }
  switch (epi) {
    case EPI_F16: return launch_epi<EPI_F16>(bn, kc, ta, tb, p, fmt, grid, st);
    case EPI_XPROJ: return launch_epi<EPI_XPROJ>(bn, kc, ta, tb, p, fmt, grid, st);
    case EPI_SOFTPLUS: return launch_epi<EPI_SOFTPLUS>(bn, kc, ta, tb, p, fmt, grid, st);
    case EPI_F32: return launch_epi<EPI_F32>(bn, kc, ta, tb, p, fmt, grid, st);
    case EPI_PARTIAL: return launch_epi<EPI_PARTIAL>(bn, kc, ta, tb, p, fmt, grid, st);
    case EPI_ATOMIC: return launch_epi<EPI_ATOMIC>(bn, kc, ta, tb, p, fmt, grid, st);
    case EPI_GEGLU: return launch_epi<EPI_GEGLU>(bn, kc, ta, tb, p, fmt, grid, st);
    default: return HYMBA_ERR_INVALID;
  }
}

}  // namespace hy
