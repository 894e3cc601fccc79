// Decode-step attention over the meta prefix and the sliding-window ring
// ("Hymba: A Hybrid-head Architecture for Small Language Models", section 2.2
// window and section 2.3 meta tokens) for bf16 caches: one new query row per
// sequence, GQA heads grouped per KV head.
//
// The step is bound by reading the cache (K and V of every visible key once),
// so the kernel is built to keep HBM busy:
//   - persistent warps; each warp owns a 2-stage ring of 64-key chunks and
//     streams K [64 x dh] and V [64 x dv] tiles into it with TMA
//     (128-byte swizzle), prefetching the next chunk while it computes on the
//     current one;
//   - the work is cut into units (sequence b, KV head g, key split sp); a
//     warp walks its units back to back, so its ring never drains between
//     them;
//   - the G = Hq/Hkv query heads of a KV head are the rows of one m16 mma
//     tile: S = Q K^T and O += P V run on mma.sync (bf16 in, fp32 out), the
//     softmax is online in registers (log2 domain: Q is prescaled by
//     log2(e)/sqrt(dh)), and P goes from the S accumulators to the A
//     operand without touching shared memory.
// Keys: meta rows 0..M-1 (one copy for the batch), then the visible ring
// slots, which form at most two contiguous slot ranges.  Each unit writes its
// partial (max m, sum l, unnormalised O) per head; a combine kernel merges the
// splits.  Every wait is bounded.
#include <algorithm>

#include "decode.cuh"

namespace hy {
namespace {

constexpr int DK = 64;          // keys per chunk
constexpr int DA_WARPS = 4;     // warps per CTA (one CTA per SM)
constexpr int DA_STAGES = 2;    // ring stages per warp
constexpr int DA_DH = 64;       // supported QK head dim
constexpr int DA_DV_MAX = 128;  // supported V head dims: 64, 128
constexpr int K_TILE = DK * DA_DH * 2;          // 8 KB
constexpr int V_BOX = DK * 64 * 2;              // one 64-column V box, 8 KB
constexpr int STAGE_BYTES = K_TILE + (DA_DV_MAX / 64) * V_BOX;  // 24 KB
constexpr int WARP_BYTES = DA_STAGES * STAGE_BYTES;

struct DaArgs {
  int B, M, Hq, Hkv, dv, window, cap, nsplit, n_units;
  const __half* q;
  long long ldq;
  const int32_t* pos;
  float* part;  // [B][Hq][nsplit][dv + 2]
  int32_t* status;
  uint64_t wait_ns;
};

// Key layout of one unit: chunk c of the unit's (b, g) key list.
struct KeyPlan {
  int nm, n1, n2;   // chunks of meta, first slot range, second slot range
  int s0, len1, len2;
  int c_lo, c_hi;   // this split's chunks
};

HY_DEV KeyPlan key_plan(const DaArgs& a, int b, int sp) {
  KeyPlan k;
  const int p = a.pos[b];
  int n_vis = a.window > 0 ? min(p + 1, a.window) : p + 1;
  n_vis = min(n_vis, a.cap);
  const int first = p - n_vis + 1;  // oldest visible token
  k.s0 = a.window > 0 ? first % a.cap : first;
  k.len1 = min(n_vis, a.cap - k.s0);
  k.len2 = n_vis - k.len1;
  k.nm = (a.M + DK - 1) / DK;
  k.n1 = (k.len1 + DK - 1) / DK;
  k.n2 = (k.len2 + DK - 1) / DK;
  const int nc = k.nm + k.n1 + k.n2;
  const int per = (nc + a.nsplit - 1) / a.nsplit;
  k.c_lo = min(nc, sp * per);
  k.c_hi = min(nc, k.c_lo + per);
  return k;
}

// chunk c -> (is_meta, first row in its tensor, valid keys)
HY_DEV void chunk_rows(const KeyPlan& k, const DaArgs& a, int b, int c, bool& meta, int& row, int& cnt) {
  if (c < k.nm) {
    meta = true;
    row = c * DK;
    cnt = min(DK, a.M - row);
  } else if (c < k.nm + k.n1) {
    meta = false;
    const int o = (c - k.nm) * DK;
    row = b * a.cap + k.s0 + o;
    cnt = min(DK, k.len1 - o);
  } else {
    meta = false;
    const int o = (c - k.nm - k.n1) * DK;
    row = b * a.cap + o;
    cnt = min(DK, k.len2 - o);
  }
}

HY_DEV void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
HY_DEV void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
HY_DEV void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
HY_DEV uint32_t pack_bf162(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
// byte offset of 16-byte chunk `c` of row `r` in a 128-byte-swizzled tile
HY_DEV uint32_t sw128(int r, int c) { return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4)); }

template <int DV>
__global__ void __launch_bounds__(DA_WARPS * 32, 1)
    decode_attn_tc_kernel(const __grid_constant__ CUtensorMap tmKr, const __grid_constant__ CUtensorMap tmVr,
                          const __grid_constant__ CUtensorMap tmKm, const __grid_constant__ CUtensorMap tmVm,
                          const DaArgs a) {
  constexpr int NVB = DV / 64;        // V boxes per chunk
  constexpr int NOT = DV / 8;         // O n-tiles
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem<1024>(smem_raw);
  __shared__ __align__(8) uint64_t bars[DA_WARPS][DA_STAGES];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane >> 2, tig = lane & 3;
  if (threadIdx.x == 0) {
    for (int w = 0; w < DA_WARPS; ++w)
      for (int s = 0; s < DA_STAGES; ++s) mbar_init(smem_u32(&bars[w][s]), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const WaitCtl wc{&abort_flag, a.status, a.wait_ns};
  uint8_t* ring = smem + warp * WARP_BYTES;
  const int G = a.Hq / a.Hkv;
  const int gw = blockIdx.x * DA_WARPS + warp;
  const int n_warps = gridDim.x * DA_WARPS;

  // producer cursor (lane 0): next (unit, chunk) to load
  int pu = gw, pc = 0;
  KeyPlan pk{};
  bool p_valid = false;
  auto p_seek = [&]() {
    // advance to a unit with chunks left
    while (pu < a.n_units) {
      const int sp = pu % a.nsplit, g_b = pu / a.nsplit;
      pk = key_plan(a, g_b / a.Hkv, sp);
      if (pc == 0) pc = pk.c_lo;
      if (pc < pk.c_hi) { p_valid = true; return; }
      pu += n_warps;
      pc = 0;
    }
    p_valid = false;
  };
  int issued = 0;
  auto p_issue = [&]() {
    if (!p_valid) return;
    const int g_b = pu / a.nsplit;
    const int b = g_b / a.Hkv, g = g_b % a.Hkv;
    bool meta;
    int row, cnt;
    chunk_rows(pk, a, b, pc, meta, row, cnt);
    const int s = issued % DA_STAGES;
    uint8_t* st = ring + s * STAGE_BYTES;
    const uint32_t bar = smem_u32(&bars[warp][s]);
    mbar_arrive_expect_tx(bar, K_TILE + NVB * V_BOX);
    tma_load_2d(smem_u32(st), meta ? &tmKm : &tmKr, bar, g * DA_DH, row);
#pragma unroll
    for (int vb = 0; vb < NVB; ++vb)
      tma_load_2d(smem_u32(st + K_TILE + vb * V_BOX), meta ? &tmVm : &tmVr, bar, g * DV + vb * 64, row);
    ++issued;
    ++pc;
    if (pc >= pk.c_hi) {
      pu += n_warps;
      pc = 0;
    }
    p_seek();
  };
  if (lane == 0) {
    p_seek();
    for (int j = 0; j < DA_STAGES; ++j) p_issue();
  }

  int consumed = 0;
  bool ok = true;
  for (int u = gw; u < a.n_units && ok; u += n_warps) {
    const int sp = u % a.nsplit, g_b = u / a.nsplit;
    const int b = g_b / a.Hkv, g = g_b % a.Hkv;
    const KeyPlan kp = key_plan(a, b, sp);
    // Q fragments: rows = heads of group g (rows >= G are zero), k = head dim
    uint32_t qf[DA_DH / 16][4];
    {
      const float qs = 1.4426950408889634f * rsqrtf(static_cast<float>(DA_DH));
      const bool row_ok = grp < G;
      const __half* qr = a.q + b * a.ldq + (g * G + (row_ok ? grp : 0)) * DA_DH;
#pragma unroll
      for (int ks = 0; ks < DA_DH / 16; ++ks) {
        const __half2 lo = *reinterpret_cast<const __half2*>(qr + ks * 16 + 2 * tig);
        const __half2 hi = *reinterpret_cast<const __half2*>(qr + ks * 16 + 8 + 2 * tig);
        const float2 fl = __half22float2(lo), fh = __half22float2(hi);
        qf[ks][0] = row_ok ? pack_bf162(fl.x * qs, fl.y * qs) : 0u;
        qf[ks][1] = 0u;
        qf[ks][2] = row_ok ? pack_bf162(fh.x * qs, fh.y * qs) : 0u;
        qf[ks][3] = 0u;
      }
    }
    float o[NOT][4];
#pragma unroll
    for (int nt = 0; nt < NOT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;  // row grp (rows >= 8 are never read)
    for (int c = kp.c_lo; c < kp.c_hi; ++c) {
      bool meta;
      int row, cnt;
      chunk_rows(kp, a, b, c, meta, row, cnt);
      const int s = consumed % DA_STAGES;
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars[warp][s]), (consumed / DA_STAGES) & 1, wc))) {
        ok = false;
        break;
      }
      const uint8_t* st = ring + s * STAGE_BYTES;
      const uint32_t kb = smem_u32(st), vb0 = smem_u32(st + K_TILE);
      // A partial chunk's tail rows hold other slots (unwritten ones may be
      // anything, NaN included) and get weight 0: clear their V rows so that
      // 0 * V stays 0.  Their scores are masked to -inf below.
      const bool partial = cnt < DK;
      if (partial) {
        const int per_box = (DK - cnt) * 8;  // 16-byte pieces of the tail rows
        for (int i = lane; i < per_box * NVB; i += 32) {
          const int box = i / per_box, r = cnt + (i % per_box) / 8, c16 = i % 8;
          *reinterpret_cast<uint4*>(const_cast<uint8_t*>(st) + K_TILE + box * V_BOX + r * 128 + c16 * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();  // these stores come before the stage's next TMA write
        __syncwarp();
      }
      // ---- S = Q K^T over 64 keys: 8 n-tiles x 4 k-steps
      float sc[DK / 8][4];
#pragma unroll
      for (int nt = 0; nt < DK / 8; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
      for (int nt = 0; nt < DK / 8; ++nt) {
#pragma unroll
        for (int kp2 = 0; kp2 < 2; ++kp2) {  // two k-steps per ldmatrix.x4
          uint32_t bf[4];
          const int key = nt * 8 + (lane & 7);
          ldsm_x4(kb + sw128(key, kp2 * 4 + (lane >> 3)), bf);
          mma_bf16(sc[nt], qf[2 * kp2], bf[0], bf[1]);
          mma_bf16(sc[nt], qf[2 * kp2 + 1], bf[2], bf[3]);
        }
      }
      // ---- online softmax on row grp (columns 2*tig, 2*tig+1 of each n-tile)
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < DK / 8; ++nt) {
        const int j = nt * 8 + 2 * tig;
        if (j >= cnt) sc[nt][0] = -INFINITY;
        if (j + 1 >= cnt) sc[nt][1] = -INFINITY;
        mx = fmaxf(mx, fmaxf(sc[nt][0], sc[nt][1]));
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run, mx);
      const float alpha = ex2_approx(m_run - m_new);
      m_run = m_new;
      float ls = 0.f;
      uint32_t pa[DK / 16][4];  // P as A fragments, one per 16-key k-step
#pragma unroll
      for (int nt = 0; nt < DK / 8; ++nt) {
        const float p0 = ex2_approx(sc[nt][0] - m_new), p1 = ex2_approx(sc[nt][1] - m_new);
        ls += p0 + p1;
        // C layout (row grp, cols 2tig..) of n-tiles 2k, 2k+1 = A layout of k-step k
        pa[nt >> 1][(nt & 1) * 2] = pack_bf162(p0, p1);
        pa[nt >> 1][(nt & 1) * 2 + 1] = 0u;  // rows 8..15
      }
      l_run = l_run * alpha + ls;
#pragma unroll
      for (int nt = 0; nt < NOT; ++nt) {
        o[nt][0] *= alpha;
        o[nt][1] *= alpha;
      }
      // ---- O += P V: 4 k-steps x NOT n-tiles, V fragments by ldmatrix.trans
#pragma unroll
      for (int ks = 0; ks < DK / 16; ++ks) {
#pragma unroll
        for (int np = 0; np < NOT / 2; ++np) {  // pairs of n-tiles = 16 V columns
          uint32_t bf[4];
          const int key = ks * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
          const int chunk = np * 2 + (lane >> 4);  // 16-byte chunk of 8 V columns
          const uint32_t vb = vb0 + (chunk >> 3) * V_BOX;
          ldsm_x4_t(vb + sw128(key, chunk & 7), bf);
          mma_bf16(o[2 * np], pa[ks], bf[0], bf[1]);
          mma_bf16(o[2 * np + 1], pa[ks], bf[2], bf[3]);
        }
      }
      __syncwarp();
      ++consumed;
      if (lane == 0) p_issue();  // the stage just read gets the chunk two ahead
    }
    if (!ok) break;
    // ---- partial result of this unit: rows 0..G-1
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    if (grp < G) {
      float* dst = a.part + ((static_cast<long long>(b) * a.Hq + g * G + grp) * a.nsplit + sp) * (DV + 2);
      const bool empty = kp.c_hi <= kp.c_lo;
      if (tig == 0) {
        dst[0] = empty ? -INFINITY : m_run;
        dst[1] = empty ? 0.f : l_run;
      }
#pragma unroll
      for (int nt = 0; nt < NOT; ++nt)
        *reinterpret_cast<float2*>(dst + 2 + nt * 8 + 2 * tig) = make_float2(o[nt][0], o[nt][1]);
    }
  }
  // a warp that gave up may still have loads in flight: let them land
  if (!ok && lane == 0)
    for (int j = max(0, issued - DA_STAGES); j < issued; ++j)
      mbar_wait_drain(smem_u32(&bars[warp][j % DA_STAGES]), (j / DA_STAGES) & 1, 1000000);
}

bool map_rows(CUtensorMap* m, const void* base, long long rows, int cols, int box_cols) {
  const uint64_t dims[2] = {static_cast<uint64_t>(cols), static_cast<uint64_t>(rows)};
  const uint64_t str[1] = {static_cast<uint64_t>(cols) * 2};
  const uint32_t box[2] = {static_cast<uint32_t>(box_cols), static_cast<uint32_t>(DK)};
  return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

bool decode_attn_tc_supported(int Hq, int Hkv, int dh, int dv) {
  return dh == DA_DH && (dv == 64 || dv == 128) && Hq % Hkv == 0 && Hq / Hkv <= 8;
}

int decode_attn_tc_splits(int B, int Hkv, int num_sms) {
  const long long pairs = static_cast<long long>(B) * Hkv;
  const long long want = 4LL * num_sms * DA_WARPS;  // ~4 units per warp
  return static_cast<int>(std::max(1LL, std::min(16LL, (want + pairs - 1) / pairs)));
}

hymba_status decode_attention_tc(int B, int M, int Hq, int Hkv, int dh, int dv, int window, int cap, int nsplit,
                                 const __half* q, long long ldq, const __nv_bfloat16* k_meta,
                                 const __nv_bfloat16* v_meta, const __nv_bfloat16* k_ring,
                                 const __nv_bfloat16* v_ring, const int32_t* pos, float* part, __half* out,
                                 long long ldo, int num_sms, int32_t* status, uint64_t wait_ns, cudaStream_t st) {
  if (!decode_attn_tc_supported(Hq, Hkv, dh, dv)) return HYMBA_ERR_UNSUPPORTED;
  const uintptr_t al = reinterpret_cast<uintptr_t>(k_ring) | reinterpret_cast<uintptr_t>(v_ring) |
                       reinterpret_cast<uintptr_t>(k_meta) | reinterpret_cast<uintptr_t>(v_meta);
  if (al & 15) return HYMBA_ERR_INVALID;
  CUtensorMap mKr, mVr, mKm, mVm;
  const long long ring_rows = static_cast<long long>(B) * cap;
  if (!map_rows(&mKr, k_ring, ring_rows, Hkv * dh, DA_DH) || !map_rows(&mVr, v_ring, ring_rows, Hkv * dv, 64))
    return HYMBA_ERR_CUDA;
  if (M > 0) {
    if (!map_rows(&mKm, k_meta, M, Hkv * dh, DA_DH) || !map_rows(&mVm, v_meta, M, Hkv * dv, 64)) return HYMBA_ERR_CUDA;
  } else {
    mKm = mKr;  // never read: there are no meta chunks
    mVm = mVr;
  }
  DaArgs a{B, M, Hq, Hkv, dv, window, cap, nsplit, B * Hkv * nsplit, q, ldq, pos, part, status, wait_ns};
  const int smem = DA_WARPS * WARP_BYTES + 1024;
  const int grid = std::max(1, std::min(num_sms, (a.n_units + DA_WARPS - 1) / DA_WARPS));
  if (dv == 128) {
    if (cudaFuncSetAttribute(decode_attn_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return HYMBA_ERR_CUDA;
    if (launch_pdl(decode_attn_tc_kernel<128>, dim3(grid), dim3(DA_WARPS * 32), smem, st, mKr, mVr, mKm, mVm, a) !=
        cudaSuccess)
      return HYMBA_ERR_CUDA;
  } else {
    if (cudaFuncSetAttribute(decode_attn_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return HYMBA_ERR_CUDA;
    if (launch_pdl(decode_attn_tc_kernel<64>, dim3(grid), dim3(DA_WARPS * 32), smem, st, mKr, mVr, mKm, mVm, a) !=
        cudaSuccess)
      return HYMBA_ERR_CUDA;
  }
  if (cudaGetLastError() != cudaSuccess) return HYMBA_ERR_CUDA;
  return decode_attn_combine(B, Hq, dv, nsplit, part, out, ldo, st);
}

}  // namespace hy
