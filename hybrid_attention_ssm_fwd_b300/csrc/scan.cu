// Selective scan + gate of the SSM branch on the bf16 path, and the
// bounded-wait probe.
//
// Recurrence (per batch b, channel c, state n), run literally in time:
//     h_t = exp(delta_t * A) * h_{t-1} + (delta_t * u_t) * B_t
//     y_t = C_t . h_t + D * u_t,   g_t = y_t * silu(z_t),   A = -exp(A_log)
// The state stays in registers for the whole sequence.  Two threads share a
// channel (8 states each) and combine C.h with one shuffle; a block of 64
// threads owns 32 channels of one sequence.  Time is walked in chunks of 32
// rows whose delta / u / z / [B|C] tiles arrive by TMA into a 2-stage shared
// memory ring, so every global read is a full coalesced tile and the scan
// itself only touches shared memory.  g is staged per chunk and written back
// with 16-byte stores.
#include "scan.cuh"
#include "simt.cuh"

namespace hy {
namespace {

constexpr int SC_CH = 32;      // channels per block
constexpr int SC_T = 32;       // time rows per chunk
constexpr int SC_THREADS = 64;

template <int NH>  // states per thread (N = 2 * NH)
struct ScanCfg {
  static constexpr int N = 2 * NH;
  static constexpr int D_BYTES = SC_T * SC_CH * 4;
  static constexpr int U_BYTES = SC_T * SC_CH * 2;
  static constexpr int Z_BYTES = SC_T * SC_CH * 2;
  static constexpr int BC_BYTES = SC_T * 2 * N * 4;
  static constexpr int STAGE = D_BYTES + U_BYTES + Z_BYTES + BC_BYTES;
  static constexpr int OFF_G = 2 * STAGE;
  static constexpr int OFF_BAR = OFF_G + SC_T * SC_CH * 2;
  static constexpr int SMEM = 128 + OFF_BAR + 64;
};

template <int NH>
__global__ void __launch_bounds__(SC_THREADS)
    scan_tc_kernel(const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmU,
                   const __grid_constant__ CUtensorMap tmZ, const __grid_constant__ CUtensorMap tmBC, int L, int di,
                   const float* __restrict__ A_log, const float* __restrict__ Dp, __half* __restrict__ g,
                   const float* __restrict__ h0, float* __restrict__ h_out, int32_t* status, uint64_t wait_ns) {
  using Cfg = ScanCfg<NH>;
  constexpr int N = Cfg::N;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
  __shared__ int abort_flag;
  __half* sg = reinterpret_cast<__half*>(smem + Cfg::OFF_G);

  const int tid = threadIdx.x;
  const int cl = tid >> 1;          // channel within block
  const int half = tid & 1;         // which 8 states
  const int c0 = blockIdx.x * SC_CH;
  const int b = blockIdx.y;
  const int c = c0 + cl;
  const long long row0 = static_cast<long long>(b) * L;
  const int n_chunks = (L + SC_T - 1) / SC_T;

  if (tid == 0) {
    mbar_init(smem_u32(&bars[0]), 1);
    mbar_init(smem_u32(&bars[1]), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtl wc{&abort_flag, status, wait_ns};

  auto issue = [&](int k) {
    const int s = k & 1;
    uint8_t* st = smem + s * Cfg::STAGE;
    const uint32_t bar = smem_u32(&bars[s]);
    const int r = static_cast<int>(row0) + k * SC_T;
    mbar_arrive_expect_tx(bar, Cfg::STAGE);
    tma_load_2d(smem_u32(st), &tmD, bar, c0, r);
    tma_load_2d(smem_u32(st + Cfg::D_BYTES), &tmU, bar, c0, r);
    tma_load_2d(smem_u32(st + Cfg::D_BYTES + Cfg::U_BYTES), &tmZ, bar, c0, r);
    tma_load_2d(smem_u32(st + Cfg::D_BYTES + Cfg::U_BYTES + Cfg::Z_BYTES), &tmBC, bar, 0, r);
  };
  if (tid == 0) {
    issue(0);
    if (n_chunks > 1) issue(1);
  }

  // per-thread constants: A * log2(e) for its states, D, initial state
  float A2[NH], h[NH];
#pragma unroll
  for (int n = 0; n < NH; ++n) {
    A2[n] = -__expf(A_log[c * N + half * NH + n]) * 1.4426950408889634f;
    h[n] = h0 ? h0[(static_cast<long long>(b) * di + c) * N + half * NH + n] : 0.f;
  }
  const float Dc = Dp[c];

  int kfail = -1;
  for (int k = 0; k < n_chunks; ++k) {
    const int s = k & 1;
    bool got = mbar_wait(smem_u32(&bars[s]), (k >> 1) & 1, wc);
    if (!__syncthreads_and(got)) {
      kfail = k;
      break;
    }
    const uint8_t* st = smem + s * Cfg::STAGE;
    const float* sD = reinterpret_cast<const float*>(st);
    const __half* sU = reinterpret_cast<const __half*>(st + Cfg::D_BYTES);
    const __half* sZ = reinterpret_cast<const __half*>(st + Cfg::D_BYTES + Cfg::U_BYTES);
    const float* sBC = reinterpret_cast<const float*>(st + Cfg::D_BYTES + Cfg::U_BYTES + Cfg::Z_BYTES);
    const int nt = min(SC_T, L - k * SC_T);
#pragma unroll 2
    for (int t = 0; t < nt; ++t) {
      const float dt = sD[t * SC_CH + cl];
      const float uu = __half2float(sU[t * SC_CH + cl]);
      const float du = dt * uu;
      const float4* Bp = reinterpret_cast<const float4*>(sBC + t * 2 * N + half * NH);
      const float4* Cp = reinterpret_cast<const float4*>(sBC + t * 2 * N + N + half * NH);
      float Bv[NH], Cv[NH];
#pragma unroll
      for (int q = 0; q < NH / 4; ++q) {
        const float4 bb = Bp[q], cc = Cp[q];
        Bv[4 * q] = bb.x; Bv[4 * q + 1] = bb.y; Bv[4 * q + 2] = bb.z; Bv[4 * q + 3] = bb.w;
        Cv[4 * q] = cc.x; Cv[4 * q + 1] = cc.y; Cv[4 * q + 2] = cc.z; Cv[4 * q + 3] = cc.w;
      }
      float yp = 0.f;
#pragma unroll
      for (int n = 0; n < NH; ++n) {
        const float a = ex2_approx(dt * A2[n]);
        h[n] = fmaf(a, h[n], du * Bv[n]);
        yp = fmaf(Cv[n], h[n], yp);
      }
      yp += __shfl_xor_sync(0xffffffffu, yp, 1);
      if (half == 0) {
        const float zz = __half2float(sZ[t * SC_CH + cl]);
        const float y = fmaf(Dc, uu, yp);
        sg[t * SC_CH + cl] = __float2half_rn(y * zz / (1.0f + __expf(-zz)));
      }
    }
    __syncthreads();
    // stage s is consumed: refill it with chunk k + 2 while g is written back
    if (tid == 0 && k + 2 < n_chunks) issue(k + 2);
    // g rows of this chunk: nt x 32 fp16 = nt x 64 bytes, 16 bytes per thread-step
    for (int idx = tid; idx < nt * 4; idx += SC_THREADS) {
      const int t = idx >> 2, q = idx & 3;
      *reinterpret_cast<uint4*>(g + (row0 + k * SC_T + t) * di + c0 + q * 8) =
          *reinterpret_cast<const uint4*>(sg + t * SC_CH + q * 8);
    }
    __syncthreads();
  }
  if (kfail < 0) {
    if (h_out) {
#pragma unroll
      for (int n = 0; n < NH; ++n) h_out[(static_cast<long long>(b) * di + c) * N + half * NH + n] = h[n];
    }
  } else if (tid == 0) {
    // chunks kfail and kfail + 1 may still be landing: let them finish
    for (int kk = kfail; kk < min(kfail + 2, n_chunks); ++kk)
      mbar_wait_drain(smem_u32(&bars[kk & 1]), (kk >> 1) & 1, 1000000);
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
          long long ld, int box_c, int box_r) {
  const uint64_t dims[2] = {static_cast<uint64_t>(cols), static_cast<uint64_t>(rows)};
  const uint64_t str[1] = {static_cast<uint64_t>(ld) * esize};
  const uint32_t box[2] = {static_cast<uint32_t>(box_c), static_cast<uint32_t>(box_r)};
  return encode_tmap(m, dt, 2, base, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

template <int NH>
hymba_status launch_scan(int B, int L, int di, const __half* u, long long ld_u, const __half* z, long long ld_z,
                         const float* delta, const float* BC, const float* A_log, const float* D, __half* g,
                         const float* h0, float* h_out, int32_t* status, uint64_t wait_ns, cudaStream_t st) {
  using Cfg = ScanCfg<NH>;
  const long long rows = static_cast<long long>(B) * L;
  CUtensorMap mD, mU, mZ, mBC;
  if (!map2(&mD, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, delta, di, rows, di, SC_CH, SC_T) ||
      !map2(&mU, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, u, di, rows, ld_u, SC_CH, SC_T) ||
      !map2(&mZ, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, z, di, rows, ld_z, SC_CH, SC_T) ||
      !map2(&mBC, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, BC, 2 * Cfg::N, rows, 2 * Cfg::N, 2 * Cfg::N, SC_T))
    return HYMBA_ERR_CUDA;
  auto kern = scan_tc_kernel<NH>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM) != cudaSuccess)
    return HYMBA_ERR_CUDA;
  dim3 grid(di / SC_CH, B);
  kern<<<grid, SC_THREADS, Cfg::SMEM, st>>>(mD, mU, mZ, mBC, L, di, A_log, D, g, h0, h_out, status, wait_ns);
  return cudaGetLastError() == cudaSuccess ? HYMBA_OK : HYMBA_ERR_CUDA;
}

}  // namespace

hymba_status scan_f16(int B, int L, int di, int N, const __half* u, long long ld_u, const __half* z,
                      long long ld_z, const float* delta, const float* BC, const float* A_log, const float* D,
                      __half* g, const float* h0, float* h_out, int32_t* status, uint64_t wait_ns,
                      cudaStream_t st) {
  auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  const bool tma_ok = di % SC_CH == 0 && ld_u % 8 == 0 && ld_z % 8 == 0 && al(u) && al(z) && al(delta) &&
                      al(BC) && al(g);
  if (tma_ok && N == 16)
    return launch_scan<8>(B, L, di, u, ld_u, z, ld_z, delta, BC, A_log, D, g, h0, h_out, status, wait_ns, st);
  if (tma_ok && N == 8)
    return launch_scan<4>(B, L, di, u, ld_u, z, ld_z, delta, BC, A_log, D, g, h0, h_out, status, wait_ns, st);
  return scan_simt<__half>(B, L, di, N, u, ld_u, z, ld_z, delta, di, BC, BC + N, 2 * N, A_log, D, g, di, h0, h_out,
                           st);
}

hymba_status wait_timeout_probe(uint32_t limit_us, int32_t* status, cudaStream_t st) {
  wait_probe_kernel<<<1, 32, 0, st>>>(static_cast<uint64_t>(limit_us) * 1000ull, status);
  return cudaGetLastError() == cudaSuccess ? HYMBA_OK : HYMBA_ERR_CUDA;
}

}  // namespace hy
