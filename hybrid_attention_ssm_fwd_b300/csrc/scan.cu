// Selective scan + gate (bf16 path) and the bounded-wait probe.
#include "scan.cuh"
#include "simt.cuh"

namespace hy {
namespace {

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

}  // namespace

hymba_status scan_f16(int B, int L, int di, int N, const __half* u, long long ld_u, const __half* z,
                      long long ld_z, const float* delta, const float* BC, const float* A_log, const float* D,
                      __half* g, const float* h0, float* h_out, cudaStream_t st) {
  return scan_simt<__half>(B, L, di, N, u, ld_u, z, ld_z, delta, di, BC, BC + N, 2 * N, A_log, D, g, di, h0, h_out,
                           st);
}

hymba_status wait_timeout_probe(uint32_t limit_us, int32_t* status, cudaStream_t st) {
  wait_probe_kernel<<<1, 32, 0, st>>>(static_cast<uint64_t>(limit_us) * 1000ull, status);
  return cudaGetLastError() == cudaSuccess ? HYMBA_OK : HYMBA_ERR_CUDA;
}

}  // namespace hy
