// Selective scan + gate of the SSM branch (bf16 path: fp16 activations,
// fp32 delta / B / C / state), and the bounded-wait probe.
#pragma once

#include "common.cuh"

namespace hy {

// g = (C.h + D u) * silu(z) with h_t = exp(delta_t A) h_{t-1} + delta_t u_t B_t,
// A = -exp(A_log).  u, z fp16 rows (strides ld_u, ld_z); delta fp32 [B, L, di];
// BC fp32 [B, L, 2N] = [B | C]; g fp16 [B, L, di]; h0/h_out [B, di, N] fp32
// (either may be null).  tpc = threads per channel (1, 2 or 4), cpt =
// channels per thread (1, or 2 with tpc 2); tpc 0 = both chosen from B * di
// and the SM count.
hymba_status scan_f16(int B, int L, int di, int N, const __half* u, long long ld_u, const __half* z,
                      long long ld_z, const float* delta, const float* BC, const float* A_log, const float* D,
                      __half* g, const float* h0, float* h_out, int32_t* status, uint64_t wait_ns, int tpc,
                      int cpt, cudaStream_t st);

// Same scan with the dt projection fused in: delta = softplus(dtr . W_dt^T +
// dt_bias) is computed per chunk inside the kernel.  dtr fp16 [B*L, ld_dtr]
// (R valid columns), W_dt bf16 [di, R].
bool scan_fused_supported(int di, int N, int R);  // di % 16 == 0, N == 16, R <= 128
hymba_status scan_fused_f16(int B, int L, int di, int N, int R, const __half* u, long long ld_u, const __half* z,
                            long long ld_z, const __half* dtr, long long ld_dtr, const __nv_bfloat16* W_dt,
                            const float* dt_bias, const float* BC, const float* A_log, const float* D, __half* g,
                            const float* h0, float* h_out, int32_t* status, uint64_t wait_ns, int tpc,
                            int cpt, cudaStream_t st, bool h0_shared = false);  // h0_shared: h0 is [di, N], one for all

// One block waits on an mbarrier nothing arrives on, bounded by limit_us,
// and records HYMBA_ERR_TIMEOUT in *status.
hymba_status wait_timeout_probe(uint32_t limit_us, int32_t* status, cudaStream_t st);

}  // namespace hy
