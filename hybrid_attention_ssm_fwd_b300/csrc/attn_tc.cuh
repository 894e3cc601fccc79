// Flash attention on tcgen05 for the attention branch: causal GQA over the
// meta prefix united with the sliding window (or global).
#pragma once

#include "common.cuh"

namespace hy {

bool attn_tc_supported(int dh, int dv);

// Q rows [B*L, ldq] (head h at column h*dh), K/V rows with strides ldk/ldv
// (KV head g at g*dh / g*dv), O [B*L, ldo] (head h at h*dv); all fp16.
hymba_status attn_tc(int B, int L, int M, int Hq, int Hkv, int dh, int dv, int window, const __half* Q,
                     long long ldq, const __half* K, long long ldk, const __half* V, long long ldv, __half* O,
                     long long ldo, int32_t* status, uint64_t wait_ns, int num_sms, cudaStream_t st);

// The same with the M meta keys taken from their own tensors Km [M, Hkv, dh]
// and Vm [M, Hkv, dv] (fp16, shared by the batch) and only the T real rows
// in Q, K, V and O ([B*T, ld]); positions stay logical (meta rows first).
// Needs M a positive multiple of 64.
hymba_status attn_tc_meta(int B, int T, int M, const __half* Km, const __half* Vm, int Hq, int Hkv, int dh, int dv,
                          int window, const __half* Q, long long ldq, const __half* K, long long ldk, const __half* V,
                          long long ldv, __half* O, long long ldo, int32_t* status, uint64_t wait_ns, int num_sms,
                          cudaStream_t st);

}  // namespace hy
