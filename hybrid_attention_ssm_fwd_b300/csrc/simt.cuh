// SIMT kernels: the fp32 path of the layer and the generic pieces shared by
// both precisions (conv + SiLU, fused norm/beta/sum, cache emission, SIMT
// attention and scan used where the tensor-core kernels do not apply).
#pragma once

#include "common.cuh"

namespace hy {

enum SimtEpi : int { SE_STORE = 0, SE_XPROJ = 1, SE_SOFTPLUS = 2, SE_RESID = 3 };

// C = A . B^T in fp32 (A [M,K] lda, B [N,K] ldb), epilogue as for the GEMM:
//   SE_STORE: C[M,N]; SE_XPROJ: col < R -> C2 (ld ldc2), else C[:, col-R];
//   SE_SOFTPLUS: softplus(acc + bias[col]); SE_RESID: acc + resid[row, col].
template <typename TA>
hymba_status gemm_simt(int M, int N, int K, const TA* A, long long lda, const TA* B, long long ldb,
                       int epi, float* C, long long ldc, float* C2, long long ldc2, int R,
                       const float* bias, const TA* resid, long long ld_resid, cudaStream_t st);

// In-place RoPE (rotate-half) on heads [0, n_heads) of width dh at column
// offset col0 of rows [rows, ld]; position = row % rows_per_seq, or
// pos_base + pos[row] when pos is given.
template <typename T>
hymba_status rope_simt(T* X, long long ld, int rows, int col0, int n_heads, int dh, float theta,
                       int rows_per_seq, const int32_t* pos, int pos_base, cudaStream_t st);

// u = silu(causal depthwise conv(x) + b); x [B, L, ld_x] at column offset 0
// (caller offsets the pointer), u [B, L, ld_u].
template <typename TI, typename TO>
hymba_status conv_silu(const TI* x, long long ld_x, TO* u, long long ld_u, int B, int L, int di, int k,
                       const float* w, const float* bias, cudaStream_t st);

// fp16 conv + SiLU fed by TMA (conv.cu): the same result as conv_silu for
// k in 2..4, di % 8 == 0, 16-byte aligned x and u, row strides % 8 == 0.
bool conv_tma_supported(int di, int k, long long ld_x, long long ld_u, const void* x, const void* u);
// tail (may be null): [di, k-1] fp32 history rows (oldest first) used in
// place of the zero padding before row 0 of every sequence.
hymba_status conv_silu_tma(const __half* x, long long ld_x, __half* u, long long ld_u, int B, int L, int di, int k,
                           const float* w, const float* bias, int32_t* status, uint64_t wait_ns, int num_sms,
                           cudaStream_t st, const float* tail = nullptr);

// Generic selective scan + gate, one thread per (b, channel), N <= 64.
// delta fp32 [B,L,di]; BC: B at Bm[row*ld_bc + n], C at Cm[row*ld_bc + n].
// h0 (may be null) initial state, h_out (may be null) final state [B,di,N].
template <typename T>
hymba_status scan_simt(int B, int L, int di, int N, const T* u, long long ld_u, const T* z,
                       long long ld_z, const float* delta, long long ld_delta, const float* Bm,
                       const float* Cm, long long ld_bc, const float* A_log, const float* D, T* g,
                       long long ld_g, const float* h0, float* h_out, cudaStream_t st);

// y = bf16(x / sqrt(mean(x^2) + eps) * w) per row of d fp32 values (d % 4 == 0,
// 16-byte aligned x and w, 8-byte aligned y).
hymba_status rmsnorm_bf16(int rows, int d, const float* x, long long ldx, const float* w, float eps,
                          __nv_bfloat16* y, long long ldy, cudaStream_t st);

// s = beta1 * att / rms(att) + beta2 * g / rms(g), rms over di (rows di wide);
// concat: s = [beta1 * att / rms(att) | beta2 * g / rms(g)] (rows 2 di wide).
template <typename T>
hymba_status fuse_norm(int rows, int di, const T* att, const T* g, const float* beta1,
                       const float* beta2, float eps, T* s, cudaStream_t st, bool concat = false);

// SIMT attention: Q rows [B, L] with row stride ldq (head h at h*dh), K/V
// with strides ldk/ldv (KV head g at g*dh / g*dv), O [B, L, ldo] (head h at
// h*dv).  Visible keys: j <= i and (window == 0 || i - j < window || j < M).
template <typename T>
hymba_status attention_simt(int B, int L, int M, int Hq, int Hkv, int dh, int dv, int window,
                            const T* Q, long long ldq, const T* K, long long ldk, const T* V,
                            long long ldv, T* O, long long ldo, cudaStream_t st);

// Strided 2-D copy with type conversion: dst[r, c] = src[r, c] for r < rows,
// c < cols (elementwise; used for K/V export and weight conversion).
template <typename TS, typename TD>
hymba_status copy2d(const TS* src, long long lds, TD* dst, long long ldd, long long rows, int cols,
                    cudaStream_t st);

// Prefill cache emission: ring K/V (last min(T, cap) tokens at slot t % cap),
// meta K/V (from sequence 0), the conv tail (last k-1 x rows, fp32; rows
// before the first from prev_tail [di, k-1] when given, else zero) and
// pos[b] = T.
template <typename TS, typename TC>
hymba_status emit_cache(int B, int L, int M, int T, int cap, int Hkv, int dh, int dv, int di, int k,
                        const TS* Kp, long long ldk, const TS* Vp, long long ldv, const TS* xp,
                        long long ldx, TC* k_ring, TC* v_ring, TC* k_meta, TC* v_meta,
                        float* conv_state, int32_t* pos, cudaStream_t st,
                        const float* prev_tail = nullptr);

}  // namespace hy
