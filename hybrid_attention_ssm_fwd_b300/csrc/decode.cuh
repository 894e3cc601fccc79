// Kernels specific to the single-token decode step.
#pragma once

#include "common.cuh"

namespace hy {

// K/V of the new token (columns k_col / v_col of proj [B, ldp]) into slot
// pos[b] % cap (window > 0) or pos[b] (global) of the ring.
template <typename TS, typename TC>
hymba_status kv_append(int B, int Hkv, int dh, int dv, int window, int cap, const TS* proj, long long ldp,
                       int k_col, int v_col, const int32_t* pos, TC* k_ring, TC* v_ring, cudaStream_t st);

// Attention of one new token per sequence over the meta K/V plus the last
// min(pos+1, window) ring entries (pos+1 when global).  q: proj rows (head h
// at h*dh), out [B, ldo] (head h at h*dv).
template <typename TQ, typename TC>
hymba_status decode_attention(int B, int M, int Hq, int Hkv, int dh, int dv, int window, int cap,
                              const TQ* q, long long ldq, const TC* k_meta, const TC* v_meta,
                              const TC* k_ring, const TC* v_ring, const int32_t* pos, TQ* out, long long ldo,
                              cudaStream_t st);

// One conv step from the carried tail: u = silu(sum w * [tail, x] + b); the
// tail is shifted in place to end with x.
template <typename T>
hymba_status conv_step(int B, int di, int k, const T* x, long long ldx, const float* w, const float* bias,
                       float* conv_state, T* u, long long ldu, cudaStream_t st);

enum ReduceEpi : int { RE_XPROJ = 0, RE_F32 = 1 };

// Sums split-K partials part[s][rows][ldp] and applies the epilogue:
//   RE_XPROJ: col < R -> dtr (fp16, ld ldd), else BC[row, col-R] (fp32, ld ldc)
//   RE_F32:   C[row, col] = sum (+ bf16 residual) (+ C itself if accumulate)
hymba_status splitk_reduce(int splits, int rows, int N, const float* part, long long ldp, int epi, int R,
                           __half* dtr, long long ldd, float* C, long long ldc, const __nv_bfloat16* resid,
                           long long ld_resid, bool accumulate, cudaStream_t st);

// Split-KV decode attention over bf16 caches (one CTA per sequence, KV group
// and key split; all query heads of a group share each K/V read), followed by
// the merge of the splits into out (fp16).  `part` is scratch of
// decode_attn_split_scratch() bytes; max_keys bounds M + visible ring entries.
bool decode_attn_split_supported(int Hq, int Hkv, int dh, int dv);
size_t decode_attn_split_scratch(int B, int Hq, int dv, int nsplit);
hymba_status decode_attention_split(int B, int M, int Hq, int Hkv, int dh, int dv, int window, int cap, int nsplit,
                                    const __half* q, long long ldq, const __nv_bfloat16* k_meta,
                                    const __nv_bfloat16* v_meta, const __nv_bfloat16* k_ring,
                                    const __nv_bfloat16* v_ring, const int32_t* pos, float* part, __half* out,
                                    long long ldo, int max_keys, cudaStream_t st);

// Merges per-split partials (m in log2 units, l, unnormalised o[dv]) into
// out [B, Hq*dv] fp16.
hymba_status decode_attn_combine(int B, int Hq, int dv, int nsplit, const float* part, __half* out, long long ldo,
                                 cudaStream_t st);

// Decode attention on persistent TMA-fed warps with mma.sync (see
// decode_attn.cu): dh == 64, dv in {64, 128}, Hq / Hkv <= 8, bf16 caches.
// part needs decode_attn_split_scratch(B, Hq, dv, nsplit) bytes; nsplit from
// decode_attn_tc_splits.
bool decode_attn_tc_supported(int Hq, int Hkv, int dh, int dv);
int decode_attn_tc_splits(int B, int Hkv, int num_sms);
hymba_status decode_attention_tc(int B, int M, int Hq, int Hkv, int dh, int dv, int window, int cap, int nsplit,
                                 const __half* q, long long ldq, const __nv_bfloat16* k_meta,
                                 const __nv_bfloat16* v_meta, const __nv_bfloat16* k_ring,
                                 const __nv_bfloat16* v_ring, const int32_t* pos, float* part, __half* out,
                                 long long ldo, int num_sms, int32_t* status, uint64_t wait_ns, cudaStream_t st);

// Decode step of the SSM branch with the dt projection fused (see decode.cu);
// pos (may be null) is advanced by one for every sequence.
bool decode_ssm_step_supported(int N, int R);
// xp [B, ld_xp] fp32 = the x projection [dt (R) | B (N) | C (N)] of each sequence.
hymba_status decode_ssm_step(int B, int di, int N, int R, const __half* u, long long ldu, const __half* z,
                             long long ldz, const float* xp, long long ld_xp, const __nv_bfloat16* W_dt, const float* dt_bias, const float* A_log, const float* D,
                             float* state, __half* g, long long ldg, int32_t* pos, cudaStream_t st);

hymba_status pos_increment(int B, int32_t* pos, cudaStream_t st);

// The ring append of the new token's K/V (when append) and the conv step in
// one launch: u = silu(conv), conv_state shifted in place.
hymba_status decode_prep(int B, int di, int k, const __half* proj, long long ldp, int x_col, int k_col, int v_col,
                         int Hkv, int dh, int dv, int window, int cap, const int32_t* pos, __nv_bfloat16* k_ring,
                         __nv_bfloat16* v_ring, const float* conv_w, const float* conv_b, float* conv_state,
                         __half* u, long long ldu, bool append, cudaStream_t st);

}  // namespace hy
