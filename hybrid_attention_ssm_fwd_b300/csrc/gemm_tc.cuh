// tcgen05/TMEM GEMM with fused epilogues: C = A . B^T, A [M, K] and B [N, K]
// both K-major (row-major activations times row-major nn.Linear weights).
#pragma once

#include "common.cuh"

namespace hy {

enum GemmEpi : int {
  EPI_F16 = 0,       // fp16 store (+ RoPE on columns < rope_cols, head_dim 64)
  EPI_XPROJ = 1,     // columns < R -> C2 fp16 (dt input); R..N-1 -> C fp32 at col-R
  EPI_SOFTPLUS = 2,  // C fp32 = softplus(acc + bias[col])
  EPI_F32 = 3,       // C fp32 = acc (+ bf16 or fp32 residual); also C2 fp16 = the same value when C2 is set
  EPI_PARTIAL = 4,   // C fp32 + split*M*ldc = acc (split-K partial sums)
  EPI_ATOMIC = 5,    // C fp32 += acc with vector atomics (split-K into a cleared or residual C)
  EPI_GEGLU = 6,     // columns (2j, 2j+1) = (gate j, up j): C fp16 [., N/2] = GeLU(gate) * up (N % 16 == 0)
};

struct GemmParams {
  int M, N, K;
  int tiles_m, tiles_n, n_kb, splits, kb_per_split, total_tiles;
  void* C;
  long long ldc;
  void* C2;
  long long ldc2;
  const float* bias;
  const __nv_bfloat16* resid;   // EPI_F32: + bf16 residual (ld_resid)
  const float* resid_f32;       // EPI_F32: + fp32 residual (ld_resid); may alias C
  long long ld_resid;
  int xproj_R;
  int rope_cols;          // 0 = no RoPE
  float rope_log2_step;   // log2(inv_freq[i]) = i * rope_log2_step
  int rows_per_seq;       // position = pos_base + row % rows_per_seq when pos == nullptr
  const int32_t* pos;     // decode: position = pos_base + pos[row]
  int pos_base;
  int32_t* status;
  uint64_t wait_ns;
  int cvt_b;  // B is bf16 in memory: converted to fp16 in shared memory before the MMA (A fp16)
  int total_pairs;  // CTA-pair launch: 256-row tile pairs = ceil(tiles_m / 2) * tiles_n
  int pdl;          // 1: programmatic dependent launch (the decode step's GEMMs)
};

// Launch C = A . B^T with the given epilogue.  ab_fmt: 0 fp16, 1 bf16.
// lda/ldb in elements.  bn = 0 picks a tile width; splits >= 1 (EPI_PARTIAL
// only for splits > 1).
hymba_status gemm_tc(int ab_fmt, const void* A, long long lda, const void* B, long long ldb,
                     int epi, GemmParams p, int bn, int splits, int num_sms, cudaStream_t st);

int gemm_pick_bn(int N, bool small_m);

}  // namespace hy
