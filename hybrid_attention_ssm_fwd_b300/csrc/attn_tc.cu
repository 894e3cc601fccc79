#include "attn_tc.cuh"

namespace hy {

bool attn_tc_supported(int, int) { return false; }

hymba_status attn_tc(int, int, int, int, int, int, int, int, const __half*, long long, const __half*, long long,
                     const __half*, long long, __half*, long long, int32_t*, uint64_t, int, cudaStream_t) {
  return HYMBA_ERR_UNSUPPORTED;
}

}  // namespace hy
