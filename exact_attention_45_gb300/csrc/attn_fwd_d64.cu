// attn_fwd_d64.cu -- BF16/FP16 forward instantiations for head dim 64.
#include "fwd_launch.cuh"

namespace attn45 {
cudaError_t launch_fwd_f16_d64(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                               const CUtensorMap& o,
                               const FwdParams& p, bool causal, bool varlen, bool bf16, int sm_count,
                               cudaStream_t s) {
  return launch_f16_dispatch<64, f16_block_n(64), 4>(q, k, v, o, p, causal, varlen, bf16, sm_count, s);
}
}  // namespace attn45
