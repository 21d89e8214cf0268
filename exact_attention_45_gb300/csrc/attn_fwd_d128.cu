// attn_fwd_d128.cu -- BF16/FP16 forward instantiations for head dim 128.
#include "fwd_launch.cuh"

namespace attn45 {
cudaError_t launch_fwd_f16_d128(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const CUtensorMap& o,
                               const FwdParams& p, bool causal, bool varlen, bool bf16, int sm_count,
                               cudaStream_t s) {
  return launch_f16_dispatch<128, f16_block_n(128), 2>(q, k, v, o, p, causal, varlen, bf16, sm_count, s);
}
}  // namespace attn45
