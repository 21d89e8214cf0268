// attn_fwd_fp8.cu -- FP8 (e4m3) forward instantiations: head dim 128 on the
// two-tile kernel (fixed length and packed sequences), head dim 256 on CTA
// pairs (fixed length).
#include "fp8_launchers.h"
#include "fwd_launch.cuh"

namespace attn45 {
cudaError_t launch_fwd_fp8_d128(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const CUtensorMap& o, const FwdParams& p, bool causal, bool varlen, int sm_count,
                                cudaStream_t s) {
  if (varlen) {
    if (causal) return launch_pair<128, 128, 4, true, true, KIND_E4M3>(q, k, v, o, p, sm_count, s);
    return launch_pair<128, 128, 4, false, true, KIND_E4M3>(q, k, v, o, p, sm_count, s);
  }
  if (causal) return launch_pair<128, 128, 4, true, false, KIND_E4M3>(q, k, v, o, p, sm_count, s);
  return launch_pair<128, 128, 4, false, false, KIND_E4M3>(q, k, v, o, p, sm_count, s);
}

cudaError_t launch_fwd_fp8_d256(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const CUtensorMap& o, const FwdParams& p, bool causal, int sm_count, cudaStream_t s) {
  if (causal) return launch_cta_pair<256, true, false, KIND_E4M3>(q, k, v, o, p, sm_count, s);
  return launch_cta_pair<256, false, false, KIND_E4M3>(q, k, v, o, p, sm_count, s);
}
}  // namespace attn45
