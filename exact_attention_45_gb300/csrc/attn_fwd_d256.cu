// attn_fwd_d256.cu -- BF16/FP16 forward instantiations for head dim 256: the
// CTA-pair kernel (attn_fwd_pair_kernel.cuh).
#include "fwd_launch.cuh"

namespace attn45 {
cudaError_t launch_fwd_f16_d256(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const CUtensorMap& o, const FwdParams& p, bool causal, bool varlen, bool bf16,
                                int sm_count, cudaStream_t s) {
#define ATTN45_L(CA, VL, BF) return launch_cta_pair<256, CA, VL, BF ? KIND_BF16 : KIND_FP16>(q, k, v, o, p, sm_count, s)
  if (causal) {
    if (varlen) { if (bf16) ATTN45_L(true, true, true); else ATTN45_L(true, true, false); }
    else        { if (bf16) ATTN45_L(true, false, true); else ATTN45_L(true, false, false); }
  } else {
    if (varlen) { if (bf16) ATTN45_L(false, true, true); else ATTN45_L(false, true, false); }
    else        { if (bf16) ATTN45_L(false, false, true); else ATTN45_L(false, false, false); }
  }
#undef ATTN45_L
}
}  // namespace attn45
