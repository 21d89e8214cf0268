// attn_decode_kt_d64.cu -- the keys-as-rows decode kernel (attn_decode_kt.cuh)
// instantiated for head dim 64.
#include "attn_decode_kt.cuh"

namespace attn45 {

cudaError_t launch_decode_kt_d64(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                 const DecodeParams& p, int grid, bool bf16, cudaStream_t s) {
  return launch_d<64>(q, k, v, p, grid, bf16, s);
}

}  // namespace attn45
