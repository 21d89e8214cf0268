// attn_decode_kt.cu -- entry points of the keys-as-rows decode kernel
// (attn_decode_kt.cuh); head dim 128 is instantiated here, head dim 64 in
// attn_decode_kt_d64.cu.
#include "attn_decode_kt.cuh"

namespace attn45 {

bool decode_kt_supported(int d, int group) {
  return (d == 64 || d == 128) && ((group >= 1 && group <= 16) || group == 24 || group == 32);
}

int decode_kt_q_rows(int group) { return group <= 16 ? 16 : 32; }

cudaError_t launch_decode_kt(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                             const DecodeParams& p, int d, int grid, bool bf16, cudaStream_t s) {
  return d == 64 ? launch_decode_kt_d64(q, k, v, p, grid, bf16, s) : launch_d<128>(q, k, v, p, grid, bf16, s);
}

}  // namespace attn45
