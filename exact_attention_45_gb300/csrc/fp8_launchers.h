// fp8_launchers.h -- host entry of the FP8 forward kernel (head dim 128).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include "attn_common.cuh"

namespace attn45 {
// q, k: e4m3 maps {d, heads, N, B} with 128 x 128-byte boxes; v: V^T map
// {ldv, d, B*Hkv, 1} with 128-key x d-row boxes; o: bf16 output map {d, H, N,
// B} with 64-element x 32-row boxes (fixed length only). varlen: q, k over
// [total, heads, d], v over [Hkv][d][128 * tmax], p.cu_seqlens, p.blk_off.
cudaError_t launch_fwd_fp8_d128(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const CUtensorMap& o, const FwdParams& p, bool causal, bool varlen, int sm_count,
                                cudaStream_t s);
}  // namespace attn45
