// fp8_launchers.h -- host entries of the FP8 forward kernels (head dims 128 and 256).
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
// Head dim 256, fixed length, on CTA pairs: q: e4m3 map {256, H, N, B} with
// 128-byte x 128-row boxes; k: the same over Hkv with 64-row boxes (each CTA
// of a pair loads 64 of a block's 128 keys); v: V^T map {ldv, 256, B*Hkv, 1}
// with 128-key x 128-channel-row boxes; o: bf16 map with 64 x 32-row boxes.
cudaError_t launch_fwd_fp8_d256(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const CUtensorMap& o, const FwdParams& p, bool causal, int sm_count, cudaStream_t s);
}  // namespace attn45
