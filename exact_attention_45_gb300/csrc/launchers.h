// launchers.h -- host-side entry points into the kernel translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include "attn_common.cuh"

namespace attn45 {

// Key-block rows (BN) of the BF16/FP16 forward kernel for head dim d; the
// K/V tensor maps use this as their box height.
constexpr int f16_block_n(int d) { return d == 256 ? 64 : 128; }
constexpr int F16_THREADS = 192;

// o: output map {d, heads, rows, batch} with 64-element x 32-row boxes (bulk
// stores of the epilogue; fixed-length launches only).
cudaError_t launch_fwd_f16_d64(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                               const CUtensorMap& o, const FwdParams& p, bool causal, bool varlen, bool bf16, int sm_count,
                               cudaStream_t s);
cudaError_t launch_fwd_f16_d128(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const CUtensorMap& o, const FwdParams& p, bool causal, bool varlen, bool bf16, int sm_count,
                                cudaStream_t s);
// Split-KV decode units of the two-tile kernel (head dim 64 or 128): fp32
// partial O [splits][B][H][d] to p.o and partial lse [splits][B][H] to p.lse.
cudaError_t launch_decode_f16(int d, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                              const FwdParams& p, bool bf16, int sm_count, cudaStream_t s);
// Decode units with the keys on the TMEM lanes (head dim 128, group = H/Hkv
// <= 16): one CTA per (sequence, KV head, split), p.ntiles of them; k, v maps
// with 64-element x 128-row boxes; writes the same partials as
// launch_decode_f16.
bool decode_kt_supported(int d, int group);
cudaError_t launch_decode_kt(int group, const CUtensorMap& k, const CUtensorMap& v, const void* q,
                             const FwdParams& p, bool bf16, cudaStream_t s);
// Merge of per-split partials into O (bf16/fp16) and lse; splits with lse =
// -inf are skipped without reading their O.
cudaError_t launch_combine(const float* o_parts, const float* lse_parts, void* o, float* lse, int splits, int rows,
                           int d, bool bf16, cudaStream_t s);

cudaError_t launch_fwd_f16_d256(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const CUtensorMap& o, const FwdParams& p, bool causal, bool varlen, bool bf16, int sm_count,
                                cudaStream_t s);

}  // namespace attn45
