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
cudaError_t launch_fwd_f16_d256(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const CUtensorMap& o, const FwdParams& p, bool causal, bool varlen, bool bf16, int sm_count,
                                cudaStream_t s);

}  // namespace attn45
