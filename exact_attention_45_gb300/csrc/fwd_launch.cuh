// fwd_launch.cuh -- launch helper for one BF16/FP16 forward instantiation.
#pragma once
#include "attn_fwd_kernel.cuh"
#include "launchers.h"

namespace attn45 {

template <int D, int BN, int ST, bool CAUSAL, bool VARLEN, bool BF16>
cudaError_t launch_f16_variant(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                               const FwdParams& p, int grid, cudaStream_t stream) {
  static_assert(BN == f16_block_n(D), "tensor-map box height and kernel BN must agree");
  using T = Bf16Traits<D, BN, ST>;
  auto kern = attn_fwd_f16_kernel<D, BN, ST, CAUSAL, VARLEN, BF16>;
  const int smem = T::SMEM_FIXED + (VARLEN ? 4 * (p.nseq + 1) : 0);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, F16_THREADS, smem, stream>>>(q, k, v, p);
  return cudaGetLastError();
}

template <int D, int BN, int ST>
cudaError_t launch_f16_dispatch(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const FwdParams& p, bool causal, bool varlen, bool bf16, int grid,
                                cudaStream_t s) {
#define ATTN45_L(CA, VL, BF) return launch_f16_variant<D, BN, ST, CA, VL, BF>(q, k, v, p, grid, s)
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
