// fwd_launch.cuh -- launch helpers for the BF16/FP16 forward instantiations.
#pragma once
#include "attn_fwd2_kernel.cuh"
#include "attn_fwd_kernel.cuh"
#include "launchers.h"

namespace attn45 {

// Persistent grid: one CTA per SM, or fewer when there are fewer work units.
inline int persistent_grid(const FwdParams& p, bool varlen, int rows_per_unit, int sm_count, int* ntiles) {
  long long units;
  if (varlen) {
    *ntiles = 0;  // counted on the device from cu_seqlens
    units = (long long)p.H * ((p.total + rows_per_unit - 1) / rows_per_unit + p.nseq);
  } else {
    units = (long long)p.nseq * p.H * ((p.N + rows_per_unit - 1) / rows_per_unit);
    *ntiles = (int)units;
  }
  return (int)(units < sm_count ? units : sm_count);
}

// One 128-row query tile per CTA (used for head dim 256; O leaves through plain
// stores, so it takes no output map).
template <int D, int BN, int ST, bool CAUSAL, bool VARLEN, bool BF16>
cudaError_t launch_f16_single(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, FwdParams p,
                              int sm_count, cudaStream_t stream) {
  static_assert(BN == f16_block_n(D), "tensor-map box height and kernel BN must agree");
  using T = Bf16Traits<D, BN, ST>;
  auto kern = attn_fwd_f16_kernel<D, BN, ST, CAUSAL, VARLEN, BF16>;
  const int grid = persistent_grid(p, VARLEN, BLOCK_M, sm_count, &p.ntiles);
  const int smem = T::SMEM_FIXED + (VARLEN ? 4 * (p.nseq + 1) : 0);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, 192, smem, stream>>>(q, k, v, p);
  return cudaGetLastError();
}

// Two 128-row query tiles per CTA (head dims 64 and 128).
// DECODE: p.ntiles holds the number of (sequence, KV head, split) units.
template <int D, int BN, int ST, bool CAUSAL, bool VARLEN, int KIND, bool DECODE = false>
cudaError_t launch_pair(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& o,
                        FwdParams p, int sm_count, cudaStream_t stream) {
  static_assert(BN == f16_block_n(D), "tensor-map box height and kernel BN must agree");
  using T = Pair2Traits<D, BN, ST, KIND == KIND_E4M3 ? 1 : 2, !VARLEN && !DECODE>;
  auto kern = attn_fwd2_kernel<D, BN, ST, CAUSAL, VARLEN, KIND, DECODE>;
  const int grid = DECODE ? (p.ntiles < sm_count ? p.ntiles : sm_count)
                          : persistent_grid(p, VARLEN, SUPER_M, sm_count, &p.ntiles);
  const int smem = T::SMEM_FIXED + (VARLEN ? 4 * (p.nseq + 1) : 0);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, 384, smem, stream>>>(q, k, v, o, p);
  return cudaGetLastError();
}

template <int D, int BN, int ST, bool PAIR, bool CA, bool VL, bool BF>
cudaError_t launch_f16_one(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& o,
                           const FwdParams& p, int sm_count, cudaStream_t s) {
  if constexpr (PAIR) return launch_pair<D, BN, ST, CA, VL, BF ? KIND_BF16 : KIND_FP16>(q, k, v, o, p, sm_count, s);
  else return launch_f16_single<D, BN, ST, CA, VL, BF>(q, k, v, p, sm_count, s);
}

template <int D, int BN, int ST, bool PAIR>
cudaError_t launch_f16_dispatch(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const CUtensorMap& o, const FwdParams& p, bool causal, bool varlen, bool bf16, int sm_count,
                                cudaStream_t s) {
#define ATTN45_L(CA, VL, BF) return launch_f16_one<D, BN, ST, PAIR, CA, VL, BF>(q, k, v, o, p, sm_count, s)
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
