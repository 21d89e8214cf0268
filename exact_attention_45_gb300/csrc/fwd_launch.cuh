// fwd_launch.cuh -- launch helpers for the BF16/FP16 forward instantiations.
#pragma once
#include "attn_fwd2_kernel.cuh"
#include "attn_fwd_pair_kernel.cuh"
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

// CTA pairs (clusters of 2, head dim 256): persistent clusters, at most as
// many as fit on the device at once (cudaOccupancyMaxActiveClusters, looked up
// once per device and instantiation), each walking 256-row units.
template <int D, bool CAUSAL, bool VARLEN, int KIND>
cudaError_t launch_cta_pair(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& o,
                            FwdParams p, int sm_count, cudaStream_t stream) {
  using T = PairTraits<D, KIND == KIND_E4M3 ? 1 : 2>;
  auto kern = attn_fwd_pair_kernel<D, CAUSAL, VARLEN, KIND>;
  const int smem = T::SMEM_FIXED + (VARLEN ? 4 * (p.nseq + 1) : 0);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(T::THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  static int max_clusters[64] = {};     // 0 = not looked up yet
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (max_clusters[dev] == 0) {
    int n = 0;
    cfg.gridDim = dim3(2 * (sm_count / 2), 1, 1);
    if ((e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg)) != cudaSuccess) return e;
    if (n < 1) return cudaErrorLaunchOutOfResources;
    max_clusters[dev] = n;
  }
  int clusters = persistent_grid(p, VARLEN, SUPER_M, max_clusters[dev], &p.ntiles);
  if (clusters < 1) clusters = 1;
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  return cudaLaunchKernelEx(&cfg, kern, q, k, v, o, p);
}

template <int D, int BN, int ST>
cudaError_t launch_f16_dispatch(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const CUtensorMap& o, const FwdParams& p, bool causal, bool varlen, bool bf16, int sm_count,
                                cudaStream_t s) {
#define ATTN45_L(CA, VL, BF) return launch_pair<D, BN, ST, CA, VL, BF ? KIND_BF16 : KIND_FP16>(q, k, v, o, p, sm_count, s)
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
