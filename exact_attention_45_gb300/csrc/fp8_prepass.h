// fp8_prepass.h -- arguments of the FP8 pre-pass kernels.
#pragma once
#include <cuda_bf16.h>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace attn45 {

struct PrepassArgs {
  const __nv_bfloat16 *q, *k, *v;  // [B,N,H,d], [B,N,Hkv,d], [B,N,Hkv,d]
  uint8_t *q8, *k8, *vt8;          // codes; vt8 is [B,Hkv,d,ldv]
  float *sq, *sk, *sv;             // scales (hold amax values during the call)
  int B, N, H, Hkv, nblk, ldv;     // nblk = ceil(N/128)
  int block_mode, rotate;
  float inv_sqrt_d;                // fl32(1/sqrt(d))
  uint32_t sign_bits[8];           // bit c set <=> sigma_c = -1 (d <= 256)
  unsigned long long timeout_ns;   // bound for device waits
  unsigned int* err;               // device error word
  // packed sequences (varlen != 0): inputs THD [total, heads, d], sequence s
  // owns tokens [cu[s], cu[s+1]); blk_off [nseq+1] is written by the pre-pass;
  // scales sq [H, tmax], sk [Hkv, tmax], sv [nseq, Hkv, d]; vt8 [Hkv, d, ldv]
  // with ldv = 128 * tmax and sequence s's keys from column 128 * blk_off[s].
  int varlen, nseq, tmax;
  const int* cu;
  int* blk_off;
};

// Tensor maps of the TMA-fed pre-pass kernels (head dim 128, and head dims 64
// and 256 with block scales): bf16 inputs (Q, K, V) {d, heads, N, B} with 64 x
// 128-row boxes, e4m3 outputs {d, heads, N, B} with 128 x 128-row boxes
// (per-tensor scales, d = 128), and (fixed length) the transposed V codes
// {ldv, d, B * Hkv} with 128 keys x min(d, 128) channel-row boxes; 128-byte
// swizzle.
struct Prepass128Maps {
  CUtensorMap in_q, in_k, in_v, out_q, out_k, out_vt;
};

// memsets of the scale outputs, two passes of the pre-pass kernels, finalise.
// maps: required for the TMA-fed kernels (nullptr selects the generic ones).
cudaError_t launch_fp8_prepass(const PrepassArgs& a, int d, const Prepass128Maps* maps, int sm_count,
                               cudaStream_t s);
// Packed sequences: block offsets, two passes, finalise. maps (head dim 128,
// inputs only, over [total, heads, 128] with 64 x 128-row boxes): the fast
// kernels; nullptr: the generic ones.
cudaError_t launch_fp8_prepass_varlen(const PrepassArgs& a, int d, const Prepass128Maps* maps, cudaStream_t s);

}  // namespace attn45
