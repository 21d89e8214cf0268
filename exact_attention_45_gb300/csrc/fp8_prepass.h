// fp8_prepass.h -- arguments of the FP8 pre-pass kernels.
#pragma once
#include <cuda_bf16.h>
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
};

// memsets of the scale outputs, two passes of the pre-pass kernel, finalise.
cudaError_t launch_fp8_prepass(const PrepassArgs& a, int d, cudaStream_t s);

}  // namespace attn45
