// bwd_launchers.h -- host entry points of the attention backward kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

namespace attn45 {

struct BwdParams {
  const float* lse;        // forward logsumexp [B,H,N] (natural log, scale included)
  const float* dvec;       // D = rowsum(dO * O) [B,H,N]
  float* dq_acc;           // fp32 dQ accumulator [B,N,H,d], zeroed before the launch
  void* dk;                // [B,N,Hkv,d] in the input dtype
  void* dv;                // [B,N,Hkv,d]
  int B, N, H, Hkv, group; // group = H / Hkv
  int nunits;              // B * Hkv * ceil(N / 128) (batch, KV head, key block) units
  float scale;             // softmax scale
  float scale_log2;        // scale * log2(e)
  unsigned long long timeout_ns;
  unsigned int* err;       // device error word
};

// q, k, v, dout: maps {d, heads, N, B} with 64-element x 128-row boxes; dq:
// fp32 accumulator map {d, H, N, B} with 32-element x 128-row boxes (bulk
// reductions), all with 128-byte swizzle.
cudaError_t launch_bwd(int d, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                       const CUtensorMap& dout, const CUtensorMap& dq, const BwdParams& p, bool causal, bool bf16,
                       int sm_count, cudaStream_t s);
cudaError_t launch_bwd_dvec(int d, const void* o, const void* dout, float* dvec, int B, int N, int H, bool bf16,
                            cudaStream_t s);
cudaError_t launch_bwd_dq_convert(const float* acc, void* dq, long long n, bool bf16, cudaStream_t s);

}  // namespace attn45
