// attn_decode.cu -- split-KV decode (one query token per sequence and query
// head over a key/value cache) for the shapes the keys-as-rows kernel
// (attn_decode_kt.cu: head dim 64 or 128 with 1-16, 24 or 32 query heads per
// KV head, see decode_kt_supported) does not take, and the merge of per-split
// partial results.
//
// Decode units run on the two-tile forward kernel: the H/Hkv query heads that
// share one KV head form the rows of tile A (tile B stays empty) and stream
// one key range of the cache, so each unit writes a partial O normalised by
// its own sum and the partial's log-sum-exp. The merge applies the online
// softmax rescaling once across splits ("Related papers: FlashAttention-4"
// page, online-softmax teaser: running maximum and normaliser):
//     lse = m + ln sum_s exp(lse_s - m),  O = sum_s exp(lse_s - lse) O_s.
// Decode-phase attention itself is the setting of the FlashAttention-3 page's
// references [49] (Lean attention, decode phase) and [51] (fast transformer
// decoding with one shared key/value head).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include "fwd_launch.cuh"

namespace attn45 {

cudaError_t launch_decode_f16(int d, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                              const FwdParams& p, bool bf16, int sm_count, cudaStream_t s) {
  // the output map is not read by decode units (partials leave as fp32 rows)
  if (d == 64) {
    if (bf16) return launch_pair<64, 128, 4, false, false, KIND_BF16, true>(q, k, v, q, p, sm_count, s);
    return launch_pair<64, 128, 4, false, false, KIND_FP16, true>(q, k, v, q, p, sm_count, s);
  }
  if (bf16) return launch_pair<128, 128, 2, false, false, KIND_BF16, true>(q, k, v, q, p, sm_count, s);
  return launch_pair<128, 128, 2, false, false, KIND_FP16, true>(q, k, v, q, p, sm_count, s);
}

namespace {

// One block per output row (b, h); each thread owns channels tid, tid + 128.
template <bool BF16>
__global__ void __launch_bounds__(128) combine_kernel(const float* __restrict__ o_parts,
                                                      const float* __restrict__ lse_parts, void* __restrict__ o,
                                                      float* __restrict__ lse, int splits, int rows, int d) {
  const int row = blockIdx.x;
  float m = -INFINITY;
  for (int s = 0; s < splits; ++s) m = fmaxf(m, __ldg(lse_parts + (size_t)s * rows + row));
  float tot = 0.f;
  if (m != -INFINITY)
    for (int s = 0; s < splits; ++s) {
      const float ls = __ldg(lse_parts + (size_t)s * rows + row);
      if (ls != -INFINITY) tot += expf(ls - m);
    }
  const float lse_out = tot > 0.f ? m + logf(tot) : -INFINITY;
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    float acc = 0.f;
    if (tot > 0.f)
      for (int s = 0; s < splits; ++s) {
        const float ls = __ldg(lse_parts + (size_t)s * rows + row);
        if (ls == -INFINITY) continue;            // empty split: its O was never written
        acc += expf(ls - lse_out) * __ldg(o_parts + ((size_t)s * rows + row) * d + c);
      }
    if constexpr (BF16) reinterpret_cast<__nv_bfloat16*>(o)[(size_t)row * d + c] = __float2bfloat16_rn(acc);
    else reinterpret_cast<__half*>(o)[(size_t)row * d + c] = __float2half_rn(acc);
  }
  if (threadIdx.x == 0) lse[row] = lse_out;
}

}  // namespace

cudaError_t launch_combine(const float* o_parts, const float* lse_parts, void* o, float* lse, int splits, int rows,
                           int d, bool bf16, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  if (bf16) combine_kernel<true><<<rows, 128, 0, s>>>(o_parts, lse_parts, o, lse, splits, rows, d);
  else combine_kernel<false><<<rows, 128, 0, s>>>(o_parts, lse_parts, o, lse, splits, rows, d);
  return cudaGetLastError();
}

}  // namespace attn45
