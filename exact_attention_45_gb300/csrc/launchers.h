// launchers.h -- host-side entry points into the kernel translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include "attn_common.cuh"

namespace attn45 {

// Rows of the K tensor map's boxes of the BF16/FP16 forward for head dim d:
// the key block (BN = 128) for d = 64, 128; for d = 256 (CTA pairs, 128-key
// blocks) each CTA loads 64 of a block's keys.
constexpr int f16_block_n(int d) { return d == 256 ? 64 : 128; }
// Rows of the V tensor map's boxes: 128 keys (d = 256: each CTA of a pair
// loads 128 keys x its 128 channels).
constexpr int f16_v_box_rows(int d) { return d == 256 ? 128 : f16_block_n(d); }

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
// Decode with the keys on the TMEM lanes (head dim 64/128, group = H/Hkv <= 32).
// The tiles of all (sequence, KV head) units, in that order, are cut into
// `grid` equal contiguous ranges, one per CTA. A CTA holding a whole unit
// writes its O and lse; otherwise each run of a range inside unit u leaves a
// partial (fp32 O normalised by its own sum, and its lse) in slot u + cta,
// rows slot * group + head-in-group, and the CTA that completes the unit's
// count merges them. Counters hold (epoch << 32) | pieces counted, so a new
// epoch per call needs no reset.
struct DecodeParams {
  float* o_parts;                 // [slots * group][d]
  float* lse_parts;               // [slots * group]
  unsigned long long* counters;   // [B * Hkv]
  void* o;                        // [B, H, d], bf16 / fp16
  float* lse;                     // [B, H]
  const int* seqlens;             // [B], clamped to [0, Nmax]
  int B, H, Hkv, group, Nmax;
  unsigned int epoch;             // != 0, different for every call sharing the counters
  float scale_log2;
  unsigned long long timeout_ns;
  unsigned int* err;
};
constexpr int DECODE_KT_MAX_GRID = 256;
// Shapes the kernel takes: d = 64 or 128, group in 1..16, 24 or 32.
bool decode_kt_supported(int d, int group);
// Rows of the q map's boxes: the group's heads padded to the MMA's N (16 or 32).
int decode_kt_q_rows(int group);
// q: [B*H, d] map with 64 x decode_kt_q_rows(group)-row boxes; k, v: cache
// maps with 64 x 128-row boxes; 1 <= grid <= DECODE_KT_MAX_GRID.
cudaError_t launch_decode_kt(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                             const DecodeParams& p, int d, int grid, bool bf16, cudaStream_t s);
// Merge of per-split partials into O (bf16/fp16) and lse; splits with lse =
// -inf are skipped without reading their O.
cudaError_t launch_combine(const float* o_parts, const float* lse_parts, void* o, float* lse, int splits, int rows,
                           int d, bool bf16, cudaStream_t s);

cudaError_t launch_fwd_f16_d256(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const CUtensorMap& o, const FwdParams& p, bool causal, bool varlen, bool bf16, int sm_count,
                                cudaStream_t s);

}  // namespace attn45
