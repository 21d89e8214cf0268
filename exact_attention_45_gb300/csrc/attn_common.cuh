// attn_common.cuh -- launch parameters shared by the forward kernels (BF16/FP16,
// FP8, decode units). The persistent tile schedulers live beside the kernels
// (attn_fwd2_kernel.cuh: tile2_fixed, tile2_varlen, tile2_decode): work units
// are independent, persistent CTAs walk the unit list with a fixed stride, and
// causal lists run the heaviest units first (longest-processing-time-first;
// "FlashAttention-3: Fast and Accurate Attention with Asynchrony and
// Low-precision", reference list footnote on the benchmark setup: the FP16
// kernel is persistent with a load-balancing strategy).
#pragma once
#include <cuda.h>
#include <cstdint>

namespace attn45 {

constexpr int BLOCK_M = 128;     // query rows per tile (= TMEM lanes)
constexpr int MAX_VARLEN_SEQS = 2048;

struct FwdParams {
  void* o;                 // output rows, same token layout as q
  float* lse;              // fixed: [B,H,N]; varlen: [H,total]
  const int* cu_seqlens;   // varlen only (device, nseq+1); nullptr = fixed length
  const float* sq;         // FP8 only: Q scales
  const float* sk;         // FP8 only: K scales
  const float* sv;         // FP8 only: V scales
  int nseq;                // fixed: B; varlen: number of sequences
  int N;                   // fixed: sequence length; varlen: unused
  int total;               // tokens in q/k/v (fixed: B*N)
  int H, Hkv, group;       // group = H / Hkv
  int ntiles;              // fixed: work units (set by the launcher); varlen: counted on the device
  int vt_ld;               // FP8 only: row stride (keys) of transposed V
  int fp8_block;           // FP8 only: 1 = per-block/per-channel scales, 0 = per-tensor
  int fp8_d;               // FP8 only: head dim of the e4m3 data (0 = the kernel's); 64 runs on the
                           // head-dim-128 kernel: the copies zero-fill channels 64-127, which are not stored
  float scale_log2;        // softmax scale * log2(e)
  const int* seqlens;      // decode only: cached keys per sequence (device, nseq)
  int num_splits;          // decode only: key-range splits per (sequence, KV head)
  const int* blk_off;      // FP8 packed sequences: first 128-row block of each sequence
  int tmax;                // FP8 packed sequences: columns of the block-scale rows
  int split_chunk;         // decode only: keys per split (a multiple of 128)
  unsigned long long timeout_ns;
  unsigned int* err;       // device error word
};

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

}  // namespace attn45
