// attn_common.cuh -- launch parameters and the persistent tile scheduler
// shared by the BF16/FP16 and FP8 forward kernels.
//
// A "tile" is 128 query rows of one (sequence, query head). Tiles are
// independent, so persistent CTAs walk the tile list with a fixed stride
// (tile = blockIdx.x, blockIdx.x + gridDim.x, ...). The list is ordered so
// the heaviest tiles come first when the mask is causal (longest-processing-
// time-first): "FlashAttention-3: Fast and Accurate Attention with Asynchrony
// and Low-precision", reference list footnote on the benchmark setup (the
// FP16 kernel is persistent with a load-balancing strategy). Query heads are
// the fastest-moving index so the H/Hkv query heads that share one K/V head
// (grouped-query attention) run at the same time and share K/V through L2.
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
  int ntiles;              // fixed: B*H*ceil(N/128); varlen: computed on device
  int vt_ld;               // FP8 only: row stride (keys) of transposed V
  int fp8_block;           // FP8 only: 1 = per-block/per-channel scales, 0 = per-tensor
  float scale_log2;        // softmax scale * log2(e)
  const int* seqlens;      // decode only: cached keys per sequence (device, nseq)
  int num_splits;          // decode only: key-range splits per (sequence, KV head)
  const int* blk_off;      // FP8 packed sequences: first 128-row block of each sequence
  int tmax;                // FP8 packed sequences: columns of the block-scale rows
  int split_chunk;         // decode only: keys per split (a multiple of 128)
  unsigned long long timeout_ns;
  unsigned int* err;       // device error word
};

struct Tile {
  int seq;       // batch index (fixed) or sequence index (varlen)
  int h;         // query head
  int qblk;      // 128-row block index within the sequence
  int n;         // sequence length
  int tok0;      // token index of the sequence's first row
  int tma_row0;  // TMA row coordinate of the sequence start (fixed: 0, varlen: tok0)
  int tma_b;     // TMA batch coordinate (fixed: b, varlen: 0)
};

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Fixed length: tile t -> (qblk descending, batch, head).
__device__ __forceinline__ Tile tile_fixed(const FwdParams& p, int t) {
  const int nqb = ceil_div(p.N, BLOCK_M);
  const int bh_count = p.nseq * p.H;
  Tile T;
  T.qblk = nqb - 1 - t / bh_count;
  const int bh = t % bh_count;
  T.seq = bh / p.H;
  T.h = bh % p.H;
  T.n = p.N;
  T.tok0 = T.seq * p.N;
  T.tma_row0 = 0;
  T.tma_b = T.seq;
  return T;
}

// Varlen: tile t -> sequence by binary search over the per-sequence tile
// prefix (prefix[s] = H * sum_{s' < s} ceil(n_s'/128)), then (qblk
// descending, head) within the sequence.
__device__ __forceinline__ Tile tile_varlen(const FwdParams& p, const int* prefix, int t) {
  int lo = 0, hi = p.nseq - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= t) lo = mid; else hi = mid - 1;
  }
  Tile T;
  T.seq = lo;
  const int r = t - prefix[lo];
  const int a = __ldg(p.cu_seqlens + lo), b = __ldg(p.cu_seqlens + lo + 1);
  T.n = b - a;
  const int nqb = ceil_div(T.n, BLOCK_M);
  T.qblk = nqb - 1 - r / p.H;
  T.h = r % p.H;
  T.tok0 = a;
  T.tma_row0 = a;
  T.tma_b = 0;
  return T;
}

// Fills prefix[0..nseq] (shared memory) from cu_seqlens; all threads of the
// block must call it. Uses warp 0 for the scan.
__device__ __forceinline__ void build_varlen_prefix(const FwdParams& p, int* prefix) {
  for (int s = threadIdx.x; s < p.nseq; s += blockDim.x) {
    const int n = __ldg(p.cu_seqlens + s + 1) - __ldg(p.cu_seqlens + s);
    prefix[s + 1] = (n > 0 ? ceil_div(n, BLOCK_M) : 0) * p.H;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int carry = 0;
    for (int base = 0; base < p.nseq; base += 32) {
      const int s = base + lane;
      int v = s < p.nseq ? prefix[s + 1] : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += u;
      }
      if (s < p.nseq) prefix[s + 1] = v + carry;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) prefix[0] = 0;
  }
  __syncthreads();
}

}  // namespace attn45
