// attn_fwd2_kernel.cuh -- BF16/FP16 (and FP8) forward, two 128-row query tiles
// per CTA (head dims 64 and 128).
//
// Fused exact attention forward, O = softmax(Q K^T * scale [+ causal mask]) V
// with the per-row logsumexp, tiled over query rows and streamed over key
// blocks so the N x N scores never leave the chip ("FlashAttention: Fast and
// Memory-Efficient Exact Attention with IO-Awareness", abstract), organised so
// the tensor core never waits for a softmax: a CTA owns a 256-row "super tile" of one (sequence,
// head), split into tile A (rows 0-127) and tile B (rows 128-255), which share
// every K/V block loaded into shared memory. Each tile has one TMEM S buffer
// (P is written back over it) and one TMEM O accumulator. The MMA thread
// issues, per key block j,
//     O_A += P_A(j-1) V_{j-1},  S_A(j) = Q_A K_j^T,  O_B += P_B(j-1) V_{j-1},  S_B(j) = Q_B K_j^T
// so while softmax warpgroup A turns S_A(j) into P_A(j) the tensor core runs
// tile B's two GEMMs, and the other way round ("FlashAttention-3: Fast and
// Accurate Attention with Asynchrony and Low-precision", abstract: warp
// specialisation and block-wise interleaving of matmul and softmax; here the
// interleaving is between two tiles through TMEM instead of Hopper registers).
//
// Online softmax ("Related papers: FlashAttention-4" page, online-softmax
// teaser: running maximum and normaliser): the running maximum m is only
// raised when a block's maximum exceeds it by more than 2^8; otherwise the
// stale m keeps being used, P stays <= 2^8 and neither O nor l is rescaled.
// The final O / l and logsumexp are unchanged by this (both use the same m).
//
// Warps 0-3: softmax/correction/epilogue of tile A; warps 4-7: tile B (thread
// r of a warpgroup owns row r = TMEM lane r); warp 8: TMA; warp 9: MMA;
// warp 10: slot watcher; warp 11 idle. Every thread keeps the launch's 168
// registers: moving registers between warpgroups (setmaxnreg) was measured to
// slow the MMA issue loop by more than the softmax gains.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include "attn_common.cuh"
#include "ptx.cuh"

namespace attn45 {

// two floats -> one 32-bit word of bf16 or fp16 (round to nearest even)
__device__ __forceinline__ uint32_t pack2(float lo, float hi, bool bf16) {
  if (bf16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

constexpr int SUPER_M = 2 * BLOCK_M;          // query rows per CTA work unit
// Raise m only past this margin (log2 units). P <= 2^8 then fits 16-bit P and
// encodes to e4m3 without saturation (codes <= 256 < 448) for the FP8 path.
constexpr float LAZY_RESCALE_LOG2 = 8.0f;

// Element kinds of the two-tile kernel.
enum : int { KIND_FP16 = 0, KIND_BF16 = 1, KIND_E4M3 = 2 };

// STAGE_OUT: the epilogue stages each warp's 32 output rows (64 columns at a
// time, 128-byte swizzle) in shared memory and writes them with bulk tensor
// stores; without it (varlen, where a tile's last rows may belong to the next
// sequence) every thread stores its own row.
template <int D, int BN, int STAGES, int ELEM = 2, bool STAGE_OUT = false>
struct Pair2Traits {
  static constexpr int NC = D * ELEM / 128;              // 128-byte chunks per Q/K row
  static constexpr int Q_CHUNK = BLOCK_M * 128;
  static constexpr int KV_CHUNK = BN * 128;
  static constexpr int Q_BYTES = BLOCK_M * D * ELEM;
  static constexpr int KV_BYTES = BN * D * ELEM;          // one K block, or one V (V^T) block
  static constexpr int OFF_Q = 0;                        // Q_A then Q_B
  static constexpr int OFF_K = 2 * Q_BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * KV_BYTES;
  static constexpr int OFF_STAGE = OFF_V + STAGES * KV_BYTES;  // 8 softmax warps x 4 KB
  static constexpr int STAGE_BYTES = STAGE_OUT ? 8 * 4096 : 0;
  static constexpr int OFF_BARS = OFF_STAGE + STAGE_BYTES;
  static constexpr int BARS_BYTES = 512;
  static constexpr int OFF_PREFIX = OFF_BARS + BARS_BYTES;
  static constexpr int SMEM_FIXED = OFF_PREFIX + 1024;
  static constexpr int TMEM_S = 0;                       // + BN * tile
  static constexpr int TMEM_O = 2 * BN;                  // + D * tile
  static constexpr int TMEM_COLS = 512;
  static_assert(2 * BN + 2 * D <= TMEM_COLS, "TMEM budget");
};

// Ring slot j of a super tile holds K_j and V_{j-1} (slots 0..nkv), so each
// key block costs one full and one empty barrier.
struct Bars2 {
  uint64_t q_full, q_empty;
  uint64_t slot_full[4], slot_empty[4];
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t p_part[2][3];                         // P of a block's key parts 0..NP-2 is in TMEM
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars2) <= 512, "barrier block");

// n: keys (= query rows for the square problems); nq: query rows.
// Decode units: h is the KV head, the rows are its H/Hkv query heads
// (qrow0 = first of them), n the keys of split `split`.
struct Tile2 {
  int seq, h, sblk, n, nq, qrow0, split, tok0, tma_row0, tma_b;
};

// Fixed length. Non-causal: head-major (all super tiles of one (b,h) are
// adjacent, so CTAs running together share that head's K/V in L2). Causal:
// longest first (super-tile index descending), heads fastest.
template <bool CAUSAL>
__device__ __forceinline__ Tile2 tile2_fixed(const FwdParams& p, int t) {
  const int nsb = ceil_div(p.N, SUPER_M);
  Tile2 T;
  int bh;
  if (CAUSAL) {
    const int cnt = p.nseq * p.H;
    T.sblk = nsb - 1 - t / cnt;
    bh = t % cnt;
  } else {
    bh = t / nsb;
    T.sblk = t % nsb;
  }
  T.seq = bh / p.H;
  T.h = bh % p.H;
  T.n = p.N;
  T.nq = p.N;
  T.qrow0 = 0;
  T.split = 0;
  T.tok0 = T.seq * p.N;
  T.tma_row0 = 0;
  T.tma_b = T.seq;
  return T;
}

// Varlen: prefix[s] = H * sum_{s'<s} ceil(n_s'/256); inside a sequence,
// super tiles run longest first with heads fastest.
__device__ __forceinline__ Tile2 tile2_varlen(const FwdParams& p, const int* prefix, int t) {
  int lo = 0, hi = p.nseq - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= t) lo = mid; else hi = mid - 1;
  }
  Tile2 T;
  T.seq = lo;
  const int r = t - prefix[lo];
  const int a = __ldg(p.cu_seqlens + lo), b = __ldg(p.cu_seqlens + lo + 1);
  T.n = b - a;
  T.nq = T.n;
  T.qrow0 = 0;
  T.split = 0;
  T.sblk = ceil_div(T.n, SUPER_M) - 1 - r / p.H;
  T.h = r % p.H;
  T.tok0 = a;
  T.tma_row0 = a;
  T.tma_b = 0;
  return T;
}

// Split-KV decode: unit t -> (sequence b, KV head, split s), splits fastest.
// The unit's rows are the H/Hkv query heads of that KV head (one token each),
// its keys the cache range [s * chunk, (s + 1) * chunk) clipped to the
// sequence's cached length (clamped to the cache size); a split past the end
// has no keys.
__device__ __forceinline__ Tile2 tile2_decode(const FwdParams& p, int t) {
  Tile2 T;
  T.split = t % p.num_splits;
  const int bk = t / p.num_splits;
  T.seq = bk / p.Hkv;
  T.h = bk % p.Hkv;
  const int n = min(max(__ldg(p.seqlens + T.seq), 0), p.N);
  const int s0 = min(T.split * p.split_chunk, n);
  T.n = min(s0 + p.split_chunk, n) - s0;
  T.nq = p.group;
  T.qrow0 = T.h * p.group;
  T.sblk = 0;
  T.tok0 = 0;
  T.tma_row0 = s0;
  T.tma_b = T.seq;
  return T;
}

__device__ __forceinline__ void build_varlen_prefix2(const FwdParams& p, int* prefix) {
  for (int s = threadIdx.x; s < p.nseq; s += blockDim.x) {
    const int n = __ldg(p.cu_seqlens + s + 1) - __ldg(p.cu_seqlens + s);
    prefix[s + 1] = (n > 0 ? ceil_div(n, SUPER_M) : 0) * p.H;
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

// Key blocks tile x (0 = A, 1 = B) of a super tile visits; 0 if it has no rows.
template <bool CAUSAL, int BN>
__device__ __forceinline__ int tile2_blocks(const Tile2& tl, int x) {
  const int r0 = tl.sblk * SUPER_M + x * BLOCK_M;
  if (r0 >= tl.nq) return 0;
  int kend = tl.n;
  if (CAUSAL) kend = min(kend, r0 + BLOCK_M);
  return ceil_div(kend, BN);
}

// max of three floats in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

// KIND_BF16 / KIND_FP16: Q, K, V in that type, V tiles MN-major (rows of
// keys). KIND_E4M3: e4m3 codes with scales (FP8 path): S = Q8 K8^T is
// dequantised by the per-block scalar sq * sk folded into the softmax scale,
// P (<= 2^8 under the lazy maximum) is rounded to e4m3 for O += P V^T with V
// given transposed (rows of channels, K-major), and the epilogue applies the
// V channel scale.
template <int D, int BN, int STAGES, bool CAUSAL, bool VARLEN, int KIND, bool DECODE = false>
__global__ void __launch_bounds__(384, 1)
attn_fwd2_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                 const FwdParams p) {
  constexpr bool FP8 = KIND == KIND_E4M3;
  constexpr bool BF16 = KIND == KIND_BF16;
  constexpr int ELEM = FP8 ? 1 : 2;
  // P V in NP parts of KP keys (PCOLS TMEM columns of P each). Halves: with
  // quarters the tensor pipe waited between the 16-bit parts (BF16 d = 128
  // 1835 -> 1555 TFLOP/s)
  constexpr int NP = 2;
  constexpr int KP = BN / NP;
  constexpr int PCOLS = FP8 ? KP / 4 : KP / 2;
  static_assert(NP <= 4 && BN % NP == 0 && (PCOLS == 16 || PCOLS == 32), "P parts");
  constexpr bool STAGE_OUT = !VARLEN && !DECODE;
  static_assert(!DECODE || (!CAUSAL && !VARLEN && !FP8), "decode units are non-causal 16-bit fixed-cache");
  // Slot watcher (16-bit kinds): measured to help when the GEMMs are long
  // (BF16/FP16) and to cost a little with the shorter FP8 GEMMs, where the MMA
  // thread waits for the slot itself.
  constexpr bool WATCH = !FP8;
  using T = Pair2Traits<D, BN, STAGES, ELEM, STAGE_OUT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sQ = smem + T::OFF_Q;
  uint8_t* sK = smem + T::OFF_K;
  uint8_t* sV = smem + T::OFF_V;
  Bars2* bars = reinterpret_cast<Bars2*>(smem + T::OFF_BARS);
  int* prefix = reinterpret_cast<int*>(smem + T::OFF_PREFIX);
  volatile int* abort_flag = &bars->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars->slot_full[s], 1);
      mbar_init(&bars->slot_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars->s_full[x], 1);
      mbar_init(&bars->o_done[x], 1);
    }
    // tile A's first-part-of-P barrier also carries "slot j has landed" from
    // the watcher warp, so the MMA thread waits once for both
    for (int x = 0; x < 2; ++x)
      for (int q = 0; q < 3; ++q) mbar_init(&bars->p_part[x][q], (x == 0 && q == 0 && WATCH) ? 129 : 128);
    mbar_init(&bars->p_full[0], 128);
    mbar_init(&bars->p_full[1], 128);
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(&bars->tmem_base, T::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    if (STAGE_OUT) tma_prefetch_desc(&tmO);
  }
  int ntiles = p.ntiles;
  if constexpr (VARLEN) {
    build_varlen_prefix2(p, prefix);
    ntiles = prefix[p.nseq];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const uint64_t tmo = p.timeout_ns;

  auto get_tile = [&](int t) -> Tile2 {
    if constexpr (VARLEN) return tile2_varlen(p, prefix, t);
    else if constexpr (DECODE) return tile2_decode(p, t);
    else return tile2_fixed<CAUSAL>(p, t);
  };
  // KV head of a unit (decode units carry it directly)
  auto kv_head = [&](const Tile2& tl) -> int { return DECODE ? tl.h : tl.h / p.group; };

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int slot_it = 0, tile_i = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        const Tile2 tl = get_tile(t);
        const int hk = kv_head(tl);
        const int nkv = max(tile2_blocks<CAUSAL, BN>(tl, 0), tile2_blocks<CAUSAL, BN>(tl, 1));
        if (nkv == 0) continue;                       // a decode split past the sequence end
        ok = mbar_wait(&bars->q_empty, (tile_i & 1) ^ 1, tmo, abort_flag, p.err);
        if (!ok) break;
        mbar_expect_tx(&bars->q_full, 2 * T::Q_BYTES);
#pragma unroll
        for (int x = 0; x < 2; ++x)
#pragma unroll
          for (int c = 0; c < T::NC; ++c) {
            // Q map: {d, H, N, B} rows of one head; decode: {d, 1, H, B}, the
            // rows being the query heads of the unit's KV head
            if constexpr (DECODE)
              tma_load_4d(&tmQ, &bars->q_full, sQ + x * T::Q_BYTES + c * T::Q_CHUNK, c * (128 / ELEM), 0,
                          tl.qrow0 + x * BLOCK_M, tl.tma_b);
            else
              tma_load_4d(&tmQ, &bars->q_full, sQ + x * T::Q_BYTES + c * T::Q_CHUNK, c * (128 / ELEM), tl.h,
                          tl.tma_row0 + tl.sblk * SUPER_M + x * BLOCK_M, tl.tma_b);
          }
        ++tile_i;
        // slot j: K_j (j < nkv) and V_{j-1} (j >= 1)
        for (int j = 0; j <= nkv; ++j, ++slot_it) {
          // 16-bit kinds: the next unit's Q tiles are prefetched into L2 four key
          // blocks before this unit ends, so their copy (issued once this unit's
          // last Q K^T has run) does not wait on HBM between units (measured
          // +1.6 % at d = 128; no gain for FP8)
          if (!FP8 && !DECODE && j == max(nkv - 4, 0) && t + (int)gridDim.x < ntiles) {
            const Tile2 tn = get_tile(t + gridDim.x);
#pragma unroll
            for (int x = 0; x < 2; ++x)
#pragma unroll
              for (int c = 0; c < T::NC; ++c)
                tma_prefetch_l2_4d(&tmQ, c * (128 / ELEM), tn.h, tn.tma_row0 + tn.sblk * SUPER_M + x * BLOCK_M, tn.tma_b);
          }
          const int st = slot_it % STAGES;
          ok = mbar_wait(&bars->slot_empty[st], ((slot_it / STAGES) & 1) ^ 1, tmo, abort_flag, p.err);
          if (!ok) break;
          mbar_expect_tx(&bars->slot_full[st], (j < nkv ? T::KV_BYTES : 0) + (j >= 1 ? T::KV_BYTES : 0));
          if (j < nkv) {
#pragma unroll
            for (int c = 0; c < T::NC; ++c)
              tma_load_4d(&tmK, &bars->slot_full[st], sK + st * T::KV_BYTES + c * T::KV_CHUNK, c * (128 / ELEM),
                          hk, tl.tma_row0 + j * BN, tl.tma_b);
          }
          if (j >= 1) {
            if constexpr (FP8) {
              // V^T block: 128 keys x D channel rows of (batch, kv head)
              // V^T block: 128 keys x D channel rows; fixed: [B*Hkv][D][ldv];
              // packed sequences: [Hkv][D][ldv] from column 128 * blk_off[seq]
              if constexpr (VARLEN)
                tma_load_4d(&tmV, &bars->slot_full[st], sV + st * T::KV_BYTES,
                            (__ldg(p.blk_off + tl.seq) + j - 1) * BN, 0, hk, 0);
              else
                tma_load_4d(&tmV, &bars->slot_full[st], sV + st * T::KV_BYTES, (j - 1) * BN, 0, tl.seq * p.Hkv + hk, 0);
            } else {
#pragma unroll
              for (int c = 0; c < T::NC; ++c)
                tma_load_4d(&tmV, &bars->slot_full[st], sV + st * T::KV_BYTES + c * T::KV_CHUNK, c * 64, hk,
                            tl.tma_row0 + (j - 1) * BN, tl.tma_b);
            }
          }
        }
      }
      // never leave with copies in flight
      for (int it = (slot_it > STAGES ? slot_it - STAGES : 0); it < slot_it; ++it)
        mbar_wait_drain(&bars->slot_full[it % STAGES], (it / STAGES) & 1, tmo, p.err);
      if (tile_i > 0) mbar_wait_drain(&bars->q_full, (tile_i - 1) & 1, tmo, p.err);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // One thread issues, in this order per key block j,
    //   O_A += P_A(j-1) V_{j-1}, S_A(j) = Q_A K_j^T, O_B += P_B(j-1) V_{j-1}, S_B(j)
    // so tile A's softmax of block j overlaps tile B's two GEMMs and vice
    // versa. The issuing thread waits as little as possible (a wait on a
    // barrier costs the tensor pipe idle time even when it is already
    // complete): twice per block and tile, for the first half of P (for tile
    // A together with the slot's data, see the watcher) and for the rest.
    // The whole warp runs the loop (convergent control flow); one elected
    // lane issues each MMA and commit.
    {
      constexpr uint32_t idesc_s = FP8 ? idesc_kind_f8_e4m3(BLOCK_M, BN) : idesc_kind_f16(BLOCK_M, BN, BF16, false);
      constexpr uint32_t idesc_o = FP8 ? idesc_kind_f8_e4m3(BLOCK_M, D) : idesc_kind_f16(BLOCK_M, D, BF16, true);
      constexpr int PV_STEPS = BN * ELEM / 32;               // 32-byte K steps of P V
      constexpr int S_STEPS = D * ELEM / 32;                 // 32-byte K steps of Q K^T
      // descriptor low halves of the operands' first bytes; every MMA's
      // descriptor is one of these plus a constant (the issue path between
      // S_B(j) and P_A(j) V_j has no descriptor arithmetic left to do)
      const uint32_t q_lo = sdesc_lo_kmajor_sw128(smem_u32(sQ));
      const uint32_t k_lo = sdesc_lo_kmajor_sw128(smem_u32(sK));
      const uint32_t v_lo = FP8 ? sdesc_lo_kmajor_sw128(smem_u32(sV)) : sdesc_lo_mnmajor_sw128(smem_u32(sV), T::KV_CHUNK);
      int slot_it = 0, tile_i = 0;
      int p_cnt0 = 0, p_cnt1 = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        const Tile2 tl = get_tile(t);
        const int nb[2] = {tile2_blocks<CAUSAL, BN>(tl, 0), tile2_blocks<CAUSAL, BN>(tl, 1)};
        const int nkv = max(nb[0], nb[1]);
        if (nkv == 0) continue;
        ok = mbar_wait_warp(&bars->q_full, tile_i & 1, tmo, abort_flag, p.err);
        ++tile_i;
        if (!ok) break;
        for (int j = 0; j <= nkv && ok; ++j, ++slot_it) {
          const int st = slot_it % STAGES;
          const uint32_t vb_lo = v_lo + st * (T::KV_BYTES >> 4);
          const uint32_t kb_lo = k_lo + st * (T::KV_BYTES >> 4);
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            if (!ok) continue;
            const bool pv = j >= 1 && j - 1 < nb[x];
            int& pc = x == 0 ? p_cnt0 : p_cnt1;
            if (x == 0 && (!WATCH || !pv))
              ok = mbar_wait_warp(&bars->slot_full[st], (slot_it / STAGES) & 1, tmo, abort_flag, p.err);
            // P(j-1) V goes out in NP parts of BN / NP keys, each as soon as
            // the softmax has stored that part's P (it stores them as its loop
            // goes); the last part waits for the whole tile
            if (ok && pv) ok = mbar_wait_warp(&bars->p_part[x][0], pc & 1, tmo, abort_flag, p.err);
            if (!ok) continue;
            tc_fence_after();
            const uint32_t s_tmem = tmem + T::TMEM_S + x * BN;
            if (pv) {
              const uint32_t o_tmem = tmem + T::TMEM_O + x * D;
#pragma unroll
              for (int k = 0; k < PV_STEPS; ++k) {
                if (k > 0 && k % (PV_STEPS / NP) == 0) {
                  const int part = k / (PV_STEPS / NP);
                  ok = mbar_wait_warp(part == NP - 1 ? &bars->p_full[x] : &bars->p_part[x][part], pc & 1, tmo,
                                      abort_flag, p.err);
                  if (!ok) break;
                  tc_fence_after();
                }
                // each K step is 8 TMEM columns of P (16 x 16-bit or 32 x 8-bit)
                if constexpr (FP8)
                  umma_f8_ts_lo_w(o_tmem, s_tmem + k * 8, vb_lo + k * (32 >> 4), idesc_o, (j > 1 || k > 0) ? 1u : 0u);
                else
                  umma_f16_ts_lo_w(o_tmem, s_tmem + k * 8, vb_lo + k * (2048 >> 4), idesc_o, (j > 1 || k > 0) ? 1u : 0u);
              }
              ++pc;
              if (!ok) continue;
              if (j == nb[x]) umma_commit_w(&bars->o_done[x]);   // last P V of this tile
            }
            if (j < nb[x]) {
#pragma unroll
              for (int k = 0; k < S_STEPS; ++k) {
                const uint32_t qo = (x * T::Q_BYTES + (k >> 2) * T::Q_CHUNK + (k & 3) * 32) >> 4;
                const uint32_t ko = ((k >> 2) * T::KV_CHUNK + (k & 3) * 32) >> 4;
                if constexpr (FP8)
                  umma_f8_ss_lo_w(s_tmem, q_lo + qo, kb_lo + ko, idesc_s, k > 0 ? 1u : 0u);
                else
                  umma_f16_ss_lo_w(s_tmem, q_lo + qo, kb_lo + ko, idesc_s, k > 0 ? 1u : 0u);
              }
              umma_commit_w(&bars->s_full[x]);
            }
          }
          if (!ok) break;
          umma_commit_w(&bars->slot_empty[st]);
          if (j == nkv - 1) umma_commit_w(&bars->q_empty);
        }
      }
      umma_commit_w(&bars->mma_done);
      mbar_wait_drain(&bars->mma_done, 0, tmo, p.err);
    }
    __syncwarp();
  } else if (warp == 10 && WATCH) {
    // ------------------------------------------------------------ slot watcher
    // For every slot j >= 1 that tile A consumes together with P_A(j-1), wait
    // until its K/V data has landed and add one arrival to tile A's P-ready
    // barrier (after the barrier's previous phase completed, so the arrival
    // lands in the phase of block j-1).
    if (lane == 0) {
      int slot_it = 0, arrivals = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        const Tile2 tl = get_tile(t);
        const int na = tile2_blocks<CAUSAL, BN>(tl, 0);
        const int nkv = max(na, tile2_blocks<CAUSAL, BN>(tl, 1));
        if (nkv == 0) continue;                       // no slots for an empty unit
        for (int j = 0; j <= nkv; ++j, ++slot_it) {
          // Every slot is waited for, in order, even those this warp does not
          // report: a parity wait is only unambiguous while the waiter is at
          // most one phase behind, and skipping slots of a short ring would
          // let it run two phases ahead of a slot still in flight.
          ok = mbar_wait(&bars->slot_full[slot_it % STAGES], (slot_it / STAGES) & 1, tmo, abort_flag, p.err);
          if (!ok) break;
          if (j >= 1 && j - 1 < na) {
            if (arrivals > 0) ok = mbar_wait(&bars->p_part[0][0], (arrivals - 1) & 1, tmo, abort_flag, p.err);
            if (!ok) break;
            mbar_arrive(&bars->p_part[0][0]);
            ++arrivals;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------- softmax / correction / epilogue
    const int x = warp >> 2;                           // 0 = tile A, 1 = tile B
    const int r = threadIdx.x & 127;                   // row within the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t ts = tmem + lane_off + T::TMEM_S + x * BN;
    const uint32_t to = tmem + lane_off + T::TMEM_O + x * D;
    constexpr float lazy = LAZY_RESCALE_LOG2;
    int s_cnt = 0, o_tiles = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
      const Tile2 tl = get_tile(t);
      const int nblk = tile2_blocks<CAUSAL, BN>(tl, x);
      const int row0 = tl.sblk * SUPER_M + x * BLOCK_M;  // first row of this tile
      const int i_row = row0 + r;
      if (nblk == 0) {                                // tile B past the sequence end
        // a decode split with no keys: its partial has lse = -inf (weight 0)
        if (DECODE && x == 0 && i_row < tl.nq)
          p.lse[((size_t)tl.split * p.nseq + tl.seq) * p.H + tl.qrow0 + i_row] = -INFINITY;
        continue;
      }
      const int hk = kv_head(tl);
      // FP8 block scales: fixed [B][heads][ceil(N/128)]; packed sequences
      // [heads][tmax] from column blk_off[seq]
      const int nb128 = VARLEN ? p.tmax : ceil_div(tl.n, BLOCK_M);
      const size_t sblk0 = VARLEN ? (size_t)(FP8 ? __ldg(p.blk_off + tl.seq) : 0) : 0;
      const size_t sq_row = VARLEN ? (size_t)tl.h * nb128 + sblk0 : ((size_t)tl.seq * p.H + tl.h) * nb128;
      const size_t sk_row = VARLEN ? (size_t)hk * nb128 + sblk0 : ((size_t)tl.seq * p.Hkv + hk) * nb128;
      float sq_x = 1.f, sk_j = 1.f;
      if constexpr (FP8) {
        sq_x = p.fp8_block ? __ldg(p.sq + sq_row + (row0 >> 7)) : __ldg(p.sq);
        sk_j = p.fp8_block ? __ldg(p.sk + sk_row) : __ldg(p.sk);
      }
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < nblk; ++j) {
        float sl2 = p.scale_log2;
        if constexpr (FP8) {
          sl2 *= sq_x * sk_j;
          // the next key block's scale is loaded one block ahead
          if (p.fp8_block && j + 1 < nblk) sk_j = __ldg(p.sk + sk_row + j + 1);
        }
        ok = mbar_wait(&bars->s_full[x], s_cnt & 1, tmo, abort_flag, p.err);
        ++s_cnt;
        if (!ok) break;
        tc_fence_after();
        static_assert(BN == 128, "softmax path assumes 128-column S tiles");
        float s[BN];
        float mx;                                     // row maximum of the block's scores
        {
          uint32_t u[BN];
          tmem_ld128_max(ts, u, mx);
#pragma unroll
          for (int i = 0; i < BN; ++i) s[i] = __uint_as_float(u[i]);
        }
        const int col0 = j * BN;
        if ((col0 + BN > tl.n) || (CAUSAL && col0 + BN - 1 > row0)) {
          int limit = tl.n - col0;
          if (CAUSAL) limit = min(limit, i_row - col0 + 1);
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (c >= limit) s[c] = -INFINITY;
          // the load's maximum may come from a masked key: recompute it
          float mxa = fmax3(s[0], s[1], s[2]), mxb = fmax3(s[3], s[4], s[5]);
          float mxc = fmax3(s[6], s[7], s[8]), mxd = fmax3(s[9], s[10], s[11]);
#pragma unroll
          for (int c = 12; c < BN - 4; c += 8) {
            mxa = fmax3(mxa, s[c], s[c + 1]);
            mxb = fmax3(mxb, s[c + 2], s[c + 3]);
            mxc = fmax3(mxc, s[c + 4], s[c + 5]);
            mxd = fmax3(mxd, s[c + 6], s[c + 7]);
          }
          mxa = fmax3(mxa, s[BN - 4], s[BN - 3]);
          mxb = fmax3(mxb, s[BN - 2], s[BN - 1]);
          mx = fmaxf(fmaxf(mxa, mxb), fmaxf(mxc, mxd));
        }
        mx *= sl2;
        // raise the running max only when it moved by more than the margin
        const bool raise = mx > m + lazy;
        const float m_new = raise ? mx : m;
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = raise ? ex2_approx(m - m_use) : 1.f;
        // O_x is rescaled (below) when any row of the warp raised its maximum;
        // such a warp reports its parts of P only after the rescale, so no
        // P V of this block reaches O_x before it
        const bool corr = j > 0 && __any_sync(0xffffffffu, raise);
        // p = 2^(s * scale * log2(e) - m): the affine step and the row sum run
        // as packed f32x2 operations, the exponentials on the MUFU unit
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
        const uint64_t negm2 = f2_pack(-m_use, -m_use);
        uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = acc0;
        // P packed as it is produced (e4m3 quads, or 16-bit pairs), so the
        // fp32 scores die early and the softmax fits its registers
        static_assert(BN == 128, "P tile is one (FP8) or two (16-bit) 32-column stores");
        constexpr int PW = FP8 ? BN / 4 : BN / 2;
        uint32_t pk[PW];
#pragma unroll
        for (int c = 0; c < BN; c += 4) {
          float a0, a1, b0, b1;
          f2_unpack(f2_fma(f2_pack(s[c], s[c + 1]), sl2x2, negm2), a0, a1);
          f2_unpack(f2_fma(f2_pack(s[c + 2], s[c + 3]), sl2x2, negm2), b0, b1);
          a0 = ex2_approx(a0);
          a1 = ex2_approx(a1);
          b0 = ex2_approx(b0);
          b1 = ex2_approx(b1);
          acc0 = f2_add(acc0, f2_pack(a0, a1));
          acc1 = f2_add(acc1, f2_pack(b0, b1));
          if constexpr (FP8) {
            pk[c / 4] = pack_e4m3x4(a0, a1, b0, b1);     // P as e4m3, four per TMEM column
          } else {
            pk[c / 2] = pack2(a0, a1, BF16);
            pk[c / 2 + 1] = pack2(b0, b1, BF16);
          }
          if ((c + 4) % KP == 0) {
            // a part's P leaves for TMEM as soon as it is complete; but for the
            // last, the MMA thread may start on it
            const int part = c / KP;
            if constexpr (PCOLS == 16) tmem_st16(ts + part * 16, &pk[part * 16]);
            else tmem_st32(ts + part * 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[part * 32]));
            if (!corr && part < NP - 1) {
              tmem_st_wait();
              tc_fence_before();
              mbar_arrive(&bars->p_part[x][part]);
            }
          }
        }
        float sum0, sum1, sum2, sum3;
        f2_unpack(acc0, sum0, sum1);
        f2_unpack(acc1, sum2, sum3);
        l = l * alpha + ((sum0 + sum1) + (sum2 + sum3));
        m = m_new;
        // the stores read their source registers asynchronously: completing
        // them here frees those registers for the (rare) correction below
        tmem_st_wait();
        // correction: O_x += P(j-1) V has completed (it was issued before
        // S_x(j), whose completion we just observed), so O_x is stable.
        if (corr) {
#pragma unroll 1
          for (int c = 0; c < D / 64; ++c) {
            uint32_t u[64];
            tmem_ld64(to + c * 64, u);
#pragma unroll
            for (int i = 0; i < 64; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
            tmem_st32(to + c * 64, *reinterpret_cast<uint32_t(*)[32]>(&u[0]));
            tmem_st32(to + c * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&u[32]));
          }
          tmem_st_wait();
          tc_fence_before();
#pragma unroll
          for (int q = 0; q < NP - 1; ++q) mbar_arrive(&bars->p_part[x][q]);
        }
        tc_fence_before();
        mbar_arrive(&bars->p_full[x]);
      }
      if (!ok) break;
      ok = mbar_wait(&bars->o_done[x], o_tiles & 1, tmo, abort_flag, p.err);
      ++o_tiles;
      if (!ok) break;
      tc_fence_after();
      const bool valid = i_row < tl.nq;
      const float inv_l = 1.f / l;
      const size_t tok = (size_t)tl.tok0 + (size_t)(valid ? i_row : 0);
      uint4* orow = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.o) + (tok * p.H + tl.h) * D);
      // channels of the output (FP8 head dim 64 runs here with zero channels 64-127)
      const int dch = (FP8 && p.fp8_d > 0) ? p.fp8_d : D;
      const float* svp = FP8 ? (p.fp8_block ? p.sv + ((size_t)tl.seq * p.Hkv + hk) * dch : p.sv) : nullptr;
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        if (FP8 && c * 64 >= dch) break;
        uint32_t u[64];
        tmem_ld64(to + c * 64, u);
        if constexpr (DECODE) {
          // fp32 partial O of this split: [split][b][H][d]
          if (valid) {
            float4* prow = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.o) +
                                                     (((size_t)tl.split * p.nseq + tl.seq) * p.H + tl.qrow0 + i_row) * D);
#pragma unroll
            for (int i = 0; i < 16; ++i)
              prow[c * 16 + i] = make_float4(__uint_as_float(u[4 * i]) * inv_l, __uint_as_float(u[4 * i + 1]) * inv_l,
                                             __uint_as_float(u[4 * i + 2]) * inv_l, __uint_as_float(u[4 * i + 3]) * inv_l);
          }
          continue;
        }
        uint32_t w[32];
        if constexpr (FP8) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int ch = c * 64 + 2 * i;
            const float s0 = p.fp8_block ? __ldg(svp + ch) : __ldg(svp);
            const float s1 = p.fp8_block ? __ldg(svp + ch + 1) : s0;
            w[i] = pack2(__uint_as_float(u[2 * i]) * (s0 * inv_l), __uint_as_float(u[2 * i + 1]) * (s1 * inv_l),
                         true);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            w[i] = pack2(__uint_as_float(u[2 * i]) * inv_l, __uint_as_float(u[2 * i + 1]) * inv_l, BF16);
        }
        if constexpr (STAGE_OUT) {
          // this warp's 32 rows x 64 columns: 128-byte rows, 16-byte chunk i of
          // row `lane` at chunk position i ^ (lane % 8) (the bulk tensor
          // store's 128-byte swizzle; conflict-free shared stores), then one
          // bulk store; rows past the sequence end are clipped by the copy
          const uint32_t stg = smem_u32(smem + T::OFF_STAGE + warp * 4096);
          if (lane == 0) tma_store_wait_read();     // previous use of the buffer
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 8; ++i)
            st_shared_v4(stg + lane * 128 + ((i ^ (lane & 7)) << 4), w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_4d(&tmO, smem + T::OFF_STAGE + warp * 4096, c * 64, tl.h, row0 + (warp & 3) * 32, tl.tma_b);
            tma_store_commit();
          }
        } else if (valid) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            orow[c * 8 + i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
      if (valid) {
        const float lse = (m + lg2_approx(l)) * 0.69314718055994530942f;
        if constexpr (VARLEN) p.lse[(size_t)tl.h * p.total + tok] = lse;
        else if constexpr (DECODE) p.lse[((size_t)tl.split * p.nseq + tl.seq) * p.H + tl.qrow0 + i_row] = lse;
        else p.lse[((size_t)tl.seq * p.H + tl.h) * p.N + i_row] = lse;
      }
    }
    if (STAGE_OUT && lane == 0) tma_store_wait_all();   // no bulk store outlives the CTA
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tmem, T::TMEM_COLS);
}

}  // namespace attn45
