// attn_decode_kt.cuh -- split-KV decode with the keys on the TMEM lanes and
// the cache divided evenly between persistent CTAs.
//
// In decode a KV head meets only its G = H/Hkv query rows, so a tile of the
// forward kernel (128 query rows on the TMEM lanes) would be mostly padding.
// Here both products are transposed so the 128 keys of a tile fill the MMA's
// M dimension and the few query heads sit in N = 16:
//   S^T [128 keys x 16]  = K [128 x d] . Q^T            (A = K tile, K-major)
//   O^T [d x 16]        += V^T [d x 128 keys] . P^T      (A = V tile, MN-major)
// with K and V exactly as TMA stages them (64-channel boxes, 128-byte
// swizzle), d = 64 or 128.
//
// Work division. Unit u = (sequence b, KV head) owns ceil(n_b / 128) tiles;
// the tiles of all units, in unit order, are cut into `grid` equal contiguous
// ranges (CTA c takes [c T / grid, (c+1) T / grid)), so every CTA streams the
// same number of bytes whatever the length mix, and its TMA ring runs on
// across unit boundaries. A CTA holding a whole unit writes its O and lse.
// Otherwise each run of a range inside unit u (a piece) leaves a partial in
// slot u + c (unique: unit u+1 starts in the CTA where unit u ends or in a
// later one), and the CTA whose piece completes the unit's count merges the
// pieces with the online-softmax rescaling, so a decode call is one launch.
//
// Roles in a CTA:
//   warp 4      TMA producer: K and V tiles of 128 keys into a 3-stage ring,
//               plus the unit's Q rows (double-buffered) with a piece's
//               first tile;
//   warp 5      MMA issuer (one thread): S^T(i) into one of two TMEM buffers
//               as soon as tile i has landed, O^T += V^T(i) P^T(i) as soon as
//               P(i) is written, so the softmax of tile i+1 overlaps PV(i)
//               and a stage is released without waiting on the next copy;
//   warps 0-3   softmax, thread = key (TMEM lane): per head, the tile maximum
//               over the 128 keys (warp shuffles, then across the 4 warps in
//               shared memory), P = 2^(s - m) written as the K-major B operand
//               of the second product, running sums per thread; the running
//               maximum moves only when a tile's maximum exceeds it by more
//               than 2^8 (then O^T is rescaled in TMEM), so P <= 256. At a
//               piece's last tile, thread = channel (TMEM lane of O^T): the
//               partial O normalised by its own sum, and its lse.
// The online softmax is the "Related papers: FlashAttention-4" page's
// online-softmax teaser; the split of the key range with a final merge is
// FlashDecoding (cited by "FlashAttention-3: Fast and Accurate Attention with
// Asynchrony and Low-precision" among its references).
#pragma once
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include "fwd_launch.cuh"

namespace attn45 {
namespace {

constexpr int KT_KEYS = 128;                       // keys per tile = TMEM lanes of S^T
constexpr int KT_CHUNK = KT_KEYS * 128;            // 128 keys x 64 channels of 16 bits
constexpr int KT_MAX_STAGES = 6;
constexpr int KT_THREADS = 192;

// D: head dim 64 or 128, a row being D/64 chunks of 64 channels. NQ: the MMA's
// N, the group's query heads padded to 16 or 32. The K/V ring holds 192 KB
// with NQ = 16 (3 stages of 64 KB or 6 of 32 KB) and 128 KB with NQ = 32,
// whose Q, P and reduction buffers are twice as large.
template <int D, int NQ>
struct KtCfg {
  static constexpr int NCH = D / 64;
  static constexpr int STAGES = (NQ == 16 ? 3 : 2) * (D == 128 ? 1 : 2);
  static constexpr int STAGE = 2 * NCH * KT_CHUNK;        // K chunks, then V chunks
  static constexpr int QCH = NQ * 128;                     // one 64-channel chunk of the Q rows
  static constexpr int QBYTES = NCH * QCH;
  static constexpr int PCH = NQ * 128;                     // one 64-key chunk of the P rows
  static constexpr int PBYTES = 2 * PCH;
  static constexpr int OFF_Q = STAGES * STAGE;             // 2 Q buffers
  static constexpr int OFF_P = OFF_Q + 2 * QBYTES;         // 2 P buffers
  static constexpr int OFF_RED = OFF_P + 2 * PBYTES;       // tile maxima [2][4][NQ], sums [4][NQ], flags
  static constexpr int OFF_LIST = OFF_RED + (12 * NQ + 16) * 4;   // CTAs holding pieces of a merged unit
  static constexpr int OFF_BARS = OFF_LIST + DECODE_KT_MAX_GRID * 4;
  // the allocation also covers the 16 KB after the last stage (D = 64, below)
  static constexpr int END = OFF_BARS + 256 > OFF_Q + KT_CHUNK ? OFF_BARS + 256 : OFF_Q + KT_CHUNK;
  static constexpr int BYTES = END + 1024;                 // + alignment slack
  static constexpr uint32_t TMEM_COLS = NQ == 16 ? 64 : 128;   // S^T at 0 and NQ, O^T at 2 NQ
  static constexpr uint32_t COL_O = 2 * NQ;
  static_assert(STAGES <= KT_MAX_STAGES && BYTES <= 227 * 1024, "shared memory");
  // for D = 64 the V^T descriptor's second 64 rows read the 16 KB after the
  // last stage, which must lie inside the allocation
  static_assert(D == 128 || OFF_Q + KT_CHUNK <= BYTES - 1024, "V^T overhang");
};

struct KtBars {
  uint64_t full[KT_MAX_STAGES], empty[KT_MAX_STAGES];
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2], q_free[2], fin;
  long long start, end;                            // this CTA's tile range
  long long T;                                     // tiles of all units
  int b0, tb0;                                     // sequence holding `start`, its tile prefix
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(KtBars) <= 256, "barrier block");

__device__ __forceinline__ int seq_len(const DecodeParams& p, int b) {
  return min(max(__ldg(p.seqlens + b), 0), p.Nmax);
}

// Position in the tile list: sequence, KV head, tile within the unit.
struct KtPos {
  int b, hkv, j, nt, n;                            // n: keys of sequence b, nt = ceil(n / 128)
  __device__ void first(const DecodeParams& p, const KtBars* bars) {
    b = bars->b0;
    n = seq_len(p, b);
    nt = (n + KT_KEYS - 1) / KT_KEYS;
    const long long rem = bars->start - (long long)bars->tb0 * p.Hkv;
    hkv = (int)(rem / nt);
    j = (int)(rem % nt);
  }
  __device__ void next(const DecodeParams& p) {
    if (++j < nt) return;
    j = 0;
    if (++hkv < p.Hkv) return;
    hkv = 0;
    do {
      ++b;
      n = b < p.B ? seq_len(p, b) : 0;
      nt = (n + KT_KEYS - 1) / KT_KEYS;
    } while (nt == 0 && b < p.B);
  }
};

// TMEM <-> registers for the NQ columns of one 32-lane slice.
template <int NQ>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[NQ]) {
  if constexpr (NQ == 16) tmem_ld16(taddr, r);
  else tmem_ld32(taddr, r);
}
template <int NQ>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[NQ]) {
  if constexpr (NQ == 16) tmem_st16(taddr, r);
  else tmem_st32(taddr, r);
}

template <bool BF16>
__device__ __forceinline__ uint16_t to_bits(float x) {
  if constexpr (BF16) return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  else return __half_as_ushort(__float2half_rn(x));
}

// Finds this CTA's range: total T = Hkv * sum_b ceil(n_b / 128), the range
// [c T / grid, (c+1) T / grid), and the sequence holding its first tile, by a
// scan over the sequences in chunks of 128 (threads 0-127). Sequences with no
// cached key get o = 0 and lse = -inf here, sequence b from CTA b % grid.
template <int D, bool BF16>
__device__ void plan_range(const DecodeParams& p, KtBars* bars, int* wsum) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  int part = 0;
  for (int b = t; b < p.B; b += 128) part += (seq_len(p, b) + KT_KEYS - 1) / KT_KEYS;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
  if (lane == 0) wsum[warp] = part;
  named_bar_sync(1, 128);
  const int total = wsum[0] + wsum[1] + wsum[2] + wsum[3];
  named_bar_sync(1, 128);
  const long long T = (long long)total * p.Hkv;
  const long long start = (long long)blockIdx.x * T / gridDim.x;
  const long long end = (long long)(blockIdx.x + 1) * T / gridDim.x;
  int carry = 0;
  for (int base = 0; base < p.B; base += 128) {
    const int b = base + t;
    const int v = b < p.B ? (seq_len(p, b) + KT_KEYS - 1) / KT_KEYS : 0;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += u;
    }
    if (lane == 31) wsum[warp] = incl;
    named_bar_sync(1, 128);
    int excl = carry + incl - v;
    for (int w = 0; w < warp; ++w) excl += wsum[w];
    if (v > 0 && (long long)excl * p.Hkv <= start && start < (long long)(excl + v) * p.Hkv) {
      bars->b0 = b;
      bars->tb0 = excl;
    }
    carry += wsum[0] + wsum[1] + wsum[2] + wsum[3];
    named_bar_sync(1, 128);
  }
  for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
    if (seq_len(p, b) > 0) continue;
    uint16_t* o = static_cast<uint16_t*>(p.o) + (size_t)b * p.H * D;
    for (int i = t; i < p.H * D; i += 128) o[i] = 0;
    for (int h = t; h < p.H; h += 128) p.lse[(size_t)b * p.H + h] = -INFINITY;
  }
  if (t == 0) {
    bars->start = start;
    bars->end = end;
    bars->T = T;
  }
}

// CTA holding tile t of T split into `grid` ranges [c T / grid, (c+1) T / grid).
__device__ __forceinline__ int cta_of(long long t, long long T, int grid) {
  return (int)(((t + 1) * grid + T - 1) / T - 1);
}

// Adds one piece to unit counter c for this call's epoch; returns the pieces
// counted so far, this one included. A counter left by another epoch counts
// as 0, so counters need no reset between calls.
__device__ __forceinline__ unsigned int count_piece(unsigned long long* c, unsigned int epoch, unsigned int* err) {
  unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(c);
  for (int tries = 0; tries < (1 << 20); ++tries) {
    const unsigned int n = (unsigned int)(old >> 32) == epoch ? (unsigned int)old + 1u : 1u;
    const unsigned long long want = ((unsigned long long)epoch << 32) | n;
    const unsigned long long seen = atomicCAS(c, old, want);
    if (seen == old) return n;
    old = seen;
  }
  atomicOr(err, DEV_ERR_TIMEOUT);
  return 0;
}

template <int D, int NQ, int G, bool BF16>
__global__ void __launch_bounds__(KT_THREADS, 1) decode_kt_kernel(const __grid_constant__ CUtensorMap tmQ,
                                                                  const __grid_constant__ CUtensorMap tmK,
                                                                  const __grid_constant__ CUtensorMap tmV,
                                                                  const DecodeParams p) {
  static_assert(G >= 1 && G <= NQ, "query heads per KV head");
  using C = KtCfg<D, NQ>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  KtBars* bars = reinterpret_cast<KtBars*>(smem + C::OFF_BARS);
  float* red = reinterpret_cast<float*>(smem + C::OFF_RED);      // [2][4][NQ]
  float* red_l = red + 2 * 4 * NQ;                                 // [4][NQ]
  int* flags = reinterpret_cast<int*>(red_l + 4 * NQ);             // [2][4] per tile, [4] per piece, merge
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp < 4) plan_range<D, BF16>(p, bars, flags);
  __syncthreads();
  const long long start = bars->start, end = bars->end;
  const int ntl = (int)(end - start);              // tiles of this CTA
  if (ntl <= 0) return;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->s_free[i], 4);
      mbar_init(&bars->p_full[i], 4);
      mbar_init(&bars->pv_done[i], 1);
      mbar_init(&bars->q_free[i], 1);
    }
    mbar_init(&bars->fin, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&bars->tmem_base, C::TMEM_COLS);
    tmem_relinquish();
  }
  for (int i = threadIdx.x; i < 2 * C::PBYTES / 16; i += KT_THREADS)  // P rows >= G stay zero
    reinterpret_cast<uint4*>(smem + C::OFF_P)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const uint64_t tmo = p.timeout_ns;
  KtPos pos;
  pos.first(p, bars);

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int i = 0, k = -1;
      for (; i < ntl; ++i, pos.next(p)) {
        const int st = i % C::STAGES;
        const bool first = i == 0 || pos.j == 0;
        if (first) ++k;
        if (i >= C::STAGES && !mbar_wait(&bars->empty[st], ((i / C::STAGES) + 1) & 1, tmo, &bars->abort_flag, p.err))
          break;
        if (first && k >= 2 && !mbar_wait(&bars->q_free[k & 1], ((k - 2) >> 1) & 1, tmo, &bars->abort_flag, p.err))
          break;
        uint8_t* base = smem + st * C::STAGE;
        const int row = pos.j * KT_KEYS;
        mbar_expect_tx(&bars->full[st], C::STAGE + (first ? C::QBYTES : 0));
        if (first) {
          uint8_t* qb = smem + C::OFF_Q + (k & 1) * C::QBYTES;
          const int qrow = pos.b * p.H + pos.hkv * G;
          for (int c = 0; c < C::NCH; ++c) tma_load_4d(&tmQ, &bars->full[st], qb + c * C::QCH, c * 64, 0, qrow, 0);
        }
        for (int c = 0; c < C::NCH; ++c) {
          tma_load_4d(&tmK, &bars->full[st], base + c * KT_CHUNK, c * 64, pos.hkv, row, pos.b);
          tma_load_4d(&tmV, &bars->full[st], base + (C::NCH + c) * KT_CHUNK, c * 64, pos.hkv, row, pos.b);
        }
      }
      // every copy issued has landed before the CTA can exit (bounded)
      for (int t = max(0, i - C::STAGES); t < i; ++t)
        mbar_wait_drain(&bars->full[t % C::STAGES], (t / C::STAGES) & 1, tmo, p.err);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    // S^T(ns) goes out once its tile has landed and its S^T buffer is free;
    // PV(np) as soon as its P is written. The two are polled rather than
    // taken in a fixed order, so a stage is released (by PV) without waiting
    // for the next tile's copy to land.
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_kind_f16_ab(128, NQ, BF16, false, false);
      constexpr uint32_t id_o = idesc_kind_f16_ab(128, NQ, BF16, true, false);
      // descriptor low halves of stage 0's K and V^T, of Q and of P: every
      // MMA's descriptor is one of these plus a constant
      const uint32_t k_lo = sdesc_lo_kmajor_sw128(smem_u32(smem));
      const uint32_t v_lo = sdesc_lo_mnmajor_sw128(smem_u32(smem + C::NCH * KT_CHUNK), KT_CHUNK);
      const uint32_t q_lo = sdesc_lo_kmajor_sw128(smem_u32(smem + C::OFF_Q));
      const uint32_t p_lo = sdesc_lo_kmajor_sw128(smem_u32(smem + C::OFF_P));
      uint32_t piece_first = 0;                     // bit (tile & 31): first tile of its piece
      int ns = 0, np = 0, k = -1;
      uint64_t t0 = global_timer_ns();
      while (np < ntl) {
        bool moved = false;
        if (ns < ntl) {
          const int st = ns % C::STAGES, sb = ns & 1;
          if (mbar_try_wait(smem_u32(&bars->full[st]), (ns / C::STAGES) & 1) &&
              (ns < 2 || mbar_try_wait(smem_u32(&bars->s_free[sb]), ((ns - 2) >> 1) & 1))) {
            const bool first = ns == 0 || pos.j == 0;
            const bool last = ns == ntl - 1 || pos.j == pos.nt - 1;
            if (first) ++k;
            piece_first = first ? (piece_first | (1u << (ns & 31))) : (piece_first & ~(1u << (ns & 31)));
            tc_fence_after();
            const uint32_t kb = k_lo + st * (C::STAGE >> 4), qb = q_lo + (k & 1) * (C::QBYTES >> 4);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              umma_f16_ss_lo(tmem + sb * NQ, kb + (((kk >> 2) * KT_CHUNK + (kk & 3) * 32) >> 4),
                             qb + (((kk >> 2) * C::QCH + (kk & 3) * 32) >> 4), id_s, kk > 0 ? 1u : 0u);
            umma_commit(&bars->s_full[sb]);
            if (last) umma_commit(&bars->q_free[k & 1]);
            pos.next(p);
            ++ns;
            moved = true;
          }
        }
        if (np < ns && mbar_try_wait(smem_u32(&bars->p_full[np & 1]), (np >> 1) & 1)) {
          const int pb = np & 1, st = np % C::STAGES;
          const bool pf = (piece_first >> (np & 31)) & 1u;
          tc_fence_after();
          // V^T as A with M = 128: for D = 64 its second 64 rows read the next
          // 16 KB of shared memory (in bounds) into O^T rows that are never used
          const uint32_t vb = v_lo + st * (C::STAGE >> 4), pbl = p_lo + pb * (C::PBYTES >> 4);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_f16_ss_lo(tmem + C::COL_O, vb + kk * (2048 >> 4), pbl + (((kk >> 2) * C::PCH + (kk & 3) * 32) >> 4),
                           id_o, (pf && kk == 0) ? 0u : 1u);
          umma_commit(&bars->empty[st]);
          umma_commit(&bars->pv_done[pb]);
          ++np;
          moved = true;
        }
        if (moved) {
          t0 = global_timer_ns();
        } else if (*(volatile int*)&bars->abort_flag) {
          break;
        } else if (global_timer_ns() - t0 > tmo) {
          bars->abort_flag = 1;
          atomicOr(p.err, DEV_ERR_TIMEOUT);
          break;
        }
      }
      umma_commit(&bars->fin);                      // all MMAs issued above have completed
      mbar_wait_drain(&bars->fin, 0, tmo, p.err);
    }
  } else {
    // ------------------------------------------------------------ softmax
    // Every softmax warp runs all ntl iterations and meets every named
    // barrier; after a failed wait a warp only skips work, and each decision
    // to skip is read from flags all four warps wrote before a barrier, so it
    // is the same in every warp.
    const int key = threadIdx.x;                    // TMEM lane of S^T; channel of O^T
    const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
    float m[G], lp[G];
    bool bad = false;
    for (int i = 0; i < ntl; ++i, pos.next(p)) {
      const int sb = i & 1;
      const bool first = i == 0 || pos.j == 0;
      const bool last = i == ntl - 1 || pos.j == pos.nt - 1;
      if (first) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          m[h] = -INFINITY;
          lp[h] = 0.f;
        }
      }
      if (!bad) bad = !mbar_wait(&bars->s_full[sb], (i >> 1) & 1, tmo, &bars->abort_flag, p.err);
      bad = __any_sync(0xffffffffu, bad);
      uint32_t r[NQ];
      if (!bad) {
        tc_fence_after();
        tmem_ld_cols<NQ>(tl + sb * NQ, r);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->s_free[sb]);
      const bool valid = pos.j * KT_KEYS + key < pos.n;
      float sc[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        sc[h] = (!bad && valid) ? __uint_as_float(r[h]) * p.scale_log2 : -INFINITY;
        float x = sc[h];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
        if (lane == 0) red[(sb * 4 + warp) * NQ + h] = x;
      }
      if (lane == 0) flags[sb * 4 + warp] = bad ? 1 : 0;
      named_bar_sync(1, 128);
      if (flags[sb * 4] | flags[sb * 4 + 1] | flags[sb * 4 + 2] | flags[sb * 4 + 3]) {
        bad = true;
        continue;
      }
      bool resc = false;
      float tmax[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float* rr = red + sb * 4 * NQ + h;
        tmax[h] = fmax3(rr[0], rr[NQ], fmaxf(rr[2 * NQ], rr[3 * NQ]));
        resc |= tmax[h] > m[h] + LAZY_RESCALE_LOG2;
      }
      if (resc) {                                   // the same decision in every thread
        float alpha[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float mn = fmaxf(m[h], tmax[h]);
          alpha[h] = ex2_approx(m[h] - mn);         // 0 while m was -inf
          m[h] = mn;
          lp[h] *= alpha[h];
        }
        if (!first) {
          // O^T holds the piece's earlier tiles once PV(i-1) is done: rescale
          bad = !mbar_wait(&bars->pv_done[(i - 1) & 1], ((i - 1) >> 1) & 1, tmo, &bars->abort_flag, p.err);
          bad = __any_sync(0xffffffffu, bad);
          if (!bad) {
            tc_fence_after();
            uint32_t o[NQ];
            tmem_ld_cols<NQ>(tl + C::COL_O, o);
#pragma unroll
            for (int h = 0; h < G; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha[h]);
            tmem_st_cols<NQ>(tl + C::COL_O, o);
            tmem_st_wait();
            tc_fence_before();
          }
        }
      }
      // P buffer sb is free once PV(i-2) is done
      if (!bad && i >= 2) bad = !mbar_wait(&bars->pv_done[sb], ((i - 2) >> 1) & 1, tmo, &bars->abort_flag, p.err);
      if (!bad) {                                   // else no P arrival: the MMA issuer's wait gives up
        if (!valid) {
          // a key past the end meets P = 0, but 0 * (Inf or NaN) is not 0 in
          // the product: clear its V row (the tile has landed: S^T(i) read it)
          uint4* vr = reinterpret_cast<uint4*>(smem + (i % C::STAGES) * C::STAGE + C::NCH * KT_CHUNK + key * 128);
#pragma unroll
          for (int c = 0; c < C::NCH; ++c)
#pragma unroll
            for (int u = 0; u < 8; ++u) vr[c * (KT_CHUNK / 16) + u] = make_uint4(0u, 0u, 0u, 0u);
        }
        uint8_t* prow = smem + C::OFF_P + sb * C::PBYTES + (key >> 6) * C::PCH;
        const int kb = (key & 63) * 2;              // byte of this key within a 128-byte row
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float pk = ex2_approx(sc[h] - m[h]);  // 0 for keys past the end
          lp[h] += pk;
          *reinterpret_cast<uint16_t*>(prow + h * 128 + ((((kb >> 4) ^ (h & 7)) << 4) | (kb & 15))) =
              to_bits<BF16>(pk);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full[sb]);
      }
      if (last) {
        // ---------------------------------------------------------- piece end
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float x = lp[h];
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
          if (lane == 0) red_l[warp * NQ + h] = x;
        }
        if (lane == 0) flags[8 + warp] = bad ? 1 : 0;
        named_bar_sync(1, 128);
        bool skip = flags[8] | flags[9] | flags[10] | flags[11];
        if (!skip) skip = !mbar_wait(&bars->pv_done[sb], (i >> 1) & 1, tmo, &bars->abort_flag, p.err);
        skip = __any_sync(0xffffffffu, skip);
        if (!skip) {
          tc_fence_after();
          uint32_t o[NQ];
          tmem_ld_cols<NQ>(tl + C::COL_O, o);
          const long long g0 = start + i - pos.j;   // the unit's first tile in the list
          const long long g1 = g0 + pos.nt;
          const size_t orow0 = (size_t)pos.b * p.H + (size_t)pos.hkv * G;   // output rows of the group
          uint16_t* o_out = static_cast<uint16_t*>(p.o);
          float l[G];
#pragma unroll
          for (int h = 0; h < G; ++h) l[h] = red_l[h] + red_l[NQ + h] + red_l[2 * NQ + h] + red_l[3 * NQ + h];
          if (g0 >= start && g1 <= end) {
            // the whole unit is here: final O and lse (thread = channel)
#pragma unroll
            for (int h = 0; h < G; ++h) {
              if (key < D) o_out[(orow0 + h) * D + key] = to_bits<BF16>(__uint_as_float(o[h]) / l[h]);
              if (key == h) p.lse[orow0 + h] = (m[h] + lg2_approx(l[h])) * 0.69314718055994530942f;
            }
          } else {
            const int u = pos.b * p.Hkv + pos.hkv;
            const size_t row0 = ((size_t)u + blockIdx.x) * G;   // slot u + c
#pragma unroll
            for (int h = 0; h < G; ++h) {
              if (key < D) p.o_parts[(row0 + h) * D + key] = __uint_as_float(o[h]) / l[h];
              if (key == h) p.lse_parts[row0 + h] = (m[h] + lg2_approx(l[h])) * 0.69314718055994530942f;
            }
            __threadfence();                        // the partial is visible before it is counted
            named_bar_sync(1, 128);
            int* list = reinterpret_cast<int*>(smem + C::OFF_LIST);
            if (key == 0) {
              // the CTAs holding tiles of the unit (with grid > T some hold
              // none), and whether this piece completes the unit's count
              const long long T = bars->T;
              const int grid = gridDim.x;
              const int c_lo = cta_of(g0, T, grid), c_hi = cta_of(g1 - 1, T, grid);
              int n_own = 0;
              for (int c = c_lo; c <= c_hi; ++c)
                if ((long long)c * T / grid != (long long)(c + 1) * T / grid) list[n_own++] = c;
              const unsigned int counted = count_piece(p.counters + u, p.epoch, p.err);
              flags[12] = counted == (unsigned int)n_own ? n_own : 0;
            }
            named_bar_sync(1, 128);
            const int n_merge = flags[12];
            if (n_merge > 0 && key < D) {
              // last piece: merge all of them in one online pass over the
              // pieces (running maximum and rescaled sums, as in the softmax),
              // the loads of every head of a piece issued together
              __threadfence();
              float mm[G], ss[G], acc[G];
#pragma unroll
              for (int h = 0; h < G; ++h) {
                mm[h] = -INFINITY;
                ss[h] = 0.f;
                acc[h] = 0.f;
              }
              for (int t = 0; t < n_merge; ++t) {
                const size_t r0 = ((size_t)u + list[t]) * G;
                float lv[G], ov[G];
#pragma unroll
                for (int h = 0; h < G; ++h) {
                  lv[h] = __ldcg(p.lse_parts + r0 + h);
                  ov[h] = __ldcg(p.o_parts + (r0 + h) * D + key);
                }
#pragma unroll
                for (int h = 0; h < G; ++h) {
                  const float mn = fmaxf(mm[h], lv[h]);
                  const float a = expf(mm[h] - mn), e = expf(lv[h] - mn);
                  ss[h] = ss[h] * a + e;
                  acc[h] = acc[h] * a + e * ov[h];
                  mm[h] = mn;
                }
              }
#pragma unroll
              for (int h = 0; h < G; ++h) {
                o_out[(orow0 + h) * D + key] = to_bits<BF16>(acc[h] / ss[h]);
                if (key == h) p.lse[orow0 + h] = mm[h] + logf(ss[h]);
              }
            }
            named_bar_sync(1, 128);                 // list and flags free for the next piece end
          }
        }
        bad = bad || skip;
        tc_fence_before();
        named_bar_sync(1, 128);                     // red_l and flags free for the next piece
      }
    }
  }
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, int G, bool BF16>
cudaError_t launch_t(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const DecodeParams& p,
                     int grid, cudaStream_t s) {
  constexpr int NQ = G <= 16 ? 16 : 32;
  auto kern = decode_kt_kernel<D, NQ, G, BF16>;
  constexpr int bytes = KtCfg<D, NQ>::BYTES;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, KT_THREADS, bytes, s>>>(q, k, v, p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const DecodeParams& p,
                     int grid, bool bf16, cudaStream_t s) {
#define ATTN45_G(G) \
  case G: return bf16 ? launch_t<D, G, true>(q, k, v, p, grid, s) : launch_t<D, G, false>(q, k, v, p, grid, s)
  switch (p.group) {
    ATTN45_G(1); ATTN45_G(2); ATTN45_G(3); ATTN45_G(4); ATTN45_G(5); ATTN45_G(6); ATTN45_G(7); ATTN45_G(8);
    ATTN45_G(9); ATTN45_G(10); ATTN45_G(11); ATTN45_G(12); ATTN45_G(13); ATTN45_G(14); ATTN45_G(15);
    ATTN45_G(16); ATTN45_G(24); ATTN45_G(32);
    default: return cudaErrorInvalidValue;
  }
#undef ATTN45_G
}
}  // namespace

// Launch for head dim 64 (its own translation unit, compiled in parallel).
cudaError_t launch_decode_kt_d64(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                 const DecodeParams& p, int grid, bool bf16, cudaStream_t s);

}  // namespace attn45
