// attn_fwd_kernel.cuh -- fused exact attention forward for sm_103a, BF16/FP16.
//
// Computes O = softmax(Q K^T * scale [+ causal mask]) V and the per-row
// logsumexp, tiled over 128-row query blocks and streamed over BN-row key
// blocks with an online softmax, so the N x N score matrix never leaves the
// chip ("FlashAttention: Fast and Memory-Efficient Exact Attention with
// IO-Awareness", abstract: tiling between HBM and on-chip memory; the
// "Related papers: FlashAttention-4" page, online-softmax teaser: a running
// maximum and normaliser per row).
//
// Roles (warp specialisation, "FlashAttention-3 ...", abstract technique (1)):
//   warps 0-3  softmax + correction + epilogue; thread r owns query row r,
//              which is TMEM lane r of the S and O accumulators;
//   warp 4     TMA producer: Q tile once, K/V blocks through a STAGES ring;
//   warp 5     MMA issuer (one thread): S = Q K^T into one of two TMEM S
//              buffers, then O += P V with P read from TMEM.
// With two S buffers the tensor core computes S for block j+1 while the
// softmax warps work on block j (block-wise interleaving of matmul and
// softmax, "FlashAttention-3 ...", abstract technique (2)).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include "attn_common.cuh"
#include "ptx.cuh"

namespace attn45 {

template <int D, int BN, int STAGES>
struct Bf16Traits {
  static constexpr int NC = D / 64;                 // 128-byte column chunks per row
  static constexpr int Q_CHUNK = BLOCK_M * 128;     // bytes per Q chunk
  static constexpr int KV_CHUNK = BN * 128;         // bytes per K/V chunk
  static constexpr int Q_BYTES = BLOCK_M * D * 2;
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * KV_BYTES;
  static constexpr int OFF_BARS = OFF_V + STAGES * KV_BYTES;
  static constexpr int BARS_BYTES = 512;
  static constexpr int OFF_PREFIX = OFF_BARS + BARS_BYTES;
  static constexpr int SMEM_FIXED = OFF_PREFIX + 1024;   // + 1024 for base alignment
  static constexpr int TMEM_S0 = 0;
  static constexpr int TMEM_S1 = BN;
  static constexpr int TMEM_O = 2 * BN;
  static constexpr int TMEM_COLS = 512;
  static_assert(2 * BN + D <= TMEM_COLS, "TMEM budget");
  static_assert(D % 64 == 0 && BN % 32 == 0, "shape");
};

struct Bars {
  uint64_t q_full, q_empty;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2], p_full[2];
  uint64_t o_done, mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 512, "barrier block");

__device__ __forceinline__ uint32_t pack2(float lo, float hi, bool bf16) {
  if (bf16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

template <int D, int BN, int STAGES, bool CAUSAL, bool VARLEN, bool BF16>
__global__ void __launch_bounds__(192, 1)
attn_fwd_f16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using T = Bf16Traits<D, BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sQ = smem + T::OFF_Q;
  uint8_t* sK = smem + T::OFF_K;
  uint8_t* sV = smem + T::OFF_V;
  Bars* bars = reinterpret_cast<Bars*>(smem + T::OFF_BARS);
  int* prefix = reinterpret_cast<int*>(smem + T::OFF_PREFIX);
  volatile int* abort_flag = &bars->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->p_full[b], 128);
    }
    mbar_init(&bars->o_done, 1);
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&bars->tmem_base, T::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  int ntiles = p.ntiles;
  if constexpr (VARLEN) {
    build_varlen_prefix(p, prefix);   // contains __syncthreads
    ntiles = prefix[p.nseq];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const uint64_t tmo = p.timeout_ns;

  auto get_tile = [&](int t) -> Tile {
    if constexpr (VARLEN) return tile_varlen(p, prefix, t);
    else return tile_fixed(p, t);
  };
  // number of key blocks a tile visits, and whether block j needs masking
  auto kv_blocks = [&](const Tile& tl) -> int {
    int kend = tl.n;
    if (CAUSAL) kend = min(kend, (tl.qblk + 1) * BLOCK_M);
    return ceil_div(kend, BN);
  };

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int kv_it = 0, tile_i = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++tile_i) {
        const Tile tl = get_tile(t);
        const int hk = tl.h / p.group;
        const int nblk = kv_blocks(tl);
        ok = mbar_wait(&bars->q_empty, (tile_i & 1) ^ 1, tmo, abort_flag, p.err);
        if (!ok) break;
        mbar_expect_tx(&bars->q_full, T::Q_BYTES);
#pragma unroll
        for (int c = 0; c < T::NC; ++c)
          tma_load_4d(&tmQ, &bars->q_full, sQ + c * T::Q_CHUNK, c * 64, tl.h,
                      tl.tma_row0 + tl.qblk * BLOCK_M, tl.tma_b);
        for (int j = 0; j < nblk; ++j, ++kv_it) {
          const int st = kv_it % STAGES;
          const uint32_t ph = (kv_it / STAGES) & 1;
          const int krow = tl.tma_row0 + j * BN;
          ok = mbar_wait(&bars->k_empty[st], ph ^ 1, tmo, abort_flag, p.err);
          if (!ok) break;
          mbar_expect_tx(&bars->k_full[st], T::KV_BYTES);
#pragma unroll
          for (int c = 0; c < T::NC; ++c)
            tma_load_4d(&tmK, &bars->k_full[st], sK + st * T::KV_BYTES + c * T::KV_CHUNK, c * 64, hk, krow,
                        tl.tma_b);
          ok = mbar_wait(&bars->v_empty[st], ph ^ 1, tmo, abort_flag, p.err);
          if (!ok) { ++kv_it; break; }
          mbar_expect_tx(&bars->v_full[st], T::KV_BYTES);
#pragma unroll
          for (int c = 0; c < T::NC; ++c)
            tma_load_4d(&tmV, &bars->v_full[st], sV + st * T::KV_BYTES + c * T::KV_CHUNK, c * 64, hk, krow,
                        tl.tma_b);
        }
      }
      // Never leave with copies in flight: wait for the last armed phase of
      // every stage (already complete on the normal path).
      const int last = kv_it;
      for (int it = (last > STAGES ? last - STAGES : 0); it < last; ++it) {
        const int st = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        mbar_wait_drain(&bars->k_full[st], ph, tmo, p.err);
        mbar_wait_drain(&bars->v_full[st], ph, tmo, p.err);
      }
      if (tile_i > 0) mbar_wait_drain(&bars->q_full, (tile_i - 1) & 1, tmo, p.err);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_kind_f16(BLOCK_M, BN, BF16, false);
      constexpr uint32_t idesc_o = idesc_kind_f16(BLOCK_M, D, BF16, true);
      const uint32_t qa = smem_u32(sQ);
      const uint32_t ka = smem_u32(sK);
      const uint32_t va = smem_u32(sV);
      int kv_it = 0, s_it = 0, tile_i = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++tile_i) {
        const Tile tl = get_tile(t);
        const int nblk = kv_blocks(tl);
        ok = mbar_wait(&bars->q_full, tile_i & 1, tmo, abort_flag, p.err);
        if (!ok) break;
        int prev_st = 0;
        for (int j = 0; j <= nblk && ok; ++j) {
          if (j < nblk) {
            // S(j) = Q K_j^T into S buffer s_it & 1
            const int st = kv_it % STAGES;
            ok = mbar_wait(&bars->k_full[st], (kv_it / STAGES) & 1, tmo, abort_flag, p.err);
            if (!ok) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem + ((s_it & 1) ? T::TMEM_S1 : T::TMEM_S0);
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
              const uint32_t off = (k >> 2) * T::Q_CHUNK + (k & 3) * 32;
              const uint32_t koff = (k >> 2) * T::KV_CHUNK + (k & 3) * 32;
              umma_f16_ss(d_tmem, sdesc_kmajor_sw128(qa + off),
                          sdesc_kmajor_sw128(ka + st * T::KV_BYTES + koff), idesc_s, k > 0 ? 1u : 0u);
            }
            umma_commit(&bars->s_full[s_it & 1]);
            umma_commit(&bars->k_empty[st]);
            if (j == nblk - 1) umma_commit(&bars->q_empty);
          }
          if (j > 0) {
            // O += P(j-1) V_{j-1}; P lives in the S buffer it was computed in
            const int ps = s_it - 1;
            ok = mbar_wait(&bars->p_full[ps & 1], (ps >> 1) & 1, tmo, abort_flag, p.err);
            if (!ok) break;
            ok = mbar_wait(&bars->v_full[prev_st], ((kv_it - 1) / STAGES) & 1, tmo, abort_flag, p.err);
            if (!ok) break;
            tc_fence_after();
            const uint32_t a_tmem = tmem + ((ps & 1) ? T::TMEM_S1 : T::TMEM_S0);
            const uint32_t vbase = va + prev_st * T::KV_BYTES;
#pragma unroll
            for (int k = 0; k < BN / 16; ++k) {
              umma_f16_ts(tmem + T::TMEM_O, a_tmem + k * 8, sdesc_mnmajor_sw128(vbase + k * 2048, T::KV_CHUNK),
                          idesc_o, (j > 1 || k > 0) ? 1u : 0u);
            }
            umma_commit(&bars->o_done);
            umma_commit(&bars->v_empty[prev_st]);
          }
          if (j < nblk) {
            prev_st = kv_it % STAGES;
            ++kv_it;
            ++s_it;
          }
        }
      }
      umma_commit(&bars->mma_done);
      mbar_wait_drain(&bars->mma_done, 0, tmo, p.err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------- softmax / correction / epilogue
    const int r = threadIdx.x;                       // query row within the tile
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const float sl2 = p.scale_log2;
    int s_it = 0, pv_cnt = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
      const Tile tl = get_tile(t);
      const int nblk = kv_blocks(tl);
      const int i_row = tl.qblk * BLOCK_M + r;       // row index within the sequence
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < nblk; ++j, ++s_it) {
        const int sb = s_it & 1;
        ok = mbar_wait(&bars->s_full[sb], (s_it >> 1) & 1, tmo, abort_flag, p.err);
        if (!ok) break;
        tc_fence_after();
        const uint32_t ts = tmem + lane_off + (sb ? T::TMEM_S1 : T::TMEM_S0);
        float s[BN];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t u[32];
          tmem_ld32(ts + c * 32, u);
#pragma unroll
          for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(u[i]);
        }
        // mask: keys past the sequence end, and (causal) keys after the row
        const int col0 = j * BN;
        const bool need_mask = (col0 + BN > tl.n) || (CAUSAL && col0 + BN - 1 > tl.qblk * BLOCK_M);
        if (need_mask) {
          int limit = tl.n - col0;
          if (CAUSAL) limit = min(limit, i_row - col0 + 1);
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (c >= limit) s[c] = -INFINITY;
        }
        float mx = s[0];
#pragma unroll
        for (int c = 1; c < BN; ++c) mx = fmaxf(mx, s[c]);
        const float m_new = fmaxf(m, mx * sl2);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = ex2_approx(m - m_use);   // 0 on the first block
        float rowsum = 0.f;
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          s[c] = ex2_approx(fmaf(s[c], sl2, -m_use));
          rowsum += s[c];
        }
        l = l * alpha + rowsum;
        m = m_new;
        // P (16-bit pairs) overwrites the first BN/2 columns of this S buffer
#pragma unroll
        for (int c = 0; c < BN / 64; ++c) {
          uint32_t u[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) u[i] = pack2(s[c * 64 + 2 * i], s[c * 64 + 2 * i + 1], BF16);
          tmem_st32(ts + c * 32, u);
        }
        if constexpr ((BN / 2) % 32 != 0) {
          uint32_t u[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            u[i] = pack2(s[(BN / 64) * 64 + 2 * i], s[(BN / 64) * 64 + 2 * i + 1], BF16);
          tmem_st16(ts + (BN / 64) * 32, u);
        }
        if (j > 0) {
          // correction: wait until O += P(j-1) V has landed, then rescale O
          ok = mbar_wait(&bars->o_done, pv_cnt & 1, tmo, abort_flag, p.err);
          ++pv_cnt;
          if (!ok) break;
          tc_fence_after();
          if (__any_sync(0xffffffffu, alpha != 1.f)) {
            const uint32_t to = tmem + lane_off + T::TMEM_O;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t u[32];
              tmem_ld32(to + c * 32, u);
#pragma unroll
              for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
              tmem_st32(to + c * 32, u);
            }
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&bars->p_full[sb]);
      }
      if (!ok) break;
      // epilogue: wait for the last O += P V, then O / l and the logsumexp
      ok = mbar_wait(&bars->o_done, pv_cnt & 1, tmo, abort_flag, p.err);
      ++pv_cnt;
      if (!ok) break;
      tc_fence_after();
      const bool valid = i_row < tl.n;
      const float inv_l = 1.f / l;
      const size_t tok = (size_t)tl.tok0 + (size_t)(valid ? i_row : 0);
      uint4* orow = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.o) + (tok * p.H + tl.h) * D);
      const uint32_t to = tmem + lane_off + T::TMEM_O;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t u[32];
        tmem_ld32(to + c * 32, u);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack2(__uint_as_float(u[2 * i]) * inv_l, __uint_as_float(u[2 * i + 1]) * inv_l, BF16);
        if (valid) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            orow[c * 4 + i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
      if (valid) {
        const float lse = (m + lg2_approx(l)) * 0.69314718055994530942f;
        if constexpr (VARLEN) p.lse[(size_t)tl.h * p.total + tok] = lse;
        else p.lse[((size_t)tl.seq * p.H + tl.h) * p.N + i_row] = lse;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, T::TMEM_COLS);
}

}  // namespace attn45
