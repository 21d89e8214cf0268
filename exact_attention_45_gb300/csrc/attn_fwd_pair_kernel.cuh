// attn_fwd_pair_kernel.cuh -- forward for head dim 256 on pairs of CTAs that
// share their tensor-core work (tcgen05 cta_group::2): BF16/FP16, and FP8
// (e4m3 codes with block scales, fixed length).
//
// Same computation as the other forward kernels (tiling so the scores never
// reach HBM: "FlashAttention: Fast and Memory-Efficient Exact Attention with
// IO-Awareness", abstract; online softmax with a running maximum and
// normaliser: "Related papers: FlashAttention-4" page, online-softmax teaser).
// The variant is the 2-CTA one the FlashAttention-3 page lists after its
// Hopper kernel (reference list, appendix B.3 fragment, "3-Stage Pipelining"):
// at head dim 256 a single CTA fits only 64-key blocks (Q, K and V tiles of
// 256 columns fill its shared memory), and its N = 64 products keep the tensor
// core waiting on the issuing thread. Two CTAs of a cluster own one 256-row
// unit of one (sequence, head): the even CTA ("leader") rows 0-127, the odd
// CTA rows 128-255. Each key block has 128 keys:
//   S = Q K^T   one M = 256, N = 128 pair MMA per 16 channels: each CTA feeds
//               its own 128 Q rows and 64 of the 128 keys (its K half);
//   O += P V    one M = 256, N = 256 pair MMA per 16 keys: P from each CTA's
//               TMEM, V's channels split 128 / 128 between the CTAs.
// Per CTA, TMEM holds two S buffers (2 x 128 columns) and O (256 columns), so
// S of block j+1 is computed while the softmax turns block j into P.
// 16-bit: K and V halves stream through rings of their own (2 + 2 stages), a
// K stage released as soon as its Q K^T has run and K copied two blocks ahead
// of V, so a V copy waits for the Q K^T two blocks back instead of competing
// with the K copies; shared memory per CTA Q 64 KB + 2 x 32 KB + 2 x 32 KB +
// output staging 16 KB. FP8 halves the operand tiles (V comes transposed,
// channels as rows, so both products are K-major) and streams them through
// three shared slots, slot j holding K_j and V_{j-1}, released after step j's
// P V (the separate rings measured 5-9 % slower there). FP8 follows the two-tile kernel's FP8 path: the dequantisation
// scalar sq * sk of a 128 x 128 score block is folded into the softmax scale,
// P (<= 2^8 under the lazy maximum) is rounded to e4m3, four per TMEM column,
// and the epilogue applies V's channel scales.
//
// Roles per CTA (192 threads): warps 0-3 softmax / correction / epilogue of
// this CTA's 128 rows (thread r owns row r = TMEM lane r); warp 4 TMA
// producer; warp 5 allocates TMEM (both CTAs) and, in the leader, issues every
// MMA of the pair. Barrier protocol:
//   q_full, k_full, v_full, slot_full  (leader)  both CTAs' copies count
//                      their bytes on the leader's barrier; only the leader
//                      posts the total;
//   q_empty, k_empty, v_empty, slot_empty, s_full, o_done  (both)  multicast
//                      commits of the leader's MMAs;
//   p_full[2] (leader) one arrival per softmax warp of both CTAs (8) once
//                      its P stores are complete, after the previous P V has
//                      landed (so O is stable for the rare correction); the
//                      P stores are ordered before the MMAs by tcgen05.wait::st
//                      and the tcgen05 fences on both sides of this barrier,
//                      so its arrivals carry no cluster-scope release.
// Every wait is bounded (timeout -> abort flag + device error word).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include "attn_common.cuh"
#include "attn_fwd2_kernel.cuh"
#include "ptx.cuh"

namespace attn45 {

template <int D, int ELEM = 2>
struct PairTraits {
  static constexpr int BN = 128;                      // keys per block (over the pair)
  static constexpr int NC = D * ELEM / 128;           // 128-byte chunks per Q / K row
  static constexpr int Q_CHUNK = BLOCK_M * 128;       // 128 rows x 128 bytes
  static constexpr int Q_BYTES = BLOCK_M * D * ELEM;
  static constexpr int K_ROWS = BN / 2;               // keys of a block held by one CTA
  static constexpr int K_CHUNK = K_ROWS * 128;
  static constexpr int K_BYTES = K_ROWS * D * ELEM;
  static constexpr int V_COLS = D / 2;                // channels of V held by one CTA
  // 16-bit: V tiles of 128 keys x 64 channels, MN-major; FP8: one V^T tile of
  // V_COLS channel rows x 128 keys, K-major
  static constexpr int V_NC = ELEM == 2 ? V_COLS / 64 : 1;
  static constexpr int V_CHUNK = ELEM == 2 ? BN * 128 : V_COLS * 128;
  static constexpr int V_BYTES = BN * V_COLS * ELEM;
  // 16-bit: separate K and V rings; FP8: shared slots {K_j, V_{j-1}}
  static constexpr bool SHARED_SLOTS = ELEM == 1;
  static constexpr int K_STAGES = 2, V_STAGES = 2;
  static constexpr int K_AHEAD = 2;                   // K_{j + K_AHEAD} is copied just before V_j
  static constexpr int SLOTS = 3;
  static constexpr int SLOT_BYTES = K_BYTES + V_BYTES;
  static constexpr int RING_BYTES = SHARED_SLOTS ? SLOTS * SLOT_BYTES : K_STAGES * K_BYTES + V_STAGES * V_BYTES;
  static constexpr int THREADS = 192;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = Q_BYTES;               // K ring, or the slots
  static constexpr int OFF_V = OFF_K + K_STAGES * K_BYTES;
  static constexpr int OFF_STAGE = OFF_K + RING_BYTES;  // 4 softmax warps x 4 KB
  static constexpr int STAGE_BYTES = 4 * 4096;
  static constexpr int OFF_BARS = OFF_STAGE + STAGE_BYTES;
  static constexpr int BARS_BYTES = 256;
  static constexpr int OFF_PREFIX = OFF_BARS + BARS_BYTES;
  static constexpr int SMEM_FIXED = OFF_PREFIX + 1024;  // + 1024 for base alignment
  static constexpr int TMEM_S = 0;                    // + 128 * buffer
  static constexpr int TMEM_O = 2 * BN;
  static constexpr int TMEM_COLS = 512;
  static_assert(2 * BN + D <= TMEM_COLS, "TMEM budget");
  static_assert(D % 128 == 0, "V channels split in 64-channel chunks between the pair");
};

struct BarsPair {
  uint64_t q_full, q_empty;
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
  uint64_t slot_full[3], slot_empty[3];
  uint64_t s_full[2], p_full[2];
  uint64_t o_done;
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(BarsPair) <= 256, "barrier block");

template <int D, bool CAUSAL, bool VARLEN, int KIND>
__global__ void __launch_bounds__(192, 1)
attn_fwd_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                     const FwdParams p) {
  constexpr bool FP8 = KIND == KIND_E4M3;
  constexpr bool BF16 = KIND == KIND_BF16;
  constexpr int ELEM = FP8 ? 1 : 2;
  static_assert(!(FP8 && VARLEN), "FP8 on CTA pairs takes fixed-length batches");
  using T = PairTraits<D, ELEM>;
  constexpr int BN = T::BN;
  constexpr bool STAGE_OUT = !VARLEN;
  extern __shared__ uint8_t smem_raw[];
  // the same offset in both CTAs: pair MMAs address both CTAs' operands by
  // one shared-memory offset
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sQ = smem + T::OFF_Q;
  BarsPair* bars = reinterpret_cast<BarsPair*>(smem + T::OFF_BARS);
  int* prefix = reinterpret_cast<int*>(smem + T::OFF_PREFIX);
  volatile int* abort_flag = &bars->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();            // 0 = leader (issues the MMAs)
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int s = 0; s < T::K_STAGES; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < T::V_STAGES; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int s = 0; s < T::SLOTS; ++s) {
      mbar_init(&bars->slot_full[s], 1);
      mbar_init(&bars->slot_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->p_full[b], 8);
    }
    mbar_init(&bars->o_done, 1);
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc_pair(&bars->tmem_base, T::TMEM_COLS);
    tmem_relinquish_pair();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    if (STAGE_OUT) tma_prefetch_desc(&tmO);
  }
  int ntiles = p.ntiles;
  if constexpr (VARLEN) {
    build_varlen_prefix2(p, prefix);                   // contains __syncthreads
    ntiles = prefix[p.nseq];
  }
  // both CTAs' barriers are initialised and their TMEM allocated before any
  // copy, arrival or MMA of the pair can touch them
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const uint64_t tmo = p.timeout_ns;
  const int cluster_id = blockIdx.x >> 1;
  const int nclusters = gridDim.x >> 1;

  auto get_tile = [&](int t) -> Tile2 {
    if constexpr (VARLEN) return tile2_varlen(p, prefix, t);
    else return tile2_fixed<CAUSAL>(p, t);
  };
  // key blocks the pair visits for a unit: those of its longer (later) tile
  auto pair_blocks = [&](const Tile2& tl) -> int {
    return max(tile2_blocks<CAUSAL, BN>(tl, 0), tile2_blocks<CAUSAL, BN>(tl, 1));
  };

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      const uint32_t q_full_l = mapa_shared(&bars->q_full, 0);
      int k_it = 0, v_it = 0, slot_it = 0, tile_i = 0;
      bool ok = true;
      for (int t = cluster_id; t < ntiles && ok; t += nclusters) {
        const Tile2 tl = get_tile(t);
        const int hk = tl.h / p.group;
        const int nkv = pair_blocks(tl);
        if (nkv == 0) continue;
        ok = mbar_wait(&bars->q_empty, (tile_i & 1) ^ 1, tmo, abort_flag, p.err);
        if (!ok) break;
        ++tile_i;
        if (leader) mbar_expect_tx(&bars->q_full, 2 * T::Q_BYTES);
#pragma unroll
        for (int c = 0; c < T::NC; ++c)
          tma_load_4d_pair(&tmQ, q_full_l, sQ + c * T::Q_CHUNK, c * (128 / ELEM), tl.h,
                           tl.tma_row0 + tl.sblk * SUPER_M + (int)rank * BLOCK_M, tl.tma_b);
        // K_j: this CTA's 64 keys of block j
        auto copy_k = [&](int j, uint8_t* dst, uint32_t full_l) {
#pragma unroll
          for (int c = 0; c < T::NC; ++c)
            tma_load_4d_pair(&tmK, full_l, dst + c * T::K_CHUNK, c * (128 / ELEM), hk,
                             tl.tma_row0 + j * BN + (int)rank * T::K_ROWS, tl.tma_b);
        };
        // V_j: this CTA's D / 2 channels of the block's 128 keys
        auto copy_v = [&](int j, uint8_t* dst, uint32_t full_l) {
          if constexpr (FP8) {
            // V^T [B*Hkv][D][ldv]: 128 keys of this CTA's channel rows
            tma_load_4d_pair(&tmV, full_l, dst, j * BN, (int)rank * T::V_COLS, tl.seq * p.Hkv + hk, 0);
          } else {
#pragma unroll
            for (int c = 0; c < T::V_NC; ++c)
              tma_load_4d_pair(&tmV, full_l, dst + c * T::V_CHUNK, (int)rank * T::V_COLS + c * 64, hk,
                               tl.tma_row0 + j * BN, tl.tma_b);
          }
        };
        if constexpr (T::SHARED_SLOTS) {
          // slot j: K_j (j < nkv) and V_{j-1} (j >= 1)
          for (int j = 0; j <= nkv; ++j, ++slot_it) {
            const int st = slot_it % T::SLOTS;
            ok = mbar_wait(&bars->slot_empty[st], ((slot_it / T::SLOTS) & 1) ^ 1, tmo, abort_flag, p.err);
            if (!ok) break;
            uint8_t* slot = smem + T::OFF_K + st * T::SLOT_BYTES;
            const uint32_t full_l = mapa_shared(&bars->slot_full[st], 0);
            if (leader)
              mbar_expect_tx(&bars->slot_full[st], (j < nkv ? 2 * T::K_BYTES : 0) + (j >= 1 ? 2 * T::V_BYTES : 0));
            if (j < nkv) copy_k(j, slot, full_l);
            if (j >= 1) copy_v(j - 1, slot + T::K_BYTES, full_l);
          }
        } else {
          auto load_k = [&](int j) -> bool {
            const int ks = k_it % T::K_STAGES;
            if (!mbar_wait(&bars->k_empty[ks], ((k_it / T::K_STAGES) & 1) ^ 1, tmo, abort_flag, p.err)) return false;
            if (leader) mbar_expect_tx(&bars->k_full[ks], 2 * T::K_BYTES);
            copy_k(j, smem + T::OFF_K + ks * T::K_BYTES, mapa_shared(&bars->k_full[ks], 0));
            ++k_it;
            return true;
          };
          auto load_v = [&](int j) -> bool {
            const int vs = v_it % T::V_STAGES;
            if (!mbar_wait(&bars->v_empty[vs], ((v_it / T::V_STAGES) & 1) ^ 1, tmo, abort_flag, p.err)) return false;
            if (leader) mbar_expect_tx(&bars->v_full[vs], 2 * T::V_BYTES);
            copy_v(j, smem + T::OFF_V + vs * T::V_BYTES, mapa_shared(&bars->v_full[vs], 0));
            ++v_it;
            return true;
          };
          // the order the MMAs consume them, K running K_AHEAD blocks ahead
          for (int j = 0; j < min(T::K_AHEAD, nkv) && ok; ++j) ok = load_k(j);
          for (int j = 0; j < nkv && ok; ++j) {
            if (j + T::K_AHEAD < nkv) ok = load_k(j + T::K_AHEAD);
            if (ok) ok = load_v(j);
          }
        }
      }
      // the leader's barriers count both CTAs' copies: never leave with one in
      // flight (already complete on the normal path)
      if (leader) {
        for (int it = (k_it > T::K_STAGES ? k_it - T::K_STAGES : 0); it < k_it; ++it)
          mbar_wait_drain(&bars->k_full[it % T::K_STAGES], (it / T::K_STAGES) & 1, tmo, p.err);
        for (int it = (v_it > T::V_STAGES ? v_it - T::V_STAGES : 0); it < v_it; ++it)
          mbar_wait_drain(&bars->v_full[it % T::V_STAGES], (it / T::V_STAGES) & 1, tmo, p.err);
        for (int it = (slot_it > T::SLOTS ? slot_it - T::SLOTS : 0); it < slot_it; ++it)
          mbar_wait_drain(&bars->slot_full[it % T::SLOTS], (it / T::SLOTS) & 1, tmo, p.err);
        if (tile_i > 0) mbar_wait_drain(&bars->q_full, (tile_i - 1) & 1, tmo, p.err);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer (leader only)
    // Step j: S(j) = Q K_j^T into S buffer (j-th S overall) & 1, then
    // O += P(j-1) V_{j-1} once both CTAs' P(j-1) is stored, so the tensor core
    // computes the next scores while the softmax warps work.
    // the whole warp runs the loop (convergent control flow); one elected
    // lane issues each MMA and commit
    if (leader) {
      constexpr uint32_t idesc_s = FP8 ? idesc_kind_f8_e4m3(2 * BLOCK_M, BN) : idesc_kind_f16(2 * BLOCK_M, BN, BF16, false);
      constexpr uint32_t idesc_o = FP8 ? idesc_kind_f8_e4m3(2 * BLOCK_M, D) : idesc_kind_f16(2 * BLOCK_M, D, BF16, true);
      constexpr int S_STEPS = D * ELEM / 32;               // 32-byte K steps of Q K^T
      constexpr int PV_STEPS = BN * ELEM / 32;             // 32-byte K steps of P V
      constexpr uint16_t both = 3;
      // descriptor low halves of the operands' first bytes: each MMA's
      // descriptor is one of these plus a constant, so no descriptor
      // arithmetic sits between S(j)'s last MMA and P(j-1) V's first
      const uint32_t q_lo = sdesc_lo_kmajor_sw128(smem_u32(sQ));
      const uint32_t k_lo = sdesc_lo_kmajor_sw128(smem_u32(smem + T::OFF_K));
      const uint32_t v_lo = FP8 ? sdesc_lo_kmajor_sw128(smem_u32(smem + T::OFF_V))
                                : sdesc_lo_mnmajor_sw128(smem_u32(smem + T::OFF_V), T::V_CHUNK);
      // the V of a shared slot sits K_BYTES after the slot's K (read with the
      // V operand's own layout)
      const uint32_t kv_lo = FP8 ? sdesc_lo_kmajor_sw128(smem_u32(smem + T::OFF_K) + T::K_BYTES)
                                 : sdesc_lo_mnmajor_sw128(smem_u32(smem + T::OFF_K) + T::K_BYTES, T::V_CHUNK);
      int k_it = 0, v_it = 0, slot_it = 0, tile_i = 0, s_it = 0, pv_it = 0;
      bool ok = true;
      for (int t = cluster_id; t < ntiles && ok; t += nclusters) {
        const Tile2 tl = get_tile(t);
        const int nkv = pair_blocks(tl);
        if (nkv == 0) continue;
        ok = mbar_wait_warp(&bars->q_full, tile_i & 1, tmo, abort_flag, p.err);
        ++tile_i;
        if (!ok) break;
        for (int j = 0; j <= nkv && ok; ++j, ++slot_it) {
          // shared slots: K_j and V_{j-1} arrive on one barrier
          const int st = slot_it % T::SLOTS;
          if constexpr (T::SHARED_SLOTS) {
            ok = mbar_wait_warp(&bars->slot_full[st], (slot_it / T::SLOTS) & 1, tmo, abort_flag, p.err);
            if (!ok) break;
            tc_fence_after();
          }
          if (j < nkv) {
            const int ks = k_it % T::K_STAGES;
            const uint32_t kb_lo = k_lo + (T::SHARED_SLOTS ? st * (T::SLOT_BYTES >> 4) : ks * (T::K_BYTES >> 4));
            if constexpr (!T::SHARED_SLOTS) {
              ok = mbar_wait_warp(&bars->k_full[ks], (k_it / T::K_STAGES) & 1, tmo, abort_flag, p.err);
              if (!ok) break;
              tc_fence_after();
            }
            const uint32_t s_tmem = tmem + T::TMEM_S + (s_it & 1) * BN;
#pragma unroll
            for (int k = 0; k < S_STEPS; ++k) {
              const uint32_t qo = ((k >> 2) * T::Q_CHUNK + (k & 3) * 32) >> 4;
              const uint32_t ko = ((k >> 2) * T::K_CHUNK + (k & 3) * 32) >> 4;
              if constexpr (FP8)
                umma_f8_ss_pair_lo_w(s_tmem, q_lo + qo, kb_lo + ko, idesc_s, k > 0 ? 1u : 0u);
              else
                umma_f16_ss_pair_lo_w(s_tmem, q_lo + qo, kb_lo + ko, idesc_s, k > 0 ? 1u : 0u);
            }
            umma_commit_pair_w(&bars->s_full[s_it & 1], both);
            if constexpr (!T::SHARED_SLOTS) umma_commit_pair_w(&bars->k_empty[ks], both);
            if (j == nkv - 1) umma_commit_pair_w(&bars->q_empty, both);
            ++s_it;
            ++k_it;
          }
          if (j >= 1) {
            // P(j-1) lives in the S buffer of the pv_it-th S
            const int vs = v_it % T::V_STAGES;
            const uint32_t vb_lo = T::SHARED_SLOTS ? kv_lo + st * (T::SLOT_BYTES >> 4) : v_lo + vs * (T::V_BYTES >> 4);
            ok = mbar_wait_warp(&bars->p_full[pv_it & 1], (pv_it >> 1) & 1, tmo, abort_flag, p.err);
            if constexpr (!T::SHARED_SLOTS)
              if (ok) ok = mbar_wait_warp(&bars->v_full[vs], (v_it / T::V_STAGES) & 1, tmo, abort_flag, p.err);
            if (!ok) break;
            tc_fence_after();
            const uint32_t a_tmem = tmem + T::TMEM_S + (pv_it & 1) * BN;
#pragma unroll
            for (int k = 0; k < PV_STEPS; ++k) {
              // each K step is 8 TMEM columns of P (16 x 16-bit or 32 x 8-bit)
              if constexpr (FP8)
                umma_f8_ts_pair_lo_w(tmem + T::TMEM_O, a_tmem + k * 8, vb_lo + k * (32 >> 4), idesc_o,
                                   (j > 1 || k > 0) ? 1u : 0u);
              else
                umma_f16_ts_pair_lo_w(tmem + T::TMEM_O, a_tmem + k * 8, vb_lo + k * (2048 >> 4), idesc_o,
                                    (j > 1 || k > 0) ? 1u : 0u);
            }
            umma_commit_pair_w(&bars->o_done, both);
            if constexpr (!T::SHARED_SLOTS) umma_commit_pair_w(&bars->v_empty[vs], both);
            ++pv_it;
            ++v_it;
          }
          if constexpr (T::SHARED_SLOTS) umma_commit_pair_w(&bars->slot_empty[st], both);
        }
      }
      umma_commit_pair_w(&bars->mma_done, 1);
      mbar_wait_drain(&bars->mma_done, 0, tmo, p.err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------- softmax / correction / epilogue (both CTAs)
    const int r = threadIdx.x;                         // row within this CTA's tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t to = tmem + lane_off + T::TMEM_O;
    const uint32_t p_full_l0 = mapa_shared(&bars->p_full[0], 0), p_full_l1 = mapa_shared(&bars->p_full[1], 0);
    constexpr float lazy = LAZY_RESCALE_LOG2;
    int s_cnt = 0, o_cnt = 0;
    bool ok = true;
    for (int t = cluster_id; t < ntiles && ok; t += nclusters) {
      const Tile2 tl = get_tile(t);
      const int nkv = pair_blocks(tl);
      if (nkv == 0) continue;
      const int row0 = tl.sblk * SUPER_M + (int)rank * BLOCK_M;   // first row of this CTA's tile
      const int i_row = row0 + r;
      const int hk = tl.h / p.group;
      // FP8 block scales [B][heads][ceil(N/128)]: this tile's Q block, key block j
      const int nb128 = ceil_div(tl.n, BLOCK_M);
      const size_t sk_row = ((size_t)tl.seq * p.Hkv + hk) * nb128;
      float sq_x = 1.f, sk_j = 1.f;
      if constexpr (FP8) {
        sq_x = p.fp8_block ? __ldg(p.sq + ((size_t)tl.seq * p.H + tl.h) * nb128 + min(row0 >> 7, nb128 - 1))
                           : __ldg(p.sq);
        sk_j = p.fp8_block ? __ldg(p.sk + sk_row) : __ldg(p.sk);
      }
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < nkv; ++j) {
        const int sb = s_cnt & 1;
        float sl2 = p.scale_log2;
        if constexpr (FP8) {
          sl2 *= sq_x * sk_j;
          if (p.fp8_block && j + 1 < nkv) sk_j = __ldg(p.sk + sk_row + j + 1);
        }
        ok = mbar_wait(&bars->s_full[sb], (s_cnt >> 1) & 1, tmo, abort_flag, p.err);
        ++s_cnt;
        if (!ok) break;
        tc_fence_after();
        const uint32_t ts = tmem + lane_off + T::TMEM_S + sb * BN;
        float s[BN];
        float mx;                                     // row maximum of the block's scores
        {
          uint32_t u[BN];
          tmem_ld128_max(ts, u, mx);
#pragma unroll
          for (int i = 0; i < BN; ++i) s[i] = __uint_as_float(u[i]);
        }
        // keys past the sequence end, and (causal) keys after the row; blocks
        // past this tile's diagonal (the pair runs its later tile's blocks)
        // mask every key, which leaves m, l and O unchanged
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
        // the running maximum moves only past the lazy margin (2^8)
        const bool raise = mx > m + lazy;
        const float m_new = raise ? mx : m;
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = raise ? ex2_approx(m - m_use) : 1.f;
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
        const uint64_t negm2 = f2_pack(-m_use, -m_use);
        uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = acc0;
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
            if (c == 60) tmem_st32(ts, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
          }
        }
        float sum0, sum1, sum2, sum3;
        f2_unpack(acc0, sum0, sum1);
        f2_unpack(acc1, sum2, sum3);
        l = l * alpha + ((sum0 + sum1) + (sum2 + sum3));
        m = m_new;
        if constexpr (FP8) tmem_st32(ts, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
        else tmem_st32(ts + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
        tmem_st_wait();
        if (j > 0) {
          // O += P(j-1) V_{j-1} was issued after S(j): wait for it before the
          // correction (and before P(j) may be consumed)
          ok = mbar_wait(&bars->o_done, o_cnt & 1, tmo, abort_flag, p.err);
          ++o_cnt;
          if (!ok) break;
          tc_fence_after();
          if (__any_sync(0xffffffffu, raise)) {
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
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(sb ? p_full_l1 : p_full_l0);
      }
      if (!ok) break;
      ok = mbar_wait(&bars->o_done, o_cnt & 1, tmo, abort_flag, p.err);
      ++o_cnt;
      if (!ok) break;
      tc_fence_after();
      const bool valid = i_row < tl.nq;
      const float inv_l = 1.f / l;
      const size_t tok = (size_t)tl.tok0 + (size_t)(valid ? i_row : 0);
      uint4* orow = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.o) + (tok * p.H + tl.h) * D);
      const float* svp = FP8 ? (p.fp8_block ? p.sv + ((size_t)tl.seq * p.Hkv + hk) * D : p.sv) : nullptr;
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        uint32_t u[64];
        tmem_ld64(to + c * 64, u);
        uint32_t w[32];
        if constexpr (FP8) {
          // O / l times V's channel scale; BF16 output
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int ch = c * 64 + 2 * i;
            const float s0 = p.fp8_block ? __ldg(svp + ch) : __ldg(svp);
            const float s1 = p.fp8_block ? __ldg(svp + ch + 1) : s0;
            w[i] = pack2(__uint_as_float(u[2 * i]) * (s0 * inv_l), __uint_as_float(u[2 * i + 1]) * (s1 * inv_l), true);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            w[i] = pack2(__uint_as_float(u[2 * i]) * inv_l, __uint_as_float(u[2 * i + 1]) * inv_l, BF16);
        }
        if constexpr (STAGE_OUT) {
          // this warp's 32 rows x 64 columns, 128-byte swizzled, one bulk
          // tensor store (rows past the sequence end are clipped by the copy)
          const uint32_t stg = smem_u32(smem + T::OFF_STAGE + warp * 4096);
          if (lane == 0) tma_store_wait_read();
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 8; ++i)
            st_shared_v4(stg + lane * 128 + ((i ^ (lane & 7)) << 4), w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_4d(&tmO, smem + T::OFF_STAGE + warp * 4096, c * 64, tl.h, row0 + warp * 32, tl.tma_b);
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
        else p.lse[((size_t)tl.seq * p.H + tl.h) * p.N + i_row] = lse;
      }
    }
    if (STAGE_OUT && lane == 0) tma_store_wait_all();
  }

  // neither CTA leaves (or frees TMEM) while the pair's MMAs, copies or
  // arrivals may still reach it
  __syncwarp();
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  if (warp == 5) tmem_dealloc_pair(tmem, T::TMEM_COLS);
}

}  // namespace attn45
