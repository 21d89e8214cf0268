// attn_bwd.cu -- BF16/FP16 attention backward (dQ, dK, dV), head dim 64/128.
//
// The backward pass of the FlashAttention papers (FA1: exact attention that
// "trains Transformers faster"; it consumes the forward's logsumexp, so P is
// recomputed from S and lse instead of stored). For a key block j of 128 keys
// and every query block i of 128 rows that sees it (every head of the group
// for grouped-query attention), with keys on the TMEM lanes:
//     S^T = K_j Q_i^T               P^T = exp(scale S^T - lse_i)  (lse per column)
//     dP^T = V_j dO_i^T             dS^T = scale P^T * (dP^T - D_i), D_i = rowsum(dO_i * O_i)
//     dV_j += P^T dO_i              dK_j += dS^T Q_i               dQ_i += dS K_j
// One CTA owns a (batch, KV head, key block) unit: dV_j and dK_j stay in TMEM
// across all its query blocks and are written once; P^T and dS^T are written
// back over S^T and dP^T in TMEM and are the A operands of dV and dK, so P never
// goes through shared memory; dS is also stored to shared memory (rows = keys)
// as dQ's A operand. dQ_i is produced per block in TMEM, staged in shared
// memory (over the dS tile and the free P tile) and added into an fp32
// accumulator in HBM by bulk tensor reductions (other key blocks add to the
// same rows); converted at the end.
//
// Roles (320 threads): warps 0-7 compute (thread r of a warpgroup owns TMEM
// lane r: key r for S^T/dP^T/dV/dK, query row r for dQ; warpgroup 0 takes
// query columns 0-63, warpgroup 1 columns 64-127), warp 8 lane 0 loads by
// TMA, warp 9 lane 0 issues the MMAs. TMEM: S^T (128 cols, reused for dQ),
// dP^T (128), dV (d), dK (d). Shared memory: K_j, V_j, two Q tiles (Q_{i+1}
// arrives while block i runs), the dO_i tile, the dS tile, the dQ staging
// half (the old P tile), and the block's lse / D per query.
// Per query block the MMA thread issues dP^T = V dO_i^T first (after the
// previous dK, which read dS^T from those columns), S^T = K Q_i^T once the
// previous dQ has been read out of S's columns, then dV and dK as soon as P^T
// and dS^T are in TMEM (while the compute warps store dS), and dQ once dS is
// stored. Each warpgroup stages its half of dQ in the chunks of the two tiles
// it writes itself and waits only for its own previous reduction.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include "api_internal.h"
#include "attn_common.cuh"
#include "bwd_launchers.h"
#include "ptx.cuh"

namespace attn45 {
namespace {

template <int D>
struct BwdTraits {
  static constexpr int CHUNK = 128 * 128;            // 128 rows x 128 bytes
  static constexpr int TILE = 128 * D * 2;           // one 128-row bf16 tile of width d
  static constexpr int PTILE = 128 * 128 * 2;        // P or dS: 128 queries x 128 keys
  static constexpr int OFF_K = 0, OFF_V = TILE, OFF_Q = 2 * TILE;   // Q: two tiles (block parity)
  static constexpr int OFF_DO = 4 * TILE;
  static constexpr int OFF_P = 5 * TILE, OFF_DS = OFF_P + PTILE;
  static constexpr int OFF_LSD = OFF_DS + PTILE;      // lse*log2(e) and D of the block's 128 queries
  static constexpr int OFF_BARS = OFF_LSD + 256 * 4;
  static constexpr int SMEM = OFF_BARS + 256 + 1024;  // + alignment slack
  static constexpr int T_S = 0, T_DP = 128, T_DV = 256, T_DK = 256 + D;
};

struct BwdBars {
  uint64_t kv_full, kv_empty, q_full[2], q_empty[2], do_full, do_empty, s_full, p_full, ds_full, dq_full, dq_empty,
      dkv_full, dkv_empty, done;
  uint32_t tmem_base;
  int abort;
};

struct BwdUnit {
  int b, hkv, j, i0, nI, nblk, rot;
};

// Units of one (batch, KV head) are adjacent, so the CTAs working on them at
// the same time share that head's Q, dO and dQ rows in L2; inside a head the
// key blocks run in order (causal: the longest, j = 0, first).
__device__ __forceinline__ BwdUnit bwd_unit(const BwdParams& p, int t, bool causal) {
  BwdUnit u;
  const int nqb = ceil_div(p.N, 128);
  u.j = t % nqb;
  const int r = t / nqb;
  u.b = r / p.Hkv;
  u.hkv = r % p.Hkv;
  u.i0 = causal ? u.j : 0;
  u.nI = nqb - u.i0;
  u.nblk = u.nI * p.group;
  // units of one head start at different query blocks, so CTAs running at
  // the same time reduce into different dQ rows
  u.rot = u.j % u.nI;
  return u;
}

// Query block of step `it` of a unit (heads of the group outermost).
__device__ __forceinline__ int bwd_qblock(const BwdUnit& u, int it) { return u.i0 + (it % u.nI + u.rot) % u.nI; }

__device__ __forceinline__ float to_f(uint32_t u) { return __uint_as_float(u); }

// Two TMEM loads of 32 lanes x 32 columns (e.g. the same rows of two regions)
// with one wait for both.
__device__ __forceinline__ void tmem_ld32x2(uint32_t ta, uint32_t (&a)[32], uint32_t tb, uint32_t (&b)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]), "=r"(a[8]),
        "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]), "=r"(a[16]),
        "=r"(a[17]), "=r"(a[18]), "=r"(a[19]), "=r"(a[20]), "=r"(a[21]), "=r"(a[22]), "=r"(a[23]), "=r"(a[24]),
        "=r"(a[25]), "=r"(a[26]), "=r"(a[27]), "=r"(a[28]), "=r"(a[29]), "=r"(a[30]), "=r"(a[31]), "=r"(b[0]),
        "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]), "=r"(b[8]), "=r"(b[9]),
        "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15]), "=r"(b[16]), "=r"(b[17]),
        "=r"(b[18]), "=r"(b[19]), "=r"(b[20]), "=r"(b[21]), "=r"(b[22]), "=r"(b[23]), "=r"(b[24]), "=r"(b[25]),
        "=r"(b[26]), "=r"(b[27]), "=r"(b[28]), "=r"(b[29]), "=r"(b[30]), "=r"(b[31])
      : "r"(ta), "r"(tb)
      : "memory");
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack16(float lo, float hi) {
  uint32_t r;
  if (BF16) asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  else asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

constexpr int BWD_THREADS = 320;
constexpr int BWD_COMPUTE = 256;

template <int D, bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(BWD_THREADS, 1)
attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                const __grid_constant__ CUtensorMap tmDQ, const BwdParams p) {
  using T = BwdTraits<D>;
  constexpr int NC = D / 64;                         // 128-byte chunks per row of a d-wide tile
  constexpr int KS = D / 16;                         // K steps over d
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + T::OFF_BARS);
  volatile int* abort_flag = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    mbar_init(&bars->kv_empty, 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars->q_full[x], 1);
      mbar_init(&bars->q_empty[x], 1);
    }
    mbar_init(&bars->do_full, 1);
    mbar_init(&bars->do_empty, 1);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->p_full, BWD_COMPUTE);
    mbar_init(&bars->ds_full, BWD_COMPUTE);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_empty, BWD_COMPUTE);
    mbar_init(&bars->dkv_full, 1);
    mbar_init(&bars->dkv_empty, BWD_COMPUTE);
    mbar_init(&bars->done, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmDO);
    tma_prefetch_desc(&tmDQ);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const uint64_t tmo = p.timeout_ns;
  const int nunits = p.nunits;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int unit_i = 0, blk_it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < nunits && ok; t += gridDim.x, ++unit_i) {
        const BwdUnit u = bwd_unit(p, t, CAUSAL);
        ok = mbar_wait(&bars->kv_empty, (unit_i & 1) ^ 1, tmo, abort_flag, p.err);
        if (!ok) break;
        mbar_expect_tx(&bars->kv_full, 2 * T::TILE);
        for (int c = 0; c < NC; ++c) {
          tma_load_4d(&tmK, &bars->kv_full, smem + T::OFF_K + c * T::CHUNK, c * 64, u.hkv, u.j * 128, u.b);
          tma_load_4d(&tmV, &bars->kv_full, smem + T::OFF_V + c * T::CHUNK, c * 64, u.hkv, u.j * 128, u.b);
        }
        for (int it = 0; it < u.nblk; ++it, ++blk_it) {
          const int h = u.hkv * p.group + it / u.nI;
          const int i = bwd_qblock(u, it);
          // Q_i into tile blk_it & 1 (free since block blk_it - 2's dK), then dO_i
          // (free since the previous block's dV)
          const int qs = blk_it & 1;
          ok = mbar_wait(&bars->q_empty[qs], ((blk_it >> 1) & 1) ^ 1, tmo, abort_flag, p.err);
          if (!ok) break;
          mbar_expect_tx(&bars->q_full[qs], T::TILE);
          for (int c = 0; c < NC; ++c)
            tma_load_4d(&tmQ, &bars->q_full[qs], smem + T::OFF_Q + qs * T::TILE + c * T::CHUNK, c * 64, h, i * 128, u.b);
          ok = mbar_wait(&bars->do_empty, (blk_it & 1) ^ 1, tmo, abort_flag, p.err);
          if (!ok) { ++blk_it; break; }
          mbar_expect_tx(&bars->do_full, T::TILE);
          for (int c = 0; c < NC; ++c)
            tma_load_4d(&tmDO, &bars->do_full, smem + T::OFF_DO + c * T::CHUNK, c * 64, h, i * 128, u.b);
        }
      }
      // never leave with copies in flight
      for (int it = (blk_it > 2 ? blk_it - 2 : 0); it < blk_it; ++it)
        mbar_wait_drain(&bars->q_full[it & 1], (it >> 1) & 1, tmo, p.err);
      if (blk_it > 0) mbar_wait_drain(&bars->do_full, (blk_it - 1) & 1, tmo, p.err);
      if (unit_i > 0) mbar_wait_drain(&bars->kv_full, (unit_i - 1) & 1, tmo, p.err);
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // the whole warp runs the loop (convergent control flow); one elected
    // lane issues each MMA and commit
    {
      constexpr uint32_t id_kk = idesc_kind_f16_ab(128, 128, BF16, false, false);   // S^T, dP^T
      constexpr uint32_t id_ts = idesc_kind_f16(128, D, BF16, true);                // dV, dK (A in TMEM)
      constexpr uint32_t id_mm = idesc_kind_f16_ab(128, D, BF16, true, true);       // dQ
      // descriptor low halves of each operand's first byte, K-major (S^T, dP^T)
      // and MN-major (dV, dK, dQ): every MMA's descriptor is one of these plus
      // a constant, so the issue path carries no descriptor arithmetic
      const uint32_t k_km = sdesc_lo_kmajor_sw128(smem_u32(smem + T::OFF_K));
      const uint32_t v_km = sdesc_lo_kmajor_sw128(smem_u32(smem + T::OFF_V));
      const uint32_t q_km = sdesc_lo_kmajor_sw128(smem_u32(smem + T::OFF_Q));
      const uint32_t do_km = sdesc_lo_kmajor_sw128(smem_u32(smem + T::OFF_DO));
      const uint32_t k_mn = sdesc_lo_mnmajor_sw128(smem_u32(smem + T::OFF_K), T::CHUNK);
      const uint32_t q_mn = sdesc_lo_mnmajor_sw128(smem_u32(smem + T::OFF_Q), T::CHUNK);
      const uint32_t do_mn = sdesc_lo_mnmajor_sw128(smem_u32(smem + T::OFF_DO), T::CHUNK);
      const uint32_t ds_mn = sdesc_lo_mnmajor_sw128(smem_u32(smem + T::OFF_DS), T::CHUNK);
      // TMEM column of K step k (16 queries) of P^T / dS^T: queries 0-63 in the
      // first 32 columns of the warpgroup-0 half, 64-127 in those of the other
      auto pcol = [](int k) -> uint32_t { return k < 4 ? 8 * k : 64 + 8 * (k - 4); };
      int unit_i = 0, blk_it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < nunits && ok; t += gridDim.x, ++unit_i) {
        const BwdUnit u = bwd_unit(p, t, CAUSAL);
        ok = mbar_wait_warp(&bars->kv_full, unit_i & 1, tmo, abort_flag, p.err);
        for (int it = 0; it < u.nblk && ok; ++it, ++blk_it) {
          const int qs = blk_it & 1;
          const uint32_t qt = qs * (T::TILE >> 4);        // Q_i's buffer, in descriptor units
          // dP^T = V_j dO_i^T (keys on the TMEM lanes): its columns held the
          // previous block's dS^T, which the previous dK has read (issued
          // before this, executed in order)
          ok = mbar_wait_warp(&bars->do_full, blk_it & 1, tmo, abort_flag, p.err);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < KS; ++k) {
            const uint32_t off = ((k >> 2) * T::CHUNK + (k & 3) * 32) >> 4;
            umma_f16_ss_lo_w(tmem + T::T_DP, v_km + off, do_km + off, id_kk, k > 0);
          }
          // S^T = K_j Q_i^T once Q_i has landed and the previous block's dQ has
          // been read out of S's columns
          ok = mbar_wait_warp(&bars->q_full[qs], (blk_it >> 1) & 1, tmo, abort_flag, p.err);
          if (ok && blk_it > 0) ok = mbar_wait_warp(&bars->dq_empty, (blk_it - 1) & 1, tmo, abort_flag, p.err);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < KS; ++k) {
            const uint32_t off = ((k >> 2) * T::CHUNK + (k & 3) * 32) >> 4;
            umma_f16_ss_lo_w(tmem + T::T_S, k_km + off, q_km + qt + off, id_kk, k > 0);
          }
          umma_commit_w(&bars->s_full);
          // P^T and dS^T in TMEM (over S^T and dP^T)
          ok = mbar_wait_warp(&bars->p_full, blk_it & 1, tmo, abort_flag, p.err);
          // the previous unit's dK/dV must have been read before they restart at zero
          if (ok && it == 0 && unit_i > 0) ok = mbar_wait_warp(&bars->dkv_empty, (unit_i - 1) & 1, tmo, abort_flag, p.err);
          if (!ok) break;
          tc_fence_after();
          // dV += P^T dO_i, dK += dS^T Q_i: A from TMEM (K = 128 queries), B
          // (dO_i, Q_i) MN-major: 16 query rows per step = 2048 bytes
#pragma unroll
          for (int k = 0; k < 8; ++k)
            umma_f16_ts_lo_w(tmem + T::T_DV, tmem + T::T_S + pcol(k), do_mn + k * (2048 >> 4), id_ts,
                           (it > 0 || k > 0) ? 1u : 0u);
          umma_commit_w(&bars->do_empty);                   // dO_i is read by nothing after dV
#pragma unroll
          for (int k = 0; k < 8; ++k)
            umma_f16_ts_lo_w(tmem + T::T_DK, tmem + T::T_DP + pcol(k), q_mn + qt + k * (2048 >> 4), id_ts,
                           (it > 0 || k > 0) ? 1u : 0u);
          umma_commit_w(&bars->q_empty[qs]);                 // Q_i is read by nothing after dK
          // dQ_i = dS K_j: A = dS in shared memory (rows = keys, queries
          // contiguous: MN-major, K = 128 keys), B = K_j MN-major (N = d)
          ok = mbar_wait_warp(&bars->ds_full, blk_it & 1, tmo, abort_flag, p.err);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 8; ++k)
            umma_f16_ss_lo_w(tmem + T::T_S, ds_mn + k * (2048 >> 4), k_mn + k * (2048 >> 4), id_mm, k > 0 ? 1u : 0u);
          umma_commit_w(&bars->dq_full);
        }
        if (!ok) break;
        umma_commit_w(&bars->dkv_full);
        umma_commit_w(&bars->kv_empty);
      }
      umma_commit_w(&bars->done);
      mbar_wait_drain(&bars->done, 0, tmo, p.err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ compute warps
    const int r = threadIdx.x & 127;                         // TMEM lane
    const int half = threadIdx.x >> 7;                       // column half this warpgroup owns
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float sl2 = p.scale_log2;
    const float scale = p.scale;
    uint8_t* tp = smem + T::OFF_P;
    uint8_t* tds = smem + T::OFF_DS;
    // row r of the dS tile (key r, queries contiguous) and of the dQ staging:
    // chunk (64 columns) at +16 KB, 16-byte unit u at u ^ (r % 8)
    const uint32_t prow = smem_u32(tp) + r * 128;
    const uint32_t dsrow = smem_u32(tds) + r * 128;
    float* lsd_base = reinterpret_cast<float*>(smem + T::OFF_LSD);
    static_assert(T::SMEM <= 227 * 1024, "backward shared memory");
    int unit_i = 0, blk_it = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < nunits && ok; t += gridDim.x, ++unit_i) {
      const BwdUnit u = bwd_unit(p, t, CAUSAL);
      const int key = u.j * 128 + r;                           // this thread's key row (S^T, dP^T)
      for (int it = 0; it < u.nblk && ok; ++it, ++blk_it) {
        const int h = u.hkv * p.group + it / u.nI;
        const int i = bwd_qblock(u, it);
        // lse * log2(e) (warpgroup 0) and D (warpgroup 1) of the block's 128
        // queries into shared memory. Rewriting them is safe: this thread has
        // passed the previous block's dQ-ready barrier, which needed every
        // thread's dS-ready arrival, made after its last read of them
        float* lsd = lsd_base;
        {
          const int qrow = i * 128 + r;
          float v = 0.f;
          if (qrow < p.N) {
            const size_t lrow = ((size_t)u.b * p.H + h) * p.N + qrow;
            v = half == 0 ? __ldg(p.lse + lrow) * 1.4426950408889634f : __ldg(p.dvec + lrow);
          }
          lsd[half * 128 + r] = v;
        }
        named_bar_sync(1, BWD_COMPUTE);
        ok = mbar_wait(&bars->s_full, blk_it & 1, tmo, abort_flag, p.err);
        if (!ok) break;
        tc_fence_after();
        // queries of this block visible to this key: [qlo, qhi)
        int qlo = 0, qhi = min(128, p.N - i * 128);
        if (CAUSAL) qlo = max(0, key - i * 128);             // query >= key
        if (key >= p.N) qhi = 0;
        {
          const int c = half;                                  // queries c*64 .. c*64+63
          uint32_t pw[32], dw[32];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            // 32 query columns at a time keep fewer registers live
            const int cb = c * 64 + hh * 32;                   // first query column of this piece
            uint32_t su[32], du[32];
            tmem_ld32x2(tmem + lane_off + T::T_S + cb, su, tmem + lane_off + T::T_DP + cb, du);
            const float4* l4 = reinterpret_cast<const float4*>(lsd + cb);
            const float4* d4 = reinterpret_cast<const float4*>(lsd + 128 + cb);
            if (qlo <= cb && qhi >= cb + 32) {
              const uint64_t sl2x2 = f2_pack(sl2, sl2), sc2 = f2_pack(scale, scale);
#pragma unroll
              for (int e4 = 0; e4 < 8; ++e4) {
                const float4 lv = l4[e4], dv4 = d4[e4];
                const float lq[4] = {lv.x, lv.y, lv.z, lv.w}, dq[4] = {dv4.x, dv4.y, dv4.z, dv4.w};
#pragma unroll
                for (int e2 = 0; e2 < 4; e2 += 2) {
                  const int e = 4 * e4 + e2;
                  float p0, p1;
                  f2_unpack(f2_fma(f2_pack(to_f(su[e]), to_f(su[e + 1])), sl2x2, f2_pack(-lq[e2], -lq[e2 + 1])), p0, p1);
                  p0 = ex2_approx(p0);
                  p1 = ex2_approx(p1);
                  const uint64_t pp = f2_pack(p0, p1);
                  float d0, d1;
                  f2_unpack(f2_mul(f2_mul(pp, sc2), f2_sub(f2_pack(to_f(du[e]), to_f(du[e + 1])), f2_pack(dq[e2], dq[e2 + 1]))),
                            d0, d1);
                  pw[hh * 16 + e / 2] = pack16<BF16>(p0, p1);
                  dw[hh * 16 + e / 2] = pack16<BF16>(d0, d1);
                }
              }
            } else {
#pragma unroll
              for (int e = 0; e < 32; e += 2) {
                const int q = cb + e;
                const bool v0 = q >= qlo && q < qhi, v1 = q + 1 >= qlo && q + 1 < qhi;
                const float p0 = v0 ? ex2_approx(to_f(su[e]) * sl2 - lsd[q]) : 0.f;
                const float p1 = v1 ? ex2_approx(to_f(su[e + 1]) * sl2 - lsd[q + 1]) : 0.f;
                const float d0 = scale * p0 * (to_f(du[e]) - lsd[128 + q]);
                const float d1 = scale * p1 * (to_f(du[e + 1]) - lsd[128 + q + 1]);
                pw[hh * 16 + e / 2] = pack16<BF16>(p0, p1);
                dw[hh * 16 + e / 2] = pack16<BF16>(d0, d1);
              }
            }
          }
          // P^T over the first 32 of this half's S^T columns, dS^T over the
          // first 32 of its dP^T columns (the A operands of dV and dK)
          tmem_st32(tmem + lane_off + T::T_S + c * 64, pw);
          tmem_st32(tmem + lane_off + T::T_DP + c * 64, dw);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&bars->p_full);
          // this warpgroup's previous dQ reduction reads chunk c of the P and
          // dS tiles as its staging: wait for it only now
          if (blk_it > 0) {
            if (r == 0) tma_store_wait_read();
            named_bar_sync(2 + half, 128);
          }
          // dS for dQ: row = key r, queries c*64 .. c*64+63 in chunk c, 16-byte unit q at q ^ (r % 8)
#pragma unroll
          for (int q = 0; q < 8; ++q)
            st_shared_v4(dsrow + c * T::CHUNK + ((q ^ (r & 7)) << 4), dw[4 * q], dw[4 * q + 1], dw[4 * q + 2], dw[4 * q + 3]);
        }
        fence_proxy_async_smem();                             // dS visible to the MMAs
        mbar_arrive(&bars->ds_full);
        // dQ_i rows: add into the fp32 accumulator
        ok = mbar_wait(&bars->dq_full, blk_it & 1, tmo, abort_flag, p.err);
        if (!ok) break;
        tc_fence_after();
        // dQ rows (query r, this warpgroup's D/2 columns) -> staging in the
        // chunks of the P and dS tiles this warpgroup writes (chunk `half` of
        // each): 32 fp32 columns per 16 KB chunk, row r, 16-byte unit v at
        // v ^ (r % 8), the bulk reduction's 128-byte swizzle
        {
          constexpr int HC = D / 2;                            // columns per warpgroup
          uint32_t qu[HC];
          if constexpr (HC == 64) tmem_ld64(tmem + lane_off + T::T_S + half * HC, qu);
          else tmem_ld32(tmem + lane_off + T::T_S + half * HC, qu);
          // dQ is in registers (the loads wait for completion): S's columns are
          // free for the next block's S while the staging and reduction go on
          tc_fence_before();
          mbar_arrive(&bars->dq_empty);
#pragma unroll
          for (int v4 = 0; v4 < HC / 4; ++v4) {
            const uint32_t base = (v4 >> 3) == 0 ? prow : dsrow;   // 32-column piece 0 / 1
            const uint32_t off = half * T::CHUNK + ((((v4 & 7) ^ (r & 7))) << 4);
            st_shared_v4(base + off, qu[4 * v4], qu[4 * v4 + 1], qu[4 * v4 + 2], qu[4 * v4 + 3]);
          }
        }
        fence_proxy_async_smem();
        named_bar_sync(2 + half, 128);
        if (r == 0) {
          // this warpgroup's columns half * D/2 ..; rows past the sequence end
          // fall outside the map and are dropped
          for (int cc = 0; cc < D / 64; ++cc)
            tma_reduce_add_4d(&tmDQ, (cc == 0 ? tp : tds) + half * T::CHUNK, half * (D / 2) + cc * 32, h, i * 128, u.b);
          tma_store_commit();
        }
      }
      if (!ok) break;
      // unit epilogue: dK_j, dV_j rows (thread r = key j*128 + r)
      ok = mbar_wait(&bars->dkv_full, unit_i & 1, tmo, abort_flag, p.err);
      if (!ok) break;
      tc_fence_after();
      const bool key_ok = key < p.N;
      const size_t krow = (((size_t)u.b * p.N + (key_ok ? key : 0)) * p.Hkv + u.hkv) * D;
      uint4* dkp = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.dk) + krow);
      uint4* dvp = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.dv) + krow);
#pragma unroll 1
      for (int c = half * (D / 64); c < (half + 1) * (D / 64); ++c) {
        uint32_t ku[32], vu[32];
        tmem_ld32(tmem + lane_off + T::T_DK + c * 32, ku);
        tmem_ld32(tmem + lane_off + T::T_DV + c * 32, vu);
        if (key_ok) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            dkp[c * 4 + e] = make_uint4(pack16<BF16>(to_f(ku[8 * e]), to_f(ku[8 * e + 1])),
                                        pack16<BF16>(to_f(ku[8 * e + 2]), to_f(ku[8 * e + 3])),
                                        pack16<BF16>(to_f(ku[8 * e + 4]), to_f(ku[8 * e + 5])),
                                        pack16<BF16>(to_f(ku[8 * e + 6]), to_f(ku[8 * e + 7])));
            dvp[c * 4 + e] = make_uint4(pack16<BF16>(to_f(vu[8 * e]), to_f(vu[8 * e + 1])),
                                        pack16<BF16>(to_f(vu[8 * e + 2]), to_f(vu[8 * e + 3])),
                                        pack16<BF16>(to_f(vu[8 * e + 4]), to_f(vu[8 * e + 5])),
                                        pack16<BF16>(to_f(vu[8 * e + 6]), to_f(vu[8 * e + 7])));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->dkv_empty);
    }
    if (r == 0) tma_store_wait_all();                        // no reduction outlives the CTA
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tmem, 512);
}

// D_i = sum_c dO_ic O_ic, one warp per (b, row, head); written [B][H][N].
template <int D>
__global__ void __launch_bounds__(256) bwd_dvec_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ dout,
                                                       float* __restrict__ dvec, int B, int N, int H, int bf16) {
  const long long wid = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wid >= (long long)B * N * H) return;
  const int h = (int)(wid % H);
  const int n = (int)((wid / H) % N);
  const int b = (int)(wid / ((long long)H * N));
  const size_t base = (size_t)wid * D;     // BSHD row (b, n, h)
  float acc = 0.f;
  for (int c = lane * 2; c < D; c += 64) {
    const uint32_t ov = *reinterpret_cast<const uint32_t*>(o + base + c);
    const uint32_t gv = *reinterpret_cast<const uint32_t*>(dout + base + c);
    float o0, o1, g0, g1;
    if (bf16) {
      o0 = __uint_as_float(ov << 16); o1 = __uint_as_float(ov & 0xffff0000u);
      g0 = __uint_as_float(gv << 16); g1 = __uint_as_float(gv & 0xffff0000u);
    } else {
      o0 = __half2float(__ushort_as_half((unsigned short)(ov & 0xffff)));
      o1 = __half2float(__ushort_as_half((unsigned short)(ov >> 16)));
      g0 = __half2float(__ushort_as_half((unsigned short)(gv & 0xffff)));
      g1 = __half2float(__ushort_as_half((unsigned short)(gv >> 16)));
    }
    acc = fmaf(o0, g0, fmaf(o1, g1, acc));
  }
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
  if (lane == 0) dvec[((size_t)b * H + h) * N + n] = acc;
}

// dQ = fp32 accumulator rounded to bf16/fp16.
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const float* __restrict__ acc, uint16_t* __restrict__ dq,
                                                             long long n, int bf16) {
  const long long i = ((long long)blockIdx.x * 256 + threadIdx.x) * 4;
  if (i >= n) return;
  const float4 a = *reinterpret_cast<const float4*>(acc + i);
  uint32_t lo, hi;
  if (bf16) {
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(lo) : "f"(a.y), "f"(a.x));
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(hi) : "f"(a.w), "f"(a.z));
  } else {
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(lo) : "f"(a.y), "f"(a.x));
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(hi) : "f"(a.w), "f"(a.z));
  }
  *reinterpret_cast<uint2*>(dq + i) = make_uint2(lo, hi);
}

template <int D, bool CAUSAL, bool BF16>
cudaError_t launch_bwd_t(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& dout,
                         const CUtensorMap& dq, const BwdParams& p, int sm_count, cudaStream_t s) {
  auto kern = attn_bwd_kernel<D, CAUSAL, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdTraits<D>::SMEM);
  if (e != cudaSuccess) return e;
  const int grid = p.nunits < sm_count ? p.nunits : sm_count;
  kern<<<grid, BWD_THREADS, BwdTraits<D>::SMEM, s>>>(q, k, v, dout, dq, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd(int d, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                       const CUtensorMap& dout, const CUtensorMap& dq, const BwdParams& p, bool causal, bool bf16,
                       int sm_count, cudaStream_t s) {
#define ATTN45_B(D, C, F) return launch_bwd_t<D, C, F>(q, k, v, dout, dq, p, sm_count, s)
  if (d == 64) {
    if (causal) { if (bf16) ATTN45_B(64, true, true); else ATTN45_B(64, true, false); }
    else        { if (bf16) ATTN45_B(64, false, true); else ATTN45_B(64, false, false); }
  }
  if (causal) { if (bf16) ATTN45_B(128, true, true); else ATTN45_B(128, true, false); }
  if (bf16) ATTN45_B(128, false, true);
  ATTN45_B(128, false, false);
#undef ATTN45_B
}

cudaError_t launch_bwd_dvec(int d, const void* o, const void* dout, float* dvec, int B, int N, int H, bool bf16,
                            cudaStream_t s) {
  const long long rows = (long long)B * N * H;
  const unsigned grid = (unsigned)((rows + 7) / 8);
  if (d == 64)
    bwd_dvec_kernel<64><<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dout), dvec,
                                             B, N, H, bf16);
  else
    bwd_dvec_kernel<128><<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dout),
                                              dvec, B, N, H, bf16);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq_convert(const float* acc, void* dq, long long n, bool bf16, cudaStream_t s) {
  const unsigned grid = (unsigned)((n / 4 + 255) / 256);
  bwd_dq_convert_kernel<<<grid, 256, 0, s>>>(acc, static_cast<uint16_t*>(dq), n, bf16);
  return cudaGetLastError();
}

}  // namespace attn45
