// attn_decode_kt.cu -- split-KV decode units with the keys on the TMEM lanes.
//
// In decode a KV head meets only its G = H/Hkv query rows, so a tile of the
// forward kernel (128 query rows on the TMEM lanes) would be mostly padding.
// Here both products are transposed so the 128 keys of a tile fill the MMA's
// M dimension and the few query heads sit in N = 16:
//   S^T [128 keys x 16]  = K [128 x d] . Q^T            (A = K tile, K-major)
//   O^T [d x 16]        += V^T [d x 128 keys] . P^T      (A = V tile, MN-major)
// with K and V exactly as TMA stages them (64-channel boxes, 128-byte
// swizzle). One CTA = one (sequence, KV head, split):
//   warp 4      TMA producer: K and V tiles of 128 keys into a 3-stage ring;
//   warp 5      MMA issuer (one thread): S^T(j) into one of two TMEM buffers,
//               then O^T += V^T(j-1) P^T(j-1), so the softmax of tile j runs
//               while the tensor core finishes the previous tile;
//   warps 0-3   softmax, thread = key (TMEM lane): per head, the tile maximum
//               over the 128 keys (warp shuffles, then across the 4 warps in
//               shared memory), P = 2^(s - m) written as the K-major B
//               operand of the second product, running sums per thread; the
//               running maximum moves only when a tile's maximum exceeds it by
//               more than 2^8 (then O^T is rescaled in TMEM), so P <= 256.
//   epilogue    thread = channel (TMEM lane of O^T): partial O normalised by
//               its own sum, and its lse, in the format attn_combine merges.
// The online softmax is the "Related papers: FlashAttention-4" page's
// online-softmax teaser; the split of the key range with a final merge is
// FlashDecoding (cited by "FlashAttention-3: Fast and Accurate Attention with
// Asynchrony and Low-precision" among its references).
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include "fwd_launch.cuh"

namespace attn45 {
namespace {

constexpr int KT_KEYS = 128;                       // keys per tile = TMEM lanes of S^T
constexpr int KT_NQ = 16;                          // MMA N: the group's query heads, padded
constexpr int KT_STAGES = 3;
constexpr int KT_CHUNK = KT_KEYS * 128;            // 128 keys x 64 channels of 16 bits
constexpr int KT_STAGE = 4 * KT_CHUNK;             // K (two channel halves), then V
constexpr int KT_OFF_Q = KT_STAGES * KT_STAGE;     // Q: 2 chunks x 16 rows x 128 B
constexpr int KT_OFF_P = KT_OFF_Q + 2 * 2048;      // P: 2 buffers x 2 key chunks x 16 rows x 128 B
constexpr int KT_OFF_RED = KT_OFF_P + 2 * 4096;    // tile maxima [2][4][16], sums [4][16], flags
constexpr int KT_OFF_BARS = KT_OFF_RED + 1024;
constexpr int KT_BYTES = KT_OFF_BARS + 256 + 1024; // + alignment slack
constexpr int KT_THREADS = 192;
constexpr uint32_t KT_TMEM_COLS = 64;              // S^T buffers at columns 0 and 16, O^T at 32
constexpr uint32_t KT_COL_O = 32;

struct KtBars {
  uint64_t full[KT_STAGES], empty[KT_STAGES];
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2], fin;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(KtBars) <= 256, "barrier block");

template <bool BF16>
__device__ __forceinline__ uint16_t to_bits(float x) {
  if constexpr (BF16) return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  else return __half_as_ushort(__float2half_rn(x));
}

template <int G, bool BF16>
__global__ void __launch_bounds__(KT_THREADS, 1) decode_kt_kernel(const __grid_constant__ CUtensorMap tmK,
                                                                  const __grid_constant__ CUtensorMap tmV,
                                                                  const uint16_t* q, const FwdParams p) {
  static_assert(G >= 1 && G <= KT_NQ, "query heads per KV head");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  KtBars* bars = reinterpret_cast<KtBars*>(smem + KT_OFF_BARS);
  float* red = reinterpret_cast<float*>(smem + KT_OFF_RED);      // [2][4][16]
  float* red_l = red + 2 * 4 * 16;                                 // [4][16]
  int* flags = reinterpret_cast<int*>(red_l + 4 * 16);             // [2][4] per tile, [4] at the end
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x % p.num_splits;
  const int bk = blockIdx.x / p.num_splits;
  const int b = bk / p.Hkv, hkv = bk % p.Hkv;
  const int n = min(max(__ldg(p.seqlens + b), 0), p.N);
  const int s0 = min(split * p.split_chunk, n);
  const int nk = min(s0 + p.split_chunk, n) - s0;
  const size_t prow0 = ((size_t)split * p.nseq + b) * p.H + (size_t)hkv * G;  // first partial row
  if (nk <= 0) {                                    // empty split: weight 0 in the merge
    if (threadIdx.x < G) p.lse[prow0 + threadIdx.x] = -INFINITY;
    return;
  }
  const int ntiles = (nk + KT_KEYS - 1) / KT_KEYS;
  if (threadIdx.x == 0) {
    for (int s = 0; s < KT_STAGES; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->s_free[i], 4);
      mbar_init(&bars->p_full[i], 4);
      mbar_init(&bars->pv_done[i], 1);
    }
    mbar_init(&bars->fin, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&bars->tmem_base, KT_TMEM_COLS);
    tmem_relinquish();
  }
  // Q rows of the group as the K-major B operand (rows >= G zero), P buffers zeroed
  for (int u = threadIdx.x; u < KT_NQ * 16; u += KT_THREADS) {
    const int r = u >> 4, c16 = u & 15;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (r < G) val = *reinterpret_cast<const uint4*>(q + ((size_t)b * p.H + (size_t)hkv * G + r) * 128 + c16 * 8);
    *reinterpret_cast<uint4*>(smem + KT_OFF_Q + (c16 >> 3) * 2048 + r * 128 + (((c16 & 7) ^ (r & 7)) << 4)) = val;
  }
  for (int i = threadIdx.x; i < 2 * 4096 / 16; i += KT_THREADS)
    reinterpret_cast<uint4*>(smem + KT_OFF_P)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const uint64_t tmo = p.timeout_ns;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int j = 0;
      for (; j < ntiles; ++j) {
        const int st = j % KT_STAGES;
        if (j >= KT_STAGES && !mbar_wait(&bars->empty[st], ((j / KT_STAGES) + 1) & 1, tmo, &bars->abort_flag, p.err))
          break;
        uint8_t* base = smem + st * KT_STAGE;
        const int row = s0 + j * KT_KEYS;
        mbar_expect_tx(&bars->full[st], KT_STAGE);
        tma_load_4d(&tmK, &bars->full[st], base, 0, hkv, row, b);
        tma_load_4d(&tmK, &bars->full[st], base + KT_CHUNK, 64, hkv, row, b);
        tma_load_4d(&tmV, &bars->full[st], base + 2 * KT_CHUNK, 0, hkv, row, b);
        tma_load_4d(&tmV, &bars->full[st], base + 3 * KT_CHUNK, 64, hkv, row, b);
      }
      // every copy issued has landed before the CTA can exit (bounded)
      for (int i = max(0, j - KT_STAGES); i < j; ++i)
        mbar_wait_drain(&bars->full[i % KT_STAGES], (i / KT_STAGES) & 1, tmo, p.err);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_kind_f16_ab(128, KT_NQ, BF16, false, false);
      constexpr uint32_t id_o = idesc_kind_f16_ab(128, KT_NQ, BF16, true, false);
      const uint32_t sq = smem_u32(smem + KT_OFF_Q), sp = smem_u32(smem + KT_OFF_P);
      auto pv = [&](int j) -> bool {                // O^T += V^T(j) P^T(j)
        const int pb = j & 1, st = j % KT_STAGES;
        if (!mbar_wait(&bars->p_full[pb], (j >> 1) & 1, tmo, &bars->abort_flag, p.err)) return false;
        tc_fence_after();
        const uint32_t sv = smem_u32(smem + st * KT_STAGE + 2 * KT_CHUNK);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_f16_ss(tmem + KT_COL_O, sdesc_mnmajor_sw128(sv + kk * 2048, KT_CHUNK),
                      sdesc_kmajor_sw128(sp + pb * 4096 + (kk >> 2) * 2048 + (kk & 3) * 32), id_o,
                      (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&bars->empty[st]);
        umma_commit(&bars->pv_done[pb]);
        return true;
      };
      bool ok = true;
      for (int j = 0; j < ntiles && ok; ++j) {
        const int st = j % KT_STAGES, sb = j & 1;
        ok = mbar_wait(&bars->full[st], (j / KT_STAGES) & 1, tmo, &bars->abort_flag, p.err);
        if (ok && j >= 2) ok = mbar_wait(&bars->s_free[sb], ((j - 2) >> 1) & 1, tmo, &bars->abort_flag, p.err);
        if (!ok) break;
        tc_fence_after();
        const uint32_t sk = smem_u32(smem + st * KT_STAGE);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_f16_ss(tmem + sb * KT_NQ, sdesc_kmajor_sw128(sk + (kk >> 2) * KT_CHUNK + (kk & 3) * 32),
                      sdesc_kmajor_sw128(sq + (kk >> 2) * 2048 + (kk & 3) * 32), id_s, kk > 0 ? 1u : 0u);
        umma_commit(&bars->s_full[sb]);
        if (j > 0) ok = pv(j - 1);
      }
      if (ok) pv(ntiles - 1);
      umma_commit(&bars->fin);                      // all MMAs issued above have completed
      mbar_wait_drain(&bars->fin, 0, tmo, p.err);
    }
  } else {
    // ------------------------------------------------------------ softmax
    // Every softmax warp runs all ntiles iterations and meets every named
    // barrier; after a failed wait a warp only skips work, and the decision
    // to skip a tile is read from flags all four warps wrote before the
    // barrier, so it is the same in every warp.
    const int key = threadIdx.x;                    // TMEM lane of S^T; channel of O^T
    const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
    float m[G], lp[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m[h] = -INFINITY;
      lp[h] = 0.f;
    }
    bool bad = false;
    for (int j = 0; j < ntiles; ++j) {
      const int sb = j & 1;
      if (!bad) bad = !mbar_wait(&bars->s_full[sb], (j >> 1) & 1, tmo, &bars->abort_flag, p.err);
      bad = __any_sync(0xffffffffu, bad);
      uint32_t r[16];
      if (!bad) {
        tc_fence_after();
        tmem_ld16(tl + sb * KT_NQ, r);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->s_free[sb]);
      const bool valid = j * KT_KEYS + key < nk;
      float sc[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        sc[h] = (!bad && valid) ? __uint_as_float(r[h]) * p.scale_log2 : -INFINITY;
        float x = sc[h];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
        if (lane == 0) red[(sb * 4 + warp) * 16 + h] = x;
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
        const float* rr = red + sb * 64 + h;
        tmax[h] = fmax3(rr[0], rr[16], fmaxf(rr[32], rr[48]));
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
        if (j > 0) {
          // O^T holds tiles 0 .. j-1 once PV(j-1) is done: rescale its columns
          bad = !mbar_wait(&bars->pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, tmo, &bars->abort_flag, p.err);
          bad = __any_sync(0xffffffffu, bad);
          if (!bad) {
            tc_fence_after();
            uint32_t o[16];
            tmem_ld16(tl + KT_COL_O, o);
#pragma unroll
            for (int h = 0; h < G; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha[h]);
            tmem_st16(tl + KT_COL_O, o);
            tmem_st_wait();
            tc_fence_before();
          }
        }
      }
      // P buffer sb is free once PV(j-2) is done
      if (!bad && j >= 2) bad = !mbar_wait(&bars->pv_done[sb], ((j - 2) >> 1) & 1, tmo, &bars->abort_flag, p.err);
      if (bad) continue;                            // no P arrival: the MMA issuer's wait gives up
      if (!valid) {
        // a key past the end meets P = 0, but 0 * (Inf or NaN) is not 0 in
        // the product: clear its V row (the tile has landed: S^T(j) read it)
        uint4* vr = reinterpret_cast<uint4*>(smem + (j % KT_STAGES) * KT_STAGE + 2 * KT_CHUNK + key * 128);
#pragma unroll
        for (int i = 0; i < 8; ++i) vr[i] = vr[i + KT_CHUNK / 16] = make_uint4(0u, 0u, 0u, 0u);
      }
      uint8_t* prow = smem + KT_OFF_P + sb * 4096 + (key >> 6) * 2048;
      const int kb = (key & 63) * 2;                // byte of this key within a 128-byte row
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float pk = ex2_approx(sc[h] - m[h]);  // 0 for keys past the end
        lp[h] += pk;
        *reinterpret_cast<uint16_t*>(prow + h * 128 + ((((kb >> 4) ^ (h & 7)) << 4) | (kb & 15))) = to_bits<BF16>(pk);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[sb]);
    }
    // ------------------------------------------------------------ epilogue
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float x = lp[h];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
      if (lane == 0) red_l[warp * 16 + h] = x;
    }
    if (lane == 0) flags[8 + warp] = bad ? 1 : 0;
    named_bar_sync(1, 128);
    bad = flags[8] | flags[9] | flags[10] | flags[11];
    if (!bad) bad = !mbar_wait(&bars->pv_done[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1, tmo, &bars->abort_flag, p.err);
    bad = __any_sync(0xffffffffu, bad);
    if (!bad) {
      tc_fence_after();
      uint32_t o[16];
      tmem_ld16(tl + KT_COL_O, o);
      float* o_part = reinterpret_cast<float*>(p.o);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float l = red_l[h] + red_l[16 + h] + red_l[32 + h] + red_l[48 + h];
        o_part[(prow0 + h) * 128 + key] = __uint_as_float(o[h]) / l;
        if (key == h) p.lse[prow0 + h] = (m[h] + lg2_approx(l)) * 0.69314718055994530942f;
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, KT_TMEM_COLS);
  }
}

template <int G, bool BF16>
cudaError_t launch_t(const CUtensorMap& k, const CUtensorMap& v, const void* q, const FwdParams& p, cudaStream_t s) {
  auto kern = decode_kt_kernel<G, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, KT_BYTES);
  if (e != cudaSuccess) return e;
  kern<<<p.ntiles, KT_THREADS, KT_BYTES, s>>>(k, v, static_cast<const uint16_t*>(q), p);
  return cudaGetLastError();
}

}  // namespace

bool decode_kt_supported(int d, int group) { return d == 128 && group >= 1 && group <= KT_NQ; }

cudaError_t launch_decode_kt(int group, const CUtensorMap& k, const CUtensorMap& v, const void* q,
                             const FwdParams& p, bool bf16, cudaStream_t s) {
#define ATTN45_G(G) \
  case G: return bf16 ? launch_t<G, true>(k, v, q, p, s) : launch_t<G, false>(k, v, q, p, s)
  switch (group) {
    ATTN45_G(1); ATTN45_G(2); ATTN45_G(3); ATTN45_G(4); ATTN45_G(5); ATTN45_G(6); ATTN45_G(7); ATTN45_G(8);
    ATTN45_G(9); ATTN45_G(10); ATTN45_G(11); ATTN45_G(12); ATTN45_G(13); ATTN45_G(14); ATTN45_G(15);
    ATTN45_G(16);
    default: return cudaErrorInvalidValue;
  }
#undef ATTN45_G
}

}  // namespace attn45
