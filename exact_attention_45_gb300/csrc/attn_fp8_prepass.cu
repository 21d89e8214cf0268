// attn_fp8_prepass.cu -- FP8 (e4m3) pre-pass: incoherent processing of Q and
// K fused with block quantisation, and per-channel quantisation of V written
// transposed (keys contiguous) for the P V product.
//
// "FlashAttention-3: Fast and Accurate Attention with Asynchrony and
// Low-precision", abstract technique (3): block quantization, and incoherent
// processing that multiplies Q and K by a random orthogonal matrix so that
// outlier features spread over all channels while Q K^T stays unchanged.
// The orthogonal matrix is M = diag(sigma) H_d / sqrt(d): H_d the Sylvester
// Hadamard matrix applied by the fast Walsh-Hadamard butterflies (spans 1, 2,
// ..., d/2, each stage one fp32 add or subtract per element), sigma_c =
// 1 - 2*(splitmix64(seed + c) & 1) computed on the host.
//
// Scales are amax / 448 (448 = largest finite e4m3), 1 for an all-zero group;
// codes are e4m3(RNE, saturating) of x / scale with the division one IEEE
// fp32 rounding, so results are reproducible bit for bit.
//
// HBM-bound. For head dim 128 (the FP8 forward's), Q and K blocks use
// qk128_kernel: the 128-row block is staged by TMA, each thread rotates one
// whole row in registers (all butterfly stages without shuffles, packed f32x2
// adds) and the codes leave by a TMA store. Other head dims and V use the
// warp-per-rows kernel below.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fp8_prepass.h"
#include "ptx.cuh"

namespace attn45 {

namespace {

constexpr int ROWS = 128;        // rows per quantisation block
constexpr int THREADS = 256;     // 8 warps x 16 rows
constexpr int ROWS_PER_WARP = ROWS / (THREADS / 32);
constexpr float E4M3_MAX = 448.0f;

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

__device__ __forceinline__ float scale_from_amax(float amax) {
  return amax == 0.f ? 1.f : __fdiv_rn(amax, E4M3_MAX);
}

// Correctly rounded x / s from the correctly rounded reciprocal r = RN(1/s):
// q0 = RN(x r), e = x - q0 s (exact with one FMA), q = RN(q0 + e r)
// (Markstein's division correction, as used for IEEE division on IA-64).
// Valid for normal s and r; callers check that once per scale.
struct Divider {
  float s, r;
  bool fast;
  __device__ __forceinline__ Divider() : s(1.f), r(1.f), fast(true) {}
  __device__ __forceinline__ explicit Divider(float s_) : s(s_) {
    r = __frcp_rn(s_);
    fast = isfinite(r) && fabsf(s_) >= 1.17549435e-38f && fabsf(r) >= 1.17549435e-38f;
  }
  __device__ __forceinline__ float div(float x) const {
    if (!fast) return __fdiv_rn(x, s);
    const float q0 = __fmul_rn(x, r);
    const float e = __fmaf_rn(-q0, s, x);
    return __fmaf_rn(e, r, q0);
  }
};

// Loads E = d/32 consecutive bf16 of one row for this lane.
template <int E>
__device__ __forceinline__ void load_row(const __nv_bfloat16* src, float (&x)[E]) {
  if constexpr (E == 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(src);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
  } else if constexpr (E == 4) {
    const uint2 v = *reinterpret_cast<const uint2*>(src);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
  } else {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(src));
    x[0] = f.x;
    x[1] = f.y;
  }
}

// In-place x -> (x * sigma) H_d * fl32(1/sqrt(d)) for the row spread over a
// warp (lane holds elements E*lane .. E*lane+E-1). Butterfly pair (i, i+h)
// with bit h of i clear becomes (x_i + x_{i+h}, x_i - x_{i+h}).
template <int E>
__device__ __forceinline__ void rotate_row(float (&x)[E], uint32_t sign_bits_lane, float inv_sqrt_d, int lane) {
#pragma unroll
  for (int e = 0; e < E; ++e)
    if ((sign_bits_lane >> e) & 1u) x[e] = -x[e];
  // spans inside the lane
#pragma unroll
  for (int h = 1; h < E; h <<= 1) {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      if ((e & h) == 0) {
        const float a = x[e], b = x[e + h];
        x[e] = __fadd_rn(a, b);
        x[e + h] = __fsub_rn(a, b);
      }
    }
  }
  // spans across lanes: partner lane holds element i ^ h at the same slot
#pragma unroll
  for (int hl = 1; hl < 32; hl <<= 1) {
    const bool upper = (lane & hl) != 0;   // this lane holds the i + h side
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float other = __shfl_xor_sync(0xffffffffu, x[e], hl);
      x[e] = upper ? __fsub_rn(other, x[e]) : __fadd_rn(x[e], other);
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) x[e] = __fmul_rn(x[e], inv_sqrt_d);
}

template <int E>
__device__ __forceinline__ void store_codes(uint8_t* dst, const float (&x)[E], const Divider& dv) {
  float y[E];
#pragma unroll
  for (int e = 0; e < E; ++e) y[e] = dv.div(x[e]);
  if constexpr (E == 8) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(e4m3x4(y[0], y[1], y[2], y[3]), e4m3x4(y[4], y[5], y[6], y[7]));
  } else if constexpr (E == 4) {
    *reinterpret_cast<uint32_t*>(dst) = e4m3x4(y[0], y[1], y[2], y[3]);
  } else {
    uint16_t c;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c) : "f"(y[1]), "f"(y[0]));
    *reinterpret_cast<uint16_t*>(dst) = c;
  }
}

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  const int warp = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[warp] = v;
  __syncthreads();
  float m = red[0];
#pragma unroll
  for (int w = 1; w < THREADS / 32; ++w) m = fmaxf(m, red[w]);
  return m;
}

// Q or K row block: rows [blk*128, blk*128+128) of a sequence whose row 0 is
// token tok0 and which has nrows rows; the block's scale goes to sc[sc_idx].
// phase 0, block mode : rotate, block amax -> scale, codes, scale written.
// phase 0, tensor mode: rotate, block amax -> atomicMax into amax_out[0].
// phase 1, tensor mode: rotate, codes with the tensor amax in amax_out[0].
template <int E>
__device__ void qk_block(const PrepassArgs& a, bool is_q, size_t tok0, int nrows, int head, int blk, size_t sc_idx,
                         int phase) {
  __shared__ float red[THREADS / 32];
  const int Hx = is_q ? a.H : a.Hkv;
  const __nv_bfloat16* src = is_q ? a.q : a.k;
  uint8_t* dst = is_q ? a.q8 : a.k8;
  float* sc = is_q ? a.sq : a.sk;
  const int d = E * 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sign_lane = (a.sign_bits[(E * lane) >> 5] >> ((E * lane) & 31)) & ((1u << E) - 1u);
  float x[ROWS_PER_WARP][E];
  float amax = 0.f;
#pragma unroll
  for (int rr = 0; rr < ROWS_PER_WARP; ++rr) {
    const int n = blk * ROWS + warp * ROWS_PER_WARP + rr;
    if (n < nrows) {
      const size_t row = (tok0 + n) * Hx + head;
      load_row<E>(src + row * d + E * lane, x[rr]);
      if (a.rotate) rotate_row<E>(x[rr], sign_lane, a.inv_sqrt_d, lane);
#pragma unroll
      for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(x[rr][e]));
    }
  }
  float s;
  if (a.block_mode) {
    amax = block_max(amax, red);
    s = scale_from_amax(amax);
    if (threadIdx.x == 0) sc[sc_idx] = s;
  } else if (phase == 0) {
    amax = block_max(amax, red);
    if (threadIdx.x == 0) atomicMax(reinterpret_cast<unsigned int*>(sc), __float_as_uint(amax));
    return;
  } else {
    s = scale_from_amax(__uint_as_float(*reinterpret_cast<volatile unsigned int*>(sc)));
  }
  const Divider dv(s);
#pragma unroll
  for (int rr = 0; rr < ROWS_PER_WARP; ++rr) {
    const int n = blk * ROWS + warp * ROWS_PER_WARP + rr;
    if (n < nrows) {
      const size_t row = (tok0 + n) * Hx + head;
      store_codes<E>(dst + row * d + E * lane, x[rr], dv);
    }
  }
}

// V row block of (sequence, kv head): rows as in qk_block; sv_row = first of
// the D per-channel amax values of (sequence, kv head). phase 0: per-channel
// (block mode) or whole tensor amax -> atomicMax into sv. phase 1: codes with
// those amax values, written transposed through shared memory into rows
// vt_row0 + c (row length a.ldv) from column vt_col.
template <int E>
__device__ void v_block(const PrepassArgs& a, size_t tok0, int nrows, int head, int blk, size_t sv_row, size_t vt_row0,
                        size_t vt_col, int phase) {
  constexpr int D = E * 32;
  constexpr int TP = ROWS + 4;                      // padded row of the transposed tile
  __shared__ __align__(16) uint8_t tile[D * TP];
  __shared__ float red[THREADS / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float x[ROWS_PER_WARP][E];
  float amax_c[E];
#pragma unroll
  for (int e = 0; e < E; ++e) amax_c[e] = 0.f;
#pragma unroll
  for (int rr = 0; rr < ROWS_PER_WARP; ++rr) {
    const int n = blk * ROWS + warp * ROWS_PER_WARP + rr;
    if (n < nrows) {
      const size_t row = (tok0 + n) * a.Hkv + head;
      load_row<E>(a.v + row * D + E * lane, x[rr]);
#pragma unroll
      for (int e = 0; e < E; ++e) amax_c[e] = fmaxf(amax_c[e], fabsf(x[rr][e]));
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) x[rr][e] = 0.f;
    }
  }
  float* sv = a.sv;
  if (phase == 0) {
    if (a.block_mode) {
      // per channel: reduce over the 8 warps through shared memory
      __shared__ float part[THREADS / 32][D];
#pragma unroll
      for (int e = 0; e < E; ++e) part[warp][E * lane + e] = amax_c[e];
      __syncthreads();
      if (threadIdx.x < D) {
        float m = part[0][threadIdx.x];
#pragma unroll
        for (int w = 1; w < THREADS / 32; ++w) m = fmaxf(m, part[w][threadIdx.x]);
        atomicMax(reinterpret_cast<unsigned int*>(sv + sv_row + threadIdx.x), __float_as_uint(m));
      }
    } else {
      float m = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) m = fmaxf(m, amax_c[e]);
      m = block_max(m, red);
      if (threadIdx.x == 0) atomicMax(reinterpret_cast<unsigned int*>(sv), __float_as_uint(m));
    }
    return;
  }
  float s[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const unsigned int bits = a.block_mode
        ? *reinterpret_cast<volatile unsigned int*>(sv + sv_row + E * lane + e)
        : *reinterpret_cast<volatile unsigned int*>(sv);
    s[e] = scale_from_amax(__uint_as_float(bits));
  }
  Divider dv[E];
#pragma unroll
  for (int e = 0; e < E; ++e) dv[e] = Divider(s[e]);
  // codes into the transposed tile: tile[c][n_local]
#pragma unroll
  for (int rr = 0; rr < ROWS_PER_WARP; ++rr) {
    const int nl = warp * ROWS_PER_WARP + rr;
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      uint16_t c2;
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
          : "=h"(c2)
          : "f"(dv[e + 1].div(x[rr][e + 1])), "f"(dv[e].div(x[rr][e])));
      tile[(E * lane + e) * TP + nl] = (uint8_t)(c2 & 0xFF);
      tile[(E * lane + e + 1) * TP + nl] = (uint8_t)(c2 >> 8);
    }
  }
  __syncthreads();
  // rows of vt8: 128 keys = 32 lanes x 4 bytes; pad keys (n >= nrows) hold code 0
  for (int c = warp; c < D; c += THREADS / 32) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(&tile[c * TP + 4 * lane]);
    *reinterpret_cast<uint32_t*>(a.vt8 + (vt_row0 + c) * a.ldv + vt_col + 4 * lane) = w;
  }
}

// Packed sequences: the sequence holding global 128-row block gb (the last s
// with blk_off[s] <= gb).
__device__ __forceinline__ int varlen_seq(const PrepassArgs& a, int gb) {
  int lo = 0, hi = a.nseq - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(a.blk_off + mid) <= gb) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <int E>
__global__ void __launch_bounds__(THREADS) prepass_kernel(const PrepassArgs a, int phase, int block_offset) {
  constexpr int D = E * 32;
  int id = blockIdx.x + block_offset;
  if (a.varlen) {
    // blocks: [Q: H x tmax][K: Hkv x tmax][V: Hkv x tmax] of global block
    // indices gb; sequence s owns gb in [blk_off[s], blk_off[s+1])
    int kind, head, gb;
    if (id < a.H * a.tmax) { kind = 0; head = id / a.tmax; gb = id % a.tmax; }
    else if ((id -= a.H * a.tmax) < a.Hkv * a.tmax) { kind = 1; head = id / a.tmax; gb = id % a.tmax; }
    else { id -= a.Hkv * a.tmax; kind = 2; head = id / a.tmax; gb = id % a.tmax; }
    if (gb >= __ldg(a.blk_off + a.nseq)) return;
    if (kind < 2 && phase == 1 && a.block_mode) return;
    const int s = varlen_seq(a, gb);
    const int blk = gb - __ldg(a.blk_off + s);
    const size_t tok0 = (size_t)__ldg(a.cu + s);
    const int nrows = __ldg(a.cu + s + 1) - __ldg(a.cu + s);
    if (kind < 2) {
      qk_block<E>(a, kind == 0, tok0, nrows, head, blk, (size_t)head * a.tmax + gb, phase);
    } else {
      v_block<E>(a, tok0, nrows, head, blk, ((size_t)s * a.Hkv + head) * D, (size_t)head * D, (size_t)gb * ROWS,
                 phase);
    }
    return;
  }
  // blocks: [Q blocks][K blocks][V blocks], each B * heads * nblk
  const int nq = a.B * a.H * a.nblk, nk = a.B * a.Hkv * a.nblk;
  if (id < nq) {
    if (phase == 1 && a.block_mode) return;   // Q done in phase 0
    const int blk = id % a.nblk, bh = id / a.nblk;
    const int b = bh / a.H, h = bh % a.H;
    qk_block<E>(a, true, (size_t)b * a.N, a.N, h, blk, ((size_t)b * a.H + h) * a.nblk + blk, phase);
    return;
  }
  id -= nq;
  if (id < nk) {
    if (phase == 1 && a.block_mode) return;
    const int blk = id % a.nblk, bh = id / a.nblk;
    const int b = bh / a.Hkv, h = bh % a.Hkv;
    qk_block<E>(a, false, (size_t)b * a.N, a.N, h, blk, ((size_t)b * a.Hkv + h) * a.nblk + blk, phase);
    return;
  }
  id -= nk;
  const int blk = id % a.nblk, bh = id / a.nblk;
  const int b = bh / a.Hkv, h = bh % a.Hkv;
  v_block<E>(a, (size_t)b * a.N, a.N, h, blk, ((size_t)b * a.Hkv + h) * D, ((size_t)b * a.Hkv + h) * D,
             (size_t)blk * ROWS, phase);
}

// blk_off[s] = sum over s' < s of ceil(n_s' / 128), s = 0..nseq (one CTA).
__global__ void __launch_bounds__(1024) varlen_block_offsets_kernel(const int* cu, int nseq, int* blk_off) {
  __shared__ int part[1024];
  const int per = (nseq + 1023) / 1024;
  const int s0 = threadIdx.x * per;
  int sum = 0;
  for (int s = s0; s < s0 + per && s < nseq; ++s) sum += (__ldg(cu + s + 1) - __ldg(cu + s) + ROWS - 1) / ROWS;
  part[threadIdx.x] = sum;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {          // inclusive scan of the per-thread sums
    const int v = threadIdx.x >= off ? part[threadIdx.x - off] : 0;
    __syncthreads();
    part[threadIdx.x] += v;
    __syncthreads();
  }
  int run = threadIdx.x > 0 ? part[threadIdx.x - 1] : 0;
  for (int s = s0; s < s0 + per && s < nseq; ++s) {
    blk_off[s] = run;
    run += (__ldg(cu + s + 1) - __ldg(cu + s) + ROWS - 1) / ROWS;
  }
  if (threadIdx.x == 1023) blk_off[nseq] = part[1023];
}


// ---------------------------------------------------------------- head dim 128
// One CTA = one 128-row block of Q or K; thread r owns row r.
constexpr int QK128_SMEM = 1024 + 2 * 16384 + 16384;   // alignment + bf16 tile + code tile

// Butterfly stage with span h >= 2 over E elements: pairs (i, i+h) and
// (i+1, i+1+h) share one f32x2 op.
template <int E>
__device__ __forceinline__ void butterfly_pairs(float (&x)[E], int h) {
#pragma unroll
  for (int i = 0; i < E; i += 2) {
    if ((i & h) == 0) {
      const uint64_t a = f2_pack(x[i], x[i + 1]);
      const uint64_t b = f2_pack(x[i + h], x[i + h + 1]);
      f2_unpack(f2_add(a, b), x[i], x[i + 1]);
      f2_unpack(f2_sub(a, b), x[i + h], x[i + h + 1]);
    }
  }
}

// One CTA = one 128-row block of Q or K, 256 threads: lanes 2i and 2i+1 of a
// warp hold elements 0-63 and 64-127 of one row (row = warp * 16 + lane / 2).
// Spans 1..32 run inside a thread; span 64 pairs the two halves by a shuffle.
__global__ void __launch_bounds__(256, 3) qk128_kernel(const __grid_constant__ CUtensorMap in_q,
                                                    const __grid_constant__ CUtensorMap in_k,
                                                    const __grid_constant__ CUtensorMap out_q,
                                                    const __grid_constant__ CUtensorMap out_k, const PrepassArgs a,
                                                    int phase) {
  extern __shared__ uint8_t raw[];
  uint8_t* tile = raw + ((1024 - (smem_u32(raw) & 1023)) & 1023);   // 2 x [128 rows][128 B], swizzled
  uint8_t* codes = tile + 2 * 16384;                                  // [128 rows][128 B], swizzled
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  __shared__ float red[8];
  __shared__ uint32_t xmask[64];
  // fixed length: [Q: B x H x nblk][K: B x Hkv x nblk]; packed sequences:
  // [Q: H x tmax][K: Hkv x tmax] global blocks (those past the last exit)
  const int nq = a.varlen ? a.H * a.tmax : a.B * a.H * a.nblk;
  int id = blockIdx.x;
  const bool is_q = id < nq;
  if (!is_q) id -= nq;
  const int Hx = is_q ? a.H : a.Hkv;
  int b, head, row0, nvalid;                  // TMA batch, head; first row; rows of the sequence in the block
  size_t sc_idx;
  if (a.varlen) {
    const int gb = id % a.tmax;
    head = id / a.tmax;
    if (gb >= __ldg(a.blk_off + a.nseq)) return;
    const int seq = varlen_seq(a, gb);
    row0 = __ldg(a.cu + seq) + (gb - __ldg(a.blk_off + seq)) * ROWS;
    nvalid = min(ROWS, __ldg(a.cu + seq + 1) - row0);
    b = 0;
    sc_idx = (size_t)head * a.tmax + gb;
  } else {
    const int blk = id % a.nblk, bh = id / a.nblk;
    b = bh / Hx;
    head = bh % Hx;
    row0 = blk * ROWS;
    nvalid = min(ROWS, a.N - row0);
    sc_idx = ((size_t)b * Hx + head) * a.nblk + blk;
  }
  float* sc = is_q ? a.sq : a.sk;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int r = warp * 16 + (lane >> 1);      // row in the block
  const int half = lane & 1;                  // elements [64*half, 64*half + 64)
  if (t == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (t < 64) {
    // sign flips as XOR masks on bf16 pairs (elements 2t, 2t+1)
    const uint32_t w = a.sign_bits[(2 * t) >> 5] >> ((2 * t) & 31);
    xmask[t] = a.rotate ? (((w & 1u) << 15) | (((w >> 1) & 1u) << 31)) : 0u;
  }
  __syncthreads();
  if (t == 0) {
    const CUtensorMap* m = is_q ? &in_q : &in_k;
    mbar_expect_tx(&bar, 2 * 16384);
    tma_load_4d(m, &bar, tile, 0, head, row0, b);
    tma_load_4d(m, &bar, tile + 16384, 64, head, row0, b);
  }
  mbar_wait(&bar, 0, a.timeout_ns, &abort_flag, a.err);
  // element e (0..63 of this half) of row r: chunk `half`, piece e/8 swizzled by r%8
  float x[64];
  const uint8_t* src = tile + half * 16384 + r * 128;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint4 v = *reinterpret_cast<const uint4*>(src + ((j ^ (r & 7)) << 4));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = j * 8 + 2 * i;
      const uint32_t u = w[i] ^ xmask[(half * 64 + e) >> 1];
      x[e] = __uint_as_float(u << 16);
      x[e + 1] = __uint_as_float(u & 0xFFFF0000u);
    }
  }
  if (a.rotate) {
#pragma unroll
    for (int i = 0; i < 64; i += 2) {
      const float p0 = x[i], p1 = x[i + 1];
      x[i] = __fadd_rn(p0, p1);
      x[i + 1] = __fsub_rn(p0, p1);
    }
    butterfly_pairs<64>(x, 2);
    butterfly_pairs<64>(x, 4);
    butterfly_pairs<64>(x, 8);
    butterfly_pairs<64>(x, 16);
    butterfly_pairs<64>(x, 32);
    // span 64: (x_i, x_{i+64}) -> (x_i + x_{i+64}, x_i - x_{i+64}); half 0 holds x_i
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, x[i], 1);
      x[i] = half ? __fsub_rn(o, x[i]) : __fadd_rn(x[i], o);
    }
    const uint64_t c2 = f2_pack(a.inv_sqrt_d, a.inv_sqrt_d);
#pragma unroll
    for (int i = 0; i < 64; i += 2) f2_unpack(f2_mul(f2_pack(x[i], x[i + 1]), c2), x[i], x[i + 1]);
  }
  const bool valid = r < nvalid;                // rows past the sequence do not count
  float m0 = 0.f, m1 = 0.f, m2 = 0.f, m3 = 0.f;
  if (valid) {
#pragma unroll
    for (int i = 0; i < 64; i += 4) {
      m0 = fmaxf(m0, fabsf(x[i]));
      m1 = fmaxf(m1, fabsf(x[i + 1]));
      m2 = fmaxf(m2, fabsf(x[i + 2]));
      m3 = fmaxf(m3, fabsf(x[i + 3]));
    }
  }
  float amax = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
  if (a.block_mode || phase == 0) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (lane == 0) red[warp] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) amax = fmaxf(amax, red[w]);
  }
  float s;
  if (a.block_mode) {
    s = scale_from_amax(amax);
    if (t == 0) sc[sc_idx] = s;
  } else if (phase == 0) {
    if (t == 0) atomicMax(reinterpret_cast<unsigned int*>(sc), __float_as_uint(amax));
    return;
  } else {
    s = scale_from_amax(__uint_as_float(*reinterpret_cast<volatile unsigned int*>(sc)));
  }
  const Divider dv(s);
  if (dv.fast) {
    // Markstein correction, hoisted branch
    const uint64_t r2 = f2_pack(dv.r, dv.r), ns2 = f2_pack(-dv.s, -dv.s);
#pragma unroll
    for (int i = 0; i < 64; i += 2) {
      const uint64_t xv = f2_pack(x[i], x[i + 1]);
      const uint64_t q0 = f2_mul(xv, r2);
      const uint64_t e = f2_fma(q0, ns2, xv);
      f2_unpack(f2_fma(e, r2, q0), x[i], x[i + 1]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 64; ++i) x[i] = __fdiv_rn(x[i], dv.s);
  }
  // packed sequences: a block may end inside the next sequence's rows, so
  // only this sequence's rows are stored, straight from registers
  uint8_t* gdst = (is_q ? a.q8 : a.k8) + ((size_t)(row0 + r) * Hx + head) * 128 + half * 64;
  uint8_t* dst = codes + r * 128;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = j * 16;
    const uint4 w = make_uint4(e4m3x4(x[e], x[e + 1], x[e + 2], x[e + 3]), e4m3x4(x[e + 4], x[e + 5], x[e + 6], x[e + 7]),
                               e4m3x4(x[e + 8], x[e + 9], x[e + 10], x[e + 11]),
                               e4m3x4(x[e + 12], x[e + 13], x[e + 14], x[e + 15]));
    if (a.varlen) {
      if (valid) reinterpret_cast<uint4*>(gdst)[j] = w;
    } else {
      const int piece = half * 4 + j;
      *reinterpret_cast<uint4*>(dst + ((piece ^ (r & 7)) << 4)) = w;
    }
  }
  if (a.varlen) return;
  fence_proxy_async_smem();
  __syncthreads();
  if (t == 0) {
    tma_store_4d(is_q ? &out_q : &out_k, codes, 0, head, row0, b);
    tma_store_commit();
    tma_store_wait_all();
  }
}

// V block (b, kv head, 128 rows) for head dim 128; thread c owns channel c.
// phase 0: per-channel (block mode) or whole-tensor amax -> atomicMax into sv.
// phase 1: codes x / scale_c written transposed: vt8[b][head][c][n0 .. n0+127].
constexpr int V128_SMEM = 1024 + 2 * 16384;

__global__ void __launch_bounds__(128) v128_kernel(const __grid_constant__ CUtensorMap in_v, const PrepassArgs a,
                                                   int phase) {
  extern __shared__ uint8_t raw[];
  uint8_t* tile = raw + ((1024 - (smem_u32(raw) & 1023)) & 1023);   // 2 x [128 rows][64 ch] bf16, swizzled
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  __shared__ float red[4];
  // fixed length: B x Hkv x nblk blocks; packed sequences: Hkv x tmax global
  // blocks (those past the last exit), V^T columns from 128 * gb
  int b, head, row0, nvalid;
  size_t sv_row, vt_row, vt_col;
  if (a.varlen) {
    const int gb = blockIdx.x % a.tmax;
    head = blockIdx.x / a.tmax;
    if (gb >= __ldg(a.blk_off + a.nseq)) return;
    const int seq = varlen_seq(a, gb);
    row0 = __ldg(a.cu + seq) + (gb - __ldg(a.blk_off + seq)) * ROWS;
    nvalid = min(ROWS, __ldg(a.cu + seq + 1) - row0);
    b = 0;
    sv_row = ((size_t)seq * a.Hkv + head) * 128;
    vt_row = (size_t)head * 128;
    vt_col = (size_t)gb * ROWS;
  } else {
    const int blk = blockIdx.x % a.nblk, bh = blockIdx.x / a.nblk;
    b = bh / a.Hkv;
    head = bh % a.Hkv;
    row0 = blk * ROWS;
    nvalid = min(ROWS, a.N - row0);
    sv_row = vt_row = ((size_t)b * a.Hkv + head) * 128;
    vt_col = (size_t)blk * ROWS;
  }
  const int c = threadIdx.x;
  if (c == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (c == 0) {
    mbar_expect_tx(&bar, 2 * 16384);
    tma_load_4d(&in_v, &bar, tile, 0, head, row0, b);
    tma_load_4d(&in_v, &bar, tile + 16384, 64, head, row0, b);
  }
  mbar_wait(&bar, 0, a.timeout_ns, &abort_flag, a.err);
  // channel c of row n: chunk c/64, 16-byte piece ((c%64)/8) ^ (n%8), element c%8
  const uint8_t* col = tile + (c >> 6) * 16384 + (c & 7) * 2;
  const int piece = (c & 63) >> 3;
  float* sv_c = a.block_mode ? a.sv + sv_row + c : a.sv;
  if (phase == 0) {
    float m0 = 0.f, m1 = 0.f;
#pragma unroll 8
    for (int n = 0; n < ROWS; n += 2) {
      const float v0 = __uint_as_float((uint32_t)*reinterpret_cast<const uint16_t*>(col + n * 128 + ((piece ^ (n & 7)) << 4)) << 16);
      const float v1 = __uint_as_float((uint32_t)*reinterpret_cast<const uint16_t*>(col + (n + 1) * 128 + ((piece ^ ((n + 1) & 7)) << 4)) << 16);
      if (n < nvalid) m0 = fmaxf(m0, fabsf(v0));
      if (n + 1 < nvalid) m1 = fmaxf(m1, fabsf(v1));
    }
    float m = fmaxf(m0, m1);
    if (a.block_mode) {
      atomicMax(reinterpret_cast<unsigned int*>(sv_c), __float_as_uint(m));
    } else {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      if ((c & 31) == 0) red[c >> 5] = m;
      __syncthreads();
      if (c == 0) atomicMax(reinterpret_cast<unsigned int*>(sv_c), __float_as_uint(fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]))));
    }
    return;
  }
  const Divider dv(scale_from_amax(__uint_as_float(*reinterpret_cast<volatile unsigned int*>(sv_c))));
  uint4* dst = reinterpret_cast<uint4*>(a.vt8 + (vt_row + c) * a.ldv + vt_col);
#pragma unroll
  for (int g = 0; g < 8; ++g) {             // 16 rows -> 16 codes -> one 16-byte store
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float y[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int n = g * 16 + i * 4 + t;
        const float v = __uint_as_float((uint32_t)*reinterpret_cast<const uint16_t*>(col + n * 128 + ((piece ^ (n & 7)) << 4)) << 16);
        y[t] = n < nvalid ? dv.div(v) : 0.f;    // pad keys past N hold code 0
      }
      w[i] = e4m3x4(y[0], y[1], y[2], y[3]);
    }
    dst[g] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// ---------------------------------------------------------------- head dims 64, 128, 256, persistent (block scales)
// Two persistent launches replace the per-block kernels for fixed-length
// block quantisation (tiles of 128 rows x D channels arrive by TMA into a
// ring, 64-channel boxes; thread 0 issues the copy of tile k + stages as soon
// as the CTA barrier that follows the reads of tile k has passed, so no
// producer warp takes registers away; three CTAs of 8 warps per SM at D = 64,
// two at D = 128, one at D = 256):
//  prep_main_kernel: work list ordered by 128-row block (batch, block) and
//    inside it [Q heads][K heads][V heads], so the V tiles (per-channel amax,
//    atomicMax into sv) keep HBM busy while other CTAs do the Q/K arithmetic:
//    sign flips, Walsh-Hadamard butterflies, block amax -> scale, e4m3 codes
//    stored from registers (each thread writes its half row). The Q/K
//    arithmetic bounds this kernel.
//  prep_vcodes_kernel: re-reads the V tiles (part of V is still in L2) and
//    writes the codes transposed (keys contiguous): each thread turns 4 rows x
//    8 channels of each 64-channel chunk into words of 4 keys by byte
//    permutes in a swizzled code tile that leaves by TMA stores (128 channel
//    rows each).
constexpr int P_THREADS = 256;
template <int D>
struct PrepTraits {
  static constexpr int TILE = ROWS * D * 2;                 // bf16 tile bytes
  static constexpr int NCH = D / 64;                        // 64-channel boxes of 16 KB
  static constexpr int MAIN_STAGES = 3;
  static constexpr int V_STAGES = 2;
  static constexpr int MAIN_SMEM = 1024 + MAIN_STAGES * TILE;
  static constexpr int CODE_TILE = D * ROWS;                // u8 [D channels][128 keys]
  static constexpr int V_SMEM = 1024 + V_STAGES * TILE + 2 * CODE_TILE;
  static constexpr int MIN_CTAS = D == 64 ? 3 : (D == 128 ? 2 : 1);
  static constexpr int E = D / 2;                           // Q/K elements per thread (two threads per row)
};

template <int S>
struct PrepRing {
  uint64_t full[S];
  int abort;
};

enum : int { ORDER_MAIN = 0, ORDER_V = 1 };

// item -> kind (0 Q, 1 K, 2 V), batch, head, 128-row block; by (batch, row
// block), heads fastest. ORDER_MAIN: [Q heads][K heads][V heads] per row
// block; ORDER_V: V heads only.
__device__ __forceinline__ void prep_item(const PrepassArgs& a, int id, int order, int& kind, int& b, int& head,
                                          int& blk) {
  const int per = order == ORDER_V ? a.Hkv : a.H + 2 * a.Hkv;
  const int rb = id / per;
  int w = id - rb * per;
  blk = rb % a.nblk;
  b = rb / a.nblk;
  if (order == ORDER_V) { kind = 2; head = w; return; }
  if (w < a.H) { kind = 0; head = w; }
  else if ((w -= a.H) < a.Hkv) { kind = 1; head = w; }
  else { kind = 2; head = w - a.Hkv; }
}

// Copy of the CTA's k-th tile (item blockIdx.x + k * gridDim.x) into stage k % S.
template <int D, int S>
__device__ __forceinline__ void prep_load(const PrepassArgs& a, PrepRing<S>& sh, uint8_t* ring, int k, int total,
                                          int order, const CUtensorMap* mq, const CUtensorMap* mk,
                                          const CUtensorMap* mv) {
  using P = PrepTraits<D>;
  const int id = blockIdx.x + k * gridDim.x;
  if (id >= total) return;
  int kind, b, head, blk;
  prep_item(a, id, order, kind, b, head, blk);
  const CUtensorMap* m = kind == 0 ? mq : (kind == 1 ? mk : mv);
  const int st = k % S;
  uint8_t* tile = ring + st * P::TILE;
  mbar_expect_tx(&sh.full[st], P::TILE);
#pragma unroll
  for (int c = 0; c < P::NCH; ++c) tma_load_4d(m, &sh.full[st], tile + c * 16384, c * 64, head, blk * ROWS, b);
}

// On the way out after an abort: wait (bounded) for copies still in flight.
template <int S>
__device__ __forceinline__ void prep_drain(const PrepassArgs& a, PrepRing<S>& sh, int k_done, int total) {
  for (int k = k_done; k < k_done + S; ++k)
    if ((int)blockIdx.x + k * (int)gridDim.x < total)
      mbar_wait_drain(&sh.full[k % S], (k / S) & 1, a.timeout_ns, a.err);
}

template <int D>
__global__ void __launch_bounds__(P_THREADS, PrepTraits<D>::MIN_CTAS) prep_main_kernel(
    const __grid_constant__ CUtensorMap in_q, const __grid_constant__ CUtensorMap in_k,
    const __grid_constant__ CUtensorMap in_v, const PrepassArgs a) {
  using P = PrepTraits<D>;
  constexpr int S = P::MAIN_STAGES;
  constexpr int E = P::E;
  constexpr int U = D / 8;                         // 16-byte units of a row (8 channels each)
  constexpr int G = P_THREADS / U;                 // row groups of the V amax
  constexpr int GR = ROWS / G;                     // rows per group
  extern __shared__ uint8_t raw[];
  uint8_t* ring = raw + ((1024 - (smem_u32(raw) & 1023)) & 1023);   // stages x NCH x [128 rows][128 B], swizzled
  __shared__ PrepRing<S> sh;
  __shared__ float red[2][8];
  __shared__ float vred[2][8][D];                  // V amax: per warp and channel
  __shared__ uint32_t xmask[D / 2];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int total = (a.B * a.H + 2 * a.B * a.Hkv) * a.nblk;
  if (t == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&sh.full[s], 1);
    sh.abort = 0;
    fence_mbar_init();
  }
  if (t < D / 2) {
    // sign flips as XOR masks on bf16 pairs (elements 2t, 2t+1)
    const uint32_t w = a.sign_bits[(2 * t) >> 5] >> ((2 * t) & 31);
    xmask[t] = a.rotate ? (((w & 1u) << 15) | (((w >> 1) & 1u) << 31)) : 0u;
  }
  __syncthreads();
  if (t == 0) {
    for (int k = 0; k < S; ++k) prep_load<D, S>(a, sh, ring, k, total, ORDER_MAIN, &in_q, &in_k, &in_v);
  }
  // Q/K: lanes 2i, 2i+1 of a warp hold elements [0, E) / [E, D) of row warp * 16 + i
  const int r = warp * 16 + (lane >> 1);
  const int half = lane & 1;
  int k = 0;
  bool ok = true;
  for (int id = blockIdx.x; id < total; id += gridDim.x, ++k) {
    const int st = k % S;
    const int pb = k & 1;
    ok = mbar_wait(&sh.full[st], (k / S) & 1, a.timeout_ns, &sh.abort, a.err);
    if (!ok) break;
    int kind, b, head, blk;
    prep_item(a, id, ORDER_MAIN, kind, b, head, blk);
    const uint8_t* tile = ring + st * P::TILE;
    const int row0 = blk * ROWS;
    const int nvalid = min(ROWS, a.N - row0);
    if (kind == 2) {
      // V: per-channel amax of the block's valid rows. Thread t reads the 8
      // channels of unit o = t % U (16-byte unit o % 8 of chunk o / 8) in
      // rows GR * g .. + GR - 1 (g = t / U); lanes of a warp with the same
      // unit combine by a shuffle (D = 128), the 8 warps through shared memory.
      const int o = t % U, g = t / U;
      const uint8_t* base = tile + (o >> 3) * 16384;
      float cm[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) cm[i] = 0.f;
#pragma unroll
      for (int i = 0; i < GR; ++i) {
        const int n = g * GR + i;
        if (n < nvalid) {
          const uint4 v = *reinterpret_cast<const uint4*>(base + n * 128 + (((o & 7) ^ (n & 7)) << 4));
          const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            cm[2 * m] = fmaxf(cm[2 * m], fabsf(__uint_as_float(w4[m] << 16)));
            cm[2 * m + 1] = fmaxf(cm[2 * m + 1], fabsf(__uint_as_float(w4[m] & 0xFFFF0000u)));
          }
        }
      }
#pragma unroll
      for (int off = U; off < 32; off <<= 1)
#pragma unroll
        for (int i = 0; i < 8; ++i) cm[i] = fmaxf(cm[i], __shfl_xor_sync(0xffffffffu, cm[i], off));
      if (lane < U) {
#pragma unroll
        for (int i = 0; i < 8; ++i) vred[pb][warp][8 * o + i] = cm[i];
      }
      __syncthreads();                                  // every thread has read the tile
      if (t == 0) prep_load<D, S>(a, sh, ring, k + S, total, ORDER_MAIN, &in_q, &in_k, &in_v);
      if (t < D) {
        float m = vred[pb][0][t];
#pragma unroll
        for (int w8 = 1; w8 < 8; ++w8) m = fmaxf(m, vred[pb][w8][t]);
        atomicMax(reinterpret_cast<unsigned int*>(a.sv + ((size_t)b * a.Hkv + head) * D + t), __float_as_uint(m));
      }
      continue;
    }
    // Q/K: rotate, block amax -> scale, codes
    const bool is_q = kind == 0;
    float x[E];
#pragma unroll
    for (int j = 0; j < E / 8; ++j) {
      // 16-byte unit j of this half row: elements e0 .. e0+7 of the row, in
      // 64-channel chunk e0 / 64 at unit (e0 / 8) % 8
      const int e0 = half * E + j * 8;
      const uint8_t* src = tile + (e0 >> 6) * 16384 + r * 128;
      const uint4 v = *reinterpret_cast<const uint4*>(src + ((((e0 >> 3) & 7) ^ (r & 7)) << 4));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int e = j * 8 + 2 * i;
        const uint32_t u = w[i] ^ xmask[(half * E + e) >> 1];
        x[e] = __uint_as_float(u << 16);
        x[e + 1] = __uint_as_float(u & 0xFFFF0000u);
      }
    }
    if (a.rotate) {
      // spans 1 .. E/2 inside the thread, span E across the lane pair
#pragma unroll
      for (int i = 0; i < E; i += 2) {
        const float p0 = x[i], p1 = x[i + 1];
        x[i] = __fadd_rn(p0, p1);
        x[i + 1] = __fsub_rn(p0, p1);
      }
#pragma unroll
      for (int h = 2; h < E; h *= 2) butterfly_pairs<E>(x, h);
#pragma unroll
      for (int i = 0; i < E; ++i) {
        const float o = __shfl_xor_sync(0xffffffffu, x[i], 1);
        x[i] = half ? __fsub_rn(o, x[i]) : __fadd_rn(x[i], o);
      }
      const uint64_t c2 = f2_pack(a.inv_sqrt_d, a.inv_sqrt_d);
#pragma unroll
      for (int i = 0; i < E; i += 2) f2_unpack(f2_mul(f2_pack(x[i], x[i + 1]), c2), x[i], x[i + 1]);
    }
    float m0 = 0.f, m1 = 0.f, m2 = 0.f, m3 = 0.f;
    if (r < nvalid) {
#pragma unroll
      for (int i = 0; i < E; i += 4) {
        m0 = fmaxf(m0, fabsf(x[i]));
        m1 = fmaxf(m1, fabsf(x[i + 1]));
        m2 = fmaxf(m2, fabsf(x[i + 2]));
        m3 = fmaxf(m3, fabsf(x[i + 3]));
      }
    }
    float amax = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (lane == 0) red[pb][warp] = amax;
    __syncthreads();                                    // every thread has read the tile
    if (t == 0) prep_load<D, S>(a, sh, ring, k + S, total, ORDER_MAIN, &in_q, &in_k, &in_v);
    amax = red[pb][0];
#pragma unroll
    for (int w = 1; w < 8; ++w) amax = fmaxf(amax, red[pb][w]);
    const float s = scale_from_amax(amax);
    if (t == 0) {
      const int Hx = is_q ? a.H : a.Hkv;
      (is_q ? a.sq : a.sk)[((size_t)b * Hx + head) * a.nblk + blk] = s;
    }
    const Divider dv(s);
    if (dv.fast) {
      const uint64_t r2 = f2_pack(dv.r, dv.r), ns2 = f2_pack(-dv.s, -dv.s);
#pragma unroll
      for (int i = 0; i < E; i += 2) {
        const uint64_t xv = f2_pack(x[i], x[i + 1]);
        const uint64_t q0 = f2_mul(xv, r2);
        const uint64_t e = f2_fma(q0, ns2, xv);
        f2_unpack(f2_fma(e, r2, q0), x[i], x[i + 1]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < E; ++i) x[i] = __fdiv_rn(x[i], dv.s);
    }
    if (r < nvalid) {
      const int Hx = is_q ? a.H : a.Hkv;
      uint4* dst = reinterpret_cast<uint4*>((is_q ? a.q8 : a.k8) + (((size_t)b * a.N + row0 + r) * Hx + head) * D +
                                            half * E);
#pragma unroll
      for (int j = 0; j < E / 16; ++j) {
        const int e = j * 16;
        dst[j] = make_uint4(e4m3x4(x[e], x[e + 1], x[e + 2], x[e + 3]), e4m3x4(x[e + 4], x[e + 5], x[e + 6], x[e + 7]),
                            e4m3x4(x[e + 8], x[e + 9], x[e + 10], x[e + 11]),
                            e4m3x4(x[e + 12], x[e + 13], x[e + 14], x[e + 15]));
      }
    }
  }
  if (t == 0 && !ok) prep_drain(a, sh, k, total);
}

template <int D>
__global__ void __launch_bounds__(P_THREADS, PrepTraits<D>::MIN_CTAS) prep_vcodes_kernel(
    const __grid_constant__ CUtensorMap in_v, const __grid_constant__ CUtensorMap out_vt, const PrepassArgs a) {
  using P = PrepTraits<D>;
  constexpr int S = P::V_STAGES;
  extern __shared__ uint8_t raw[];
  uint8_t* ring = raw + ((1024 - (smem_u32(raw) & 1023)) & 1023);   // stages x NCH x [128 rows][128 B], swizzled
  uint8_t* codes = ring + S * P::TILE;             // 2 x [D channels][128 keys] u8, 128-byte swizzled
  __shared__ PrepRing<S> sh;
  __shared__ float vdiv_s[2][D], vdiv_r[2][D];     // per-channel scale and RN(1/scale)
  __shared__ int vdiv_slow[2];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int total = a.B * a.Hkv * a.nblk;
  if (t == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&sh.full[s], 1);
    sh.abort = 0;
    fence_mbar_init();
  }
  if (t == 32) tma_prefetch_desc(&out_vt);
  __syncthreads();
  if (t == 0) {
    for (int k = 0; k < S; ++k) prep_load<D, S>(a, sh, ring, k, total, ORDER_V, &in_v, &in_v, &in_v);
  }
  // thread (warp w, lane q): rows 4q .. 4q+3 and the 8 channels of 16-byte
  // unit o = (w + q) % 8 in every 64-channel chunk; over the CTA every (row
  // quad, unit) pair is taken once, and both the unit loads and the
  // transposed 32-bit stores are free of shared-memory bank conflicts
  const int q = lane, o = (warp + lane) & 7;
  int k = 0, n_v = 0;
  bool ok = true;
  for (int id = blockIdx.x; id < total; id += gridDim.x, ++k) {
    const int st = k % S;
    const int pb = k & 1;
    ok = mbar_wait(&sh.full[st], (k / S) & 1, a.timeout_ns, &sh.abort, a.err);
    if (!ok) break;
    int kind, b, head, blk;
    prep_item(a, id, ORDER_V, kind, b, head, blk);
    const uint8_t* tile = ring + st * P::TILE;
    const int nvalid = min(ROWS, a.N - blk * ROWS);
    if (t < D) {
      // divisor of channel t: scale from the channel amax, and its reciprocal
      const Divider dv(scale_from_amax(
          __uint_as_float(*reinterpret_cast<volatile const unsigned int*>(a.sv + ((size_t)b * a.Hkv + head) * D + t))));
      vdiv_s[pb][t] = dv.s;
      vdiv_r[pb][t] = dv.r;
      if (t == 0) vdiv_slow[pb] = 0;
    }
    uint8_t* ct = codes + (n_v & 1) * P::CODE_TILE;
    ++n_v;
    if (t == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");   // ct's previous stores have read it
    __syncthreads();
    if (t < D && !Divider(vdiv_s[pb][t]).fast) vdiv_slow[pb] = 1;
    __syncthreads();
    const bool slow = vdiv_slow[pb] != 0;
#pragma unroll
    for (int ck = 0; ck < P::NCH; ++ck) {
      const int c0 = ck * 64 + 8 * o;                 // first of this thread's 8 channels
      uint32_t cw[4][4];                              // [row i][channel pair m]: e4m3 codes (lo, hi)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int n = 4 * q + i;
        const uint4 v = *reinterpret_cast<const uint4*>(tile + ck * 16384 + n * 128 + ((o ^ (n & 7)) << 4));
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          float y0 = __uint_as_float(w4[m] << 16), y1 = __uint_as_float(w4[m] & 0xFFFF0000u);
          const float s0 = vdiv_s[pb][c0 + 2 * m], s1 = vdiv_s[pb][c0 + 2 * m + 1];
          if (!slow) {
            const uint64_t xv = f2_pack(y0, y1);
            const uint64_t r2 = f2_pack(vdiv_r[pb][c0 + 2 * m], vdiv_r[pb][c0 + 2 * m + 1]);
            const uint64_t q0 = f2_mul(xv, r2);
            const uint64_t e = f2_fma(q0, f2_pack(-s0, -s1), xv);
            f2_unpack(f2_fma(e, r2, q0), y0, y1);
          } else {
            y0 = __fdiv_rn(y0, s0);
            y1 = __fdiv_rn(y1, s1);
          }
          if (n >= nvalid) y0 = y1 = 0.f;              // pad keys past N hold code 0
          uint16_t c2;
          asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c2) : "f"(y1), "f"(y0));
          cw[i][m] = c2;
        }
      }
      // transpose: channel c0 + 2m gets the low bytes of rows 0-3, c0 + 2m + 1
      // the high bytes; one 32-bit word (4 keys) per channel row
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const uint32_t lo01 = cw[0][m] | (cw[1][m] << 16), lo23 = cw[2][m] | (cw[3][m] << 16);
        uint32_t even, odd;
        asm("prmt.b32 %0, %1, %2, 0x6420;" : "=r"(even) : "r"(lo01), "r"(lo23));
        asm("prmt.b32 %0, %1, %2, 0x7531;" : "=r"(odd) : "r"(lo01), "r"(lo23));
        const int ce = c0 + 2 * m, co = ce + 1;
        *reinterpret_cast<uint32_t*>(ct + ce * 128 + ((((4 * q) >> 4) ^ (ce & 7)) << 4) + ((4 * q) & 15)) = even;
        *reinterpret_cast<uint32_t*>(ct + co * 128 + ((((4 * q) >> 4) ^ (co & 7)) << 4) + ((4 * q) & 15)) = odd;
      }
    }
    fence_proxy_async_smem();
    __syncthreads();                                  // tile read, code tile written
    if (t == 0) {
      prep_load<D, S>(a, sh, ring, k + S, total, ORDER_V, &in_v, &in_v, &in_v);
      // one bulk group per tile: up to 128 channel rows per store
#pragma unroll
      for (int h = 0; h < (D + 127) / 128; ++h)
        tma_store_4d(&out_vt, ct + h * 16384, blk * ROWS, h * 128, b * a.Hkv + head, 0);
      tma_store_commit();
    }
  }
  if (t == 0) {
    if (!ok) prep_drain(a, sh, k, total);
    tma_store_wait_all();
  }
}

// Turns the amax values left in the scale outputs into scales.
__global__ void finalize_kernel(float* sq, float* sk, float* sv, int nsv, int tensor_mode) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < nsv) sv[i] = scale_from_amax(sv[i]);
  if (tensor_mode && i == 0) {
    sq[0] = scale_from_amax(sq[0]);
    sk[0] = scale_from_amax(sk[0]);
  }
}

}  // namespace

// Packed sequences (a.varlen): block offsets, then the kernels over H x tmax,
// Hkv x tmax and Hkv x tmax global blocks (those past the last sequence exit
// at once): the head-dim-128 kernels when `maps` is given, else the generic.
cudaError_t launch_fp8_prepass_varlen(const PrepassArgs& a, int d, const Prepass128Maps* maps, cudaStream_t s) {
  const size_t nsv = a.block_mode ? (size_t)a.nseq * a.Hkv * d : 1;
  cudaError_t e = cudaMemsetAsync(a.sv, 0, nsv * sizeof(float), s);
  if (e != cudaSuccess) return e;
  if (!a.block_mode) {
    if ((e = cudaMemsetAsync(a.sq, 0, sizeof(float), s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(a.sk, 0, sizeof(float), s)) != cudaSuccess) return e;
  }
  // V^T pad keys of each sequence's last block are written as code 0 by the
  // V kernel; columns past the last block are never read
  varlen_block_offsets_kernel<<<1, 1024, 0, s>>>(a.cu, a.nseq, a.blk_off);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int blocks = (a.H + 2 * a.Hkv) * a.tmax;
  const bool fast = d == 128 && maps != nullptr;
  if (fast) {
    e = cudaFuncSetAttribute(qk128_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, QK128_SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(v128_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, V128_SMEM);
    if (e != cudaSuccess) return e;
  }
  for (int phase = 0; phase < 2; ++phase) {
    if (fast) {
      // codes leave by plain stores in this mode: the output maps are not used
      if (phase == 0 || !a.block_mode) {
        qk128_kernel<<<(a.H + a.Hkv) * a.tmax, 256, QK128_SMEM, s>>>(maps->in_q, maps->in_k, maps->in_q, maps->in_k,
                                                                     a, phase);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
      }
      v128_kernel<<<a.Hkv * a.tmax, 128, V128_SMEM, s>>>(maps->in_v, a, phase);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
      continue;
    }
    switch (d) {
      case 64: prepass_kernel<2><<<blocks, THREADS, 0, s>>>(a, phase, 0); break;
      case 128: prepass_kernel<4><<<blocks, THREADS, 0, s>>>(a, phase, 0); break;
      default: prepass_kernel<8><<<blocks, THREADS, 0, s>>>(a, phase, 0); break;
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // amax values -> scales (phase 1 derived its divisors from the amax values)
  finalize_kernel<<<(int)((nsv + 255) / 256), 256, 0, s>>>(a.sq, a.sk, a.sv, (int)nsv, a.block_mode ? 0 : 1);
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_prep_persistent(const PrepassArgs& a, const Prepass128Maps& maps, int nqk, int nv,
                                          int sm_count, cudaStream_t s) {
  using P = PrepTraits<D>;
  cudaError_t e = cudaFuncSetAttribute(prep_main_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, P::MAIN_SMEM);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(prep_vcodes_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, P::V_SMEM);
  if (e != cudaSuccess) return e;
  const int g1 = min(nqk + nv, P::MIN_CTAS * sm_count), g2 = min(nv, P::MIN_CTAS * sm_count);
  prep_main_kernel<D><<<g1, P_THREADS, P::MAIN_SMEM, s>>>(maps.in_q, maps.in_k, maps.in_v, a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  prep_vcodes_kernel<D><<<g2, P_THREADS, P::V_SMEM, s>>>(maps.in_v, maps.out_vt, a);
  return cudaGetLastError();
}

cudaError_t launch_fp8_prepass(const PrepassArgs& a, int d, const Prepass128Maps* maps, int sm_count,
                               cudaStream_t s) {
  const size_t nsv = a.block_mode ? (size_t)a.B * a.Hkv * d : 1;
  cudaError_t e = cudaMemsetAsync(a.sv, 0, nsv * sizeof(float), s);
  if (e != cudaSuccess) return e;
  if (!a.block_mode) {
    if ((e = cudaMemsetAsync(a.sq, 0, sizeof(float), s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(a.sk, 0, sizeof(float), s)) != cudaSuccess) return e;
  }
  const int nqk = (a.B * a.H + a.B * a.Hkv) * a.nblk;
  const int nv = a.B * a.Hkv * a.nblk;
  const bool fast_qk = d == 128 && maps != nullptr;
  if (maps != nullptr && a.block_mode) {
    // persistent kernels: Q/K codes and V channel amax in one pass, V codes in
    // a second one, then the amax values become scales
    e = d == 64 ? launch_prep_persistent<64>(a, *maps, nqk, nv, sm_count, s)
                : (d == 128 ? launch_prep_persistent<128>(a, *maps, nqk, nv, sm_count, s)
                            : launch_prep_persistent<256>(a, *maps, nqk, nv, sm_count, s));
    if (e != cudaSuccess) return e;
    finalize_kernel<<<(int)((nsv + 255) / 256), 256, 0, s>>>(a.sq, a.sk, a.sv, (int)nsv, 0);
    return cudaGetLastError();
  }
  if (fast_qk) {
    e = cudaFuncSetAttribute(qk128_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, QK128_SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(v128_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, V128_SMEM);
    if (e != cudaSuccess) return e;
  }
  for (int phase = 0; phase < 2; ++phase) {
    if (fast_qk) {
      if (phase == 0 || !a.block_mode) {
        qk128_kernel<<<nqk, 256, QK128_SMEM, s>>>(maps->in_q, maps->in_k, maps->out_q, maps->out_k, a, phase);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
      }
      v128_kernel<<<nv, 128, V128_SMEM, s>>>(maps->in_v, a, phase);
    } else {
      const int blocks = nqk + nv;
      switch (d) {
        case 64: prepass_kernel<2><<<blocks, THREADS, 0, s>>>(a, phase, 0); break;
        case 128: prepass_kernel<4><<<blocks, THREADS, 0, s>>>(a, phase, 0); break;
        default: prepass_kernel<8><<<blocks, THREADS, 0, s>>>(a, phase, 0); break;
      }
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  finalize_kernel<<<(int)((nsv + 255) / 256), 256, 0, s>>>(a.sq, a.sk, a.sv, (int)nsv, a.block_mode ? 0 : 1);
  return cudaGetLastError();
}

}  // namespace attn45
