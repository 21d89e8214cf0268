// attn_fp8_api.cu -- C ABI of the FP8 path: pre-pass (rotation + block
// quantisation), FP8 forward, and the two combined over a caller workspace.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "api_internal.h"
#include "attn_common.cuh"
#include "attn45.h"
#include "fp8_launchers.h"
#include "fp8_prepass.h"

using namespace attn45;

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// SplitMix64 (Vigna): first output of the generator whose state is x.
uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

// Fixed device scratch for attn_fwd_fp8_auto_noalloc: a file-scope device
// array, so every GPU that loads this library holds these 16 MiB until the
// process exits. Host code must not use the symbol as a pointer (it is a
// host-side stand-in); its device address comes from cudaGetSymbolAddress,
// looked up once per device with that device current.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
static __device__ __align__(256) uint8_t g_fp8_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxScratchDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxScratchDevices] = {};

int noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return api_cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxScratchDevices) return api_fail(ATTN_ERR_UNSUPPORTED, "device index out of range");
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_fp8_noalloc_scratch);
    if (e != cudaSuccess || !ptr) return api_cuda_fail(e, "cudaGetSymbolAddress(fixed FP8 scratch)");
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return ATTN_OK;
}

struct Fp8Layout {
  size_t q8, k8, vt8, sq, sk, sv, total;
};

Fp8Layout fp8_layout(int B, int H, int Hkv, int N, int d, int mode) {
  const size_t nb = (size_t)((N + 127) / 128);
  const size_t ldv = (size_t)attn_fp8_vt_ld(N);
  Fp8Layout L;
  size_t off = 0;
  L.q8 = off; off += up256((size_t)B * N * H * d);
  L.k8 = off; off += up256((size_t)B * N * Hkv * d);
  L.vt8 = off; off += up256((size_t)B * Hkv * d * ldv);
  const bool blk = mode == ATTN_FP8_PER_BLOCK;
  L.sq = off; off += up256(4 * (blk ? (size_t)B * H * nb : 1));
  L.sk = off; off += up256(4 * (blk ? (size_t)B * Hkv * nb : 1));
  L.sv = off; off += up256(4 * (blk ? (size_t)B * Hkv * d : 1));
  L.total = off;
  return L;
}

int check_shape(int B, int H, int Hkv, int N, int d, int mode) {
  if (B < 1 || N < 1 || H < 1 || Hkv < 1 || H % Hkv != 0)
    return api_fail(ATTN_ERR_INVALID_ARG, "need B, N, H, Hkv >= 1 and H % Hkv == 0");
  if (d != 64 && d != 128 && d != 256) return api_fail(ATTN_ERR_UNSUPPORTED, "head dim not in {64,128,256}");
  if (mode != ATTN_FP8_PER_TENSOR && mode != ATTN_FP8_PER_BLOCK)
    return api_fail(ATTN_ERR_INVALID_ARG, "unknown FP8 scaling mode");
  if ((long long)B * N * (H > Hkv ? H : Hkv) > 0x7fffffffLL || (long long)(B * (long long)H + 2LL * B * Hkv) * ((N + 127) / 128) > 0x7fffffffLL)
    return api_fail(ATTN_ERR_INVALID_ARG, "problem too large for int32 indexing");
  return ATTN_OK;
}

// Checks of the forward step's own arguments, made by the combined calls
// before the pre-pass runs, so a call that is bound to fail writes nothing.
int check_fwd_fp8_args(int d, int causal, float scale, const void* o, const float* lse) {
  if (d != 64 && d != 128 && d != 256) return api_fail(ATTN_ERR_UNSUPPORTED, "head dim not in {64,128,256}");
  if (causal != 0 && causal != 1) return api_fail(ATTN_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (!(scale > 0.f) || !std::isfinite(scale)) return api_fail(ATTN_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (!o || !lse) return api_fail(ATTN_ERR_INVALID_ARG, "null pointer");
  if (!aligned(o, 16) || !aligned(lse, 4))
    return api_fail(ATTN_ERR_INVALID_ARG, "o must be 16-byte aligned, lse 4-byte aligned");
  return ATTN_OK;
}

}  // namespace

extern "C" {

int attn_fp8_vt_ld(int N) { return N <= 0 ? 0 : ((N + 127) / 128) * 128; }

size_t attn_fp8_workspace_size(int B, int H, int Hkv, int N, int d, int mode) {
  if (check_shape(B, H, Hkv, N, d, mode)) return 0;
  return fp8_layout(B, H, Hkv, N, d, mode).total;
}

int attn_fp8_prepass(const void* q, const void* k, const void* v, void* q8, void* k8, void* vt8, float* sq,
                     float* sk, float* sv, int B, int H, int Hkv, int N, int d, int mode, int rotate,
                     uint64_t hadamard_seed, void* stream) {
  int rc = check_shape(B, H, Hkv, N, d, mode);
  if (rc) return rc;
  if (rotate != 0 && rotate != 1) return api_fail(ATTN_ERR_INVALID_ARG, "rotate must be 0 or 1");
  if (!q || !k || !v || !q8 || !k8 || !vt8 || !sq || !sk || !sv) return api_fail(ATTN_ERR_INVALID_ARG, "null pointer");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(q8, 16) || !aligned(k8, 16) ||
      !aligned(vt8, 16) || !aligned(sq, 4) || !aligned(sk, 4) || !aligned(sv, 4))
    return api_fail(ATTN_ERR_INVALID_ARG, "tensors must be 16-byte aligned, scales 4-byte aligned");
  int sm = 0;
  unsigned int* err = nullptr;
  if ((rc = api_device(&sm, &err))) return rc;
  PrepassArgs a;
  memset(&a, 0, sizeof(a));
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.q8 = static_cast<uint8_t*>(q8);
  a.k8 = static_cast<uint8_t*>(k8);
  a.vt8 = static_cast<uint8_t*>(vt8);
  a.sq = sq;
  a.sk = sk;
  a.sv = sv;
  a.B = B;
  a.N = N;
  a.H = H;
  a.Hkv = Hkv;
  a.nblk = (N + 127) / 128;
  a.ldv = attn_fp8_vt_ld(N);
  a.block_mode = mode == ATTN_FP8_PER_BLOCK;
  a.rotate = rotate;
  a.inv_sqrt_d = (float)(1.0 / std::sqrt((double)d));
  for (int c = 0; c < d; ++c)
    if (splitmix64(hadamard_seed + (uint64_t)c) & 1ull) a.sign_bits[c >> 5] |= 1u << (c & 31);
  a.timeout_ns = api_timeout_ns();
  a.err = err;
  Prepass128Maps maps;
  const Prepass128Maps* mp = nullptr;
  if (d == 128 || mode == ATTN_FP8_PER_BLOCK) {
    if ((rc = api_make_map(&maps.in_q, false, q, d, H, N, B, 64, 128))) return rc;
    if ((rc = api_make_map(&maps.in_k, false, k, d, Hkv, N, B, 64, 128))) return rc;
    if ((rc = api_make_map(&maps.in_v, false, v, d, Hkv, N, B, 64, 128))) return rc;
    if ((rc = api_make_map(&maps.out_q, true, q8, d, H, N, B, 128, 128))) return rc;
    if ((rc = api_make_map(&maps.out_k, true, k8, d, Hkv, N, B, 128, 128))) return rc;
    if ((rc = api_make_map_rows(&maps.out_vt, vt8, attn_fp8_vt_ld(N), d, (uint64_t)B * Hkv, 128, d < 128 ? d : 128)))
      return rc;
    mp = &maps;
  }
  cudaError_t e = launch_fp8_prepass(a, d, mp, sm, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return api_cuda_fail(e, "attn_fp8_prepass launch");
  return ATTN_OK;
}

int attn_fwd_fp8(const void* q8, const void* k8, const void* vt8, const float* sq, const float* sk,
                 const float* sv, void* o, float* lse, int B, int H, int Hkv, int N, int d, int causal,
                 float scale, int mode, void* stream) {
  int rc = check_shape(B, H, Hkv, N, d, mode);
  if (rc) return rc;
  if (causal != 0 && causal != 1) return api_fail(ATTN_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (!(scale > 0.f) || !std::isfinite(scale)) return api_fail(ATTN_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (!q8 || !k8 || !vt8 || !sq || !sk || !sv || !o || !lse) return api_fail(ATTN_ERR_INVALID_ARG, "null pointer");
  if (!aligned(q8, 16) || !aligned(k8, 16) || !aligned(vt8, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
      !aligned(sq, 4) || !aligned(sk, 4) || !aligned(sv, 4))
    return api_fail(ATTN_ERR_INVALID_ARG, "tensors must be 16-byte aligned, scales and lse 4-byte aligned");
  int sm = 0;
  unsigned int* err = nullptr;
  if ((rc = api_device(&sm, &err))) return rc;
  const int ldv = attn_fp8_vt_ld(N);
  CUtensorMap mq, mk, mv, mo;
  // head dim 256 runs on CTA pairs: each CTA of a pair loads 64 keys of a
  // 128-key block and 128 of V's channel rows. Head dim 64 runs on the
  // head-dim-128 kernel: its 128-byte boxes reach past the 64 channels of a
  // row (and the 64 channel rows of V^T), which the copies fill with zeros.
  const bool pair = d == 256;
  if ((rc = api_make_map(&mq, true, q8, d, H, N, B, 128, 128))) return rc;
  if ((rc = api_make_map(&mk, true, k8, d, Hkv, N, B, 128, pair ? 64 : 128))) return rc;
  // V^T codes: [B*Hkv][d][ldv] read as boxes of (128 keys) x (128 channel rows)
  if ((rc = api_make_map_rows(&mv, vt8, ldv, d, (uint64_t)B * Hkv, 128, 128))) return rc;
  // bf16 output: 64 columns x 32 rows per bulk store (one warp's rows)
  if ((rc = api_make_map(&mo, false, o, d, H, N, B, 64, 32))) return rc;
  FwdParams p;
  memset(&p, 0, sizeof(p));
  p.o = o;
  p.lse = lse;
  p.sq = sq;
  p.sk = sk;
  p.sv = sv;
  p.nseq = B;
  p.N = N;
  p.total = B * N;
  p.H = H;
  p.Hkv = Hkv;
  p.group = H / Hkv;
  p.vt_ld = ldv;
  p.fp8_block = mode == ATTN_FP8_PER_BLOCK;
  p.fp8_d = d;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.timeout_ns = api_timeout_ns();
  p.err = err;
  cudaError_t e = pair ? launch_fwd_fp8_d256(mq, mk, mv, mo, p, causal != 0, sm, static_cast<cudaStream_t>(stream))
                       : launch_fwd_fp8_d128(mq, mk, mv, mo, p, causal != 0, false, sm, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return api_cuda_fail(e, "attn_fwd_fp8 launch");
  return ATTN_OK;
}

int attn_fwd_fp8_auto(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
                      size_t workspace_bytes, int B, int H, int Hkv, int N, int d, int causal, float scale,
                      int mode, int rotate, uint64_t hadamard_seed, void* stream) {
  int rc = check_shape(B, H, Hkv, N, d, mode);
  if (rc) return rc;
  if ((rc = check_fwd_fp8_args(d, causal, scale, o, lse))) return rc;
  const Fp8Layout L = fp8_layout(B, H, Hkv, N, d, mode);
  if (!workspace || !aligned(workspace, 256)) return api_fail(ATTN_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (workspace_bytes < L.total) return api_fail(ATTN_ERR_INVALID_ARG, "workspace smaller than attn_fp8_workspace_size()");
  uint8_t* w = static_cast<uint8_t*>(workspace);
  float* sq = reinterpret_cast<float*>(w + L.sq);
  float* sk = reinterpret_cast<float*>(w + L.sk);
  float* sv = reinterpret_cast<float*>(w + L.sv);
  rc = attn_fp8_prepass(q, k, v, w + L.q8, w + L.k8, w + L.vt8, sq, sk, sv, B, H, Hkv, N, d, mode, rotate,
                        hadamard_seed, stream);
  if (rc) return rc;
  return attn_fwd_fp8(w + L.q8, w + L.k8, w + L.vt8, sq, sk, sv, o, lse, B, H, Hkv, N, d, causal, scale, mode,
                      stream);
}

int attn_fp8_varlen_tmax(int total, int nseq) {
  if (total < 0 || nseq < 1) return 0;
  return (total + 127) / 128 + nseq;
}

int attn_fp8_prepass_varlen(const void* q, const void* k, const void* v, const int* cu_seqlens, void* q8, void* k8,
                            void* vt8, float* sq, float* sk, float* sv, int* blk_off, int nseq, int total, int H,
                            int Hkv, int d, int mode, int rotate, uint64_t hadamard_seed, void* stream) {
  if (nseq < 1 || nseq > MAX_VARLEN_SEQS) return api_fail(ATTN_ERR_INVALID_ARG, "nseq must be in [1, 2048]");
  if (total < 0) return api_fail(ATTN_ERR_INVALID_ARG, "total must be >= 0");
  if (H < 1 || Hkv < 1 || H % Hkv != 0) return api_fail(ATTN_ERR_INVALID_ARG, "need H % Hkv == 0");
  if (d != 64 && d != 128 && d != 256) return api_fail(ATTN_ERR_UNSUPPORTED, "head dim not in {64,128,256}");
  if (mode != ATTN_FP8_PER_TENSOR && mode != ATTN_FP8_PER_BLOCK) return api_fail(ATTN_ERR_INVALID_ARG, "unknown FP8 mode");
  if (rotate != 0 && rotate != 1) return api_fail(ATTN_ERR_INVALID_ARG, "rotate must be 0 or 1");
  const int tmax = attn_fp8_varlen_tmax(total, nseq);
  if ((long long)(H + 2 * Hkv) * tmax > 0x7fffffffLL || (long long)total * H * d > 0x7fffffffffLL)
    return api_fail(ATTN_ERR_INVALID_ARG, "problem too large");
  if (!q || !k || !v || !cu_seqlens || !q8 || !k8 || !vt8 || !sq || !sk || !sv || !blk_off)
    return api_fail(ATTN_ERR_INVALID_ARG, "null pointer");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(q8, 16) || !aligned(k8, 16) ||
      !aligned(vt8, 16) || !aligned(sq, 4) || !aligned(sk, 4) || !aligned(sv, 4) || !aligned(blk_off, 4) ||
      !aligned(cu_seqlens, 4))
    return api_fail(ATTN_ERR_INVALID_ARG, "tensors must be 16-byte aligned, scales and indices 4-byte aligned");
  int sm = 0;
  unsigned int* err = nullptr;
  int rc;
  if ((rc = api_device(&sm, &err))) return rc;
  PrepassArgs a;
  memset(&a, 0, sizeof(a));
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.q8 = static_cast<uint8_t*>(q8);
  a.k8 = static_cast<uint8_t*>(k8);
  a.vt8 = static_cast<uint8_t*>(vt8);
  a.sq = sq;
  a.sk = sk;
  a.sv = sv;
  a.H = H;
  a.Hkv = Hkv;
  a.ldv = 128 * tmax;
  a.block_mode = mode == ATTN_FP8_PER_BLOCK;
  a.rotate = rotate;
  a.inv_sqrt_d = (float)(1.0 / std::sqrt((double)d));
  for (int c = 0; c < d; ++c)
    if (splitmix64(hadamard_seed + (uint64_t)c) & 1ull) a.sign_bits[c >> 5] |= 1u << (c & 31);
  a.timeout_ns = api_timeout_ns();
  a.err = err;
  a.varlen = 1;
  a.nseq = nseq;
  a.tmax = tmax;
  a.cu = cu_seqlens;
  a.blk_off = blk_off;
  Prepass128Maps maps;
  const Prepass128Maps* mp = nullptr;
  if (d == 128 && total > 0) {
    if ((rc = api_make_map(&maps.in_q, false, q, d, H, total, 1, 64, 128))) return rc;
    if ((rc = api_make_map(&maps.in_k, false, k, d, Hkv, total, 1, 64, 128))) return rc;
    if ((rc = api_make_map(&maps.in_v, false, v, d, Hkv, total, 1, 64, 128))) return rc;
    mp = &maps;
  }
  cudaError_t e = launch_fp8_prepass_varlen(a, d, mp, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return api_cuda_fail(e, "attn_fp8_prepass_varlen launch");
  return ATTN_OK;
}

int attn_fwd_fp8_varlen(const void* q8, const void* k8, const void* vt8, const float* sq, const float* sk,
                        const float* sv, const int* blk_off, const int* cu_seqlens, void* o, float* lse, int nseq,
                        int total, int H, int Hkv, int d, int causal, float scale, int mode, void* stream) {
  if (nseq < 1 || nseq > MAX_VARLEN_SEQS) return api_fail(ATTN_ERR_INVALID_ARG, "nseq must be in [1, 2048]");
  if (total < 0) return api_fail(ATTN_ERR_INVALID_ARG, "total must be >= 0");
  if (H < 1 || Hkv < 1 || H % Hkv != 0) return api_fail(ATTN_ERR_INVALID_ARG, "need H % Hkv == 0");
  if (d != 128) return api_fail(ATTN_ERR_UNSUPPORTED, "the FP8 forward is built for head dim 128");
  if (mode != ATTN_FP8_PER_TENSOR && mode != ATTN_FP8_PER_BLOCK) return api_fail(ATTN_ERR_INVALID_ARG, "unknown FP8 mode");
  if (causal != 0 && causal != 1) return api_fail(ATTN_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (!(scale > 0.f) || !std::isfinite(scale)) return api_fail(ATTN_ERR_INVALID_ARG, "scale must be finite and > 0");
  if ((long long)H * ((long long)total / 128 + nseq + 1) > 0x7fffffffLL)
    return api_fail(ATTN_ERR_INVALID_ARG, "problem too large for int32 indexing");
  if (total == 0) return ATTN_OK;
  if (!q8 || !k8 || !vt8 || !sq || !sk || !sv || !blk_off || !cu_seqlens || !o || !lse)
    return api_fail(ATTN_ERR_INVALID_ARG, "null pointer");
  if (!aligned(q8, 16) || !aligned(k8, 16) || !aligned(vt8, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
      !aligned(sq, 4) || !aligned(sk, 4) || !aligned(sv, 4) || !aligned(blk_off, 4) || !aligned(cu_seqlens, 4))
    return api_fail(ATTN_ERR_INVALID_ARG, "tensors must be 16-byte aligned, scales and indices 4-byte aligned");
  int sm = 0;
  unsigned int* err = nullptr;
  int rc;
  if ((rc = api_device(&sm, &err))) return rc;
  const int tmax = attn_fp8_varlen_tmax(total, nseq);
  CUtensorMap mq, mk, mv;
  if ((rc = api_make_map(&mq, true, q8, d, H, total, 1, 128, 128))) return rc;
  if ((rc = api_make_map(&mk, true, k8, d, Hkv, total, 1, 128, 128))) return rc;
  // V^T codes: [Hkv][d][128 * tmax] read as boxes of (128 keys) x (d channel rows)
  if ((rc = api_make_map_rows(&mv, vt8, 128 * (uint64_t)tmax, d, Hkv, 128, d))) return rc;
  FwdParams p;
  memset(&p, 0, sizeof(p));
  p.o = o;
  p.lse = lse;
  p.cu_seqlens = cu_seqlens;
  p.sq = sq;
  p.sk = sk;
  p.sv = sv;
  p.blk_off = blk_off;
  p.tmax = tmax;
  p.nseq = nseq;
  p.total = total;
  p.H = H;
  p.Hkv = Hkv;
  p.group = H / Hkv;
  p.ntiles = 0;          // counted on the device from cu_seqlens
  p.vt_ld = 128 * tmax;
  p.fp8_block = mode == ATTN_FP8_PER_BLOCK;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.timeout_ns = api_timeout_ns();
  p.err = err;
  // packed sequences store O row by row: the output-map argument is not read
  cudaError_t e = launch_fwd_fp8_d128(mq, mk, mv, mq, p, causal != 0, true, sm, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return api_cuda_fail(e, "attn_fwd_fp8_varlen launch");
  return ATTN_OK;
}

// Same computation as attn_fwd_fp8_auto, for callers that are not allowed to
// allocate device memory: the quantised Q/K/V and their scales go to the
// library's fixed 16 MiB device scratch instead of a caller workspace. Nothing
// here allocates (no cudaMalloc/cudaFree, no allocating library routine).
int attn_fwd_fp8_auto_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                              int Hkv, int N, int d, int causal, float scale, int mode, int rotate,
                              uint64_t hadamard_seed, void* stream) {
  int rc = check_shape(B, H, Hkv, N, d, mode);
  if (rc) return rc;
  const size_t need = fp8_layout(B, H, Hkv, N, d, mode).total;
  if (need > kNoAllocScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "this shape needs %zu bytes of FP8 scratch; the fixed scratch of attn_fwd_fp8_auto_noalloc holds %zu "
             "(use attn_fwd_fp8_auto with a caller workspace)",
             need, kNoAllocScratchBytes);
    return api_fail(ATTN_ERR_INVALID_ARG, msg);
  }
  // reject what the forward step would reject before the shared scratch is touched
  if ((rc = check_fwd_fp8_args(d, causal, scale, o, lse))) return rc;
  void* scratch = nullptr;
  if ((rc = noalloc_scratch(&scratch))) return rc;
  return attn_fwd_fp8_auto(q, k, v, o, lse, scratch, kNoAllocScratchBytes, B, H, Hkv, N, d, causal, scale, mode,
                           rotate, hadamard_seed, stream);
}

}  // extern "C"
