/*
 * attn45.h -- C ABI of the GB300 (sm_103a) fused exact attention forward
 * library, libattn45.so.
 *
 * What is computed ("FlashAttention: Fast and Memory-Efficient Exact
 * Attention with IO-Awareness", abstract: exact attention, tiled so the score
 * matrix never goes to HBM; "FlashAttention-3: Fast and Accurate Attention
 * with Asynchrony and Low-precision", abstract: the same layer with
 * asynchronous data movement and an FP8 path):
 *
 *   O[i,h,:]  = sum_j softmax_j(scale * q[i,h,:] . k[j,hk,:]) v[j,hk,:]
 *   lse[h,i]  = ln sum_j exp(scale * q[i,h,:] . k[j,hk,:])
 *
 * over the keys j of row i's own sequence (j <= i when causal), with kv head
 * hk = h / (H / Hkv): H/Hkv consecutive query heads share one K/V head
 * (grouped-query / multi-query attention).
 *
 * Conventions for every call
 *  - All tensor pointers are DEVICE pointers owned by the caller, 16-byte
 *    aligned, contiguous in the layouts stated per call. The library never
 *    frees or keeps them.
 *  - Every call is asynchronous on `stream` (a cudaStream_t passed as void*,
 *    NULL = legacy default stream) and never synchronises the host, except
 *    attn_get_device_error().
 *  - Head dim d must be 64, 128 or 256; H % Hkv == 0; scale > 0 and finite.
 *  - Errors are returned as attn_status codes, never thrown or trapped; a
 *    one-line description of the last failing call on this thread is
 *    available from attn_last_error_message().
 *  - Every device-side wait is bounded. If one gives up (a bug, never
 *    expected), the kernel sets a device error word and exits cleanly;
 *    attn_get_device_error() reports it as ATTN_ERR_TIMEOUT.
 *  - Needs a compute capability 10.3 (GB300) device: ATTN_ERR_UNSUPPORTED
 *    otherwise.
 */
#ifndef ATTN45_H
#define ATTN45_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ATTN45_API __attribute__((visibility("default")))
#else
#define ATTN45_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1, /* bad pointer, alignment, shape or value */
  ATTN_ERR_UNSUPPORTED = 2, /* valid request this build does not serve (device, head dim) */
  ATTN_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
  ATTN_ERR_TIMEOUT = 4      /* a device-side bounded wait gave up */
} attn_status;

typedef enum { ATTN_BF16 = 0, ATTN_FP16 = 1 } attn_dtype;

typedef enum {
  ATTN_FP8_PER_TENSOR = 0, /* one scale per tensor for Q, K and V */
  ATTN_FP8_PER_BLOCK = 1   /* Q, K: one scale per (b, head, 128-row block); V: per (b, kv head, channel) */
} attn_fp8_mode;

/*
 * attn_fwd -- fixed-length BF16/FP16 forward.
 *   q   [B, N, H,   d]  dtype (BSHD, contiguous)
 *   k,v [B, N, Hkv, d]  dtype
 *   o   [B, N, H,   d]  dtype, written
 *   lse [B, H, N]       fp32, natural-log logsumexp of the scaled scores, written
 *   causal: 0 or 1 (row i attends keys j <= i).
 * B, N >= 1 (B*N*H must fit in int32).
 */
ATTN45_API int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv, int N,
             int d, int causal, float scale, int dtype, void* stream);

/*
 * attn_fwd_varlen -- packed variable-length BF16/FP16 forward.
 *   q [total, H, d], k,v [total, Hkv, d], o [total, H, d] (THD, contiguous);
 *   lse [H, total] fp32;
 *   cu_seqlens: DEVICE int32[nseq+1], cu_seqlens[0] = 0, non-decreasing,
 *   cu_seqlens[nseq] = total; sequence s owns tokens [cu[s], cu[s+1]).
 *   Causal masking is per sequence (local row i attends local keys j <= i).
 *   1 <= nseq <= 2048. max_seqlen is accepted for interface symmetry and
 *   unused. Empty sequences are allowed. Rows of each sequence see only keys
 *   of that sequence.
 */
ATTN45_API int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens,
                    int nseq, int max_seqlen, int total, int H, int Hkv, int d, int causal, float scale,
                    int dtype, void* stream);

/*
 * FP8 (e4m3) path. "FlashAttention-3 ...", abstract technique (3): block
 * quantization plus incoherent processing (Q and K multiplied by a random
 * orthogonal matrix, which leaves Q K^T unchanged and spreads outliers).
 *
 * attn_fp8_prepass -- quantise BF16 Q, K, V (BSHD as in attn_fwd).
 *   rotate != 0: Q and K rows are first mapped x -> (x * sigma) H_d / sqrt(d)
 *     (Sylvester Hadamard H_d, butterfly stages of span 1, 2, ..., d/2 in
 *     fp32; sigma_c = 1 - 2 * (splitmix64(hadamard_seed + c) & 1), the same
 *     signs for every batch and head). V is never rotated.
 *   scale = amax / 448 (1 when amax = 0); code = e4m3 RNE-satfinite(x / scale).
 *   Outputs (device, caller-owned):
 *     q8 [B,N,H,d], k8 [B,N,Hkv,d] uint8 e4m3 codes;
 *     vt8 [B,Hkv,d,ldv] uint8: V codes transposed (keys contiguous),
 *         ldv = attn_fp8_vt_ld(N) (padding columns written as 0);
 *     mode PER_BLOCK:  sq [B,H,ceil(N/128)], sk [B,Hkv,ceil(N/128)], sv [B,Hkv,d] fp32;
 *     mode PER_TENSOR: sq, sk, sv each one fp32.
 *   sv is also used as scratch for the per-channel amax during the call.
 */
ATTN45_API int attn_fp8_vt_ld(int N);
ATTN45_API int attn_fp8_prepass(const void* q, const void* k, const void* v, void* q8, void* k8, void* vt8, float* sq,
                     float* sk, float* sv, int B, int H, int Hkv, int N, int d, int mode, int rotate,
                     uint64_t hadamard_seed, void* stream);

/*
 * attn_fwd_fp8 -- forward on pre-pass outputs (same layouts as above).
 *   o [B,N,H,d] BF16 and lse [B,H,N] fp32 (of the scaled, dequantised scores).
 *   Online softmax over 128-key blocks with a lazy running maximum m: m is
 *   raised only when a block's maximum exceeds it by more than 8 (log2
 *   units), so every p = 2^(t - m) is <= 2^8. p is rounded to e4m3 with no
 *   extra multiplier (codes <= 256 < 448, never saturated) for the P*V
 *   product; the row normaliser sums the unrounded p. d = 64, 128 or 256
 *   (256 runs on pairs of CTAs that share each tensor-core product; 64 runs
 *   on the head-dim-128 kernel, whose copies zero-fill channels 64-127).
 */
ATTN45_API int attn_fwd_fp8(const void* q8, const void* k8, const void* vt8, const float* sq, const float* sk,
                 const float* sv, void* o, float* lse, int B, int H, int Hkv, int N, int d, int causal,
                 float scale, int mode, void* stream);

/*
 * attn_fwd_fp8_auto -- pre-pass + FP8 forward in one call, with the
 * quantised tensors placed in a caller-provided device workspace of at least
 * attn_fp8_workspace_size() bytes (256-byte aligned). Every argument the
 * forward step checks (causal, scale, o, lse) is checked before the
 * pre-pass runs, so a rejected call writes nothing.
 */
ATTN45_API size_t attn_fp8_workspace_size(int B, int H, int Hkv, int N, int d, int mode);
ATTN45_API int attn_fwd_fp8_auto(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
                      size_t workspace_bytes, int B, int H, int Hkv, int N, int d, int causal, float scale,
                      int mode, int rotate, uint64_t hadamard_seed, void* stream);

/*
 * attn_fwd_fp8_auto_noalloc -- attn_fwd_fp8_auto for callers that may not
 * allocate device memory (for example a host framework that owns every byte
 * of device memory through its own pool and forbids cudaMalloc/cudaFree,
 * whose implicit device-wide synchronisation and possible out-of-memory
 * failure it cannot accept on its request path). Nothing in the pages has a
 * counterpart to this call; it is an interface convenience.
 *   Same arguments, layouts and results as attn_fwd_fp8_auto, without the
 *   workspace: the quantised tensors live in one fixed device scratch array
 *   of 16 MiB (16777216 bytes) inside this library, which every GPU that
 *   loads the library holds until the process exits. Shapes whose
 *   attn_fp8_workspace_size() exceeds that return ATTN_ERR_INVALID_ARG.
 *   The first call on a device looks up the scratch address for that device
 *   (with it current); make that first call before any stream capture.
 *   Every call uses the same scratch: calls that may overlap on the GPU
 *   (different streams, or several host threads) race and must be
 *   serialised by the caller. Parts that must start at zero are cleared by
 *   each call. Allocates nothing.
 */
/*   Arguments are checked as in attn_fwd_fp8_auto before the scratch is
 *   looked up or written. */
ATTN45_API int attn_fwd_fp8_auto_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                                         int H, int Hkv, int N, int d, int causal, float scale, int mode, int rotate,
                                         uint64_t hadamard_seed, void* stream);

/*
 * FP8 over packed variable-length sequences (THD, as attn_fwd_varlen).
 * Every sequence is quantised on its own (128-row blocks never cross a
 * sequence boundary; V's channel scales are per (sequence, KV head)).
 *   tmax = attn_fp8_varlen_tmax(total, nseq) = ceil(total/128) + nseq bounds
 *   the number of 128-row blocks over all sequences.
 * attn_fp8_prepass_varlen -- bf16 q [total,H,d], k, v [total,Hkv,d] ->
 *   q8 [total,H,d], k8 [total,Hkv,d] (e4m3 codes); vt8 [Hkv, d, 128*tmax]
 *   (V codes transposed, sequence s's keys from column 128*blk_off[s], the
 *   pad keys of its last block code 0; columns from 128*blk_off[nseq] on are
 *   neither written nor read); block mode: sq [H, tmax],
 *   sk [Hkv, tmax] (sequence s's block b in column blk_off[s] + b),
 *   sv [nseq, Hkv, d]; tensor mode: sq, sk, sv one float each; blk_off:
 *   DEVICE int32 [nseq+1] written here, blk_off[s] = sum over s' < s of
 *   ceil(n_s'/128). d in {64, 128, 256}; cu_seqlens as in attn_fwd_varlen.
 *   d = 128 runs the head-dim-128 kernels of attn_fp8_prepass (TMA loads of
 *   128-row blocks starting at each sequence's rows, codes of the sequence's
 *   own rows stored from registers); d = 64, 256 the generic kernels.
 * attn_fwd_fp8_varlen -- the FP8 forward over those outputs (d = 128):
 *   o [total, H, d] bf16, lse [H, total] fp32; causal masking per sequence.
 */
ATTN45_API int attn_fp8_varlen_tmax(int total, int nseq);
ATTN45_API int attn_fp8_prepass_varlen(const void* q, const void* k, const void* v, const int* cu_seqlens, void* q8,
                                       void* k8, void* vt8, float* sq, float* sk, float* sv, int* blk_off, int nseq,
                                       int total, int H, int Hkv, int d, int mode, int rotate, uint64_t hadamard_seed,
                                       void* stream);
ATTN45_API int attn_fwd_fp8_varlen(const void* q8, const void* k8, const void* vt8, const float* sq, const float* sk,
                                   const float* sv, const int* blk_off, const int* cu_seqlens, void* o, float* lse,
                                   int nseq, int total, int H, int Hkv, int d, int causal, float scale, int mode,
                                   void* stream);

/*
 * Split-KV decode: one query token per sequence and query head attends to
 * the first seqlens[b] keys of its KV head's cache (the decode phase of
 * "FlashAttention-3 ..." references [49] and [51]; the merge of partial
 * results is the online-softmax rescaling of the "Related papers:
 * FlashAttention-4" page's online-softmax teaser, applied across splits).
 *
 * attn_decode -- BF16/FP16, head dim 64 or 128, H % Hkv == 0, H/Hkv <= 128.
 *   q [B, H, d]; k_cache, v_cache [B, Nmax, Hkv, d] (BSHD, contiguous);
 *   seqlens: DEVICE int32[B], keys cached per sequence (values are clamped to
 *   [0, Nmax]; 0 gives o = 0 and lse = -inf); o [B, H, d] in q's dtype;
 *   lse [B, H] fp32 (natural log, scale included).
 *   H/Hkv in 1..16, 24 or 32 (one kernel launch, head dim 64 or 128): the 128-key tiles of
 *   all (sequence, KV head) pairs are divided evenly between min(SMs, 256,
 *   num_splits * B * Hkv) persistent CTAs, whatever the length mix; each CTA
 *   puts the keys on the tensor core's 128 rows (S^T = K Q^T,
 *   O^T += V^T P^T) and clears the V rows at or past seqlens[b], so those
 *   rows may hold anything. A pair held by one CTA is written directly;
 *   otherwise each CTA leaves a partial result in `workspace` and the last
 *   one to finish (a per-pair counter tagged with a per-call epoch) merges
 *   them. Other groups: the cache of every sequence is cut into num_splits
 *   ranges of ceil(Nmax / num_splits) keys rounded up to 128, each (sequence,
 *   KV head, range) a unit of the forward kernel with the query heads as
 *   rows, where rows past seqlens[b] meet P = 0 in the product and must be
 *   finite; a second kernel merges the partials. The merge is the
 *   online-softmax rescaling: lse = m + ln sum_s e^(lse_s - m),
 *   O = sum_s e^(lse_s - lse) O_s. num_splits <= 0 picks
 *   attn_decode_num_splits().
 *   workspace: DEVICE, 256-byte aligned, >= attn_decode_workspace_size(B, H,
 *   d, num_splits) bytes, owned by the caller, used by one call at a time;
 *   its contents are scratch (no initialisation needed).
 */
ATTN45_API int attn_decode(const void* q, const void* k_cache, const void* v_cache, const int* seqlens, void* o,
                           float* lse, void* workspace, size_t workspace_bytes, int B, int H, int Hkv, int Nmax,
                           int d, int num_splits, float scale, int dtype, void* stream);
/* Splits attn_decode picks for num_splits <= 0: about four (sequence, KV
 * head, range) units per SM, at most one split per 128 cached keys. With the
 * persistent keys-as-rows kernel the value only bounds its grid
 * (min(SMs, 256, num_splits * B * Hkv)) and the workspace. */
ATTN45_API int attn_decode_num_splits(int B, int Hkv, int Nmax);
/* Bytes of attn_decode's workspace: fp32 partial O [(num_splits + 1) B H][d],
 * partial lse [(num_splits + 1) B H], per-pair counters uint64 [B H], each
 * padded to 256 bytes; 0 for bad sizes. */
ATTN45_API size_t attn_decode_workspace_size(int B, int H, int d, int num_splits);
/*
 * attn_combine -- merge results computed over disjoint key subsets:
 *   o_parts [num_splits][rows][d] fp32, lse_parts [num_splits][rows] fp32
 *   (DEVICE) -> o [rows][d] (dtype: ATTN_BF16 / ATTN_FP16), lse [rows] fp32:
 *   lse = m + ln sum_s exp(lse_s - m) (m = max_s lse_s),
 *   o = sum_s exp(lse_s - lse) o_s. A part with lse_s = -inf is skipped
 *   without reading its o_s; if every part is empty, o = 0 and lse = -inf.
 *   1 <= d <= 1024; o 2-byte, other pointers 4-byte aligned.
 */
ATTN45_API int attn_combine(const float* o_parts, const float* lse_parts, void* o, float* lse, int num_splits,
                            int rows, int d, int dtype, void* stream);

/*
 * attn_bwd -- gradients of sum(dO * O) for the BF16/FP16 forward (head dim 64
 * or 128, fixed length, causal or not, H % Hkv == 0). The backward pass of the
 * FlashAttention papers: P is recomputed from S and the forward's lse;
 * dV = P^T dO, dS = scale P (dO V^T - rowsum(dO * O)), dK = dS^T Q, dQ = dS K;
 * dK, dV of a KV head sum over its query heads.
 *   q, o, dout [B, N, H, d]; k, v [B, N, Hkv, d] (BSHD, the forward's inputs
 *   and output); lse [B, H, N] fp32 as the forward wrote it; dq [B, N, H, d],
 *   dk, dv [B, N, Hkv, d] outputs in the input dtype.
 *   workspace: DEVICE, 256-byte aligned, >= attn_bwd_workspace_size(B, H, N,
 *   d) bytes (an fp32 dQ accumulator and the row sums), owned by the caller.
 *   Launches: a row-sum kernel, the main kernel (one CTA per (batch, KV head,
 *   128-key block) unit: five tcgen05 GEMMs per query block, dK/dV kept in
 *   TMEM, dQ added into the fp32 accumulator), a dQ conversion kernel.
 */
ATTN45_API int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                        const void* dout, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                        int B, int H, int Hkv, int N, int d, int causal, float scale, int dtype, void* stream);
/* Bytes of attn_bwd's workspace: fp32 [B,N,H,d] then fp32 [B,H,N], each
 * padded to 256 bytes; 0 for bad sizes. */
ATTN45_API size_t attn_bwd_workspace_size(int B, int H, int N, int d);

/* Synchronises `stream`, reads and clears the current device's error word.
 * ATTN_OK, ATTN_ERR_TIMEOUT (a bounded device wait gave up) or ATTN_ERR_CUDA. */
ATTN45_API int attn_get_device_error(void* stream);

/* Bound for every device-side wait, in nanoseconds (default 2e9). Values
 * outside [1e3, 6e10] are rejected with ATTN_ERR_INVALID_ARG. */
ATTN45_API int attn_set_wait_timeout_ns(uint64_t ns);

/* Test hook for the bounded-wait machinery: launches one CTA that waits on a
 * barrier nothing will ever complete, with the given bound. Returns ATTN_OK
 * once launched; the caller then sees ATTN_ERR_TIMEOUT from
 * attn_get_device_error(). No fault, trap or hang is involved. */
ATTN45_API int attn_debug_timeout_probe(uint64_t ns, void* stream);

ATTN45_API const char* attn_status_string(int status);
ATTN45_API const char* attn_last_error_message(void);
ATTN45_API int attn_version(void);

#ifdef __cplusplus
}
#endif
#endif /* ATTN45_H */
