// attn45_api.cu -- the C ABI (include/attn45.h): argument checks, TMA tensor
// map encoding, grid sizing and launches. No allocation happens per call; the
// only device state the library owns is one error word per device (a
// __device__ variable, so nothing is allocated for it either).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "attn45.h"
#include "attn_common.cuh"
#include "api_internal.h"
#include "bwd_launchers.h"
#include "launchers.h"
#include "ptx.cuh"

namespace attn45 {

__device__ unsigned int g_err_word;

namespace {

thread_local char g_msg[512] = "";
unsigned long long g_timeout_ns = 2000000000ull;

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(ATTN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

struct DeviceInfo {
  bool ready = false;
  bool supported = false;
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
  unsigned int* err = nullptr;
};

constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Current device's info, filled once. Returns ATTN_OK or an error code.
int device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_UNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    cudaDeviceProp prop;
    e = cudaGetDeviceProperties(&prop, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
    d.cc_major = prop.major;
    d.cc_minor = prop.minor;
    d.sm_count = prop.multiProcessorCount;
    d.supported = (prop.major == 10 && prop.minor == 3);
    void* sym = nullptr;
    e = cudaGetSymbolAddress(&sym, g_err_word);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
    d.err = static_cast<unsigned int*>(sym);
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled entry point not found");
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    d.ready = true;
  }
  if (!d.supported)
    return fail(ATTN_ERR_UNSUPPORTED, "device %d has compute capability %d.%d; this library needs 10.3 (GB300)",
                dev, d.cc_major, d.cc_minor);
  *out = &d;
  return ATTN_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// 4-D tiled map over a [batch][rows][heads][inner] tensor with dims listed
// innermost first {inner, heads, rows, batch}; box = {box_inner, 1, box_rows,
// 1}; 128-byte swizzle, out-of-bounds rows read as zero.
int make_map(CUtensorMap* m, CUtensorMapDataType dt, int elem_bytes, const void* base, uint64_t inner,
             uint64_t heads, uint64_t rows, uint64_t batch, uint32_t box_inner, uint32_t box_rows) {
  cuuint64_t dims[4] = {inner, heads, rows, batch};
  cuuint64_t strides[3] = {inner * elem_bytes, heads * inner * elem_bytes, rows * heads * inner * elem_bytes};
  cuuint32_t box[4] = {box_inner, 1, box_rows, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, dt, 4, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return ATTN_OK;
}

int check_common(int H, int Hkv, int d, int causal, float scale, int dtype) {
  if (H < 1 || Hkv < 1 || H % Hkv != 0) return fail(ATTN_ERR_INVALID_ARG, "need H >= 1, Hkv >= 1, H %% Hkv == 0 (H=%d Hkv=%d)", H, Hkv);
  if (d != 64 && d != 128 && d != 256) return fail(ATTN_ERR_UNSUPPORTED, "head dim %d not in {64,128,256}", d);
  if (causal != 0 && causal != 1) return fail(ATTN_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(ATTN_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (dtype != ATTN_BF16 && dtype != ATTN_FP16) return fail(ATTN_ERR_INVALID_ARG, "dtype %d unknown", dtype);
  return ATTN_OK;
}

cudaError_t launch_f16(int d, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                       const CUtensorMap& o, const FwdParams& p, bool causal, bool varlen, bool bf16,
                       int sm_count, cudaStream_t s) {
  switch (d) {
    case 64: return launch_fwd_f16_d64(q, k, v, o, p, causal, varlen, bf16, sm_count, s);
    case 128: return launch_fwd_f16_d128(q, k, v, o, p, causal, varlen, bf16, sm_count, s);
    default: return launch_fwd_f16_d256(q, k, v, o, p, causal, varlen, bf16, sm_count, s);
  }
}

__global__ void timeout_probe_kernel(unsigned long long ns, unsigned int* err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, ns, &abort_flag, err);  // nothing ever arrives
  __syncthreads();
}

}  // namespace

// Shared with the FP8 translation unit (api_internal.h).
int api_fail(int code, const char* msg) { return fail(code, "%s", msg); }
int api_cuda_fail(cudaError_t e, const char* what) { return cuda_fail(e, what); }
unsigned long long api_timeout_ns() { return g_timeout_ns; }
int api_device(int* sm_count, unsigned int** err) {
  DeviceInfo* d = nullptr;
  int rc = device_info(&d);
  if (rc) return rc;
  *sm_count = d->sm_count;
  *err = d->err;
  return ATTN_OK;
}
int api_make_map_rows(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t batch,
                      uint32_t box_inner, uint32_t box_rows) {
  // u8 [batch][rows][inner] as {inner, rows, batch, 1}, box {box_inner, box_rows, 1, 1}
  cuuint64_t dims[4] = {inner, rows, batch, 1};
  cuuint64_t strides[3] = {inner, rows * inner, batch * rows * inner};
  cuuint32_t box[4] = {box_inner, box_rows, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return ATTN_OK;
}
int api_make_map(CUtensorMap* m, bool u8, const void* base, uint64_t inner, uint64_t heads, uint64_t rows,
                 uint64_t batch, uint32_t box_inner, uint32_t box_rows) {
  return make_map(m, u8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, u8 ? 1 : 2, base,
                  inner, heads, rows, batch, box_inner, box_rows);
}

}  // namespace attn45

using namespace attn45;

extern "C" {

int attn_version(void) { return 1; }

const char* attn_status_string(int s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

const char* attn_last_error_message(void) { return g_msg; }

int attn_set_wait_timeout_ns(uint64_t ns) {
  if (ns < 1000ull || ns > 60000000000ull) return fail(ATTN_ERR_INVALID_ARG, "timeout %llu ns out of range", (unsigned long long)ns);
  g_timeout_ns = ns;
  return ATTN_OK;
}

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv, int N,
             int d, int causal, float scale, int dtype, void* stream) {
  int rc = check_common(H, Hkv, d, causal, scale, dtype);
  if (rc) return rc;
  if (B < 1 || N < 1) return fail(ATTN_ERR_INVALID_ARG, "need B >= 1 and N >= 1 (B=%d N=%d)", B, N);
  if ((long long)B * N > 0x7fffffffLL || (long long)B * H * ((N + 127) / 128) > 0x7fffffffLL)
    return fail(ATTN_ERR_INVALID_ARG, "problem too large for int32 indexing");
  if (!q || !k || !v || !o || !lse) return fail(ATTN_ERR_INVALID_ARG, "null pointer");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return fail(ATTN_ERR_INVALID_ARG, "q, k, v, o must be 16-byte aligned and lse 4-byte aligned");
  DeviceInfo* dev = nullptr;
  if ((rc = device_info(&dev))) return rc;
  const int bn = f16_block_n(d);
  const CUtensorMapDataType dt = dtype == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap mq, mk, mv, mo;
  if ((rc = make_map(&mq, dt, 2, q, d, H, N, B, 64, BLOCK_M))) return rc;
  if ((rc = make_map(&mk, dt, 2, k, d, Hkv, N, B, 64, bn))) return rc;
  if ((rc = make_map(&mv, dt, 2, v, d, Hkv, N, B, 64, f16_v_box_rows(d)))) return rc;
  // output: 64 columns x 32 rows per bulk store (one warp's rows)
  if ((rc = make_map(&mo, dt, 2, o, d, H, N, B, 64, 32))) return rc;
  FwdParams p;
  memset(&p, 0, sizeof(p));
  p.o = o;
  p.lse = lse;
  p.nseq = B;
  p.N = N;
  p.total = B * N;
  p.H = H;
  p.Hkv = Hkv;
  p.group = H / Hkv;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.timeout_ns = g_timeout_ns;
  p.err = dev->err;
  cudaError_t e = launch_f16(d, mq, mk, mv, mo, p, causal != 0, false, dtype == ATTN_BF16, dev->sm_count,
                             static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "attn_fwd launch");
  return ATTN_OK;
}

int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens,
                    int nseq, int max_seqlen, int total, int H, int Hkv, int d, int causal, float scale,
                    int dtype, void* stream) {
  (void)max_seqlen;
  int rc = check_common(H, Hkv, d, causal, scale, dtype);
  if (rc) return rc;
  if (nseq < 1 || nseq > MAX_VARLEN_SEQS) return fail(ATTN_ERR_INVALID_ARG, "nseq must be in [1, %d]", MAX_VARLEN_SEQS);
  if (total < 0) return fail(ATTN_ERR_INVALID_ARG, "total must be >= 0");
  if ((long long)H * ((long long)total / 128 + nseq + 1) > 0x7fffffffLL)
    return fail(ATTN_ERR_INVALID_ARG, "problem too large for int32 indexing");
  if (!cu_seqlens || !aligned(cu_seqlens, 4)) return fail(ATTN_ERR_INVALID_ARG, "cu_seqlens must be a 4-byte aligned device pointer");
  if (total == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !lse) return fail(ATTN_ERR_INVALID_ARG, "null pointer");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return fail(ATTN_ERR_INVALID_ARG, "q, k, v, o must be 16-byte aligned and lse 4-byte aligned");
  DeviceInfo* dev = nullptr;
  if ((rc = device_info(&dev))) return rc;
  const int bn = f16_block_n(d);
  const CUtensorMapDataType dt = dtype == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap mq, mk, mv;
  if ((rc = make_map(&mq, dt, 2, q, d, H, total, 1, 64, BLOCK_M))) return rc;
  if ((rc = make_map(&mk, dt, 2, k, d, Hkv, total, 1, 64, bn))) return rc;
  if ((rc = make_map(&mv, dt, 2, v, d, Hkv, total, 1, 64, f16_v_box_rows(d)))) return rc;
  FwdParams p;
  memset(&p, 0, sizeof(p));
  p.o = o;
  p.lse = lse;
  p.cu_seqlens = cu_seqlens;
  p.nseq = nseq;
  p.total = total;
  p.H = H;
  p.Hkv = Hkv;
  p.group = H / Hkv;
  p.ntiles = 0;  // computed on the device from cu_seqlens
  p.scale_log2 = scale * 1.4426950408889634f;
  p.timeout_ns = g_timeout_ns;
  p.err = dev->err;
  // varlen stores O row by row (a tile's last rows may belong to the next
  // sequence), so the output-map argument is not read
  cudaError_t e = launch_f16(d, mq, mk, mv, mq, p, causal != 0, true, dtype == ATTN_BF16, dev->sm_count,
                             static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "attn_fwd_varlen launch");
  return ATTN_OK;
}

int attn_decode_num_splits(int B, int Hkv, int Nmax) {
  if (B < 1 || Hkv < 1 || Nmax < 1) return 1;
  DeviceInfo* dev = nullptr;
  const int sm = device_info(&dev) == ATTN_OK ? dev->sm_count : 148;
  // about four units per SM (one CTA per SM walks them; measured best on
  // 8 x 8 KV heads with 1k-32k cached keys), at most one split per 128 keys
  const long long units = (long long)B * Hkv;
  long long s = (4LL * sm + units - 1) / units;
  const long long smax = (Nmax + 127) / 128;
  if (s > smax) s = smax;
  return (int)(s < 1 ? 1 : s);
}

namespace {
// Partial rows the decode workspace holds: num_splits + 1 rows per output row
// (the balanced division leaves at most units + grid - 1 pieces, grid <=
// num_splits * units).
size_t decode_part_rows(int B, int H, int num_splits) { return (size_t)(num_splits + 1) * B * H; }
size_t pad256(size_t x) { return (x + 255) & ~size_t(255); }
}  // namespace

size_t attn_decode_workspace_size(int B, int H, int d, int num_splits) {
  if (B < 1 || H < 1 || d < 1 || num_splits < 1) return 0;
  const size_t rows = decode_part_rows(B, H, num_splits);
  return pad256(rows * d * 4) + pad256(rows * 4) + pad256((size_t)B * H * 8);
}

int attn_combine(const float* o_parts, const float* lse_parts, void* o, float* lse, int num_splits, int rows, int d,
                 int dtype, void* stream) {
  if (num_splits < 1 || rows < 0 || d < 1 || d > 1024) return fail(ATTN_ERR_INVALID_ARG, "need num_splits >= 1, rows >= 0, 1 <= d <= 1024");
  if (dtype != ATTN_BF16 && dtype != ATTN_FP16) return fail(ATTN_ERR_INVALID_ARG, "dtype %d unknown", dtype);
  if (rows == 0) return ATTN_OK;
  if (!o_parts || !lse_parts || !o || !lse) return fail(ATTN_ERR_INVALID_ARG, "null pointer");
  if (!aligned(o_parts, 4) || !aligned(lse_parts, 4) || !aligned(o, 2) || !aligned(lse, 4))
    return fail(ATTN_ERR_INVALID_ARG, "misaligned pointer");
  DeviceInfo* dev = nullptr;
  int rc = device_info(&dev);
  if (rc) return rc;
  cudaError_t e = launch_combine(o_parts, lse_parts, o, lse, num_splits, rows, d, dtype == ATTN_BF16,
                                 static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "attn_combine launch");
  return ATTN_OK;
}

int attn_decode(const void* q, const void* k_cache, const void* v_cache, const int* seqlens, void* o, float* lse,
                void* workspace, size_t workspace_bytes, int B, int H, int Hkv, int Nmax, int d, int num_splits,
                float scale, int dtype, void* stream) {
  int rc = check_common(H, Hkv, d, 0, scale, dtype);
  if (rc) return rc;
  if (d == 256) return fail(ATTN_ERR_UNSUPPORTED, "decode is built for head dims 64 and 128");
  if (H / Hkv > BLOCK_M) return fail(ATTN_ERR_UNSUPPORTED, "at most %d query heads per KV head", BLOCK_M);
  if (B < 1 || Nmax < 1) return fail(ATTN_ERR_INVALID_ARG, "need B >= 1 and Nmax >= 1 (B=%d Nmax=%d)", B, Nmax);
  if (num_splits <= 0) num_splits = attn_decode_num_splits(B, Hkv, Nmax);
  if ((long long)B * Hkv * num_splits > 0x7fffffffLL || (long long)B * Nmax > 0x7fffffffLL)
    return fail(ATTN_ERR_INVALID_ARG, "problem too large for int32 indexing");
  if (!q || !k_cache || !v_cache || !seqlens || !o || !lse || !workspace) return fail(ATTN_ERR_INVALID_ARG, "null pointer");
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
      !aligned(seqlens, 4) || !aligned(workspace, 256))
    return fail(ATTN_ERR_INVALID_ARG, "q, caches, o 16-byte, lse and seqlens 4-byte, workspace 256-byte aligned");
  const size_t need = attn_decode_workspace_size(B, H, d, num_splits);
  if (workspace_bytes < need) return fail(ATTN_ERR_INVALID_ARG, "workspace of %zu bytes < %zu needed", workspace_bytes, need);
  DeviceInfo* dev = nullptr;
  if ((rc = device_info(&dev))) return rc;
  const CUtensorMapDataType dt = dtype == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const bool bf16 = dtype == ATTN_BF16;
  const int group = H / Hkv;
  CUtensorMap mq, mk, mv;
  if ((rc = make_map(&mk, dt, 2, k_cache, d, Hkv, Nmax, B, 64, 128))) return rc;
  if ((rc = make_map(&mv, dt, 2, v_cache, d, Hkv, Nmax, B, 64, 128))) return rc;
  const size_t part_rows = decode_part_rows(B, H, num_splits);
  float* o_parts = static_cast<float*>(workspace);
  float* lse_parts = reinterpret_cast<float*>(static_cast<char*>(workspace) + pad256(part_rows * d * 4));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (decode_kt_supported(d, group)) {
    // q [B*H][d] in boxes of 16 or 32 rows: the group's rows (and zero-weighted neighbours)
    if ((rc = make_map(&mq, dt, 2, q, d, 1, (uint64_t)B * H, 1, 64, decode_kt_q_rows(group)))) return rc;
    static std::atomic<unsigned int> epoch{0};
    DecodeParams p;
    memset(&p, 0, sizeof(p));
    p.o_parts = o_parts;
    p.lse_parts = lse_parts;
    p.counters = reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(lse_parts) + pad256(part_rows * 4));
    p.o = o;
    p.lse = lse;
    p.seqlens = seqlens;
    p.B = B;
    p.H = H;
    p.Hkv = Hkv;
    p.group = group;
    p.Nmax = Nmax;
    do p.epoch = ++epoch; while (p.epoch == 0);
    p.scale_log2 = scale * 1.4426950408889634f;
    p.timeout_ns = g_timeout_ns;
    p.err = dev->err;
    const long long units = (long long)B * Hkv;
    const int grid = (int)std::min<long long>(std::min(dev->sm_count, DECODE_KT_MAX_GRID), (long long)num_splits * units);
    cudaError_t e = launch_decode_kt(mq, mk, mv, p, d, grid, bf16, st);
    if (e != cudaSuccess) return cuda_fail(e, "attn_decode launch");
    return ATTN_OK;
  }
  // q [B][H][d] as rows of one "head": the query heads of a KV head are rows
  if ((rc = make_map(&mq, dt, 2, q, d, 1, H, B, 64, BLOCK_M))) return rc;
  int chunk = (Nmax + num_splits - 1) / num_splits;
  chunk = (chunk + 127) / 128 * 128;
  FwdParams p;
  memset(&p, 0, sizeof(p));
  p.o = o_parts;
  p.lse = lse_parts;
  p.nseq = B;
  p.N = Nmax;
  p.total = B * Nmax;
  p.H = H;
  p.Hkv = Hkv;
  p.group = group;
  p.ntiles = B * Hkv * num_splits;
  p.seqlens = seqlens;
  p.num_splits = num_splits;
  p.split_chunk = chunk;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.timeout_ns = g_timeout_ns;
  p.err = dev->err;
  cudaError_t e = launch_decode_f16(d, mq, mk, mv, p, bf16, dev->sm_count, st);
  if (e != cudaSuccess) return cuda_fail(e, "attn_decode launch");
  e = launch_combine(o_parts, lse_parts, o, lse, num_splits, B * H, d, bf16, st);
  if (e != cudaSuccess) return cuda_fail(e, "attn_decode combine launch");
  return ATTN_OK;
}

size_t attn_bwd_workspace_size(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
  const size_t rows = (size_t)B * N * H;
  return ((rows * d * 4 + 255) & ~size_t(255)) + ((rows * 4 + 255) & ~size_t(255));
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout, void* dq,
             void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int H, int Hkv, int N, int d,
             int causal, float scale, int dtype, void* stream) {
  int rc = check_common(H, Hkv, d, causal, scale, dtype);
  if (rc) return rc;
  if (d == 256) return fail(ATTN_ERR_UNSUPPORTED, "the backward is built for head dims 64 and 128");
  if (B < 1 || N < 1) return fail(ATTN_ERR_INVALID_ARG, "need B >= 1 and N >= 1 (B=%d N=%d)", B, N);
  if ((long long)B * N * H > 0x7fffffffLL) return fail(ATTN_ERR_INVALID_ARG, "problem too large for int32 indexing");
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace) return fail(ATTN_ERR_INVALID_ARG, "null pointer");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dout, 16) ||
      !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4) || !aligned(workspace, 256))
    return fail(ATTN_ERR_INVALID_ARG, "tensors 16-byte, lse 4-byte, workspace 256-byte aligned");
  const size_t need = attn_bwd_workspace_size(B, H, N, d);
  if (workspace_bytes < need) return fail(ATTN_ERR_INVALID_ARG, "workspace of %zu bytes < %zu needed", workspace_bytes, need);
  DeviceInfo* dev = nullptr;
  if ((rc = device_info(&dev))) return rc;
  const CUtensorMapDataType dt = dtype == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap mq, mk, mv, mdo;
  if ((rc = make_map(&mq, dt, 2, q, d, H, N, B, 64, 128))) return rc;
  if ((rc = make_map(&mk, dt, 2, k, d, Hkv, N, B, 64, 128))) return rc;
  if ((rc = make_map(&mv, dt, 2, v, d, Hkv, N, B, 64, 128))) return rc;
  if ((rc = make_map(&mdo, dt, 2, dout, d, H, N, B, 64, 128))) return rc;
  const size_t rows = (size_t)B * N * H;
  float* dq_acc = static_cast<float*>(workspace);
  float* dvec = reinterpret_cast<float*>(static_cast<char*>(workspace) + ((rows * d * 4 + 255) & ~size_t(255)));
  CUtensorMap mdq;
  if ((rc = make_map(&mdq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dq_acc, d, H, N, B, 32, 128))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool bf16 = dtype == ATTN_BF16;
  cudaError_t e = cudaMemsetAsync(dq_acc, 0, rows * d * 4, st);
  if (e != cudaSuccess) return cuda_fail(e, "zeroing the dQ accumulator");
  e = launch_bwd_dvec(d, o, dout, dvec, B, N, H, bf16, st);
  if (e != cudaSuccess) return cuda_fail(e, "attn_bwd row-sum launch");
  BwdParams p;
  memset(&p, 0, sizeof(p));
  p.lse = lse;
  p.dvec = dvec;
  p.dq_acc = dq_acc;
  p.dk = dk;
  p.dv = dv;
  p.B = B;
  p.N = N;
  p.H = H;
  p.Hkv = Hkv;
  p.group = H / Hkv;
  p.nunits = B * Hkv * ((N + 127) / 128);
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.timeout_ns = g_timeout_ns;
  p.err = dev->err;
  e = launch_bwd(d, mq, mk, mv, mdo, mdq, p, causal != 0, bf16, dev->sm_count, st);
  if (e != cudaSuccess) return cuda_fail(e, "attn_bwd launch");
  e = launch_bwd_dq_convert(dq_acc, dq, (long long)rows * d, bf16, st);
  if (e != cudaSuccess) return cuda_fail(e, "attn_bwd dQ conversion launch");
  return ATTN_OK;
}

int attn_get_device_error(void* stream) {
  DeviceInfo* dev = nullptr;
  int rc = device_info(&dev);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned int word = 0;
  e = cudaMemcpyFromSymbol(&word, g_err_word, sizeof(word));
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  if (word) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_err_word, &zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
    if (word & DEV_ERR_TIMEOUT) return fail(ATTN_ERR_TIMEOUT, "a device-side wait exceeded its bound");
  }
  return ATTN_OK;
}

int attn_debug_timeout_probe(uint64_t ns, void* stream) {
  if (ns < 1000ull || ns > 60000000000ull) return fail(ATTN_ERR_INVALID_ARG, "timeout out of range");
  DeviceInfo* dev = nullptr;
  int rc = device_info(&dev);
  if (rc) return rc;
  timeout_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(ns, dev->err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "timeout probe launch");
  return ATTN_OK;
}

}  // extern "C"
