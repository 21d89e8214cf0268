// attn_fp8_api.cu -- C ABI of the FP8 path (pre-pass and FP8 forward).
#include "../../include/attn45.h"
#include "api_internal.h"

using namespace attn45;

extern "C" {

int attn_fp8_vt_ld(int N) { return N <= 0 ? 0 : ((N + 127) / 128) * 128; }

size_t attn_fp8_workspace_size(int B, int H, int Hkv, int N, int d, int mode) {
  (void)B; (void)H; (void)Hkv; (void)N; (void)d; (void)mode;
  return 0;
}

int attn_fp8_prepass(const void*, const void*, const void*, void*, void*, void*, float*, float*, float*, int, int,
                     int, int, int, int, int, uint64_t, void*) {
  return api_fail(ATTN_ERR_UNSUPPORTED, "FP8 pre-pass not built yet");
}

int attn_fwd_fp8(const void*, const void*, const void*, const float*, const float*, const float*, void*, float*,
                 int, int, int, int, int, int, float, int, void*) {
  return api_fail(ATTN_ERR_UNSUPPORTED, "FP8 forward not built yet");
}

int attn_fwd_fp8_auto(const void*, const void*, const void*, void*, float*, void*, size_t, int, int, int, int, int,
                      int, float, int, int, uint64_t, void*) {
  return api_fail(ATTN_ERR_UNSUPPORTED, "FP8 forward not built yet");
}

}  // extern "C"
