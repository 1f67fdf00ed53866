// paged_attention_prefill (placeholder until the tcgen05 kernel lands).
#include "device.cuh"
#include "host_util.h"

extern "C" int pkv_prefill_workspace_bytes(int32_t S, int32_t total_q, int32_t Hq, int32_t D,
                                           size_t* out) {
  PKV_REQUIRE(out, "pkv_prefill_workspace_bytes: out is NULL");
  *out = 256;
  return pkv::ok();
}

extern "C" int pkv_paged_attention_prefill(void*, const void*, const int32_t*, const int32_t*,
                                           const void*, const void*, const int32_t*, int32_t,
                                           int32_t, int32_t, int32_t, int32_t, int32_t, int32_t,
                                           int32_t, int32_t, int32_t, float, void*, size_t,
                                           int32_t*, void*) {
  return pkv::fail(PKV_EINVAL, "pkv_paged_attention_prefill: not built yet");
}
