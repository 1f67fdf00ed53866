// The GPU side of one continuous-batching iteration in one call.
//
// "Deep Dive: continuous batching", sections Iteration-level scheduling and
// The prefill/decode mix: every iteration runs the new tokens' cache writes,
// the prompt chunks' prefill attention and the running requests' decode
// attention over one rebuilt batch. pkv_iteration_prepare writes the batch's
// metadata into one host buffer; once the caller has copied it to the
// device, this call launches, in stream order, the copy-on-write copies, the
// append of every new token, the prefill and the decode, reading each
// kernel's arrays from that one device buffer. It adds no kernel of its own:
// it only saves the host the per-kernel argument handling of separate calls.
#include <cstdint>

#include "internal.h"

using pkv::fail;
using pkv::ok;

extern "C" int pkv_iteration_run(const void* meta, const pkv_iteration_layout* layout,
                                 int32_t n_prefill, int32_t n_decode,
                                 int32_t max_blocks_per_seq, const void* q, const void* k_new,
                                 const void* v_new, void* out, void* k_cache, void* v_cache,
                                 int32_t num_blocks, int32_t Hq, int32_t Hkv, int32_t D,
                                 int32_t block_size, float scale, int32_t partition_size,
                                 void* decode_ws, size_t decode_ws_bytes, void* prefill_ws,
                                 size_t prefill_ws_bytes, int32_t* dev_status, void* stream) {
  const char* who = "pkv_iteration_run";
  PKV_REQUIRE(layout, "%s: layout is NULL", who);
  PKV_REQUIRE(n_prefill >= 0 && n_decode >= 0 && max_blocks_per_seq > 0, "%s: bad sizes", who);
  const int32_t T = layout->n_tokens;
  if (T == 0 && layout->n_cow == 0) return ok();
  PKV_REQUIRE(meta, "%s: meta is NULL", who);
  PKV_REQUIRE(Hkv > 0 && Hq > 0 && Hq % Hkv == 0 && D > 0, "%s: bad head shape", who);
  const uint8_t* m = static_cast<const uint8_t*>(meta);
  auto sec = [m](int64_t off) { return reinterpret_cast<const int32_t*>(m + off); };
  if (layout->n_cow > 0) {
    if (int rc = pkv_block_copy(k_cache, v_cache, sec(layout->cow_pairs), layout->n_cow,
                                num_blocks, Hkv, D, block_size, dev_status, stream))
      return rc;
  }
  if (T > 0) {
    if (int rc = pkv_kv_append(k_new, v_new, sec(layout->slot_mapping), T, k_cache, v_cache,
                               num_blocks, Hkv, D, block_size, dev_status, stream))
      return rc;
  }
  // prefill rows come first in q and out, one per prompt token
  const int32_t n_pre_rows = T - n_decode;
  const size_t row_bytes = (size_t)Hq * D * 2;
  if (n_prefill > 0) {
    if (int rc = pkv_paged_attention_prefill(
            out, q, sec(layout->cu_q_lens), sec(layout->prefill_lens), k_cache, v_cache,
            sec(layout->prefill_tables), max_blocks_per_seq, n_prefill, n_pre_rows,
            layout->max_q_len, layout->max_prefill_len, Hq, Hkv, D, block_size, num_blocks,
            scale, prefill_ws, prefill_ws_bytes, dev_status, stream))
      return rc;
  }
  if (n_decode > 0) {
    if (int rc = pkv_paged_attention_decode(
            static_cast<uint8_t*>(out) + (size_t)n_pre_rows * row_bytes,
            static_cast<const uint8_t*>(q) + (size_t)n_pre_rows * row_bytes, k_cache, v_cache,
            sec(layout->decode_tables), max_blocks_per_seq, sec(layout->decode_lens),
            layout->max_decode_len, n_decode, Hq, Hkv, D, block_size, num_blocks, scale,
            partition_size, decode_ws, decode_ws_bytes, dev_status, stream))
      return rc;
  }
  return ok();
}
