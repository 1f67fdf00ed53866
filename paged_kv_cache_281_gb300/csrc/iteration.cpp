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
//
// The prefill and the decode of one iteration touch different sequences and
// only read the cache the append wrote, so they run side by side: the
// prefill on a second stream of the library's (one per device) forked from
// the caller's stream after the append and joined back into it after the
// prefill. The prefill is tensor-bound and the decode HBM-bound, so each
// fills what the other leaves idle, and the calls' starts and last waves
// overlap.
#include <cstdint>
#include <mutex>

#include "host_util.h"

using pkv::fail;
using pkv::ok;

namespace {

// The second stream of a device and the events that fork it from and join it
// into the caller's stream. The mutex keeps one call's record / wait pairs
// together when several host threads launch on the same device.
struct SideStream {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  std::mutex mu;
};
constexpr int kMaxDevices = 64;
SideStream g_side[kMaxDevices];

int side_stream(SideStream** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return pkv::cuda_fail(err, "pkv_iteration_run: current device");
  if (dev < 0 || dev >= kMaxDevices) return fail(PKV_ECUDA, "pkv_iteration_run: device %d", dev);
  SideStream& sd = g_side[dev];
  std::call_once(sd.once, [&sd]() {
    sd.err = cudaStreamCreateWithFlags(&sd.stream, cudaStreamNonBlocking);
    if (sd.err == cudaSuccess) sd.err = cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming);
    if (sd.err == cudaSuccess) sd.err = cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming);
  });
  if (sd.err != cudaSuccess) return pkv::cuda_fail(sd.err, "pkv_iteration_run: side stream");
  *out = &sd;
  return PKV_OK;
}

}  // namespace

extern "C" int pkv_iteration_run(const void* meta, const pkv_iteration_layout* layout,
                                 int32_t n_prefill, int32_t n_decode, const void* q,
                                 const void* k_new,
                                 const void* v_new, void* out, void* k_cache, void* v_cache,
                                 int32_t num_blocks, int32_t Hq, int32_t Hkv, int32_t D,
                                 int32_t block_size, float scale, int32_t partition_size,
                                 void* decode_ws, size_t decode_ws_bytes, void* prefill_ws,
                                 size_t prefill_ws_bytes, int32_t* dev_status, void* stream) {
  const char* who = "pkv_iteration_run";
  PKV_REQUIRE(layout, "%s: layout is NULL", who);
  PKV_REQUIRE(n_prefill >= 0 && n_decode >= 0, "%s: bad sizes", who);
  const int32_t T = layout->n_tokens;
  if (T == 0 && layout->n_cow == 0) return ok();
  PKV_REQUIRE(meta, "%s: meta is NULL", who);
  const int32_t max_blocks_per_seq = layout->table_width;
  PKV_REQUIRE(max_blocks_per_seq > 0, "%s: layout has no table width", who);
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
  auto prefill = [&](void* on) {
    return pkv_paged_attention_prefill(
        out, q, sec(layout->cu_q_lens), sec(layout->prefill_lens), k_cache, v_cache,
        sec(layout->prefill_tables), max_blocks_per_seq, n_prefill, n_pre_rows,
        layout->max_q_len, layout->max_prefill_len, Hq, Hkv, D, block_size, num_blocks, scale,
        prefill_ws, prefill_ws_bytes, dev_status, on);
  };
  auto decode = [&]() {
    return pkv_paged_attention_decode(
        static_cast<uint8_t*>(out) + (size_t)n_pre_rows * row_bytes,
        static_cast<const uint8_t*>(q) + (size_t)n_pre_rows * row_bytes, k_cache, v_cache,
        sec(layout->decode_tables), max_blocks_per_seq, sec(layout->decode_lens),
        layout->max_decode_len, n_decode, Hq, Hkv, D, block_size, num_blocks, scale,
        partition_size, decode_ws, decode_ws_bytes, dev_status, stream);
  };
  if (n_prefill == 0 || n_decode == 0) {
    if (n_prefill > 0)
      if (int rc = prefill(stream)) return rc;
    if (n_decode > 0)
      if (int rc = decode()) return rc;
    return ok();
  }
  SideStream* sd = nullptr;
  if (int rc = side_stream(&sd)) return rc;
  cudaStream_t caller = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(sd->mu);
  cudaError_t err = cudaEventRecord(sd->fork, caller);
  if (err == cudaSuccess) err = cudaStreamWaitEvent(sd->stream, sd->fork, 0);
  if (err != cudaSuccess) return pkv::cuda_fail(err, "pkv_iteration_run: fork");
  const int rc_pre = prefill(sd->stream);
  // joined back whatever the prefill call returned, so that `stream` waits
  // for all of it (and a stream capture stays whole)
  err = cudaEventRecord(sd->join, sd->stream);
  const int rc_dec = rc_pre ? rc_pre : decode();
  if (err == cudaSuccess) err = cudaStreamWaitEvent(caller, sd->join, 0);
  if (err != cudaSuccess) return pkv::cuda_fail(err, "pkv_iteration_run: join");
  return rc_dec ? rc_dec : ok();
}

// Both halves of an iteration in one call: the host work of
// pkv_iteration_prepare into the caller's pinned buffer, one asynchronous
// copy of it to the caller's device buffer, and pkv_iteration_run from there.
extern "C" int pkv_iteration_step(pkv_alloc* a, const int64_t* seqs, const int32_t* counts,
                                  int32_t n_prefill, int32_t n_decode,
                                  int32_t max_blocks_per_seq, void* host_buf,
                                  size_t host_bytes, void* dev_buf, size_t dev_bytes,
                                  const void* q, const void* k_new, const void* v_new, void* out,
                                  void* k_cache, void* v_cache, int32_t num_blocks, int32_t Hq,
                                  int32_t Hkv, int32_t D, int32_t block_size, float scale,
                                  int32_t partition_size, void* decode_ws,
                                  size_t decode_ws_bytes, void* prefill_ws,
                                  size_t prefill_ws_bytes, int32_t* dev_status, void* stream,
                                  pkv_iteration_layout* layout, int32_t* n_fit) {
  const char* who = "pkv_iteration_step";
  PKV_REQUIRE(dev_buf, "%s: dev_buf is NULL", who);
  if (int rc = pkv_iteration_prepare(a, seqs, counts, n_prefill, n_decode, max_blocks_per_seq,
                                     host_buf, host_bytes, layout, n_fit))
    return rc;
  PKV_REQUIRE(dev_bytes >= (size_t)layout->total_bytes,
              "%s: dev_buf has %zu bytes, needs %lld (the allocator work is done)", who,
              dev_bytes, (long long)layout->total_bytes);
  cudaError_t err = cudaMemcpyAsync(dev_buf, host_buf, (size_t)layout->total_bytes,
                                    cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return pkv::cuda_fail(err, "pkv_iteration_step: metadata copy");
  return pkv_iteration_run(dev_buf, layout, n_prefill, n_decode, q, k_new, v_new, out, k_cache, v_cache, num_blocks, Hq, Hkv, D, block_size,
                           scale, partition_size, decode_ws, decode_ws_bytes, prefill_ws,
                           prefill_ws_bytes, dev_status, stream);
}
