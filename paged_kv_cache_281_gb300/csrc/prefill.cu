// paged_attention_prefill: a prompt chunk attending causally over its own
// cached blocks, on the tcgen05 tensor cores.
//
// What it computes ("Deep Dive: continuous batching", sections Selective
// batching and The prefill/decode mix): sequence s owns c_s query rows, its
// last c_s tokens (already appended); row i sits at position L_s - c_s + i and
// attends keys 0 .. L_s - c_s + i of its own request, gathered page by page
// through the block table ("Batching, Scheduling, and Paging", section
// PagedAttention).
//
// How (GB300 design). One CTA of 4 warps owns a tile of 128 rows, each row a
// (query, head) pair: 128/G consecutive queries times the G query heads that
// share one kv head, so every key/value tile loaded serves all of them.
//  * Q is loaded once by a 3-D TMA box (64 columns x G heads x 128/G queries)
//    per 64-column half, 128-byte swizzled.
//  * For each 64-key tile (whole pages located through the block table, one
//    TMA box per page and half) S = Q K^T is computed by tcgen05.mma
//    (M=128, N=64, K=16 steps) into tensor memory.
//  * Thread r owns TMEM lane r = row r: it loads its 64 scores, applies the
//    causal limit, updates its running max and sum (base 2) and writes its
//    probabilities to shared memory as two bf16 parts P_hi + P_lo in the
//    swizzled K-major layout the next MMA reads. When the max moved, it
//    rescales its O row in tensor memory.
//  * O += P_hi V + P_lo V runs as tcgen05.mma with V as an MN-major operand
//    (M=128, N=D); the two parts keep the product at ~fp32 precision.
//  * The K buffer is refilled as soon as the S MMA retires and the V buffer as
//    soon as the P V MMA retires, so loads overlap the softmax.
//  * Every mbarrier wait has a time limit; on expiry the CTA records
//    PKV_ETIMEOUT, waits (with a limit) for its own copies and MMAs, frees its
//    tensor memory and returns. About 97 KB of shared memory per CTA lets two
//    CTAs share an SM (one's softmax overlaps the other's MMAs and loads); the
//    request never allows a third, so the two 256-column tensor-memory
//    allocations always fit and allocation never waits.
#include <cmath>
#include <mutex>

#include "device.cuh"
#include "host_util.h"

namespace pkv {
namespace {

constexpr int kRows = 128;       // (query, head) rows per tile = TMEM lanes
constexpr int kKeys = 64;        // keys per KV tile
constexpr int kThreadsP = 128;
constexpr uint32_t kQHalf = kRows * 128;   // one 64-column half of Q: 128 rows x 128 B
constexpr uint32_t kKVHalf = kKeys * 128;  // one 64-column half of a K or V tile
constexpr uint32_t kPTile = kRows * kKeys * 2;  // P (one part): 128 rows x 64 keys

template <int D>
struct PCfg {
  static constexpr int kHalves = D / 64;
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK = kQ + kHalves * kQHalf;
  static constexpr uint32_t kV = kK + kHalves * kKVHalf;
  static constexpr uint32_t kPhi = kV + kHalves * kKVHalf;
  static constexpr uint32_t kPlo = kPhi + kPTile;
  static constexpr uint32_t kBytes = kPlo + kPTile;
  // more than a third of an SM's shared memory: at most two CTAs per SM, whose
  // two tensor-memory allocations always fit, so allocation never waits
  static constexpr uint32_t kSmem = kBytes + 1024 > 80u * 1024 ? kBytes + 1024 : 80u * 1024;
  static constexpr uint32_t kTmemCols = 256;  // S: 64 columns, O: D columns at 128
  static constexpr uint32_t kOcol = 128;
};

struct PrefillArgs {
  __nv_bfloat16* out;
  const int32_t* cu_q_lens;
  const int32_t* context_lens;
  const int32_t* block_tables;
  int32_t max_blocks_per_seq;
  int32_t S, Hq, Hkv, num_blocks, block_size, max_context_len;
  float scale_log2;
  int32_t* status;
  uint64_t timeout_ns;
  int32_t force_timeout;
};

// Loads the pages holding keys [key0, min(key0 + 64, kv_end)) of kv head
// `kvh` from the pool behind `map` (keys or values) into `dst`; arms `bar`.
template <int D>
__device__ void load_kv_tile(const CUtensorMap* map, const PrefillArgs& a, const int32_t* bt,
                             int kvh, int key0, int kv_end, uint32_t dst, uint32_t bar) {
  using C = PCfg<D>;
  const int B = a.block_size;
  const int pages = kKeys / B;
  uint32_t bytes = 0;
  for (int pg = 0; pg < pages; ++pg) {
    const int tok = key0 + pg * B;
    if (tok >= kv_end) break;
    const int32_t blk = __ldg(bt + tok / B);
    if (blk >= 0 && blk < a.num_blocks) bytes += C::kHalves * B * 128u;
  }
  mbar_arrive_expect_tx(bar, bytes);
  for (int pg = 0; pg < pages; ++pg) {
    const int tok = key0 + pg * B;
    if (tok >= kv_end) break;
    const int32_t blk = __ldg(bt + tok / B);
    if (blk < 0 || blk >= a.num_blocks) {
      record_status(a.status, PKV_EDEVICE, blk, kKernelPrefill);
      continue;
    }
    const int row = (blk * a.Hkv + kvh) * B;
#pragma unroll
    for (int h = 0; h < C::kHalves; ++h)
      tma_load_2d(dst + h * kKVHalf + pg * B * 128, map, h * 64, row, bar);
  }
}

template <int D, int G>
__global__ void __launch_bounds__(kThreadsP, 2)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap tmap_q,
                         const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v, const PrefillArgs a) {
  using C = PCfg<D>;
  constexpr int QT = kRows / G;  // queries per tile
  constexpr uint32_t kIdescS = umma_idesc_bf16(128, kKeys, false);
  constexpr uint32_t kIdescO = umma_idesc_bf16(128, D, true);

  extern __shared__ uint8_t dsm[];
  __shared__ __align__(8) uint64_t bars[5];  // q, k, v, s, o
  __shared__ uint32_t s_tmem;

  const int tid = threadIdx.x, warp = tid >> 5;
  const int qt = blockIdx.x, kvh = blockIdx.y, s = blockIdx.z;
  const int c0 = __ldg(a.cu_q_lens + s);
  const int c = __ldg(a.cu_q_lens + s + 1) - c0;
  const int L = __ldg(a.context_lens + s);
  const int q0 = qt * QT;
  if (q0 >= c) return;
  if (L < c || L > a.max_context_len) {
    if (tid == 0) record_status(a.status, PKV_EDEVICE, L, kKernelPrefill);
    return;
  }
  const int qn = min(QT, c - q0);
  const int kv_end = L - c + q0 + qn;  // keys 0 .. kv_end-1 are visible to some row
  const int nkt = (kv_end + kKeys - 1) / kKeys;
  const int32_t* bt = a.block_tables + (int64_t)s * a.max_blocks_per_seq;

  const uint32_t raw = smem_u32(dsm);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = dsm + (base - raw);
  const uint32_t bar_of[5] = {smem_u32(&bars[0]), smem_u32(&bars[1]), smem_u32(&bars[2]),
                              smem_u32(&bars[3]), smem_u32(&bars[4])};
  enum { kBarQ = 0, kBarK = 1, kBarV = 2, kBarS = 3, kBarO = 4 };

  if (tid == 0) {
    for (int i = 0; i < 5; ++i) mbar_init(bar_of[i], 1);
    fence_barrier_init();
    prefetch_tensormap(&tmap_q);
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&s_tmem), C::kTmemCols);
    tmem_relinquish();
  }
  tcgen05_before_sync();
  __syncthreads();
  tcgen05_after_sync();
  const uint32_t tmem = s_tmem;
  const uint32_t t_s = tmem, t_o = tmem + C::kOcol;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;

  // Phases armed (by thread 0) and observed (by everyone) per barrier: at
  // most one phase of each is outstanding at any time, which is what a
  // timed-out CTA waits for before it leaves.
  int armed[5] = {0, 0, 0, 0, 0}, seen[5] = {0, 0, 0, 0, 0};
  if (tid == 0) {
    mbar_arrive_expect_tx(bar_of[kBarQ], C::kHalves * kQHalf);
#pragma unroll
    for (int h = 0; h < C::kHalves; ++h)
      tma_load_3d(base + C::kQ + h * kQHalf, &tmap_q, h * 64, kvh * G, c0 + q0,
                  bar_of[kBarQ]);
    load_kv_tile<D>(&tmap_k, a, bt, kvh, 0, kv_end, base + C::kK, bar_of[kBarK]);
    load_kv_tile<D>(&tmap_v, a, bt, kvh, 0, kv_end, base + C::kV, bar_of[kBarV]);
    armed[kBarQ] = armed[kBarK] = armed[kBarV] = 1;
  }

  // this thread's row: query qi (within the chunk) and head r % G of the group
  const int r = tid;
  const int qi = q0 + r / G;
  const bool row_valid = (r / G) < qn;
  const int limit = row_valid ? (L - c + qi + 1) : 1;  // number of visible keys
  float m = -INFINITY, l = 0.f;
  int fail_site = 0;

  // Waits for the next phase of barrier `b` on every thread; the result is
  // the same on every thread of the CTA.
  auto wait = [&](int b) {
    const bool landed = mbar_wait_bounded(bar_of[b], seen[b] & 1, a.timeout_ns, a.force_timeout);
    if (!landed) fail_site = b + 1;
    const bool all = __syncthreads_and(landed) != 0;
    if (all) ++seen[b];
    return all;
  };

  bool ok = wait(kBarQ);
  for (int kt = 0; ok && kt < nkt; ++kt) {
    const int key0 = kt * kKeys;
    ok = wait(kBarK);
    if (!ok) break;
    if (tid == 0) {
      tcgen05_after_sync();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t koff = (kk & 3) * 32;
        umma_bf16(t_s, umma_desc_sw128(base + C::kQ + (kk >> 2) * kQHalf + koff, 16, 1024),
                  umma_desc_sw128(base + C::kK + (kk >> 2) * kKVHalf + koff, 16, 1024), kIdescS,
                  kk > 0 ? 1u : 0u);
      }
      umma_commit(bar_of[kBarS]);
      ++armed[kBarS];
    }
    ok = wait(kBarS);
    if (!ok) break;
    tcgen05_after_sync();
    if (tid == 0 && kt + 1 < nkt) {
      load_kv_tile<D>(&tmap_k, a, bt, kvh, key0 + kKeys, kv_end, base + C::kK, bar_of[kBarK]);
      ++armed[kBarK];
    }

    // ---- softmax on this thread's row
    float x[kKeys];
#pragma unroll
    for (int c32 = 0; c32 < kKeys / 32; ++c32) {
      uint32_t rr[32];
      tmem_ld32(t_s + lane_off + c32 * 32, rr);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) x[c32 * 32 + i] = __uint_as_float(rr[i]) * a.scale_log2;
    }
    const int vis = min(kKeys, limit - key0);  // visible columns of this tile (may be <= 0)
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < kKeys; ++i)
      if (i < vis) mx = fmaxf(mx, x[i]);
    const float m_new = fmaxf(m, mx);          // finite: tile 0 always shows key 0
    const float alpha = fast_exp2(m - m_new);  // 0 on the first tile
    float sum = 0.f;
    uint8_t* phi = base_ptr + C::kPhi;
    uint8_t* plo = base_ptr + C::kPlo;
#pragma unroll
    for (int ch = 0; ch < kKeys / 8; ++ch) {
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i0 = ch * 8 + 2 * e;
        const float p0 = i0 < vis ? fast_exp2(x[i0] - m_new) : 0.f;
        const float p1 = i0 + 1 < vis ? fast_exp2(x[i0 + 1] - m_new) : 0.f;
        sum += p0 + p1;
        hi[e] = pack_bf16x2(p0, p1);
        lo[e] = pack_bf16x2(p0 - bf16_lo_to_f32(hi[e]), p1 - bf16_hi_to_f32(hi[e]));
      }
      const uint32_t off = swz128(r, ch);  // 64 keys: one 128-byte row per row
      *reinterpret_cast<uint4*>(phi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(plo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    l = l * alpha + sum;
    m = m_new;
    if (kt > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
      for (int c32 = 0; c32 < D / 32; ++c32) {
        uint32_t rr[32];
        tmem_ld32(t_o + lane_off + c32 * 32, rr);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
        tmem_st32(t_o + lane_off + c32 * 32, rr);
      }
      tmem_wait_st();
    }

    ok = wait(kBarV);
    if (!ok) break;
    if (key0 + kKeys > kv_end && r < kKeys && r >= kv_end - key0) {
      // keys past the last visible one: their value rows (unloaded pages, or
      // slots past the sequence end) must not reach O, not even as NaN * 0
#pragma unroll
      for (int h = 0; h < C::kHalves; ++h)
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
          *reinterpret_cast<uint4*>(base_ptr + C::kV + h * kKVHalf + r * 128 + ch * 16) =
              make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();  // P and zeroed V rows before the tensor core reads them
    tcgen05_before_sync();
    __syncthreads();
    if (tid == 0) {
      tcgen05_after_sync();
#pragma unroll
      for (int kk = 0; kk < kKeys / 16; ++kk) {
        const uint32_t poff = kk * 32;
        const uint64_t vdesc = umma_desc_sw128(base + C::kV + kk * 16 * 128, kKVHalf, 1024);
        umma_bf16(t_o, umma_desc_sw128(base + C::kPhi + poff, 16, 1024), vdesc, kIdescO,
                  (kt > 0 || kk > 0) ? 1u : 0u);
        umma_bf16(t_o, umma_desc_sw128(base + C::kPlo + poff, 16, 1024), vdesc, kIdescO, 1u);
      }
      umma_commit(bar_of[kBarO]);
      ++armed[kBarO];
    }
    ok = wait(kBarO);
    if (!ok) break;
    tcgen05_after_sync();
    if (tid == 0 && kt + 1 < nkt) {
      load_kv_tile<D>(&tmap_v, a, bt, kvh, key0 + kKeys, kv_end, base + C::kV, bar_of[kBarV]);
      ++armed[kBarV];
    }
  }

  if (ok) {
    // ---- epilogue: O / l -> bf16, row r -> (query qi, head kvh*G + r%G)
    const float inv = 1.f / l;
    __nv_bfloat16* orow = a.out + ((int64_t)(c0 + qi) * a.Hq + kvh * G + (r % G)) * D;
#pragma unroll
    for (int c32 = 0; c32 < D / 32; ++c32) {
      uint32_t rr[32];
      tmem_ld32(t_o + lane_off + c32 * 32, rr);
      tmem_wait_ld();
      if (row_valid) {
#pragma unroll
        for (int i = 0; i < 32; i += 8) {
          uint4 v;
          v.x = pack_bf16x2(__uint_as_float(rr[i + 0]) * inv, __uint_as_float(rr[i + 1]) * inv);
          v.y = pack_bf16x2(__uint_as_float(rr[i + 2]) * inv, __uint_as_float(rr[i + 3]) * inv);
          v.z = pack_bf16x2(__uint_as_float(rr[i + 4]) * inv, __uint_as_float(rr[i + 5]) * inv);
          v.w = pack_bf16x2(__uint_as_float(rr[i + 6]) * inv, __uint_as_float(rr[i + 7]) * inv);
          *reinterpret_cast<uint4*>(orow + c32 * 32 + i) = v;
        }
      }
    }
  } else {
    if (fail_site) record_status(a.status, PKV_ETIMEOUT, fail_site, kKernelPrefill);
    // Let this CTA's own copies and MMAs land before its shared and tensor
    // memory are released: wait (again with a limit) for each armed phase
    // that nobody has observed yet.
    if (tid == 0) {
      for (int b = 0; b < 5; ++b)
        if (armed[b] > seen[b]) mbar_wait_bounded(bar_of[b], seen[b] & 1, 4 * a.timeout_ns, 0);
    }
  }
  tcgen05_before_sync();
  __syncthreads();
  if (warp == 0) {
    tcgen05_after_sync();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, int G>
int launch_prefill(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                   const PrefillArgs& a, int max_q_len, cudaStream_t stream) {
  using C = PCfg<D>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, []() {
    attr_err = cudaFuncSetAttribute(paged_prefill_kernel<D, G>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  });
  if (attr_err != cudaSuccess) return cuda_fail(attr_err, "prefill kernel attributes");
  constexpr int QT = kRows / G;
  dim3 grid((unsigned)((max_q_len + QT - 1) / QT), (unsigned)a.Hkv, (unsigned)a.S);
  paged_prefill_kernel<D, G><<<grid, kThreadsP, C::kSmem, stream>>>(tq, tk, tv, a);
  return check_launch("prefill");
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" int pkv_prefill_workspace_bytes(int32_t S, int32_t total_q, int32_t Hq, int32_t D,
                                           size_t* out) {
  PKV_REQUIRE(out, "pkv_prefill_workspace_bytes: out is NULL");
  PKV_REQUIRE(S >= 0 && total_q >= 0 && Hq > 0 && (D == 64 || D == 128),
              "pkv_prefill_workspace_bytes: bad sizes");
  *out = 256;  // reserved: the kernel keeps all of its state on chip
  return ok();
}

extern "C" int pkv_paged_attention_prefill(void* out, const void* q, const int32_t* cu_q_lens,
                                           const int32_t* context_lens, const void* k_cache,
                                           const void* v_cache, const int32_t* block_tables,
                                           int32_t max_blocks_per_seq, int32_t S, int32_t total_q,
                                           int32_t max_q_len, int32_t max_context_len, int32_t Hq,
                                           int32_t Hkv, int32_t D, int32_t block_size,
                                           int32_t num_blocks, float scale, void* workspace,
                                           size_t workspace_bytes, int32_t* dev_status,
                                           void* stream) {
  PKV_REQUIRE(S >= 0 && S <= 65535, "prefill: S must be in [0, 65535]");
  PKV_REQUIRE(Hkv > 0 && Hkv <= 65535 && Hq > 0 && Hq % Hkv == 0,
              "prefill: Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
  const int G = Hq / Hkv;
  PKV_REQUIRE(G == 1 || G == 2 || G == 4 || G == 8, "prefill: Hq/Hkv must be 1, 2, 4 or 8");
  PKV_REQUIRE(D == 64 || D == 128, "prefill: D must be 64 or 128 (got %d)", D);
  PKV_REQUIRE(block_size == 8 || block_size == 16 || block_size == 32,
              "prefill: block_size must be 8, 16 or 32 (got %d)", block_size);
  PKV_REQUIRE(num_blocks > 0 && (int64_t)num_blocks * Hkv * block_size < (int64_t(1) << 31),
              "prefill: num_blocks * Hkv * block_size must be in [1, 2^31)");
  PKV_REQUIRE(total_q >= 0 && max_q_len >= 0, "prefill: sizes must be >= 0");
  PKV_REQUIRE((int64_t)max_blocks_per_seq * block_size >= max_context_len,
              "prefill: max_context_len exceeds max_blocks_per_seq * block_size");
  PKV_REQUIRE(std::isfinite(scale), "prefill: scale must be finite");
  if (S == 0 || total_q == 0 || max_q_len == 0) return ok();
  PKV_REQUIRE(max_context_len >= max_q_len, "prefill: max_context_len < max_q_len");
  PKV_REQUIRE(out && q && cu_q_lens && context_lens && k_cache && v_cache && block_tables &&
                  workspace,
              "prefill: NULL pointer");
  PKV_REQUIRE(workspace_bytes >= 256, "prefill: workspace too small");
  PKV_REQUIRE(aligned16(out) && aligned16(q) && aligned16(k_cache) && aligned16(v_cache),
              "prefill: bf16 arrays must be 16-byte aligned");
  const DeviceInfo* dev = nullptr;
  if (int rc = current_device_info(&dev)) return rc;

  CUtensorMap tq, tk, tv;
  {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)Hq, (uint64_t)total_q};
    const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)Hq * D * 2};
    const uint32_t box[3] = {64, (uint32_t)G, (uint32_t)(kRows / G)};
    if (int rc = encode_tile_map_3d(&tq, q, dims, strides, box)) return rc;
  }
  const uint64_t rows = (uint64_t)num_blocks * Hkv * block_size;
  if (int rc = encode_tile_map_2d(&tk, k_cache, D, rows, (uint64_t)D * 2, 64, block_size))
    return rc;
  if (int rc = encode_tile_map_2d(&tv, v_cache, D, rows, (uint64_t)D * 2, 64, block_size))
    return rc;

  PrefillArgs a;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.cu_q_lens = cu_q_lens;
  a.context_lens = context_lens;
  a.block_tables = block_tables;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.S = S;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.num_blocks = num_blocks;
  a.block_size = block_size;
  a.max_context_len = max_context_len;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.status = dev_status;
  const WaitConfig wc = wait_config();
  a.timeout_ns = wc.timeout_ns;
  a.force_timeout = wc.force_timeout;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int rc = PKV_OK;
#define PKV_PREFILL_CASE(DD, GG) \
  if (D == DD && G == GG) rc = launch_prefill<DD, GG>(tq, tk, tv, a, max_q_len, st);
  PKV_PREFILL_CASE(64, 1)
  PKV_PREFILL_CASE(64, 2)
  PKV_PREFILL_CASE(64, 4)
  PKV_PREFILL_CASE(64, 8)
  PKV_PREFILL_CASE(128, 1)
  PKV_PREFILL_CASE(128, 2)
  PKV_PREFILL_CASE(128, 4)
  PKV_PREFILL_CASE(128, 8)
#undef PKV_PREFILL_CASE
  if (rc) return rc;
  return ok();
}
