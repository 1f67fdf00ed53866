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
// How (GB300 design). A Q tile is 128 rows, each row a (query, head) pair:
// 128/G consecutive queries times the G query heads that share one kv head,
// so every key/value tile loaded serves all of them. A work item is (sequence,
// query group, kv head) with one Q tile; large launches run a plan
// kernel and a persistent grid that takes items from an atomic ticket (the
// key producer posts each item whole to the other warps through a small
// ring), small ones one CTA per item. The warps specialise and run as a
// pipeline over 64-key tiles:
//  * warp 0 (key producer) takes the items, loads each one's Q tile by 3-D
//    TMA boxes and streams its key tiles into a ring of NS stages; warp 7
//    (value producer) streams the value tiles into their own ring. Page
//    numbers come from block-table windows in shared memory (one per
//    producer), and lane k issues the box of page k of a tile, one 4-D box
//    per page holding all its rows and both 64-column halves (tiles sit in
//    shared memory as [8-row group][half][8 rows x 128 B], 128-byte
//    swizzled). A value stage is freed late (by the P V product two tiles
//    back), a key stage early: apart, the key producer starts the next
//    item's Q and first keys without waiting for the last value stage;
//  * warp 1 issues the score products S_j = Q K_j^T into one of two TMEM
//    score buffers, so the scores of the next tile are computed while the
//    softmax works on the current one, and warp 2 the value products
//    O += P_j V_j (both under elect.sync, from different SM
//    sub-partitions: one warp issuing both took ~70 SM clocks per MMA beside
//    the softmax warps). A score buffer is rewritten once the value product
//    that read its probabilities has completed. Warp 2 also zeroes the
//    value rows past the last visible key before its product (they may hold
//    stale or poisoned bytes, and 0 * NaN is NaN);
//  * four softmax warps, one thread per TMEM lane (= row) with the row's 64
//    scores in registers (no exchange with another thread): they read the
//    scores, apply the causal limit, keep a running sum against a reference
//    maximum (base 2, packed f32x2 arithmetic), and write the probabilities
//    back into the same TMEM columns as two bf16 parts P_hi + P_lo (~fp32
//    precision for the product), which the P V MMA reads as its A operand
//    straight from tensor memory. O is rescaled (in TMEM) only when a row's
//    maximum grows by more than 2^8, so the stored probabilities stay below
//    256 and the rescale is rare; the final division by the row sum makes
//    the result independent of the reference chosen. The same warps write
//    the item's output rows.
// Every mbarrier wait has a time limit and gives up early once another warp
// has given up; the CTA then records PKV_ETIMEOUT, waits (with a limit) for its
// own copies and MMAs, frees its tensor memory and returns.
#include <cmath>
#include <mutex>

#include "device.cuh"
#include "host_util.h"

namespace pkv {
namespace {

constexpr int kRows = 128;       // (query, head) rows per Q tile = TMEM lanes
constexpr int kKeys = 64;        // keys per KV tile
// K and V tiles sit in shared memory as [8-row group][64-column half][8 rows
// x 128 B] (128-byte swizzled), so that one TMA box brings a whole page (both
// halves) and the tensor core still sees equal strides between 8-row groups
constexpr float kRescaleLog2 = 8.f;  // rescale O when a row max grows past 2^8
constexpr int kWin = 256;            // block-table entries held in shared memory
constexpr int kItemRing = 4;         // work items handed from the key producer to the others

// One Q tile per CTA and two CTAs per SM, so that one CTA's start and end
// overlap the other's work.
template <int D, int NS>
struct PCfg {
  // key producer, score-MMA warp, P V-MMA warp, four softmax warps, value
  // producer
  static constexpr int kThreads = 96 + 128 + 32;
  static constexpr uint32_t kQHalf = kRows * 128;  // one 64-column half of the Q tile
  static constexpr int kHalves = D / 64;
  static constexpr uint32_t kGroup = kHalves * 1024;  // one 8-row group of a K or V tile
  static constexpr uint32_t kStage = (kKeys / 8) * kGroup;
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK = kQ + kHalves * kQHalf;
  static constexpr uint32_t kV = kK + NS * kStage;
  static constexpr uint32_t kBytes = kV + NS * kStage;
  // + alignment slack; padded so that at most two CTAs share an SM: their
  // TMEM allocations (256 columns each) always fit and never wait
  static constexpr uint32_t kMinSmem = 80u * 1024;
  static constexpr uint32_t kSmem = kBytes + 1024 > kMinSmem ? kBytes + 1024 : kMinSmem;
  // barriers: Q; K full/empty and V full/empty per stage; per score
  // buffer: S full, P full, PV done; output read out (O free); Q free; work
  // item posted / taken per item-ring slot; final, per MMA warp
  static constexpr int kBarQ = 0, kBarKF = 1, kBarKE = 1 + NS, kBarVF = 1 + 2 * NS,
                       kBarVE = 1 + 3 * NS, kBarSF = 1 + 4 * NS, kBarPF = kBarSF + 2,
                       kBarPV = kBarPF + 2, kBarOE = kBarPV + 2, kBarQE = kBarOE + 1,
                       kBarIF = kBarQE + 1,
                       kBarIE = kBarIF + kItemRing, kBarFin = kBarIE + kItemRing,
                       kNumBars = kBarFin + 2;
  // TMEM: S buffers at columns 0..63 and 64..127, O at 128..128+D
  static constexpr uint32_t kTmemCols = 256;
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
  int32_t qc;         // queries per work item (128 / G)
  int32_t item_cap;
  int4* items;        // (sequence, query group, kv head, -)
  int32_t* n_items;
  int32_t* ticket;    // next item to hand out
  int32_t direct;     // 1: one CTA per (query group, kv head, sequence), no plan
};

// Lists the work items (sequence, query group, kv head): for each sequence
// its query groups from the last (which sees the most keys) to the first.
// One CTA of 1024 threads: a scan over the sequences gives each one its first
// item, then each warp writes the items of every 32nd sequence with its lanes
// on consecutive items. Sequences with an inconsistent length are recorded
// and skipped.
__global__ void __launch_bounds__(1024) prefill_plan_kernel(const PrefillArgs a) {
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t s_base, s_chunk;
  __shared__ int32_t s_first[1024], s_groups[1024];  // per sequence of the chunk
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  grid_dep_launch();  // the prefill kernel may start its set-up now
  grid_dep_wait();    // launched early: whatever ran before (the append) is complete
  if (tid == 0) s_base = 0;
  __syncthreads();
  for (int c0 = 0; c0 < a.S; c0 += 1024) {
    const int s = c0 + tid;
    int ng = 0;
    if (s < a.S) {
      const int c = __ldg(a.cu_q_lens + s + 1) - __ldg(a.cu_q_lens + s);
      const int L = __ldg(a.context_lens + s);
      if (c < 0 || L < c || L > a.max_context_len) {
        if (c != 0) record_status(a.status, PKV_EDEVICE, L, kKernelPrefill);
      } else {
        ng = (c + a.qc - 1) / a.qc;
      }
    }
    const int cnt = ng * a.Hkv;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int w = warp_tot[lane];
      int wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += v;
      }
      warp_tot[lane] = wi - w;
      if (lane == 31) s_chunk = wi;
    }
    __syncthreads();
    s_first[tid] = s_base + warp_tot[warp] + incl - cnt;
    s_groups[tid] = ng;
    __syncthreads();
    const int n_seq = min(1024, a.S - c0);
    for (int j = warp; j < n_seq; j += 32) {
      const int first = s_first[j], groups = s_groups[j], n = groups * a.Hkv;
      for (int i = lane; i < n && first + i < a.item_cap; i += 32)
        a.items[first + i] = make_int4(c0 + j, groups - 1 - i / a.Hkv, i % a.Hkv, 0);
    }
    __syncthreads();
    if (tid == 0) s_base += s_chunk;
    __syncthreads();
  }
  if (tid == 0) {
    *a.n_items = min(s_base, a.item_cap);
    *a.ticket = 0;
  }
}

// Bounded wait that also gives up as soon as another warp of the CTA has
// given up (`abort` set). The first waiter to run out of time sets `abort`
// to the site where it waited.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, const PrefillArgs& a,
                                              volatile int* abort, int site) {
  if (a.force_timeout) {
    *abort = site;
    return false;
  }
  if (mbar_try_wait(bar, parity)) return true;
  // the clocks and the abort flag are read every 32nd retry only, so that a
  // retry follows a failed one closely
  const uint64_t t0 = globaltimer_ns();
  const long long c0 = clock64();
  const long long cycle_limit =
      (long long)(a.timeout_ns < (1ull << 60) ? a.timeout_ns : (1ull << 60)) * 4;
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 31) == 0) {
      if (*abort) return false;
      if (clock64() - c0 > cycle_limit || globaltimer_ns() - t0 > a.timeout_ns) {
        *abort = site;
        return false;
      }
    }
  }
}

// tcgen05.mma kind::f16 with A (M x 16, bf16 pairs per 32-bit column, row =
// lane) in tensor memory and B in shared memory.
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Packed pairs of fp32 (two lanes of one 64-bit register) and their
// arithmetic, one instruction for both lanes.
__device__ __forceinline__ uint64_t f32x2_pack(float x, float y) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
  return r;
}
__device__ __forceinline__ void f32x2_unpack(uint64_t v, float& x, float& y) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(v));
}
__device__ __forceinline__ uint64_t f32x2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f32x2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f32x2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f32x2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// 16 consecutive 32-bit columns of this thread's TMEM lane (warp-collective).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%16], {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, "
      "%10, %11, %12, %13, %14, %15};" ::"r"(r[0]),
      "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
      "r"(taddr)
      : "memory");
}

// One lane of the warp, chosen by the hardware; the branch it guards stays
// warp-uniform for the compiler, so the tcgen05 operands stay in uniform
// registers (a lane-index test made the MMA issue markedly slower).
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// One work item: queries q0 .. q0 + qc - 1 of sequence s's chunk, kv head kvh.
struct PItem {
  int s, kvh, c0, c, L, q0;
  int kv_end, nkt;  // keys visible to the item's last query, and their key tiles
};

// The item (sequence, query group, kv head) = `it` given its sequence's
// chunk offsets c0 .. c1 and context length L.
__device__ __forceinline__ PItem make_item(int4 it, int c0, int c1, int L, int QT) {
  PItem p;
  p.s = it.x;
  p.kvh = it.z;
  p.c0 = c0;
  p.c = c1 - c0;
  p.L = L;
  p.q0 = it.y * QT;
  // the tile holds queries q0 .. q0 + QT - 1 of the chunk
  p.kv_end = p.L - p.c + p.q0 + min(QT, p.c - p.q0);
  p.nkt = (p.kv_end + kKeys - 1) / kKeys;
  return p;
}

__device__ __forceinline__ PItem load_item(const PrefillArgs& a, int idx, int QT) {
  if (idx < 0) {
    // direct launches: the item is the CTA's own grid position, sequence
    // blockIdx.x and kv head blockIdx.y, its query groups counted from the
    // last (which sees the most keys) as blockIdx.z grows, so that the grid's
    // first CTAs hold every sequence's longest items
    const int s = blockIdx.x;
    const int c0 = __ldg(a.cu_q_lens + s), c1 = __ldg(a.cu_q_lens + s + 1);
    const int ng = (c1 - c0 + QT - 1) / QT;
    return make_item(make_int4(s, ng - 1 - (int)blockIdx.z, blockIdx.y, 0), c0, c1,
                     __ldg(a.context_lens + s), QT);
  }
  const int4 it = a.items[idx];
  return make_item(it, __ldg(a.cu_q_lens + it.x), __ldg(a.cu_q_lens + it.x + 1),
                   __ldg(a.context_lens + it.x), QT);
}

// Persistent: the key producer takes the next work item from a global
// ticket and posts it whole in a small shared ring that the other warps read
// in the same order; every barrier's phase follows a running count, so the
// next item's Q and first K/V tiles load while this item finishes and its
// scores are computed while this item's output is written.
template <int D, int G, int NS>
__global__ void __launch_bounds__(PCfg<D, NS>::kThreads, 2)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap tmap_q,
                         const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v, const PrefillArgs a) {
  using C = PCfg<D, NS>;
  constexpr int kQHalf = C::kQHalf;
  constexpr int QT = kRows / G;  // queries per Q tile
  constexpr uint32_t kIdescS = umma_idesc_bf16(128, kKeys, false);
  constexpr uint32_t kIdescO = umma_idesc_bf16(128, D, true);

  extern __shared__ uint8_t dsm[];
  __shared__ __align__(8) uint64_t bars[C::kNumBars];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  // windows of the current sequence's block table, one per producer warp
  __shared__ int32_t s_pages[2][kWin];
  __shared__ PItem s_item[kItemRing];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (a.direct) {
    // one item per CTA: leave at once when its query group is empty
    const int s = blockIdx.x;
    const int c = __ldg(a.cu_q_lens + s + 1) - __ldg(a.cu_q_lens + s);
    const int L = __ldg(a.context_lens + s);
    if ((int)blockIdx.z * QT >= c) return;
    if (L < c || L > a.max_context_len) {
      if (tid == 0) record_status(a.status, PKV_EDEVICE, L, kKernelPrefill);
      return;
    }
  }

  const uint32_t raw = smem_u32(dsm);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = dsm + (base - raw);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  volatile int* abort = &s_abort;
  // a wait whose outcome is the same on every lane of the warp
  auto wait_warp = [&](int b, uint32_t parity, int site) {
    return __all_sync(0xffffffffu, wait_or_abort(bar(b), parity, a, abort, site)) != 0;
  };

  if (tid == 0) {
    mbar_init(bar(C::kBarQ), 1);
    mbar_init(bar(C::kBarQE), 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(bar(C::kBarKF + i), 1);
      mbar_init(bar(C::kBarKE + i), 1);
      mbar_init(bar(C::kBarVF + i), 1);
      mbar_init(bar(C::kBarVE + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::kBarSF + i), 1);
      mbar_init(bar(C::kBarPF + i), 128);
      mbar_init(bar(C::kBarPV + i), 1);
    }
    mbar_init(bar(C::kBarOE), 128);
    for (int i = 0; i < kItemRing; ++i) {
      mbar_init(bar(C::kBarIF + i), 1);
      mbar_init(bar(C::kBarIE + i), 2 + 4 + 1);  // MMA, softmax and value-producer warps
    }
    mbar_init(bar(C::kBarFin), 1);
    mbar_init(bar(C::kBarFin + 1), 1);
    s_abort = 0;
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
  grid_dep_wait();  // the plan (and everything before it) is complete
  const int n_items = a.direct ? 1 : *reinterpret_cast<volatile int32_t*>(a.n_items);

  // The n-th item of this CTA as the key producer posted it whole (s < 0: no
  // more), so that no consuming warp waits on a global load for it; every
  // consuming warp calls it once per n, in order.
  auto take_item = [&](int n, bool& ok) -> PItem {
    const int slot = n % kItemRing;
    PItem it;
    it.s = -1;
    ok = wait_warp(C::kBarIF + slot, (n / kItemRing) & 1, 14);
    if (!ok) return it;
    const volatile PItem& v = s_item[slot];
    it.s = v.s;
    it.kvh = v.kvh;
    it.c0 = v.c0;
    it.c = v.c;
    it.L = v.L;
    it.q0 = v.q0;
    it.kv_end = v.kv_end;
    it.nkt = v.nkt;
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(C::kBarIE + slot));
    return it;
  };

  // loads this CTA issued (Q, and K and V tiles, each counted by its producer):
  // what a CTA that gives up waits for before its shared memory goes
  int issued_q = 0, issued_k = 0, issued_v = 0;

  if (warp == 0 || warp == 7) {
    // ------------------------------------------------------------ producers
    // Warp 0 takes the items, loads each one's Q tile and streams its key
    // tiles; warp 7 streams the value tiles of the same items (it reads them
    // from the ring like the other warps). A value stage is freed late (by
    // the P V product two tiles back) and a key stage early, so one warp
    // loading both would start an item's Q and first keys only after the
    // previous item's last value wait. Page numbers come from a window of the
    // block table held in shared memory (one per producer, refilled by the
    // whole warp), so no tile's loads wait for a global read; lane k issues
    // the box of page k of a tile (all rows of the page and both column
    // halves in one box).
    const bool keys = warp == 0;
    const int B = a.block_size, ppt = kKeys / B;  // pages per tile
    int32_t* const sp = s_pages[keys ? 0 : 1];
    bool ok = true;
    int jg = 0;  // tiles issued so far (ring position)
    for (int n = 0; ok; ++n) {
      PItem it;
      it.s = -1;
      if (keys) {
        // post the next item (or the end) in the ring
        const int slot = n % kItemRing;
        if (n >= kItemRing) ok = wait_warp(C::kBarIE + slot, (n / kItemRing - 1) & 1, 15);
        if (!ok) break;
        // direct launches post their own item (index -2) once, then the end
        int idx = 0;
        if (lane == 0) idx = a.direct ? (n == 0 ? -2 : n_items) : atomicAdd(a.ticket, 1);
        idx = __shfl_sync(0xffffffffu, idx, 0);
        if (idx < n_items) it = load_item(a, idx, QT);
        if (lane == 0) {
          s_item[slot] = it;
          mbar_arrive(bar(C::kBarIF + slot));  // release: the item is visible to the waiters
        }
        if (idx >= n_items) break;
      } else {
        it = take_item(n, ok);
        if (!ok || it.s < 0) break;
      }
      const int32_t* bt = a.block_tables + (int64_t)it.s * a.max_blocks_per_seq;
      const int npages = (it.kv_end + B - 1) / B;
      int win0 = 0;
      if (keys) {
        // Q of this item once the previous item's score MMAs have read theirs
        if (n > 0) ok = wait_warp(C::kBarQE, (n - 1) & 1, 12);
        if (!ok) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(C::kBarQ), C::kHalves * kQHalf);
#pragma unroll
          for (int h = 0; h < C::kHalves; ++h)
            tma_load_3d(base + C::kQ + h * kQHalf, &tmap_q, h * 64, it.kvh * G, it.c0 + it.q0,
                        bar(C::kBarQ));
        }
        ++issued_q;
      }
      // the block-table window loads while Q is in flight
      __syncwarp();
      for (int i = lane; i < kWin && i < npages; i += 32) sp[i] = __ldg(bt + i);
      __syncwarp();
      for (int j = 0; ok && j < it.nkt; ++j) {
        if (min((j + 1) * ppt, npages) > win0 + kWin) {
          // slide the window to tile j
          win0 = j * ppt;
          __syncwarp();
          for (int i = lane; i < kWin && win0 + i < npages; i += 32) sp[i] = __ldg(bt + win0 + i);
          __syncwarp();
        }
        const int g = jg + j, st = g % NS;
        if (g >= NS)
          ok = wait_warp((keys ? C::kBarKE : C::kBarVE) + st, (g / NS - 1) & 1, keys ? 1 : 2);
        if (!ok) break;
        const int p0 = j * ppt;
        const bool mine = lane < ppt && lane < npages - p0;
        const int32_t blk = mine ? sp[p0 + lane - win0] : -1;
        const bool valid = mine && blk >= 0 && blk < a.num_blocks;
        const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
        const uint32_t full = bar((keys ? C::kBarKF : C::kBarVF) + st);
        const uint32_t page_bytes = B * C::kHalves * 128u;
        if (lane == 0) mbar_arrive_expect_tx(full, __popc(vmask) * page_bytes);
        __syncwarp();
        if (mine && !valid) record_status(a.status, PKV_EDEVICE, blk, kKernelPrefill);
        if (valid)
          tma_load_4d((keys ? base + C::kK : base + C::kV) + st * C::kStage +
                          lane * (B / 8) * C::kGroup,
                      keys ? &tmap_k : &tmap_v, 0, 0, 0, (blk * a.Hkv + it.kvh) * (B / 8), full);
        if (keys)
          ++issued_k;
        else
          ++issued_v;
        __syncwarp();
      }
      jg += it.nkt;
      __syncwarp();
    }
    __syncwarp();
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ tensor core
    // Two issuing warps on different SM sub-partitions: warp 1 issues the
    // score products S_j = Q K_j^T, warp 2 the value products O += P_j V_j.
    // One warp issuing both spent most of its time issuing (an MMA took ~70
    // SM clocks to issue beside the softmax warps), and the probabilities it
    // waited for were picked up late. A score buffer is rewritten only after
    // the product that read its probabilities has completed (the two warps'
    // MMAs are not ordered with each other).
    // shared-memory descriptors of the first Q, K and V tiles; the others
    // differ only in the start address field (bytes / 16)
    const uint64_t dq = umma_desc_sw128(base + C::kQ, 16, 1024);
    const uint64_t dk = umma_desc_sw128(base + C::kK, 16, C::kGroup);
    const uint64_t dv = umma_desc_sw128(base + C::kV, 1024, C::kGroup);
    // A descriptor's start address (bytes / 16) sits in its low word and never
    // carries into the high word (shared memory is below 2^18 bytes), so an
    // offset is added to the low word alone
    auto at = [](uint64_t d, uint32_t bytes) -> uint64_t {
      uint64_t r;
      asm("mov.b64 %0, {%1, %2};"
          : "=l"(r)
          : "r"((uint32_t)d + (bytes >> 4)), "r"((uint32_t)(d >> 32)));
      return r;
    };
    const bool scores = warp == 1;
    bool ok = true;
    int jg = 0;                   // K/V ring position
    int sg = 0, oe = 0;           // score-buffer uses and finished outputs
    for (int n = 0; ok; ++n) {
      const PItem it = take_item(n, ok);
      if (!ok || it.s < 0) break;
      if (scores) {
        ok = wait_warp(C::kBarQ, n & 1, 3);
        for (int j = 0; ok && j < it.nkt; ++j) {
          const int g = jg + j, st = g % NS, u = g / NS;
          const int sj = sg + j, b = sj & 1;
          ok = wait_warp(C::kBarKF + st, u & 1, 4);
          // buffer b is free once the product of tile sj - 2 has completed
          if (ok && sj >= 2) ok = wait_warp(C::kBarPV + b, ((sj - 2) >> 1) & 1, 16);
          if (!ok) break;
          tcgen05_after_sync();
          if (elect_one()) {
            const uint32_t kst = st * C::kStage;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t koff = (kk >> 2) * 1024 + (kk & 3) * 32;
              const uint32_t qoff = (kk >> 2) * kQHalf + (kk & 3) * 32;
              umma_bf16(tmem + b * kKeys, at(dq, qoff), at(dk, kst + koff), kIdescS,
                        kk > 0 ? 1u : 0u);
            }
            umma_commit(bar(C::kBarSF + b));
            umma_commit(bar(C::kBarKE + st));
            if (j == it.nkt - 1) umma_commit(bar(C::kBarQE));  // Q may be replaced
          }
          __syncwarp();
        }
      } else {
        for (int i = 0; ok && i < it.nkt; ++i) {
          const int g = jg + i, st = g % NS, u = g / NS;
          ok = wait_warp(C::kBarVF + st, u & 1, 6);
          if (!ok) break;
          const int key0 = i * kKeys;
          if (key0 + kKeys > it.kv_end) {
            // value rows past the last visible key: stale or poisoned bytes that
            // must not reach O, not even as NaN * 0
            uint8_t* vp = base_ptr + C::kV + st * C::kStage;
            for (int r = it.kv_end - key0 + lane; r < kKeys; r += 32)
#pragma unroll
              for (int h = 0; h < C::kHalves; ++h)
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                  *reinterpret_cast<uint4*>(vp + (r >> 3) * C::kGroup + h * 1024 +
                                            (r & 7) * 128 + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
            fence_proxy_async_smem();
          }
          __syncwarp();
          const int sgi = sg + i, b = sgi & 1;
          ok = wait_warp(C::kBarPF + b, (sgi >> 1) & 1, 5);
          // the previous item's output must have been read out of O
          if (ok && i == 0 && oe > 0) ok = wait_warp(C::kBarOE, (oe - 1) & 1, 13);
          if (!ok) break;
          tcgen05_after_sync();
          if (elect_one()) {
            const uint32_t p = tmem + b * kKeys;
            const uint32_t o = tmem + 128;
            const uint32_t vst = st * C::kStage;
#pragma unroll
            for (int kk = 0; kk < kKeys / 16; ++kk) {
              const uint64_t vdesc = at(dv, vst + kk * 2 * C::kGroup);
              umma_bf16_ts(o, p + kk * 8, vdesc, kIdescO, (i > 0 || kk > 0) ? 1u : 0u);
              umma_bf16_ts(o, p + 32 + kk * 8, vdesc, kIdescO, 1u);
            }
            umma_commit(bar(C::kBarPV + b));
            umma_commit(bar(C::kBarVE + st));
          }
          __syncwarp();
        }
        oe += it.nkt > 0 ? 1 : 0;
      }
      jg += it.nkt;
      sg += it.nkt;
    }
    // every MMA (and the arrivals it triggers) is done before the CTA leaves
    const int fin = C::kBarFin + (scores ? 0 : 1);
    if (lane == 0) {
      umma_commit(bar(fin));
      mbar_wait_bounded(bar(fin), 0, 4 * a.timeout_ns, 0);
    }
    __syncwarp();
  } else if (warp >= 3 && warp <= 6) {
    // ------------------------------------------------------------ softmax
    // Four warps, one thread per TMEM lane (= row) holding the row's 64
    // scores of a tile.
    const int quarter = warp & 3;     // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t t_o = tmem + 128 + lane_off;
    const uint64_t scale2 = f32x2_pack(a.scale_log2, a.scale_log2);
    bool ok = true;
    int sg = 0;  // score-buffer uses
    for (int n = 0; ok; ++n) {
      const PItem it = take_item(n, ok);
      if (!ok || it.s < 0) break;
      const int nk = it.nkt;
      const int qi = it.q0 + r / G;
      const bool row_valid = qi < it.c;
      const int limit = row_valid ? (it.L - it.c + qi + 1) : 1;  // number of visible keys
      float m_ref = 0.f;
      uint64_t l2 = f32x2_pack(0.f, 0.f);  // the row sum, two lanes
      for (int j = 0; j < nk; ++j) {
        const int sj = sg + j, b = sj & 1, key0 = j * kKeys;
        ok = wait_warp(C::kBarSF + b, (sj >> 1) & 1, 7);
        if (!ok) break;
        tcgen05_after_sync();
        const uint32_t t_s = tmem + lane_off + b * kKeys;
        uint32_t x[kKeys];
        tmem_ld32(t_s, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
        tmem_ld32(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(&x[32]));
        tmem_wait_ld();
        const int vis = min(kKeys, limit - key0);  // visible columns (may be <= 0)
        if (!(__all_sync(0xffffffffu, vis >= kKeys) != 0)) {
#pragma unroll
          for (int i = 0; i < kKeys; ++i)
            if (i >= vis) x[i] = __float_as_uint(-INFINITY);
        }
        float m8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
          m8[e] = fmax3(__uint_as_float(x[8 * e]), __uint_as_float(x[8 * e + 1]),
                        fmax3(__uint_as_float(x[8 * e + 2]), __uint_as_float(x[8 * e + 3]),
                              fmax3(__uint_as_float(x[8 * e + 4]), __uint_as_float(x[8 * e + 5]),
                                    fmax3(__uint_as_float(x[8 * e + 6]),
                                          __uint_as_float(x[8 * e + 7]), -INFINITY))));
        const float m_tile =
            fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7])) *
            a.scale_log2;  // -inf: no visible key
        if (j == 0) m_ref = m_tile;  // key 0 is visible to every row
        const bool need = m_tile > m_ref + kRescaleLog2;
        if (__any_sync(0xffffffffu, need)) {
          // O must be complete up to tile j-1 before it is rescaled
          ok = wait_warp(C::kBarPV + ((sj - 1) & 1), ((sj - 1) >> 1) & 1, 8);
          if (!ok) break;
          tcgen05_after_sync();
          const float alpha = need ? fast_exp2(m_ref - m_tile) : 1.f;
          if (need) m_ref = m_tile;
          l2 = f32x2_mul(l2, f32x2_pack(alpha, alpha));
#pragma unroll 1
          for (int c32 = 0; c32 < D / 32; ++c32) {
            uint32_t o[32];
            tmem_ld32(t_o + c32 * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(t_o + c32 * 32, o);
          }
        }
        // p = 2^(x scale - m_ref) for two columns at a time, split into bf16
        // hi + lo parts; masked columns hold -inf and give 0. Keys 32 c ..
        // 32 c + 31: hi parts in columns 16 c .. 16 c + 15, lo parts in
        // 32 + 16 c .. 32 + 16 c + 15.
        const uint64_t negm = f32x2_pack(-m_ref, -m_ref);
#pragma unroll
        for (int c = 0; c < kKeys / 32; ++c) {
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const uint32_t* y = x + 32 * c;
            float y0, y1;
            f32x2_unpack(
                f32x2_fma(f32x2_pack(__uint_as_float(y[2 * e]), __uint_as_float(y[2 * e + 1])),
                          scale2, negm),
                y0, y1);
            const float p0 = fast_exp2(y0), p1 = fast_exp2(y1);
            const uint64_t p = f32x2_pack(p0, p1);
            l2 = f32x2_add(l2, p);
            hi[e] = pack_bf16x2(p0, p1);
            float d0, d1;
            f32x2_unpack(
                f32x2_sub(p, f32x2_pack(bf16_lo_to_f32(hi[e]), bf16_hi_to_f32(hi[e]))), d0, d1);
            lo[e] = pack_bf16x2(d0, d1);
          }
          tmem_st16(t_s + 16 * c, hi);
          tmem_st16(t_s + 32 + 16 * c, lo);
        }
        tmem_wait_st();
        tcgen05_before_sync();
        mbar_arrive(bar(C::kBarPF + b));
      }
      if (!ok || nk == 0) {
        sg += nk;
        continue;
      }
      const int sl = sg + nk - 1;
      ok = wait_warp(C::kBarPV + (sl & 1), (sl >> 1) & 1, 9);
      if (ok) {
        // ---- epilogue: O / l -> bf16, row r -> (query qi, head kvh*G + r%G)
        float l0, l1;
        f32x2_unpack(l2, l0, l1);
        const float inv = 1.f / (l0 + l1);
        tcgen05_after_sync();
        __nv_bfloat16* orow = a.out + ((int64_t)(it.c0 + qi) * a.Hq + it.kvh * G + (r % G)) * D;
#pragma unroll 1
        for (int c32 = 0; c32 < D / 32; ++c32) {
          uint32_t o[32];
          tmem_ld32(t_o + c32 * 32, o);
          tmem_wait_ld();
          if (row_valid) {
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
              uint4 v;
              v.x = pack_bf16x2(__uint_as_float(o[e + 0]) * inv, __uint_as_float(o[e + 1]) * inv);
              v.y = pack_bf16x2(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
              v.z = pack_bf16x2(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
              v.w = pack_bf16x2(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
              *reinterpret_cast<uint4*>(orow + c32 * 32 + e) = v;
            }
          }
        }
        // O may be reused by the next item
        tcgen05_before_sync();
        mbar_arrive(bar(C::kBarOE));
      }
      sg += nk;
    }
  }

  tcgen05_before_sync();
  __syncthreads();
  if (*abort) {
    if (tid == 0) record_status(a.status, PKV_ETIMEOUT, *abort, kKernelPrefill);
    // Let this CTA's own copies land before its shared memory is released:
    // wait (again with a limit) for the last phase armed on each barrier.
    // (each producer for its own loads)
    if ((warp == 0 || warp == 7) && lane == 0) {
      if (issued_q) mbar_wait_bounded(bar(C::kBarQ), (issued_q - 1) & 1, 4 * a.timeout_ns, 0);
      for (int i = 0; i < NS; ++i) {
        // tiles i, i + NS, ... went to stage i: wait for the last one's phase
        const int nk = issued_k > i ? (issued_k - 1 - i) / NS + 1 : 0;
        const int nv = issued_v > i ? (issued_v - 1 - i) / NS + 1 : 0;
        if (nk) mbar_wait_bounded(bar(C::kBarKF + i), (nk - 1) & 1, 4 * a.timeout_ns, 0);
        if (nv) mbar_wait_bounded(bar(C::kBarVF + i), (nv - 1) & 1, 4 * a.timeout_ns, 0);
      }
    }
    __syncthreads();
  }
  if (warp == 0) {
    tcgen05_after_sync();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, int G>
int launch_prefill(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                   PrefillArgs a, const DeviceInfo& dev, int total_q, int max_q_len,
                   cudaStream_t stream) {
  constexpr int NS = 2;
  using C = PCfg<D, NS>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, []() {
    attr_err = cudaFuncSetAttribute(paged_prefill_kernel<D, G, NS>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  });
  if (attr_err != cudaSuccess) return cuda_fail(attr_err, "prefill kernel attributes");
  a.qc = kRows / G;  // queries per work item
  const int slots = dev.sm_count * 2;
  // Few items (under two per resident CTA): one CTA each, straight from the
  // grid (no plan launch); more: a plan and a persistent grid that hands
  // them out.
  const int64_t items = ((int64_t)total_q / a.qc + a.S) * a.Hkv;
  const int64_t groups = ((int64_t)max_q_len + a.qc - 1) / a.qc;
  if (items < 2 * (int64_t)slots && groups <= 65535) {
    a.direct = 1;
    dim3 grid((unsigned)a.S, (unsigned)a.Hkv, (unsigned)groups);
    paged_prefill_kernel<D, G, NS><<<grid, C::kThreads, C::kSmem, stream>>>(tq, tk, tv, a);
    return check_launch("prefill");
  }
  a.direct = 0;
  // the plan may start launching while the previous kernel ends (it waits
  // for it first); the persistent grid's set-up overlaps the plan
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  {
    cudaLaunchConfig_t pc = {};
    pc.gridDim = dim3(1);
    pc.blockDim = dim3(1024);
    pc.stream = stream;
    pc.attrs = pdl;
    pc.numAttrs = 1;
    cudaError_t perr = cudaLaunchKernelEx(&pc, prefill_plan_kernel, a);
    if (perr != cudaSuccess) return cuda_fail(perr, "prefill plan launch");
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)slots);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  cudaError_t err = cudaLaunchKernelEx(&cfg, paged_prefill_kernel<D, G, NS>, tq, tk, tv, a);
  if (err != cudaSuccess) return cuda_fail(err, "prefill launch");
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

// Workspace: 256-byte header (item count, ticket), then the work items, at most one
// per 16 queries plus one per sequence, per kv head (<= Hq).
static int64_t prefill_item_cap(int64_t S, int64_t total_q, int64_t Hq) {
  return (total_q / 16 + S + 1) * Hq;
}
static size_t prefill_ws_bytes(int64_t S, int64_t total_q, int64_t Hq) {
  return 256 + (size_t)prefill_item_cap(S, total_q, Hq) * sizeof(int4);
}

extern "C" int pkv_prefill_workspace_bytes(int32_t S, int32_t total_q, int32_t Hq, int32_t D,
                                           size_t* out) {
  PKV_REQUIRE(out, "pkv_prefill_workspace_bytes: out is NULL");
  PKV_REQUIRE(S >= 0 && total_q >= 0 && Hq > 0 && (D == 64 || D == 128),
              "pkv_prefill_workspace_bytes: bad sizes");
  *out = prefill_ws_bytes(S, total_q, Hq);
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
  PKV_REQUIRE(workspace_bytes >= prefill_ws_bytes(S, total_q, Hq),
              "prefill: workspace has %zu bytes, needs %zu", workspace_bytes,
              prefill_ws_bytes(S, total_q, Hq));
  PKV_REQUIRE((reinterpret_cast<uintptr_t>(workspace) & 15u) == 0,
              "prefill: workspace must be 16-byte aligned");
  PKV_REQUIRE(prefill_item_cap(S, total_q, Hq) < (int64_t(1) << 31), "prefill: batch too large");
  PKV_REQUIRE(aligned16(out) && aligned16(q) && aligned16(k_cache) && aligned16(v_cache),
              "prefill: bf16 arrays must be 16-byte aligned");
  const DeviceInfo* dev = nullptr;
  if (int rc = current_device_info(&dev)) return rc;
  // One Q tile per CTA and two CTAs per SM, whose starts and ends overlap:
  // measured faster on GB300 than two Q tiles per CTA sharing every K/V tile,
  // with 64-key tiles and also with 128-key tiles taking turns on the tensor
  // core, for fresh prompts and for short chunks after long cached prefixes.
  CUtensorMap tq, tk, tv;
  {
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)Hq, (uint64_t)total_q};
    const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)Hq * D * 2};
    const uint32_t box[3] = {64, (uint32_t)G, (uint32_t)(kRows / G)};
    if (int rc = encode_tile_map_3d(&tq, q, dims, strides, box)) return rc;
  }
  const uint64_t rows = (uint64_t)num_blocks * Hkv * block_size;
  if (int rc = encode_row_group_map(&tk, k_cache, D, rows, block_size)) return rc;
  if (int rc = encode_row_group_map(&tv, v_cache, D, rows, block_size)) return rc;

  PrefillArgs a = {};
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
  a.item_cap = (int32_t)prefill_item_cap(S, total_q, Hq);
  a.n_items = static_cast<int32_t*>(workspace);
  a.ticket = static_cast<int32_t*>(workspace) + 1;
  a.items = reinterpret_cast<int4*>(static_cast<uint8_t*>(workspace) + 256);

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int rc = PKV_OK;
#define PKV_PREFILL_CASE(DD, GG) \
  if (D == DD && G == GG) rc = launch_prefill<DD, GG>(tq, tk, tv, a, *dev, total_q, max_q_len, st);
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
