// paged_attention_decode: one query token per sequence over its paged K/V.
//
// What it computes ("Deep Dive: continuous batching", section Selective
// batching; "Batching, Scheduling, and Paging", section PagedAttention): for
// sequence s and query head h, softmax(scale * q . K_s^T) V_s over the s-th
// request's own L_s tokens, where K_s and V_s are gathered page by page
// through its block table.
//
// How (GB300 design):
//  * Split-K. A sequence's tokens are cut into partitions of a fixed number of
//    16-token tiles. A work item is (sequence, kv head, partition); a plan
//    kernel lists the items (full partitions first, partial ones last) and a
//    persistent grid of 3 CTAs per SM pulls them from an atomic ticket. Items
//    of multi-partition sequences write an unnormalised partial state
//    (m, l, o) that a combine kernel merges with the online-softmax rule; a
//    sequence with one partition is normalised in place.
//  * Data movement. Each of the CTA's 4 warps owns every 4th tile of the item
//    and a private 2-stage ring in shared memory. The warp's lanes look up the
//    block-table entries of its tiles in parallel; lanes 0..7 issue a tile's
//    TMA loads, one box each in one instruction (two 64-column halves per
//    tensor, 128-byte swizzle, whole pages), signalling an mbarrier with the
//    byte count; the warp waits on it with a time limit. The plan is launched
//    early after the previous kernel
//    (programmatic dependent launch) and waits for it before reading; the
//    decode and combine kernels follow the same way.
//  * Arithmetic. The G query heads that share a kv head form the rows of a
//    16-row MMA operand (rows >= G are zero). Scores S = Q K^T and the update
//    O += P V run as m16n8k16 bf16 MMAs with fp32 accumulators held in
//    registers; the online softmax (running max m, running sum l) works on
//    the accumulator fragment directly, in base 2 (scale pre-multiplied by
//    log2 e). P enters the second MMA as a bf16 pair P_hi + P_lo (rows 0..7
//    and 8..15 of the operand), so the P.V product keeps ~fp32 precision.
//  * Robustness. Block-table entries outside the pool are skipped and
//    recorded; V rows past the sequence end are zeroed in shared memory so
//    that whatever the pool holds there (even NaN) cannot leak into O.
#include <cmath>
#include <mutex>

#include "device.cuh"
#include "host_util.h"

namespace pkv {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kTileTokens = 16;
constexpr int kDefaultPartition = 1024;

// two stages of 8 KB per warp at D = 128: three CTAs (12 warps) per SM
template <int D, int Stages = (D == 128 ? 2 : 4)>
struct Cfg {
  static constexpr int kHalves = D / 64;            // 128-byte swizzled column halves
  static constexpr int kHalfBytes = kTileTokens * 128;
  static constexpr int kTensorBytes = kHalves * kHalfBytes;
  static constexpr int kStageBytes = 2 * kTensorBytes;  // keys, then values
  static constexpr int kStages = Stages;
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kSmemBytes = kWarps * kRingBytes + 1024;  // + alignment slack
};

struct DecodeArgs {
  __nv_bfloat16* out;
  const __nv_bfloat16* q;
  const int32_t* block_tables;
  const int32_t* context_lens;
  int32_t max_blocks_per_seq;
  int32_t S, Hq, Hkv;
  int32_t num_blocks;
  int32_t block_size;
  int32_t max_context_len;
  int32_t partition_tiles;
  int32_t max_partitions;
  float scale_log2;
  int2* items;
  int32_t* n_items;
  int32_t* ticket;
  float2* ws_ml;
  float* ws_o;
  int32_t* status;
  uint64_t timeout_ns;
  int32_t force_timeout;
  // FP8 pages (the e4m3 variant): codes [N][Hkv][B][D], scales [N][Hkv][B]
  const uint8_t* k8;
  const uint8_t* v8;
  const float* ks;
  const float* vs;
  // shared-prefix decode: groups of sequences whose first tokens share blocks
  const int32_t* grp_start;    // [n_groups + 1]
  const int32_t* grp_members;  // sequence indices
  const int32_t* grp_shared;   // [n_groups] tokens all members share
  int32_t n_groups;
  int32_t members_per_item;    // 16 / G
  int32_t item_cap;
  int4* gitems;                // two per item (see decode_group_plan_kernel)
  int32_t* seq_shared;         // [S] shared tokens processed by group items (0: none)
};

// Lists the work items: every full partition (s, p) in sequence order, then
// the trailing partial partition of each sequence. Single CTA of 1024
// threads; up to 1024 sequences one scan of both counts places both kinds,
// more take one pass over the sequences per kind. In one pass the tails are
// listed longest first (by 16-token tiles, 64 length classes), so that the
// items handed out last are the shortest and the CTAs finish together; the
// order within a class is that of the atomics (no result depends on the
// item order: each item's arithmetic is its own and the combine merges in
// partition order).
constexpr int kTailClasses = 64;
__global__ void __launch_bounds__(1024) decode_plan_kernel(DecodeArgs a) {
  __shared__ int32_t warp_tot[2][32];
  __shared__ int32_t s_base[2], s_chunk[2];  // [0] full partitions, [1] tails
  __shared__ int32_t s_class_n[kTailClasses], s_class_at[kTailClasses];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int P = a.partition_tiles * kTileTokens;
  const bool one_pass = a.S <= 1024;
  grid_dep_launch();  // the decode kernel may start its set-up now
  grid_dep_wait();    // launched early: whatever ran before (the append) is complete
  if (tid == 0) s_base[0] = s_base[1] = 0;
  if (tid < kTailClasses) s_class_n[tid] = 0;
  __syncthreads();
  for (int pass = 0; pass < (one_pass ? 1 : 2); ++pass) {
    for (int c0 = 0; c0 < a.S; c0 += 1024) {
      const int s = c0 + tid;
      int L = 0;
      if (s < a.S) {
        L = a.context_lens[s];
        if (L < 1 || L > a.max_context_len) {
          if (pass == 0) record_status(a.status, PKV_EDEVICE, L, kKernelDecodePlan);
          L = 0;
        }
      }
      const int full = (one_pass || pass == 0) ? L / P : 0;
      const int tail = (one_pass || pass == 1) && L % P != 0 ? 1 : 0;
      int cls = 0;  // length class of the tail, 0 = the longest
      if (one_pass && tail) {
        cls = kTailClasses - min((L % P + kTileTokens - 1) / kTileTokens, kTailClasses);
        atomicAdd(&s_class_n[cls], 1);
      }
      int incl_f = full, incl_t = tail;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int vf = __shfl_up_sync(0xffffffffu, incl_f, o);
        const int vt = __shfl_up_sync(0xffffffffu, incl_t, o);
        if (lane >= o) {
          incl_f += vf;
          incl_t += vt;
        }
      }
      if (lane == 31) {
        warp_tot[0][warp] = incl_f;
        warp_tot[1][warp] = incl_t;
      }
      __syncthreads();
      if (warp < 2) {  // warp k: exclusive prefix of the warp totals of kind k
        const int w = warp_tot[warp][lane];
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, wi, o);
          if (lane >= o) wi += v;
        }
        warp_tot[warp][lane] = wi - w;
        if (lane == 31) s_chunk[warp] = wi;
      } else if (warp == 2 && one_pass) {  // first position of each length class
        static_assert(kTailClasses == 64, "two classes per lane");
        const int n0 = s_class_n[lane], n1 = s_class_n[32 + lane];
        int i0 = n0, i1 = n1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v0 = __shfl_up_sync(0xffffffffu, i0, o);
          const int v1 = __shfl_up_sync(0xffffffffu, i1, o);
          if (lane >= o) {
            i0 += v0;
            i1 += v1;
          }
        }
        s_class_at[lane] = i0 - n0;
        s_class_at[32 + lane] = __shfl_sync(0xffffffffu, i0, 31) + i1 - n1;
      }
      __syncthreads();
      const int excl_f = s_base[0] + warp_tot[0][warp] + incl_f - full;
      // the tails follow every full partition: in one pass this chunk's (by
      // length class), else those of the first pass (in sequence order)
      const int tail_base = one_pass ? s_chunk[0] : s_base[0];
      for (int i = 0; i < full; ++i) a.items[excl_f + i] = make_int2(s, i);
      if (tail) {
        const int at = one_pass ? atomicAdd(&s_class_at[cls], 1)
                                : s_base[1] + warp_tot[1][warp] + incl_t - tail;
        a.items[tail_base + at] = make_int2(s, L / P);
      }
      __syncthreads();
      if (tid == 0) {
        s_base[0] += s_chunk[0];
        s_base[1] += s_chunk[1];
      }
      __syncthreads();
    }
  }
  if (tid == 0) {
    *a.n_items = s_base[0] + s_base[1];
    *a.ticket = 0;
  }
}

// TMA box rows (at most two boxes of min(B,16) rows) holding the keys and
// values of one 16-token tile of kv head `kvh`, and the bytes they bring.
// A box past the sequence end is not loaded; a block-table entry outside the
// pool is skipped and recorded.
struct TileRows {
  int32_t row[2];
  uint32_t bytes;
};

template <int D>
__device__ __forceinline__ TileRows tile_rows(const DecodeArgs& a, const int32_t* bt, int kvh,
                                              int tile, int L) {
  using C = Cfg<D>;
  const int B = a.block_size;
  const int R = B < kTileTokens ? B : kTileTokens;  // rows per TMA box
  const int nsub = kTileTokens / R;
  TileRows tr;
  tr.row[0] = tr.row[1] = -1;
  tr.bytes = 0;
  for (int sub = 0; sub < nsub; ++sub) {
    const int tok = tile * kTileTokens + sub * R;
    if (tok >= L) break;
    const int32_t blk = __ldg(bt + tok / B);
    if (blk < 0 || blk >= a.num_blocks) {
      record_status(a.status, PKV_EDEVICE, blk, kKernelDecode);
      continue;
    }
    tr.row[sub] = (blk * a.Hkv + kvh) * B + tok % B;
    tr.bytes += 2u * C::kHalves * R * 128u;
  }
  return tr;
}

// Arms `bar` with the tile's bytes and issues its TMA loads into `stage`.
template <int D>
__device__ __forceinline__ void issue_tile_rows(const CUtensorMap* tk, const CUtensorMap* tv,
                                                int block_size, int32_t row0, int32_t row1,
                                                uint32_t bytes, uint32_t stage, uint32_t bar,
                                                int lane) {
  // warp-collective: lane 0 arms the barrier, then lane 4 sub + 2 half + v
  // issues the box of run `sub` (R rows), column half `half` of the keys
  // (v = 0) or values (v = 1), so that one warp instruction issues them all
  using C = Cfg<D>;
  const int R = block_size < kTileTokens ? block_size : kTileTokens;
  if (lane == 0) mbar_arrive_expect_tx(bar, bytes);
  __syncwarp();
  const int sub = (lane >> 2) & 1, half = (lane >> 1) & 1, v = lane & 1;
  const int32_t row = sub == 0 ? row0 : row1;
  if (lane < 8 && half < C::kHalves && row >= 0)
    tma_load_2d(stage + (v ? C::kTensorBytes : 0u) + half * C::kHalfBytes + sub * R * 128,
                v ? tv : tk, half * 64, row, bar);
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 3)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, const DecodeArgs a) {
  using C = Cfg<D>;  // three CTAs per SM (168 registers)
  constexpr int KS = D / 16;  // k-steps of the score MMA
  constexpr int NT = D / 8;   // n-tiles of the output MMA
  static_assert(256 + kWarps * G * D * 4 <= kWarps * C::kRingBytes,
                "the merge buffer reuses the rings");
  extern __shared__ uint8_t dsm[];
  __shared__ __align__(8) uint64_t bars[kWarps][C::kStages];
  __shared__ int32_t s_next;
  __shared__ int32_t s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;  // MMA fragment row / column group
  const uint32_t dsm_u32 = smem_u32(dsm);
  const uint32_t base = (dsm_u32 + 1023u) & ~1023u;
  uint8_t* base_ptr = dsm + (base - dsm_u32);
  const uint32_t ring = base + warp * C::kRingBytes;

  if (lane == 0) {
#pragma unroll
    for (int st = 0; st < C::kStages; ++st) mbar_init(smem_u32(&bars[warp][st]), 1);
    fence_barrier_init();
  }
  grid_dep_launch();  // the combine kernel may start its set-up
  grid_dep_wait();    // the plan (and, before it, the appended tokens) are complete
  if (tid == 0) {
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
    s_abort = 0;
    s_next = atomicAdd(a.ticket, 1);
  }
  __syncthreads();
  const int total = __ldg(a.n_items) * a.Hkv;
  const int P = a.partition_tiles * kTileTokens;
  uint32_t phase = 0;  // bit st: parity of the next completion of stage st
  int cur = s_next;

  while (cur < total) {
    __syncthreads();  // everyone has read s_next
    const int2 item = __ldg(a.items + cur / a.Hkv);
    const int kvh = cur % a.Hkv;
    const int s = item.x, p = item.y;
    const int L = __ldg(a.context_lens + s);
    const int t_begin = p * a.partition_tiles;
    const int t_end = min((L + kTileTokens - 1) / kTileTokens, t_begin + a.partition_tiles);
    const int n_item = t_end - t_begin;
    const int n_mine = n_item > warp ? (n_item - warp + kWarps - 1) / kWarps : 0;
    const int32_t* bt = a.block_tables + (int64_t)s * a.max_blocks_per_seq;

    // The warp's lanes look up the block-table entries of its tiles of this
    // item together (32 tiles at a time); lanes 0..7 issue a tile's copies.
    TileRows mine = {{-1, -1}, 0u};
    int chunk0 = 0;
    if (lane < n_mine) mine = tile_rows<D>(a, bt, kvh, t_begin + warp + lane * kWarps, L);
    auto issue = [&](int k, uint32_t st) {
      if (k - chunk0 >= 32) {  // next 32 tiles of this warp (warp-uniform)
        chunk0 += 32;
        mine = {{-1, -1}, 0u};
        if (chunk0 + lane < n_mine)
          mine = tile_rows<D>(a, bt, kvh, t_begin + warp + (chunk0 + lane) * kWarps, L);
      }
      const int src = k - chunk0;
      const int32_t r0 = __shfl_sync(0xffffffffu, mine.row[0], src);
      const int32_t r1 = __shfl_sync(0xffffffffu, mine.row[1], src);
      const uint32_t by = __shfl_sync(0xffffffffu, mine.bytes, src);
      issue_tile_rows<D>(&tmap_k, &tmap_v, a.block_size, r0, r1, by, ring + st * C::kStageBytes,
                         smem_u32(&bars[warp][st]), lane);
    };
    {
      const int npro = n_mine < C::kStages ? n_mine : C::kStages;
      for (int k = 0; k < npro; ++k) issue(k, k);
    }
    // the next ticket, stored at the item's end (nothing waits on it before)
    int nxt = 0;
    if (tid == 0) nxt = atomicAdd(a.ticket, 1);

    // Q fragments (A operand rows g < G; rows g+8 are always zero).
    uint32_t qa[KS][2];
    {
      const bool live = g < G;
      const __nv_bfloat16* qrow = a.q + ((int64_t)s * a.Hq + kvh * G + (live ? g : 0)) * D;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qa[ks][0] = live ? __ldg(reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 2 * t)) : 0u;
        qa[ks][1] =
            live ? __ldg(reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 8 + 2 * t)) : 0u;
      }
    }

    float m = -INFINITY, l = 0.f;
    float o[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;

    for (int k = 0; k < n_mine; ++k) {
      const int st = k % C::kStages;
      const int tile = t_begin + warp + k * kWarps;
      const uint32_t bar = smem_u32(&bars[warp][st]);
      const uint32_t par = (phase >> st) & 1u;
      const bool landed = mbar_wait_bounded(bar, par, a.timeout_ns, a.force_timeout);
      if (!__all_sync(0xffffffffu, landed)) {
        if (lane == 0) {
          record_status(a.status, PKV_ETIMEOUT, k, kKernelDecode);
          s_abort = 1;
        }
        // Let this warp's loads in flight land before leaving: tiles k .. k+stages-1.
        uint32_t ph = phase;
        const int last = min(k + C::kStages, n_mine);
        for (int j = k; j < last; ++j) {
          const int sj = j % C::kStages;
          mbar_wait_bounded(smem_u32(&bars[warp][sj]), (ph >> sj) & 1u, 4 * a.timeout_ns, 0);
          ph ^= 1u << sj;
        }
        phase = ph;
        break;
      }
      phase ^= 1u << st;
      const uint32_t stage = ring + st * C::kStageBytes;
      const int valid = min(kTileTokens, L - tile * kTileTokens);
      if (valid < kTileTokens) {
        // Rows past the sequence end hold whatever the pool holds: clear V there.
        const int n16 = (kTileTokens - valid) * C::kHalves * 8;
        for (int i = lane; i < n16; i += 32) {
          const int row = valid + i / (C::kHalves * 8);
          const int rem = i % (C::kHalves * 8);
          const uint32_t addr = stage + C::kTensorBytes + (rem >> 3) * C::kHalfBytes + row * 128 +
                                (rem & 7) * 16;
          asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u)
                       : "memory");
        }
        __syncwarp();
      }

      // S = Q K^T over this tile: two n-tiles of 8 tokens.
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      {
        const int tok = (lane & 7) + ((lane >> 4) << 3);
        const int csel = (lane >> 3) & 1;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          const int chunk = 2 * ks + csel;
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(stage + (chunk >> 3) * C::kHalfBytes + swz128(tok, chunk & 7), b0, b1, b2,
                      b3);
          mma_bf16_16816(sc[0], qa[ks][0], 0u, qa[ks][1], 0u, b0, b1);
          mma_bf16_16816(sc[1], qa[ks][0], 0u, qa[ks][1], 0u, b2, b3);
        }
      }

      // Online softmax on row g (tokens 2t, 2t+1, 8+2t, 8+2t+1 of the tile).
      float x[4];
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e)
          x[2 * j + e] = (8 * j + 2 * t + e < valid) ? sc[j][e] * a.scale_log2 : -INFINITY;
      float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m, mx);
      const float alpha = fast_exp2(m - m_new);
      float pr[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) pr[i] = fast_exp2(x[i] - m_new);
      l = l * alpha + ((pr[0] + pr[1]) + (pr[2] + pr[3]));
      m = m_new;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        o[nt][0] *= alpha;
        o[nt][1] *= alpha;
        o[nt][2] *= alpha;
        o[nt][3] *= alpha;
      }
      // P = P_hi + P_lo with both parts in bf16: P_hi drives A rows 0..7 and
      // the residual P_lo the otherwise empty rows 8..15, so one MMA gives
      // the P.V product to about 2^-17 relative precision.
      const uint32_t pa0 = pack_bf16x2(pr[0], pr[1]);
      const uint32_t pa2 = pack_bf16x2(pr[2], pr[3]);
      const uint32_t pl0 = pack_bf16x2(pr[0] - bf16_lo_to_f32(pa0), pr[1] - bf16_hi_to_f32(pa0));
      const uint32_t pl2 = pack_bf16x2(pr[2] - bf16_lo_to_f32(pa2), pr[3] - bf16_hi_to_f32(pa2));

      // O += P V: n-tiles of 8 columns, two per ldmatrix.
      {
        const int tok = (lane & 7) + (((lane >> 3) & 1) << 3);
        const int csel = lane >> 4;
#pragma unroll
        for (int n2 = 0; n2 < NT / 2; ++n2) {
          const int chunk = 2 * n2 + csel;
          uint32_t r0, r1, r2, r3;
          ldmatrix_x4_trans(
              stage + C::kTensorBytes + (chunk >> 3) * C::kHalfBytes + swz128(tok, chunk & 7), r0,
              r1, r2, r3);
          mma_bf16_16816(o[2 * n2], pa0, pl0, pa2, pl2, r0, r1);
          mma_bf16_16816(o[2 * n2 + 1], pa0, pl0, pa2, pl2, r2, r3);
        }
      }
      if (valid < kTileTokens) fence_proxy_async_smem();  // zeroing stores before TMA reuse
      __syncwarp();
      if (k + C::kStages < n_mine) issue(k + C::kStages, st);
    }

    // Merge the 4 warps' states through shared memory (the rings are drained).
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    if (tid == 0) s_next = nxt;
    __syncthreads();
    if (s_abort) return;
    float2* cml = reinterpret_cast<float2*>(base_ptr);                  // [kWarps][G]
    float* co = reinterpret_cast<float*>(base_ptr + 256);               // [kWarps][G][D]
    if (g < G) {
      if (t == 0) cml[warp * G + g] = make_float2(m, l);
      float* row = co + (warp * G + g) * D;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        *reinterpret_cast<float2*>(row + nt * 8 + 2 * t) =
            make_float2(o[nt][0] + o[nt][2], o[nt][1] + o[nt][3]);
    }
    __syncthreads();
    const int nparts = (L + P - 1) / P;
    for (int e = tid; e < G * D; e += kThreads) {
      const int h = e / D, d = e % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, cml[w * G + h].x);
      float lsum = 0.f, acc = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float sw = fast_exp2(cml[w * G + h].x - M);
        lsum += sw * cml[w * G + h].y;
        acc += sw * co[(w * G + h) * D + d];
      }
      const int64_t qh = (int64_t)s * a.Hq + kvh * G + h;
      if (nparts == 1) {
        a.out[qh * D + d] = __float2bfloat16_rn(acc / lsum);
      } else {
        const int64_t idx = qh * a.max_partitions + p;
        a.ws_o[idx * D + d] = acc;
        if (d == 0) a.ws_ml[idx] = make_float2(M, lsum);
      }
    }
    fence_proxy_async_smem();  // merge-buffer stores before the ring's next TMA writes
    __syncthreads();           // the ring is free again for the next item's loads
    cur = s_next;
  }
}

// Merges the partial states of multi-partition sequences: one warp per
// (sequence, query head).
template <int D>
__global__ void __launch_bounds__(128) decode_combine_kernel(const DecodeArgs a) {
  constexpr int E = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t sh = (int64_t)blockIdx.x * 4 + warp;
  grid_dep_wait();  // every partial state has been written
  if (sh >= (int64_t)a.S * a.Hq) return;
  const int s = (int)(sh / a.Hq);
  const int L = __ldg(a.context_lens + s);
  if (L < 1 || L > a.max_context_len) return;
  const int P = a.partition_tiles * kTileTokens;
  int np = (L + P - 1) / P;
  if (a.seq_shared) {  // shared-prefix decode: shared partitions, then private ones
    const int shr = __ldg(a.seq_shared + s);
    np = (shr + P - 1) / P + (L - shr + P - 1) / P;
  }
  if (np <= 1) return;
  const float2* ml = a.ws_ml + sh * a.max_partitions;
  float M = -INFINITY;
  for (int p = lane; p < np; p += 32) M = fmaxf(M, ml[p].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float lsum = 0.f;
  for (int p = lane; p < np; p += 32) lsum += fast_exp2(ml[p].x - M) * ml[p].y;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  const float* ob = a.ws_o + sh * a.max_partitions * D + lane * E;
  for (int p = 0; p < np; ++p) {
    const float w = fast_exp2(ml[p].x - M);
    if constexpr (E == 4) {
      const float4 v = *reinterpret_cast<const float4*>(ob + (int64_t)p * D);
      acc[0] += w * v.x;
      acc[1] += w * v.y;
      acc[2] += w * v.z;
      acc[3] += w * v.w;
    } else {
      const float2 v = *reinterpret_cast<const float2*>(ob + (int64_t)p * D);
      acc[0] += w * v.x;
      acc[1] += w * v.y;
    }
  }
  const float inv = 1.f / lsum;
  __nv_bfloat16* out = a.out + sh * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; e += 2)
    *reinterpret_cast<__nv_bfloat162*>(out + e) =
        __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
}

struct WsLayout {
  size_t items_off, ml_off, o_off, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

WsLayout ws_layout(int64_t S, int64_t Hq, int64_t D, int64_t max_parts) {
  WsLayout w;
  w.items_off = 256;
  w.ml_off = align256(w.items_off + S * max_parts * sizeof(int2));
  w.o_off = align256(w.ml_off + S * Hq * max_parts * sizeof(float2));
  w.total = align256(w.o_off + S * Hq * max_parts * D * sizeof(float));
  return w;
}

// ---------------------------------------------------------------------------
// Decode over FP8 (e4m3) pages with one fp32 scale per token row.
//
// Same work items, partitions, ring discipline and merge as the bf16 kernel;
// what differs is the tile:
//  * a tile's codes arrive by TMA (16 rows x D bytes per tensor, 128-byte
//    swizzled when D = 128) and its 16 key and 16 value scales by two small
//    bulk copies into a separate scale ring;
//  * scores run transposed, S^T = K Q^T, with the tile's 16 keys as the
//    MMA's rows and 8 score columns (query heads) as its columns. The MMA's
//    k index is a sum index, so each thread owns a contiguous D/4-byte run
//    of its two key rows (and the matching run of q, rounded to fp16 once
//    per item: exact for 2^-14 <= |q| <= 65504) instead of the columns the
//    hardware layout names; two codes widen to one fp16 pair (exact: every
//    e4m3 value is an fp16 value);
//  * values: the product runs transposed too, O^T += V^T P'^T, with 16
//    value columns as the MMA's rows. One transposing 8-bit ldmatrix per
//    16 x 16 code block hands thread (g, t) value rows 4t .. 4t+3 at
//    columns g and 8 + g, its A fragment; the keys of the score rows are
//    ordered so that a movmatrix transpose of the packed P' blocks hands the
//    same thread column g of those four keys, its B fragment;
//  * a key's scale multiplies its score and a value's scale its probability
//    (P' = p * s_v) before the P V product, so no code is rescaled element by
//    element; P' enters as fp16 hi + lo parts: for G <= 4 the score
//    columns 4..7 repeat columns 0..3 and carry the lo parts, so one MMA per
//    16 value columns takes both (G = 8 issues a second MMA for lo); O^T and
//    S^T share their columns, so every lane rescales with its own factors;
//    value rows past the sequence end are zeroed in shared memory.
template <int D>
struct Cfg8 {
  static constexpr int kTile8 = kTileTokens * D;         // codes of one tensor tile
  static constexpr int kCodeStage = 2 * kTile8;          // keys, then values
  static constexpr int kScaleStage = 2 * kTileTokens * 4;  // key scales, then value scales
  // four CTAs per SM: 4 warps x 3 stages x 4.2 KB at D = 128
  static constexpr int kStages = D == 128 ? 3 : 6;
  static constexpr int kWarpBytes =
      (kStages * (kCodeStage + kScaleStage) + 1023) / 1024 * 1024;
  static constexpr int kSmemBytes = kWarps * kWarpBytes + 1024;
  static_assert(kCodeStage % 1024 == 0, "swizzled code tiles need 1024-byte alignment");
};

// Byte offset of 16-byte chunk c of code row r inside a tile: 128-byte
// swizzled rows for D = 128 (as TMA writes them), plain rows for D = 64.
template <int D>
__device__ __forceinline__ uint32_t code_off(int r, int c) {
  if constexpr (D == 128)
    return swz128(r, c);
  else
    return r * D + c * 16;
}

struct TileRows8 {
  int32_t row[2];
  uint32_t bytes;
};

template <int D>
__device__ __forceinline__ TileRows8 tile_rows8(const DecodeArgs& a, const int32_t* bt, int kvh,
                                                int tile, int L) {
  const int B = a.block_size;
  const int R = B < kTileTokens ? B : kTileTokens;
  const int nsub = kTileTokens / R;
  TileRows8 tr;
  tr.row[0] = tr.row[1] = -1;
  tr.bytes = 0;
  for (int sub = 0; sub < nsub; ++sub) {
    const int tok = tile * kTileTokens + sub * R;
    if (tok >= L) break;
    const int32_t blk = __ldg(bt + tok / B);
    if (blk < 0 || blk >= a.num_blocks) {
      record_status(a.status, PKV_EDEVICE, blk, kKernelDecode);
      continue;
    }
    tr.row[sub] = (blk * a.Hkv + kvh) * B + tok % B;
    tr.bytes += 2u * R * (D + 4);
  }
  return tr;
}

template <int D>
__device__ __forceinline__ void issue_tile_rows8(const CUtensorMap* tk, const CUtensorMap* tv,
                                                 const DecodeArgs& a, int32_t row0, int32_t row1,
                                                 uint32_t bytes, uint32_t codes, uint32_t scales,
                                                 uint32_t bar) {
  using C = Cfg8<D>;
  const int R = a.block_size < kTileTokens ? a.block_size : kTileTokens;
  mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
  for (int sub = 0; sub < 2; ++sub) {
    const int32_t row = sub == 0 ? row0 : row1;
    if (row < 0) continue;
    tma_load_2d(codes + sub * R * D, tk, 0, row, bar);
    tma_load_2d(codes + C::kTile8 + sub * R * D, tv, 0, row, bar);
    bulk_load(scales + sub * R * 4, a.ks + row, R * 4, bar);
    bulk_load(scales + kTileTokens * 4 + sub * R * 4, a.vs + row, R * 4, bar);
  }
}

// An 8 x 8 matrix of 16-bit values, one pair per thread (thread (g, t) holds
// row g, columns 2t and 2t + 1), transposed across the warp.
__device__ __forceinline__ uint32_t movmatrix_trans_b16(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// 16 x 16 bytes at row addresses given by lanes 0..15, transposed: thread
// (g, t) receives rows 4t .. 4t+3 of column g (r0) and of column 8 + g (r1).
__device__ __forceinline__ void ldmatrix_b8_16x16_trans(uint32_t addr, uint32_t& r0,
                                                        uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m16n16.x1.trans.shared.b8 {%0, %1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 4)
    paged_decode_fp8_kernel(const __grid_constant__ CUtensorMap tmap_k,
                            const __grid_constant__ CUtensorMap tmap_v, const DecodeArgs a) {
  using C = Cfg8<D>;
  constexpr int KS = D / 16;
  constexpr int NC = D / 16;  // 16-column blocks of O^T
  // G <= 4: score column r < 4 is query head r (hi part of P'), column
  // 4 + r the same head again (lo part); G = 8: columns are heads, lo takes
  // its own MMA
  constexpr bool kLoRows = G <= 4;
  extern __shared__ uint8_t dsm[];
  __shared__ __align__(8) uint64_t bars[kWarps][C::kStages];
  __shared__ int32_t s_next;
  __shared__ int32_t s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t dsm_u32 = smem_u32(dsm);
  const uint32_t base = (dsm_u32 + 1023u) & ~1023u;
  uint8_t* base_ptr = dsm + (base - dsm_u32);
  const uint32_t ring = base + warp * C::kWarpBytes;       // code stages
  const uint32_t sring = ring + C::kStages * C::kCodeStage;  // scale stages
  uint8_t* ring_ptr = base_ptr + warp * C::kWarpBytes;
  const uint8_t* sring_ptr = ring_ptr + C::kStages * C::kCodeStage;

  if (lane == 0) {
#pragma unroll
    for (int st = 0; st < C::kStages; ++st) mbar_init(smem_u32(&bars[warp][st]), 1);
    fence_barrier_init();
  }
  grid_dep_launch();
  grid_dep_wait();
  if (tid == 0) {
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
    s_abort = 0;
    s_next = atomicAdd(a.ticket, 1);
  }
  __syncthreads();
  const int total = __ldg(a.n_items) * a.Hkv;
  const int P = a.partition_tiles * kTileTokens;
  uint32_t phase = 0;
  int cur = s_next;

  while (cur < total) {
    __syncthreads();
    if (tid == 0) s_next = atomicAdd(a.ticket, 1);
    const int2 item = __ldg(a.items + cur / a.Hkv);
    const int kvh = cur % a.Hkv;
    const int s = item.x, p = item.y;
    const int L = __ldg(a.context_lens + s);
    const int t_begin = p * a.partition_tiles;
    const int t_end = min((L + kTileTokens - 1) / kTileTokens, t_begin + a.partition_tiles);
    const int n_item = t_end - t_begin;
    const int n_mine = n_item > warp ? (n_item - warp + kWarps - 1) / kWarps : 0;
    const int32_t* bt = a.block_tables + (int64_t)s * a.max_blocks_per_seq;

    TileRows8 mine = {{-1, -1}, 0u};
    int chunk0 = 0;
    if (lane < n_mine) mine = tile_rows8<D>(a, bt, kvh, t_begin + warp + lane * kWarps, L);
    auto issue = [&](int k, uint32_t st) {
      if (k - chunk0 >= 32) {
        chunk0 += 32;
        mine = {{-1, -1}, 0u};
        if (chunk0 + lane < n_mine)
          mine = tile_rows8<D>(a, bt, kvh, t_begin + warp + (chunk0 + lane) * kWarps, L);
      }
      const int src = k - chunk0;
      const int32_t r0 = __shfl_sync(0xffffffffu, mine.row[0], src);
      const int32_t r1 = __shfl_sync(0xffffffffu, mine.row[1], src);
      const uint32_t by = __shfl_sync(0xffffffffu, mine.bytes, src);
      if (lane == 0)
        issue_tile_rows8<D>(&tmap_k, &tmap_v, a, r0, r1, by, ring + st * C::kCodeStage,
                            sring + st * C::kScaleStage, smem_u32(&bars[warp][st]));
    };
    {
      const int npro = n_mine < C::kStages ? n_mine : C::kStages;
      for (int k = 0; k < npro; ++k) issue(k, k);
    }

    // Q^T fragments in fp16 (column g holds head g, or head g & 3 when
    // G <= 4). Thread t owns d = (D/4) t + 4 ks + {0,1 | 2,3} in k-step ks
    // (see the key loads).
    uint32_t qa[KS][2];
    {
      const int qh = kLoRows ? (g & 3) : g;
      const bool live = qh < G;
      const __nv_bfloat16* qrow =
          a.q + ((int64_t)s * a.Hq + kvh * G + (live ? qh : 0)) * D + (D / 4) * t;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const uint2 w =
            live ? __ldg(reinterpret_cast<const uint2*>(qrow + 4 * ks)) : make_uint2(0u, 0u);
        qa[ks][0] = pack_f16x2(bf16_lo_to_f32(w.x), bf16_hi_to_f32(w.x));
        qa[ks][1] = pack_f16x2(bf16_lo_to_f32(w.y), bf16_hi_to_f32(w.y));
      }
    }

    // running max and sum of score columns 2t (m0, l0) and 2t + 1 (m1, l1);
    // l holds this thread's keys only until the end of the item
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    // O^T block c: thread (g, t) holds value columns 16c + g (o[c][0..1]) and
    // 16c + 8 + g (o[c][2..3]) of score columns 2t and 2t + 1
    float o[NC][4];
#pragma unroll
    for (int c = 0; c < NC; ++c) o[c][0] = o[c][1] = o[c][2] = o[c][3] = 0.f;

    for (int k = 0; k < n_mine; ++k) {
      const int st = k % C::kStages;
      const int tile = t_begin + warp + k * kWarps;
      const uint32_t bar = smem_u32(&bars[warp][st]);
      const uint32_t par = (phase >> st) & 1u;
      const bool landed = mbar_wait_bounded(bar, par, a.timeout_ns, a.force_timeout);
      if (!__all_sync(0xffffffffu, landed)) {
        if (lane == 0) {
          record_status(a.status, PKV_ETIMEOUT, k, kKernelDecode);
          s_abort = 1;
        }
        uint32_t ph = phase;
        const int last = min(k + C::kStages, n_mine);
        for (int j = k; j < last; ++j) {
          const int sj = j % C::kStages;
          mbar_wait_bounded(smem_u32(&bars[warp][sj]), (ph >> sj) & 1u, 4 * a.timeout_ns, 0);
          ph ^= 1u << sj;
        }
        phase = ph;
        break;
      }
      phase ^= 1u << st;
      const uint32_t kcodes = ring + st * C::kCodeStage;
      const uint32_t vcodes = kcodes + C::kTile8;
      const uint8_t* kptr = ring_ptr + st * C::kCodeStage;
      const int valid = min(kTileTokens, L - tile * kTileTokens);
      if (valid < kTileTokens) {
        // value rows past the sequence end hold whatever the pool holds
        for (int i = lane; i < (kTileTokens - valid) * (D / 16); i += 32) {
          const int r = valid + i / (D / 16), c = i % (D / 16);
          asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(vcodes + code_off<D>(r, c)),
                       "r"(0u)
                       : "memory");
        }
        __syncwarp();
      }
      const float* ksc = reinterpret_cast<const float*>(sring_ptr + st * C::kScaleStage);
      const float* vsc = ksc + kTileTokens;

      // S^T = K Q^T: the tile's 16 keys are the MMA rows, the 8 score
      // columns its columns. Row r holds key 4 (r >> 1) + (r & 1) for r < 8
      // and that key + 2 for row r + 8, so thread (g, t) loads keys kr0 (row
      // g) and kr1 (row g + 8) and holds their scores for columns 2t, 2t + 1;
      // after a transpose it holds columns g of keys 4t .. 4t+3, the rows its
      // value fragments cover.
      const int kr0 = 4 * (g >> 1) + (g & 1), kr1 = kr0 + 2;
      uint32_t kw0[KS], kw1[KS];
#pragma unroll
      for (int v = 0; v < KS / 4; ++v) {
        const uint4 u0 =
            *reinterpret_cast<const uint4*>(kptr + code_off<D>(kr0, (KS / 4) * t + v));
        const uint4 u1 =
            *reinterpret_cast<const uint4*>(kptr + code_off<D>(kr1, (KS / 4) * t + v));
        kw0[4 * v] = u0.x, kw0[4 * v + 1] = u0.y, kw0[4 * v + 2] = u0.z, kw0[4 * v + 3] = u0.w;
        kw1[4 * v] = u1.x, kw1[4 * v + 1] = u1.y, kw1[4 * v + 2] = u1.z, kw1[4 * v + 3] = u1.w;
      }
      float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};  // even, odd k-steps
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t x0, x1, y0, y1;
        e4m3x4_to_f16x4(kw0[ks], x0, x1);
        e4m3x4_to_f16x4(kw1[ks], y0, y1);
        if (ks & 1)
          mma_f16_16816(sb, x0, y0, x1, y1, qa[ks][0], qa[ks][1]);
        else
          mma_f16_16816(sa, x0, y0, x1, y1, qa[ks][0], qa[ks][1]);
      }

      const bool ok0 = kr0 < valid, ok1 = kr1 < valid;
      const float sk0 = ksc[kr0] * a.scale_log2, sk1 = ksc[kr1] * a.scale_log2;
      // x: (key kr0, column 2t), (kr0, 2t + 1), (kr1, 2t), (kr1, 2t + 1)
      float x[4];
      x[0] = ok0 ? (sa[0] + sb[0]) * sk0 : -INFINITY;
      x[1] = ok0 ? (sa[1] + sb[1]) * sk0 : -INFINITY;
      x[2] = ok1 ? (sa[2] + sb[2]) * sk1 : -INFINITY;
      x[3] = ok1 ? (sa[3] + sb[3]) * sk1 : -INFINITY;
      float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float al0 = fast_exp2(m0 - mn0), al1 = fast_exp2(m1 - mn1);
      float pr[4];
      pr[0] = fast_exp2(x[0] - mn0);
      pr[1] = fast_exp2(x[1] - mn1);
      pr[2] = fast_exp2(x[2] - mn0);
      pr[3] = fast_exp2(x[3] - mn1);
      l0 = l0 * al0 + (pr[0] + pr[2]);
      l1 = l1 * al1 + (pr[1] + pr[3]);
      m0 = mn0;
      m1 = mn1;
      if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {  // a running max moved
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          o[c][0] *= al0;
          o[c][1] *= al1;
          o[c][2] *= al0;
          o[c][3] *= al1;
        }
      }
      // P' = p * s_v in fp16 hi + lo; keys past the end carry p = 0 (and a
      // zero scale: their scale slots are stale) and a zeroed value row
      const float sv0 = ok0 ? vsc[kr0] : 0.f, sv1 = ok1 ? vsc[kr1] : 0.f;
      const float pv0 = pr[0] * sv0, pv1 = pr[1] * sv0, pv2 = pr[2] * sv1, pv3 = pr[3] * sv1;
      const uint32_t hA = pack_f16x2(pv0, pv1), hB = pack_f16x2(pv2, pv3);
      const uint32_t lA = pack_f16x2(pv0 - f16_lo_to_f32(hA), pv1 - f16_hi_to_f32(hA));
      const uint32_t lB = pack_f16x2(pv2 - f16_lo_to_f32(hB), pv3 - f16_hi_to_f32(hB));
      // the 8 x 8 blocks (rows 0..7 and 8..15) transposed: column g of keys
      // (4t, 4t+1) and (4t+2, 4t+3); columns 4..7 carry the lo parts (G <= 4)
      const bool lo_col = kLoRows && t >= 2;
      const uint32_t pb0 = movmatrix_trans_b16(lo_col ? lA : hA);
      const uint32_t pb2 = movmatrix_trans_b16(lo_col ? lB : hB);
      uint32_t pl0 = 0u, pl2 = 0u;
      if constexpr (!kLoRows) {
        pl0 = movmatrix_trans_b16(lA);
        pl2 = movmatrix_trans_b16(lB);
      }
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        uint32_t r0, r1;
        ldmatrix_b8_16x16_trans(vcodes + code_off<D>(lane & 15, c), r0, r1);
        // v0, v1: keys (4t, 4t+1), (4t+2, 4t+3) of value column 16c + g;
        // v2, v3: the same keys of column 16c + 8 + g
        uint32_t v0, v1, v2, v3;
        e4m3x4_to_f16x4(r0, v0, v1);
        e4m3x4_to_f16x4(r1, v2, v3);
        mma_f16_16816(o[c], v0, v2, v1, v3, pb0, pb2);
        if constexpr (!kLoRows) mma_f16_16816(o[c], v0, v2, v1, v3, pl0, pl2);
      }
      if (valid < kTileTokens) fence_proxy_async_smem();  // zeroing stores before TMA reuse
      __syncwarp();
      if (k + C::kStages < n_mine) issue(k + C::kStages, st);
    }

#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    __syncthreads();
    if (s_abort) return;
    float2* cml = reinterpret_cast<float2*>(base_ptr);
    float* co = reinterpret_cast<float*>(base_ptr + 256);
    if (g == 0 && (!kLoRows || t < 2)) {
      if (2 * t < G) cml[warp * G + 2 * t] = make_float2(m0, l0);
      if (2 * t + 1 < G) cml[warp * G + 2 * t + 1] = make_float2(m1, l1);
    }
    if constexpr (kLoRows) {
      // columns 4 + r (lo) sit two lanes up from columns r (hi)
#pragma unroll
      for (int c = 0; c < NC; ++c)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[c][e] += __shfl_down_sync(0xffffffffu, o[c][e], 2);
    }
    if (!kLoRows || t < 2) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int h = 2 * t + j;
        if (h < G) {
          float* row = co + (warp * G + h) * D;
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            row[16 * c + g] = o[c][j];
            row[16 * c + 8 + g] = o[c][2 + j];
          }
        }
      }
    }
    __syncthreads();
    const int nparts = (L + P - 1) / P;
    for (int e = tid; e < G * D; e += kThreads) {
      const int h = e / D, d = e % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, cml[w * G + h].x);
      float lsum = 0.f, acc = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float sw = fast_exp2(cml[w * G + h].x - M);
        lsum += sw * cml[w * G + h].y;
        acc += sw * co[(w * G + h) * D + d];
      }
      const int64_t qh = (int64_t)s * a.Hq + kvh * G + h;
      if (nparts == 1) {
        a.out[qh * D + d] = __float2bfloat16_rn(acc / lsum);
      } else {
        const int64_t idx = qh * a.max_partitions + p;
        a.ws_o[idx * D + d] = acc;
        if (d == 0) a.ws_ml[idx] = make_float2(M, lsum);
      }
    }
    fence_proxy_async_smem();  // merge-buffer stores before the ring's next TMA writes
    __syncthreads();
    cur = s_next;
  }
}

// ---------------------------------------------------------------------------
// Shared-prefix decode ("Batching, Scheduling, and Paging", section Block
// sharing: parallel samples point at the same physical blocks for their
// common prefix). A group's members share their first tokens' blocks, so the
// group's prefix is read once for up to 16 / G members: their (member, query
// head) pairs form the 16 rows of the MMA operand. The rest of each member's
// context is decoded as usual. A member's partial states are its shared
// partitions followed by its private ones; the combine kernel merges them.
//
// Item kinds: 1 = (group, shared partition, member chunk), 0 = (sequence,
// private partition), each written resolved as two int4 so that a CTA starts
// an item from one load: (kind, first member's sequence, first token, end
// token) and (index of the chunk's first member in grp_members, members,
// partition index within each member's partial states, 0). Built by one CTA
// with atomics (the item order does not affect any result: each item's
// arithmetic depends only on its own data and the merge runs in partition
// order).
__global__ void __launch_bounds__(1024) decode_group_plan_kernel(DecodeArgs a) {
  __shared__ int32_t s_n;
  const int tid = threadIdx.x;
  const int P = a.partition_tiles * kTileTokens;
  const int M = a.members_per_item;
  grid_dep_launch();
  grid_dep_wait();  // launched early: whatever ran before is complete
  if (tid == 0) s_n = 0;
  for (int s = tid; s < a.S; s += 1024) a.seq_shared[s] = 0;
  __syncthreads();
  for (int g = tid; g < a.n_groups; g += 1024) {
    const int b = __ldg(a.grp_start + g), e = __ldg(a.grp_start + g + 1);
    if (b < 0 || e < b) {
      record_status(a.status, PKV_EDEVICE, g, kKernelDecodePlan);
      continue;
    }
    int minL = 1 << 30;
    bool bad = false;
    for (int i = b; i < e; ++i) {
      const int s = __ldg(a.grp_members + i);
      if (s < 0 || s >= a.S) {
        bad = true;
        break;
      }
      const int L = __ldg(a.context_lens + s);
      minL = min(minL, (L < 1 || L > a.max_context_len) ? 0 : L);
    }
    if (bad || e == b) {
      if (bad) record_status(a.status, PKV_EDEVICE, g, kKernelDecodePlan);
      continue;
    }
    // whole tiles only, and never past a member's end
    const int sh = min(max(__ldg(a.grp_shared + g), 0), minL) / kTileTokens * kTileTokens;
    if (sh == 0) continue;
    for (int i = b; i < e; ++i) a.seq_shared[__ldg(a.grp_members + i)] = sh;
    const int nsp = (sh + P - 1) / P, chunks = (e - b + M - 1) / M;
    const int k = atomicAdd(&s_n, nsp * chunks);
    if (k + nsp * chunks > a.item_cap) {
      record_status(a.status, PKV_EDEVICE, g, kKernelDecodePlan);
      continue;
    }
    for (int p = 0; p < nsp; ++p)
      for (int c = 0; c < chunks; ++c) {
        const int i = 2 * (k + p * chunks + c), mb = b + c * M;
        a.gitems[i] = make_int4(1, __ldg(a.grp_members + mb), p * P, min(p * P + P, sh));
        a.gitems[i + 1] = make_int4(mb, min(M, e - mb), p, 0);
      }
  }
  __syncthreads();
  for (int s = tid; s < a.S; s += 1024) {
    const int L = __ldg(a.context_lens + s);
    if (L < 1 || L > a.max_context_len) {
      record_status(a.status, PKV_EDEVICE, L, kKernelDecodePlan);
      continue;
    }
    const int sh = a.seq_shared[s];
    const int np = (L - sh + P - 1) / P;
    if (np == 0) continue;
    const int k = atomicAdd(&s_n, np);
    if (k + np > a.item_cap) {
      record_status(a.status, PKV_EDEVICE, s, kKernelDecodePlan);
      continue;
    }
    const int nsp = (sh + P - 1) / P;
    for (int p = 0; p < np; ++p) {
      a.gitems[2 * (k + p)] = make_int4(0, s, sh + p * P, min(sh + p * P + P, L));
      a.gitems[2 * (k + p) + 1] = make_int4(0, 1, nsp + p, 0);
    }
  }
  __syncthreads();
  if (tid == 0) {
    *a.n_items = min(s_n, a.item_cap);
    *a.ticket = 0;
  }
}

// Decode of group items: up to 16 rows (member, query head) per kv head; each
// thread owns rows g and g + 8 of the MMA fragments. P enters the P V product
// as two MMAs (bf16 hi, then lo), since all 16 operand rows may be in use.
template <int D, int G>
__global__ void __launch_bounds__(kThreads, 3)
    paged_decode_group_kernel(const __grid_constant__ CUtensorMap tmap_k,
                              const __grid_constant__ CUtensorMap tmap_v, const DecodeArgs a) {
  using C = Cfg<D>;  // three CTAs per SM (168 registers)
  constexpr int KS = D / 16;
  constexpr int NT = D / 8;
  constexpr int M = 16 / G;  // members per item
  static_assert(512 + kWarps * 16 * D * 4 <= kWarps * C::kRingBytes,
                "the merge buffer reuses the rings");
  extern __shared__ uint8_t dsm[];
  __shared__ __align__(8) uint64_t bars[kWarps][C::kStages];
  __shared__ int32_t s_next;
  __shared__ int32_t s_abort;
  __shared__ int32_t s_mem[M];  // the item's members (sequences)
  __shared__ int32_t s_np[M];   // their partial-state counts
  __shared__ int32_t s_nm, s_part;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t dsm_u32 = smem_u32(dsm);
  const uint32_t base = (dsm_u32 + 1023u) & ~1023u;
  uint8_t* base_ptr = dsm + (base - dsm_u32);
  const uint32_t ring = base + warp * C::kRingBytes;

  if (lane == 0) {
#pragma unroll
    for (int st = 0; st < C::kStages; ++st) mbar_init(smem_u32(&bars[warp][st]), 1);
    fence_barrier_init();
  }
  grid_dep_launch();
  grid_dep_wait();
  if (tid == 0) {
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
    s_abort = 0;
    s_next = atomicAdd(a.ticket, 1);
  }
  __syncthreads();
  const int total = __ldg(a.n_items) * a.Hkv;
  const int P = a.partition_tiles * kTileTokens;
  uint32_t phase = 0;
  int cur = s_next;

  while (cur < total) {
    __syncthreads();  // everyone has read s_next; the rings and s_mem are free
    // The item from one load; the loads of the first tiles go out before
    // anything waits on the members or on the next ticket.
    const int4 h0 = __ldg(a.gitems + 2 * (cur / a.Hkv));
    const int4 h1 = __ldg(a.gitems + 2 * (cur / a.Hkv) + 1);
    const int kvh = cur % a.Hkv;
    const int first = h0.y, r_begin = h0.z, r_end = h0.w;  // token range
    const int nm = h1.y;                                    // members
    const int t_begin = r_begin / kTileTokens;
    const int t_end = (r_end + kTileTokens - 1) / kTileTokens;
    const int n_item = t_end - t_begin;
    const int n_mine = n_item > warp ? (n_item - warp + kWarps - 1) / kWarps : 0;
    const int32_t* bt = a.block_tables + (int64_t)first * a.max_blocks_per_seq;

    TileRows mine = {{-1, -1}, 0u};
    int chunk0 = 0;
    if (lane < n_mine) mine = tile_rows<D>(a, bt, kvh, t_begin + warp + lane * kWarps, r_end);
    auto issue = [&](int k, uint32_t st) {
      if (k - chunk0 >= 32) {
        chunk0 += 32;
        mine = {{-1, -1}, 0u};
        if (chunk0 + lane < n_mine)
          mine = tile_rows<D>(a, bt, kvh, t_begin + warp + (chunk0 + lane) * kWarps, r_end);
      }
      const int src = k - chunk0;
      const int32_t q0 = __shfl_sync(0xffffffffu, mine.row[0], src);
      const int32_t q1 = __shfl_sync(0xffffffffu, mine.row[1], src);
      const uint32_t by = __shfl_sync(0xffffffffu, mine.bytes, src);
      issue_tile_rows<D>(&tmap_k, &tmap_v, a.block_size, q0, q1, by, ring + st * C::kStageBytes,
                         smem_u32(&bars[warp][st]), lane);
    };
    {
      const int npro = n_mine < C::kStages ? n_mine : C::kStages;
      for (int k = 0; k < npro; ++k) issue(k, k);
    }
    // the members, and for the merge their context and shared lengths (not
    // waited on until then); the next ticket is stored only at the item's end
    int mem_L = 0, mem_sh = 0, nxt = 0;
    if (tid < nm) {
      const int sq = h0.x == 1 ? __ldg(a.grp_members + h1.x + tid) : first;
      s_mem[tid] = sq;
      mem_L = __ldg(a.context_lens + sq);
      mem_sh = a.seq_shared[sq];
    }
    if (tid == 0) {
      s_nm = nm;
      s_part = h1.z;
      nxt = atomicAdd(a.ticket, 1);
    }
    __syncthreads();

    // Q fragments for rows g and g + 8: row r is (member r / G, head r % G)
    uint32_t qa[KS][4];
    {
      const int r0 = g, r1 = g + 8;
      const bool l0 = r0 / G < nm, l1 = r1 / G < nm;
      const __nv_bfloat16* q0 =
          a.q + ((int64_t)s_mem[l0 ? r0 / G : 0] * a.Hq + kvh * G + r0 % G) * D;
      const __nv_bfloat16* q1 =
          a.q + ((int64_t)s_mem[l1 ? r1 / G : 0] * a.Hq + kvh * G + r1 % G) * D;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qa[ks][0] = l0 ? __ldg(reinterpret_cast<const uint32_t*>(q0 + ks * 16 + 2 * t)) : 0u;
        qa[ks][1] = l1 ? __ldg(reinterpret_cast<const uint32_t*>(q1 + ks * 16 + 2 * t)) : 0u;
        qa[ks][2] = l0 ? __ldg(reinterpret_cast<const uint32_t*>(q0 + ks * 16 + 8 + 2 * t)) : 0u;
        qa[ks][3] = l1 ? __ldg(reinterpret_cast<const uint32_t*>(q1 + ks * 16 + 8 + 2 * t)) : 0u;
      }
    }

    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    float o[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;

    for (int k = 0; k < n_mine; ++k) {
      const int st = k % C::kStages;
      const int tile = t_begin + warp + k * kWarps;
      const uint32_t bar = smem_u32(&bars[warp][st]);
      const uint32_t par = (phase >> st) & 1u;
      const bool landed = mbar_wait_bounded(bar, par, a.timeout_ns, a.force_timeout);
      if (!__all_sync(0xffffffffu, landed)) {
        if (lane == 0) {
          record_status(a.status, PKV_ETIMEOUT, k, kKernelDecode);
          s_abort = 1;
        }
        uint32_t ph = phase;
        const int last = min(k + C::kStages, n_mine);
        for (int j = k; j < last; ++j) {
          const int sj = j % C::kStages;
          mbar_wait_bounded(smem_u32(&bars[warp][sj]), (ph >> sj) & 1u, 4 * a.timeout_ns, 0);
          ph ^= 1u << sj;
        }
        phase = ph;
        break;
      }
      phase ^= 1u << st;
      const uint32_t stage = ring + st * C::kStageBytes;
      const int valid = min(kTileTokens, r_end - tile * kTileTokens);
      if (valid < kTileTokens) {
        const int n16 = (kTileTokens - valid) * C::kHalves * 8;
        for (int i = lane; i < n16; i += 32) {
          const int row = valid + i / (C::kHalves * 8);
          const int rem = i % (C::kHalves * 8);
          const uint32_t addr = stage + C::kTensorBytes + (rem >> 3) * C::kHalfBytes + row * 128 +
                                (rem & 7) * 16;
          asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u)
                       : "memory");
        }
        __syncwarp();
      }

      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      {
        const int tok = (lane & 7) + ((lane >> 4) << 3);
        const int csel = (lane >> 3) & 1;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          const int chunk = 2 * ks + csel;
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(stage + (chunk >> 3) * C::kHalfBytes + swz128(tok, chunk & 7), b0, b1, b2,
                      b3);
          mma_bf16_16816(sc[0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
          mma_bf16_16816(sc[1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
        }
      }

      // online softmax on rows g (fragment entries 0, 1) and g + 8 (2, 3)
      float pr[2][4];
      float alpha[2];
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        float x[4];
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int e = 0; e < 2; ++e)
            x[2 * j + e] =
                (8 * j + 2 * t + e < valid) ? sc[j][2 * hr + e] * a.scale_log2 : -INFINITY;
        float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m[hr], mx);
        alpha[hr] = fast_exp2(m[hr] - m_new);
#pragma unroll
        for (int i = 0; i < 4; ++i) pr[hr][i] = fast_exp2(x[i] - m_new);
        l[hr] = l[hr] * alpha[hr] + ((pr[hr][0] + pr[hr][1]) + (pr[hr][2] + pr[hr][3]));
        m[hr] = m_new;
      }
      if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          o[nt][0] *= alpha[0];
          o[nt][1] *= alpha[0];
          o[nt][2] *= alpha[1];
          o[nt][3] *= alpha[1];
        }
      }
      // P = P_hi + P_lo, each a full 16-row bf16 operand
      uint32_t ph[4], pl[4];
#pragma unroll
      for (int hr = 0; hr < 2; ++hr)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float p0 = pr[hr][2 * j], p1 = pr[hr][2 * j + 1];
          const uint32_t hi = pack_bf16x2(p0, p1);
          ph[2 * j + hr] = hi;  // a0: row g keys 2t; a1: row g+8; a2/a3: keys 8+2t
          pl[2 * j + hr] = pack_bf16x2(p0 - bf16_lo_to_f32(hi), p1 - bf16_hi_to_f32(hi));
        }
      {
        const int tok = (lane & 7) + (((lane >> 3) & 1) << 3);
        const int csel = lane >> 4;
#pragma unroll
        for (int n2 = 0; n2 < NT / 2; ++n2) {
          const int chunk = 2 * n2 + csel;
          uint32_t r0, r1, r2, r3;
          ldmatrix_x4_trans(
              stage + C::kTensorBytes + (chunk >> 3) * C::kHalfBytes + swz128(tok, chunk & 7), r0,
              r1, r2, r3);
          mma_bf16_16816(o[2 * n2], ph[0], ph[1], ph[2], ph[3], r0, r1);
          mma_bf16_16816(o[2 * n2], pl[0], pl[1], pl[2], pl[3], r0, r1);
          mma_bf16_16816(o[2 * n2 + 1], ph[0], ph[1], ph[2], ph[3], r2, r3);
          mma_bf16_16816(o[2 * n2 + 1], pl[0], pl[1], pl[2], pl[3], r2, r3);
        }
      }
      if (valid < kTileTokens) fence_proxy_async_smem();
      __syncwarp();
      if (k + C::kStages < n_mine) issue(k + C::kStages, st);
    }

#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      l[hr] += __shfl_xor_sync(0xffffffffu, l[hr], 1);
      l[hr] += __shfl_xor_sync(0xffffffffu, l[hr], 2);
    }
    if (tid < s_nm) s_np[tid] = (mem_sh + P - 1) / P + (mem_L - mem_sh + P - 1) / P;
    if (tid == 0) s_next = nxt;
    __syncthreads();
    if (s_abort) return;
    constexpr int R = 16;
    float2* cml = reinterpret_cast<float2*>(base_ptr);     // [kWarps][R]
    float* co = reinterpret_cast<float*>(base_ptr + 512);  // [kWarps][R][D]
    {
      if (t == 0) {
        cml[warp * R + g] = make_float2(m[0], l[0]);
        cml[warp * R + g + 8] = make_float2(m[1], l[1]);
      }
      float* row0 = co + (warp * R + g) * D;
      float* row1 = co + (warp * R + g + 8) * D;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        *reinterpret_cast<float2*>(row0 + nt * 8 + 2 * t) = make_float2(o[nt][0], o[nt][1]);
        *reinterpret_cast<float2*>(row1 + nt * 8 + 2 * t) = make_float2(o[nt][2], o[nt][3]);
      }
    }
    __syncthreads();
    const int rows = s_nm * G;
    for (int e = tid; e < rows * D; e += kThreads) {
      const int r = e / D, d = e % D;
      float Mx = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) Mx = fmaxf(Mx, cml[w * R + r].x);
      float lsum = 0.f, acc = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float sw = fast_exp2(cml[w * R + r].x - Mx);
        lsum += sw * cml[w * R + r].y;
        acc += sw * co[(w * R + r) * D + d];
      }
      const int sq = s_mem[r / G];
      const int nparts = s_np[r / G];
      const int part = s_part;
      const int64_t qh = (int64_t)sq * a.Hq + kvh * G + r % G;
      if (nparts == 1) {
        a.out[qh * D + d] = __float2bfloat16_rn(acc / lsum);
      } else {
        const int64_t idx = qh * a.max_partitions + part;
        a.ws_o[idx * D + d] = acc;
        if (d == 0) a.ws_ml[idx] = make_float2(Mx, lsum);
      }
    }
    fence_proxy_async_smem();
    __syncthreads();
    cur = s_next;
  }
}

// Launches a one-CTA plan kernel that may start while the previous kernel in
// the stream ends (it waits for it before touching memory).
template <typename Args>
int launch_plan(void (*kernel)(Args), const Args& a, cudaStream_t stream, const char* what) {
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(1024);
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, a);
  if (err != cudaSuccess) return cuda_fail(err, what);
  return PKV_OK;
}

template <int D, int G>
int launch_decode_group(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                        const DeviceInfo& dev, cudaStream_t stream) {
  using C = Cfg<D>;
  static std::once_flag once;
  static int blocks_per_sm = 0;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, []() {
    attr_err = cudaFuncSetAttribute(paged_decode_group_kernel<D, G>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (attr_err == cudaSuccess)
      attr_err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &blocks_per_sm, paged_decode_group_kernel<D, G>, kThreads, C::kSmemBytes);
  });
  if (attr_err != cudaSuccess) return cuda_fail(attr_err, "shared decode kernel attributes");
  if (blocks_per_sm < 1) return fail(PKV_ECUDA, "shared decode kernel does not fit on an SM");
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  if (int rc = launch_plan(decode_group_plan_kernel, a, stream, "decode plan launch")) return rc;
  if (int rc = check_launch("shared decode plan")) return rc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(dev.sm_count * blocks_per_sm));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  cudaError_t err = cudaLaunchKernelEx(&cfg, paged_decode_group_kernel<D, G>, tk, tv, a);
  if (err != cudaSuccess) return cuda_fail(err, "shared decode launch");
  const int64_t pairs = (int64_t)a.S * a.Hq;
  cfg.gridDim = dim3((unsigned)((pairs + 3) / 4));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  err = cudaLaunchKernelEx(&cfg, decode_combine_kernel<D>, a);
  if (err != cudaSuccess) return cuda_fail(err, "decode combine launch");
  return PKV_OK;
}

int resolve_partition(int32_t partition_size, int32_t* tiles) {
  const int32_t P = partition_size == 0 ? kDefaultPartition : partition_size;
  PKV_REQUIRE(P >= kTileTokens && P % kTileTokens == 0 && P <= (1 << 20),
              "partition_size must be a positive multiple of 16 (got %d)", partition_size);
  *tiles = P / kTileTokens;
  return PKV_OK;
}

template <int D, int G>
int launch_decode(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                  const DeviceInfo& dev, cudaStream_t stream) {
  using C = Cfg<D>;
  static std::once_flag once;
  static int blocks_per_sm = 0;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, []() {
    attr_err = cudaFuncSetAttribute(paged_decode_kernel<D, G>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (attr_err == cudaSuccess)
      attr_err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &blocks_per_sm, paged_decode_kernel<D, G>, kThreads, C::kSmemBytes);
  });
  if (attr_err != cudaSuccess) return cuda_fail(attr_err, "decode kernel attributes");
  if (blocks_per_sm < 1) return fail(PKV_ECUDA, "decode kernel does not fit on an SM");
  // plan -> decode -> combine, each dependent launch overlapping its set-up
  // with the end of its predecessor (programmatic stream serialisation)
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  if (int rc = launch_plan(decode_plan_kernel, a, stream, "decode plan launch")) return rc;
  if (int rc = check_launch("decode plan")) return rc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(dev.sm_count * blocks_per_sm));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  cudaError_t err = cudaLaunchKernelEx(&cfg, paged_decode_kernel<D, G>, tk, tv, a);
  if (err != cudaSuccess) return cuda_fail(err, "decode launch");
  if (a.max_partitions > 1) {
    const int64_t pairs = (int64_t)a.S * a.Hq;
    cfg.gridDim = dim3((unsigned)((pairs + 3) / 4));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    err = cudaLaunchKernelEx(&cfg, decode_combine_kernel<D>, a);
    if (err != cudaSuccess) return cuda_fail(err, "decode combine launch");
  }
  return PKV_OK;
}

template <int D, int G>
int launch_decode_fp8(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                      const DeviceInfo& dev, cudaStream_t stream) {
  using C = Cfg8<D>;
  static std::once_flag once;
  static int blocks_per_sm = 0;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, []() {
    attr_err = cudaFuncSetAttribute(paged_decode_fp8_kernel<D, G>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (attr_err == cudaSuccess)
      attr_err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &blocks_per_sm, paged_decode_fp8_kernel<D, G>, kThreads, C::kSmemBytes);
  });
  if (attr_err != cudaSuccess) return cuda_fail(attr_err, "fp8 decode kernel attributes");
  if (blocks_per_sm < 1) return fail(PKV_ECUDA, "fp8 decode kernel does not fit on an SM");
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  if (int rc = launch_plan(decode_plan_kernel, a, stream, "decode plan launch")) return rc;
  if (int rc = check_launch("decode plan")) return rc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(dev.sm_count * blocks_per_sm));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  cudaError_t err = cudaLaunchKernelEx(&cfg, paged_decode_fp8_kernel<D, G>, tk, tv, a);
  if (err != cudaSuccess) return cuda_fail(err, "fp8 decode launch");
  if (a.max_partitions > 1) {
    const int64_t pairs = (int64_t)a.S * a.Hq;
    cfg.gridDim = dim3((unsigned)((pairs + 3) / 4));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    err = cudaLaunchKernelEx(&cfg, decode_combine_kernel<D>, a);
    if (err != cudaSuccess) return cuda_fail(err, "decode combine launch");
  }
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" int pkv_decode_workspace_bytes(int32_t S, int32_t Hq, int32_t D,
                                          int32_t max_context_len, int32_t partition_size,
                                          size_t* out) {
  PKV_REQUIRE(out, "pkv_decode_workspace_bytes: out is NULL");
  PKV_REQUIRE(S >= 0 && Hq > 0 && (D == 64 || D == 128) && max_context_len >= 0,
              "pkv_decode_workspace_bytes: bad sizes");
  int32_t tiles = 0;
  if (int rc = resolve_partition(partition_size, &tiles)) return rc;
  const int64_t P = (int64_t)tiles * kTileTokens;
  const int64_t max_parts = max_context_len > 0 ? (max_context_len + P - 1) / P : 1;
  *out = ws_layout(S, Hq, D, max_parts).total;
  return ok();
}

extern "C" int pkv_paged_attention_decode(void* out, const void* q, const void* k_cache,
                                          const void* v_cache, const int32_t* block_tables,
                                          int32_t max_blocks_per_seq,
                                          const int32_t* context_lens, int32_t max_context_len,
                                          int32_t S, int32_t Hq, int32_t Hkv, int32_t D,
                                          int32_t block_size, int32_t num_blocks, float scale,
                                          int32_t partition_size, void* workspace,
                                          size_t workspace_bytes, int32_t* dev_status,
                                          void* stream) {
  PKV_REQUIRE(S >= 0, "decode: S must be >= 0");
  PKV_REQUIRE(Hkv > 0 && Hq > 0 && Hq % Hkv == 0, "decode: Hq (%d) must be a multiple of Hkv (%d)",
              Hq, Hkv);
  const int G = Hq / Hkv;
  PKV_REQUIRE(G == 1 || G == 2 || G == 4 || G == 8, "decode: Hq/Hkv must be 1, 2, 4 or 8 (got %d)",
              G);
  PKV_REQUIRE(D == 64 || D == 128, "decode: D must be 64 or 128 (got %d)", D);
  PKV_REQUIRE(block_size == 8 || block_size == 16 || block_size == 32,
              "decode: block_size must be 8, 16 or 32 (got %d)", block_size);
  PKV_REQUIRE(num_blocks > 0 && (int64_t)num_blocks * Hkv * block_size < (int64_t(1) << 31),
              "decode: num_blocks * Hkv * block_size must be in [1, 2^31)");
  PKV_REQUIRE(max_context_len >= 1, "decode: max_context_len must be >= 1");
  PKV_REQUIRE((int64_t)max_blocks_per_seq * block_size >= max_context_len,
              "decode: max_context_len %d exceeds max_blocks_per_seq * block_size", max_context_len);
  PKV_REQUIRE(std::isfinite(scale), "decode: scale must be finite");
  if (S == 0) return ok();
  PKV_REQUIRE(out && q && k_cache && v_cache && block_tables && context_lens && workspace,
              "decode: NULL pointer");
  PKV_REQUIRE(aligned16(out) && aligned16(q) && aligned16(k_cache) && aligned16(v_cache),
              "decode: bf16 arrays must be 16-byte aligned");
  PKV_REQUIRE((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0,
              "decode: workspace must be 256-byte aligned");
  int32_t tiles = 0;
  if (int rc = resolve_partition(partition_size, &tiles)) return rc;
  const int64_t P = (int64_t)tiles * kTileTokens;
  const int64_t max_parts = (max_context_len + P - 1) / P;
  const WsLayout ws = ws_layout(S, Hq, D, max_parts);
  PKV_REQUIRE(workspace_bytes >= ws.total, "decode: workspace has %zu bytes, needs %zu",
              workspace_bytes, ws.total);
  const DeviceInfo* dev = nullptr;
  if (int rc = current_device_info(&dev)) return rc;

  CUtensorMap tk, tv;
  const uint64_t rows = (uint64_t)num_blocks * Hkv * block_size;
  const uint32_t box_rows = block_size < kTileTokens ? block_size : kTileTokens;
  if (int rc = encode_tile_map_2d(&tk, k_cache, D, rows, (uint64_t)D * 2, 64, box_rows)) return rc;
  if (int rc = encode_tile_map_2d(&tv, v_cache, D, rows, (uint64_t)D * 2, 64, box_rows)) return rc;

  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  DecodeArgs a = {};
  a.out = static_cast<__nv_bfloat16*>(out);
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.S = S;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.num_blocks = num_blocks;
  a.block_size = block_size;
  a.max_context_len = max_context_len;
  a.partition_tiles = tiles;
  a.max_partitions = (int32_t)max_parts;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.ticket = reinterpret_cast<int32_t*>(wsb);
  a.n_items = reinterpret_cast<int32_t*>(wsb) + 1;
  a.items = reinterpret_cast<int2*>(wsb + ws.items_off);
  a.ws_ml = reinterpret_cast<float2*>(wsb + ws.ml_off);
  a.ws_o = reinterpret_cast<float*>(wsb + ws.o_off);
  a.status = dev_status;
  const WaitConfig wc = wait_config();
  a.timeout_ns = wc.timeout_ns;
  a.force_timeout = wc.force_timeout;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int rc = PKV_OK;
#define PKV_DECODE_CASE(DD, GG) \
  if (D == DD && G == GG) rc = launch_decode<DD, GG>(tk, tv, a, *dev, st);
  PKV_DECODE_CASE(64, 1)
  PKV_DECODE_CASE(64, 2)
  PKV_DECODE_CASE(64, 4)
  PKV_DECODE_CASE(64, 8)
  PKV_DECODE_CASE(128, 1)
  PKV_DECODE_CASE(128, 2)
  PKV_DECODE_CASE(128, 4)
  PKV_DECODE_CASE(128, 8)
#undef PKV_DECODE_CASE
  if (rc) return rc;
  return ok();
}

extern "C" int pkv_paged_attention_decode_fp8(
    void* out, const void* q, const void* k_codes, const void* v_codes, const float* k_scales,
    const float* v_scales, const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* context_lens, int32_t max_context_len, int32_t S, int32_t Hq, int32_t Hkv,
    int32_t D, int32_t block_size, int32_t num_blocks, float scale, int32_t partition_size,
    void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
  PKV_REQUIRE(S >= 0, "decode_fp8: S must be >= 0");
  PKV_REQUIRE(Hkv > 0 && Hq > 0 && Hq % Hkv == 0,
              "decode_fp8: Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
  const int G = Hq / Hkv;
  PKV_REQUIRE(G == 1 || G == 2 || G == 4 || G == 8,
              "decode_fp8: Hq/Hkv must be 1, 2, 4 or 8 (got %d)", G);
  PKV_REQUIRE(D == 64 || D == 128, "decode_fp8: D must be 64 or 128 (got %d)", D);
  PKV_REQUIRE(block_size == 8 || block_size == 16 || block_size == 32,
              "decode_fp8: block_size must be 8, 16 or 32 (got %d)", block_size);
  PKV_REQUIRE(num_blocks > 0 && (int64_t)num_blocks * Hkv * block_size < (int64_t(1) << 31),
              "decode_fp8: num_blocks * Hkv * block_size must be in [1, 2^31)");
  PKV_REQUIRE(max_context_len >= 1, "decode_fp8: max_context_len must be >= 1");
  PKV_REQUIRE((int64_t)max_blocks_per_seq * block_size >= max_context_len,
              "decode_fp8: max_context_len %d exceeds max_blocks_per_seq * block_size",
              max_context_len);
  PKV_REQUIRE(std::isfinite(scale), "decode_fp8: scale must be finite");
  if (S == 0) return ok();
  PKV_REQUIRE(out && q && k_codes && v_codes && k_scales && v_scales && block_tables &&
                  context_lens && workspace,
              "decode_fp8: NULL pointer");
  PKV_REQUIRE(aligned16(out) && aligned16(q) && aligned16(k_codes) && aligned16(v_codes) &&
                  aligned16(k_scales) && aligned16(v_scales),
              "decode_fp8: arrays must be 16-byte aligned");
  PKV_REQUIRE((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0,
              "decode_fp8: workspace must be 256-byte aligned");
  int32_t tiles = 0;
  if (int rc = resolve_partition(partition_size, &tiles)) return rc;
  const int64_t P = (int64_t)tiles * kTileTokens;
  const int64_t max_parts = (max_context_len + P - 1) / P;
  const WsLayout ws = ws_layout(S, Hq, D, max_parts);
  PKV_REQUIRE(workspace_bytes >= ws.total, "decode_fp8: workspace has %zu bytes, needs %zu",
              workspace_bytes, ws.total);
  const DeviceInfo* dev = nullptr;
  if (int rc = current_device_info(&dev)) return rc;

  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  DecodeArgs a = {};
  a.out = static_cast<__nv_bfloat16*>(out);
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.S = S;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.num_blocks = num_blocks;
  a.block_size = block_size;
  a.max_context_len = max_context_len;
  a.partition_tiles = tiles;
  a.max_partitions = (int32_t)max_parts;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.ticket = reinterpret_cast<int32_t*>(wsb);
  a.n_items = reinterpret_cast<int32_t*>(wsb) + 1;
  a.items = reinterpret_cast<int2*>(wsb + ws.items_off);
  a.ws_ml = reinterpret_cast<float2*>(wsb + ws.ml_off);
  a.ws_o = reinterpret_cast<float*>(wsb + ws.o_off);
  a.status = dev_status;
  const WaitConfig wc = wait_config();
  a.timeout_ns = wc.timeout_ns;
  a.force_timeout = wc.force_timeout;
  a.k8 = static_cast<const uint8_t*>(k_codes);
  a.v8 = static_cast<const uint8_t*>(v_codes);
  a.ks = k_scales;
  a.vs = v_scales;
  CUtensorMap tk, tv;
  const uint64_t rows = (uint64_t)num_blocks * Hkv * block_size;
  const uint32_t box_rows = block_size < kTileTokens ? block_size : kTileTokens;
  if (int rc = encode_byte_rows_map(&tk, k_codes, D, rows, box_rows, D == 128)) return rc;
  if (int rc = encode_byte_rows_map(&tv, v_codes, D, rows, box_rows, D == 128)) return rc;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int rc = PKV_OK;
#define PKV_DECODE8_CASE(DD, GG) \
  if (D == DD && G == GG) rc = launch_decode_fp8<DD, GG>(tk, tv, a, *dev, st);
  PKV_DECODE8_CASE(64, 1)
  PKV_DECODE8_CASE(64, 2)
  PKV_DECODE8_CASE(64, 4)
  PKV_DECODE8_CASE(64, 8)
  PKV_DECODE8_CASE(128, 1)
  PKV_DECODE8_CASE(128, 2)
  PKV_DECODE8_CASE(128, 4)
  PKV_DECODE8_CASE(128, 8)
#undef PKV_DECODE8_CASE
  if (rc) return rc;
  return ok();
}

// Shared-prefix decode: workspace (header, items, per-sequence shared
// lengths, partial states with one extra partition per sequence).
struct WsShared {
  size_t items_off, shared_off, ml_off, o_off, total;
  int64_t item_cap, parts;
};

WsShared ws_shared_layout(int64_t S, int64_t Hq, int64_t D, int64_t max_parts) {
  WsShared w;
  w.parts = max_parts + 1;
  w.item_cap = 2 * S * max_parts + 1;
  w.items_off = 256;
  w.shared_off = align256(w.items_off + w.item_cap * 2 * sizeof(int4));
  w.ml_off = align256(w.shared_off + S * sizeof(int32_t));
  w.o_off = align256(w.ml_off + S * Hq * w.parts * sizeof(float2));
  w.total = align256(w.o_off + S * Hq * w.parts * D * sizeof(float));
  return w;
}

extern "C" int pkv_decode_shared_workspace_bytes(int32_t S, int32_t Hq, int32_t D,
                                                 int32_t max_context_len, int32_t partition_size,
                                                 size_t* out) {
  PKV_REQUIRE(out, "pkv_decode_shared_workspace_bytes: out is NULL");
  PKV_REQUIRE(S >= 0 && Hq > 0 && (D == 64 || D == 128) && max_context_len >= 0,
              "pkv_decode_shared_workspace_bytes: bad sizes");
  int32_t tiles = 0;
  if (int rc = resolve_partition(partition_size, &tiles)) return rc;
  const int64_t P = (int64_t)tiles * kTileTokens;
  const int64_t max_parts = max_context_len > 0 ? (max_context_len + P - 1) / P : 1;
  *out = ws_shared_layout(S, Hq, D, max_parts).total;
  return ok();
}

extern "C" int pkv_paged_attention_decode_shared(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* context_lens,
    int32_t max_context_len, const int32_t* group_start, const int32_t* group_members,
    const int32_t* group_shared, int32_t n_groups, int32_t S, int32_t Hq, int32_t Hkv, int32_t D,
    int32_t block_size, int32_t num_blocks, float scale, int32_t partition_size, void* workspace,
    size_t workspace_bytes, int32_t* dev_status, void* stream) {
  PKV_REQUIRE(S >= 0 && n_groups >= 0, "decode_shared: S and n_groups must be >= 0");
  PKV_REQUIRE(Hkv > 0 && Hq > 0 && Hq % Hkv == 0,
              "decode_shared: Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
  const int G = Hq / Hkv;
  PKV_REQUIRE(G == 1 || G == 2 || G == 4 || G == 8,
              "decode_shared: Hq/Hkv must be 1, 2, 4 or 8 (got %d)", G);
  PKV_REQUIRE(D == 64 || D == 128, "decode_shared: D must be 64 or 128 (got %d)", D);
  PKV_REQUIRE(block_size == 8 || block_size == 16 || block_size == 32,
              "decode_shared: block_size must be 8, 16 or 32 (got %d)", block_size);
  PKV_REQUIRE(num_blocks > 0 && (int64_t)num_blocks * Hkv * block_size < (int64_t(1) << 31),
              "decode_shared: num_blocks * Hkv * block_size must be in [1, 2^31)");
  PKV_REQUIRE(max_context_len >= 1, "decode_shared: max_context_len must be >= 1");
  PKV_REQUIRE((int64_t)max_blocks_per_seq * block_size >= max_context_len,
              "decode_shared: max_context_len %d exceeds max_blocks_per_seq * block_size",
              max_context_len);
  PKV_REQUIRE(std::isfinite(scale), "decode_shared: scale must be finite");
  if (S == 0) return ok();
  PKV_REQUIRE(out && q && k_cache && v_cache && block_tables && context_lens && workspace &&
                  (n_groups == 0 || (group_start && group_members && group_shared)),
              "decode_shared: NULL pointer");
  PKV_REQUIRE(aligned16(out) && aligned16(q) && aligned16(k_cache) && aligned16(v_cache),
              "decode_shared: bf16 arrays must be 16-byte aligned");
  PKV_REQUIRE((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0,
              "decode_shared: workspace must be 256-byte aligned");
  int32_t tiles = 0;
  if (int rc = resolve_partition(partition_size, &tiles)) return rc;
  const int64_t P = (int64_t)tiles * kTileTokens;
  const int64_t max_parts = (max_context_len + P - 1) / P;
  const WsShared ws = ws_shared_layout(S, Hq, D, max_parts);
  PKV_REQUIRE(workspace_bytes >= ws.total, "decode_shared: workspace has %zu bytes, needs %zu",
              workspace_bytes, ws.total);
  PKV_REQUIRE(ws.item_cap < (int64_t(1) << 31) / 16, "decode_shared: batch too large");
  const DeviceInfo* dev = nullptr;
  if (int rc = current_device_info(&dev)) return rc;

  CUtensorMap tk, tv;
  const uint64_t rows = (uint64_t)num_blocks * Hkv * block_size;
  const uint32_t box_rows = block_size < kTileTokens ? block_size : kTileTokens;
  if (int rc = encode_tile_map_2d(&tk, k_cache, D, rows, (uint64_t)D * 2, 64, box_rows)) return rc;
  if (int rc = encode_tile_map_2d(&tv, v_cache, D, rows, (uint64_t)D * 2, 64, box_rows)) return rc;

  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  DecodeArgs a = {};
  a.out = static_cast<__nv_bfloat16*>(out);
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.S = S;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.num_blocks = num_blocks;
  a.block_size = block_size;
  a.max_context_len = max_context_len;
  a.partition_tiles = tiles;
  a.max_partitions = (int32_t)ws.parts;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.ticket = reinterpret_cast<int32_t*>(wsb);
  a.n_items = reinterpret_cast<int32_t*>(wsb) + 1;
  a.gitems = reinterpret_cast<int4*>(wsb + ws.items_off);
  a.seq_shared = reinterpret_cast<int32_t*>(wsb + ws.shared_off);
  a.ws_ml = reinterpret_cast<float2*>(wsb + ws.ml_off);
  a.ws_o = reinterpret_cast<float*>(wsb + ws.o_off);
  a.status = dev_status;
  const WaitConfig wc = wait_config();
  a.timeout_ns = wc.timeout_ns;
  a.force_timeout = wc.force_timeout;
  a.grp_start = group_start;
  a.grp_members = group_members;
  a.grp_shared = group_shared;
  a.n_groups = n_groups;
  a.members_per_item = 16 / G;
  a.item_cap = (int32_t)ws.item_cap;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int rc = PKV_OK;
#define PKV_DECODEG_CASE(DD, GG) \
  if (D == DD && G == GG) rc = launch_decode_group<DD, GG>(tk, tv, a, *dev, st);
  PKV_DECODEG_CASE(64, 1)
  PKV_DECODEG_CASE(64, 2)
  PKV_DECODEG_CASE(64, 4)
  PKV_DECODEG_CASE(64, 8)
  PKV_DECODEG_CASE(128, 1)
  PKV_DECODEG_CASE(128, 2)
  PKV_DECODEG_CASE(128, 4)
  PKV_DECODEG_CASE(128, 8)
#undef PKV_DECODEG_CASE
  if (rc) return rc;
  return ok();
}

// ---------------------------------------------------------------------------
// Decode without a caller-supplied workspace.
//
// Some callers cannot hand the library device scratch memory: a plugin that
// is given only its input and output buffers by the host framework, an engine
// whose KV pool already reserved every free byte of HBM, or a latency-critical
// loop that must not call cudaMalloc (which can synchronise the device). For
// them the split-K scratch lives in this fixed array, which every GPU that
// loads the library holds until the process exits.
static __device__ __align__(256) uint8_t g_decode_noalloc_scratch[PKV_DECODE_NOALLOC_SCRATCH_BYTES];

namespace pkv {
namespace {
constexpr int kNoAllocMaxDevices = 64;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};
cudaError_t g_noalloc_err[kNoAllocMaxDevices] = {};
std::once_flag g_noalloc_once[kNoAllocMaxDevices];

// Device address of the scratch array on the current device. In host code the
// array's name is only a stand-in, so the address is looked up once per
// device, with that device current, and kept for the life of the process (a
// cudaDeviceReset reloads the module, after which the kept address is stale;
// the header tells callers not to use this entry point after a reset).
int noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err, "cudaGetDevice");
  if (dev < 0 || dev >= kNoAllocMaxDevices)
    return fail(PKV_EINVAL, "decode_noalloc: device ordinal %d unsupported", dev);
  std::call_once(g_noalloc_once[dev], [dev]() {
    void* p = nullptr;
    g_noalloc_err[dev] = cudaGetSymbolAddress(&p, g_decode_noalloc_scratch);
    if (g_noalloc_err[dev] == cudaSuccess) g_noalloc_ptr[dev] = p;
  });
  if (g_noalloc_err[dev] != cudaSuccess)
    return cuda_fail(g_noalloc_err[dev], "decode_noalloc: cudaGetSymbolAddress");
  *out = g_noalloc_ptr[dev];
  return PKV_OK;
}
}  // namespace
}  // namespace pkv

extern "C" int pkv_paged_attention_decode_noalloc(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* context_lens,
    int32_t max_context_len, int32_t S, int32_t Hq, int32_t Hkv, int32_t D, int32_t block_size,
    int32_t num_blocks, float scale, int32_t partition_size, int32_t* dev_status, void* stream) {
  size_t need = 0;
  if (int rc = pkv_decode_workspace_bytes(S, Hq, D, max_context_len, partition_size, &need))
    return rc;
  if (need > (size_t)PKV_DECODE_NOALLOC_SCRATCH_BYTES)
    return fail(PKV_EINVAL,
                "decode_noalloc: this batch needs %zu bytes of scratch, more than the built-in "
                "%zu (use pkv_paged_attention_decode with a workspace, or a larger "
                "partition_size)",
                need, (size_t)PKV_DECODE_NOALLOC_SCRATCH_BYTES);
  void* scratch = nullptr;
  if (S > 0) {
    if (int rc = noalloc_scratch(&scratch)) return rc;
  }
  // The plan kernel rewrites the item list and resets the work ticket at the
  // start of every call, so nothing left in the array by an earlier call is
  // read before it is written.
  return pkv_paged_attention_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                    context_lens, max_context_len, S, Hq, Hkv, D, block_size,
                                    num_blocks, scale, partition_size, scratch,
                                    (size_t)PKV_DECODE_NOALLOC_SCRATCH_BYTES, dev_status, stream);
}
