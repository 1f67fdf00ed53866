/*
 * pagedkv.h — C ABI of the paged-KV attention library for GB300 (sm_103a).
 *
 * What the library computes, and where the pages on continuous batching and
 * PagedAttention say so:
 *
 *   "Batching, Scheduling, and Paging" (datasystem.school, module 4)
 *     section PagedAttention: each sequence's KV cache is cut into fixed-size
 *       blocks stored non-contiguously; a per-sequence block table maps logical
 *       blocks to physical ones; the CPU allocates a block only when the
 *       previous one fills and frees blocks when the request completes; the
 *       attention kernels gather K and V through the block table.
 *     section Block sharing: parallel samples point at the same physical blocks;
 *       the first divergent write does copy-on-write; reference counts keep a
 *       shared block alive until its last user finishes.
 *   "Deep Dive: continuous batching" (worksonmygpu.com)
 *     section Selective batching: attention, softmax(Q K^T / sqrt(d_k)) V, runs
 *       per request over that request's own tokens only.
 *     section The prefill/decode mix: a new request's prompt (prefill) and a
 *       running request's single new token (decode) are different shapes of
 *       work mixed in one iteration.
 *
 * Conventions
 *   - Every call returns an int status: PKV_OK (0) or a negative PKV_E* code;
 *     pkv_last_error() then describes the failure (thread-local string).
 *   - Memory layout of the KV cache (the pages fix none): two separate pools,
 *     keys and values, each bf16 [num_blocks][Hkv][block_size][D], row-major.
 *     Token j of a sequence with block table bt lives in block bt[j / B] at
 *     offset j % B. A slot is block * B + offset (int32); slot -1 means "skip".
 *   - Query head h reads key/value head h / (Hq / Hkv) (grouped heads).
 *   - bf16 pointers are passed as void*; they must be 16-byte aligned and the
 *     arrays contiguous. int32 arrays are int32_t*.
 *   - Ownership: the caller owns all device memory (the library allocates
 *     none in these calls) and the allocator handle (create/destroy).
 *   - GPU calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream). Pointers must stay valid until that work completes.
 *   - Device-side faults are never raised on purpose: a table entry or slot out
 *     of range, or a bounded wait that expires, skips the access and records a
 *     code in the caller's status block (`dev_status`, 4 int32 on the device,
 *     zeroed by pkv_status_reset); pkv_check_status() synchronises and reports.
 *     `dev_status` may be NULL, in which case such events are dropped silently.
 *   - Supported shapes: bf16 only; D in {64, 128}; block_size in {8, 16, 32};
 *     Hq / Hkv in {1, 2, 4, 8}.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  PKV_OK = 0,
  PKV_EINVAL = -1,   /* bad argument: null pointer, unsupported shape, size mismatch */
  PKV_ENOMEM = -2,   /* allocator: not enough free blocks; state unchanged          */
  PKV_ECUDA = -3,    /* a CUDA launch or API call failed                             */
  PKV_ETIMEOUT = -4, /* a device wait exceeded its time limit (reported by status)  */
  PKV_EDEVICE = -5   /* a device range check fired (reported by status)             */
};

/* Thread-local description of the last failing call on this thread. */
const char* pkv_last_error(void);
/* Library version, major * 10000 + minor * 100 + patch. */
int pkv_version(void);

/* ------------------------------------------------------------------------
 * Host block allocator ("Batching, Scheduling, and Paging", sections
 * PagedAttention and Block sharing). CPU only, single-threaded, deterministic.
 *   - Free blocks are handed out first-in first-out. The initial order is
 *     `free_order` (a permutation of 0..num_blocks-1, e.g. a seeded shuffle) or
 *     0,1,2,... when NULL; a block whose count drops to 0 joins the tail.
 *   - A new block is taken only when a sequence's last block is full.
 *   - fork shares every block of the parent and adds one reference to each.
 *   - An append whose first new token lands in a partially filled block that
 *     other sequences share copies it first (copy-on-write): a fresh block
 *     replaces it in this sequence's table, one (src, dst) pair is reported and
 *     the source loses one reference. Full shared blocks are never copied; the
 *     last remaining user writes in place. At most one pair per append.
 *   - An append that cannot get every block it needs returns PKV_ENOMEM and
 *     changes nothing.
 *   - Sequence ids are 0, 1, 2, ... in creation order; they are never reused.
 * ---------------------------------------------------------------------- */
typedef struct pkv_alloc pkv_alloc;

int pkv_alloc_create(int32_t num_blocks, int32_t block_size, const int32_t* free_order,
                     pkv_alloc** out);
int pkv_alloc_destroy(pkv_alloc* a);
int pkv_seq_create(pkv_alloc* a, int64_t* seq_id);
int pkv_seq_fork(pkv_alloc* a, int64_t parent, int64_t* child);
/* Reserve slots for n new tokens of `seq`. slots_out: n int32 (host).
 * cow_pair_out: 2 int32 (host), receives (src, dst) when *n_cow == 1. */
int pkv_seq_append_slots(pkv_alloc* a, int64_t seq, int32_t n, int32_t* slots_out,
                         int32_t* cow_pair_out, int32_t* n_cow);
/* The request completed: drop its references, freeing blocks that reach 0. */
int pkv_seq_free(pkv_alloc* a, int64_t seq);
/* Batched forms for an iteration's admissions and completions: n new empty
 * sequences (ids to seq_ids, n int64, host, in creation order); n sequences
 * freed as by pkv_seq_free. PKV_EINVAL, nothing freed, when an id is unknown
 * or listed twice. */
int pkv_seq_create_many(pkv_alloc* a, int32_t n, int64_t* seq_ids);
int pkv_seq_free_many(pkv_alloc* a, const int64_t* seqs, int32_t n);
int pkv_seq_len(pkv_alloc* a, int64_t seq, int32_t* len);
/* Copies min(cap, table length) entries to out (host); *n = table length. */
int pkv_seq_block_table(pkv_alloc* a, int64_t seq, int32_t* out, int32_t cap, int32_t* n);
int pkv_block_refcount(pkv_alloc* a, int32_t block, int32_t* out);
int pkv_num_free_blocks(pkv_alloc* a, int32_t* out);
/* Per-iteration metadata for n sequences (host arrays): tables_out is
 * [n][max_blocks_per_seq] int32, padded with 0; lens_out is [n] int32.
 * PKV_EINVAL if a table is longer than max_blocks_per_seq. */
int pkv_build_block_tables(pkv_alloc* a, const int64_t* seqs, int32_t n, int32_t* tables_out,
                           int32_t max_blocks_per_seq, int32_t* lens_out);

/* One iteration's host work in one call ("Batching, Scheduling, and Paging",
 * section Continuous batching: the batch is rebuilt every iteration and the
 * CPU work per iteration is overhead to keep small; "Deep Dive: continuous
 * batching", section Iteration-level scheduling).
 *   seqs[n], counts[n] (host), n = n_prefill + n_decode: works 0 ..
 *     n_prefill-1 are prompt chunks (counts >= 1), the rest decodes (count
 *     1). Each sequence at most once, none swapped out.
 *   Every work gets its counts[i] slots as pkv_seq_append_slots would give
 *   them, in order (the same blocks, the same copy-on-write pairs). The batch
 *   is all or nothing: if the free blocks do not cover every work, nothing
 *   changes, the call returns PKV_ENOMEM and *n_fit is the number of leading
 *   works that would fit (evict, then call again). On success *n_fit = n.
 *   buf (host memory the caller owns, e.g. pinned, of at least
 *   total_bytes as pkv_iteration_layout_bytes reports for the same sizes)
 *   receives, at the layout's byte offsets, each section starting on a
 *   64-byte boundary (W = layout->table_width, the batch's longest table
 *   after the appends, at most max_blocks_per_seq):
 *     slot_mapping   int32 [n_tokens]   (prefill works first, then decodes)
 *     cu_q_lens      int32 [n_prefill + 1]
 *     prefill_lens   int32 [n_prefill]  (context lengths after the appends)
 *     prefill_tables int32 [n_prefill][W]
 *     decode_lens    int32 [n_decode]
 *     decode_tables  int32 [n_decode][W]
 *     cow_pairs      int32 [n_cow][2]  (run pkv_block_copy on them first)
 *   (a table row holds the sequence's ceil(len / block_size) blocks; the
 *   entries after them are left as they were: no kernel reads them),
 *   so one host-to-device copy of the whole buffer feeds pkv_block_copy,
 *   pkv_kv_append, pkv_paged_attention_prefill and pkv_paged_attention_decode.
 *   PKV_EINVAL (nothing changed) for unknown, repeated or swapped-out
 *   sequences, bad counts, a table longer than max_blocks_per_seq or a short
 *   buf. */
typedef struct pkv_iteration_layout {
  int64_t slot_mapping, cu_q_lens, prefill_lens, prefill_tables, decode_lens, decode_tables,
      cow_pairs;        /* byte offsets into buf */
  int64_t total_bytes;  /* bytes of buf the layout covers */
  int32_t n_tokens;     /* sum of counts */
  int32_t n_cow;        /* copy-on-write pairs written */
  int32_t max_q_len;    /* longest prompt chunk */
  int32_t max_prefill_len, max_decode_len; /* longest context of each kind */
  int32_t table_width;  /* entries per block-table row (the layout_bytes call: its bound) */
} pkv_iteration_layout;
int pkv_iteration_layout_bytes(int32_t n_prefill, int32_t n_decode, int32_t n_tokens,
                               int32_t max_blocks_per_seq, pkv_iteration_layout* layout);
int pkv_iteration_prepare(pkv_alloc* a, const int64_t* seqs, const int32_t* counts,
                          int32_t n_prefill, int32_t n_decode, int32_t max_blocks_per_seq,
                          void* buf, size_t buf_bytes, pkv_iteration_layout* layout,
                          int32_t* n_fit);

/* The GPU side of that iteration in one call ("Deep Dive: continuous
 * batching", sections Iteration-level scheduling and The prefill/decode mix):
 * after the caller has copied the buffer pkv_iteration_prepare filled to
 * device memory `meta` (same offsets, 64-byte aligned or better), this
 * launches on `stream`, in order, pkv_block_copy of the copy pairs,
 * pkv_kv_append of every new token, pkv_paged_attention_prefill of the
 * prompt chunks and pkv_paged_attention_decode of the decodes, with the
 * arrays read from `meta` and the sizes (the block-table width included)
 * from `layout` (the host struct the prepare call returned).
 *   q, out          : bf16 [n_tokens][Hq][D] (device), prefill rows first
 *                     (one per prompt token, in work order), then one row
 *                     per decode.
 *   k_new, v_new    : bf16 [n_tokens][Hkv][D] (device), the same order.
 *   decode_ws       : pkv_decode_workspace_bytes(n_decode, Hq, D,
 *                     max_decode_len, partition_size) bytes or more.
 *   prefill_ws      : pkv_prefill_workspace_bytes(n_prefill, prefill rows,
 *                     Hq, D) bytes or more.
 * When the iteration has both prompt chunks and decodes, the prefill runs on
 * a second stream of the library's (one per device, created by the first
 * such call; the first call should not be made inside a stream capture),
 * forked from `stream` after the append and joined back into it, beside the
 * decode on `stream`: work queued on `stream` after this call still waits
 * for all of it, and a captured call captures both branches. The stream and
 * its two events do not survive cudaDeviceReset.
 * Errors are those of the four calls (the first failing one returns; the
 * launches before it stay queued). An iteration with no token and no copy
 * does nothing. */
int pkv_iteration_run(const void* meta, const pkv_iteration_layout* layout, int32_t n_prefill,
                      int32_t n_decode, const void* q,
                      const void* k_new, const void* v_new, void* out, void* k_cache,
                      void* v_cache, int32_t num_blocks, int32_t Hq, int32_t Hkv, int32_t D,
                      int32_t block_size, float scale, int32_t partition_size, void* decode_ws,
                      size_t decode_ws_bytes, void* prefill_ws, size_t prefill_ws_bytes,
                      int32_t* dev_status, void* stream);

/* Both halves of an iteration in one call: pkv_iteration_prepare into
 * host_buf, one cudaMemcpyAsync of the layout's total_bytes to dev_buf on
 * `stream`, then pkv_iteration_run from dev_buf. Arguments as in those two
 * calls; *layout and *n_fit are returned as pkv_iteration_prepare returns
 * them (on PKV_ENOMEM nothing was changed, copied or launched).
 *   host_buf : host memory the caller owns; pinned memory keeps the copy
 *              asynchronous. The copy reads it after this call returns:
 *              do not write into it again until the copy has completed (an
 *              event recorded after the call, or a ring of buffers).
 *   dev_buf  : device memory of at least total_bytes, 64-byte aligned;
 *              stream order protects it from the next iteration's copy. */
int pkv_iteration_step(pkv_alloc* a, const int64_t* seqs, const int32_t* counts,
                       int32_t n_prefill, int32_t n_decode, int32_t max_blocks_per_seq,
                       void* host_buf, size_t host_bytes, void* dev_buf, size_t dev_bytes,
                       const void* q, const void* k_new, const void* v_new, void* out,
                       void* k_cache, void* v_cache, int32_t num_blocks, int32_t Hq, int32_t Hkv,
                       int32_t D, int32_t block_size, float scale, int32_t partition_size,
                       void* decode_ws, size_t decode_ws_bytes, void* prefill_ws,
                       size_t prefill_ws_bytes, int32_t* dev_status, void* stream,
                       pkv_iteration_layout* layout, int32_t* n_fit);

/* Preemption ("Batching, Scheduling, and Paging", section PagedAttention: if
 * HBM runs out a request is evicted, swapped to CPU memory or discarded and
 * recomputed later).
 *   swap_out: the sequence gives its blocks back (table order, written to
 *     blocks_out, *n of them) and keeps its length; each block loses one
 *     reference and may be handed out again at once, so copy the blocks out
 *     (pkv_swap_blocks, on the stream that will later write into them) before
 *     the next kv_append. A swapped-out sequence cannot be appended to,
 *     forked or put in a block table until it is swapped in.
 *   swap_in: fresh blocks for all of its tokens (first in, first out), all or
 *     nothing (PKV_ENOMEM); copy the saved contents into them before use.
 *   Recompute: pkv_seq_free, then create the request again and re-append. */
int pkv_seq_swap_out(pkv_alloc* a, int64_t seq, int32_t* blocks_out, int32_t cap, int32_t* n);
int pkv_seq_swap_in(pkv_alloc* a, int64_t seq, int32_t* blocks_out, int32_t cap, int32_t* n);

/* Prefix caching ("Batching, Scheduling, and Paging", section Block sharing:
 * identical prefixes of different requests can share physical blocks;
 * "Paging the KV Cache": a system prompt common to many concurrent requests
 * occupies one set of pages that all of them reference).
 *   A full block of a sequence whose token ids are known is registered under
 *   (the block before it, or none for the first block; its block_size token
 *   ids). Entries are compared in full, never by hash alone. A registered
 *   block keeps its entry after its last user leaves; it sits in the free
 *   list as usual, a lookup can take it back from there, and it loses the
 *   entry (with the entries that chain from it) when the free list hands it
 *   out again.
 *   create_cached: a new sequence whose table starts with the registered
 *     blocks matching token_ids[0..n) block by block from the start, at most
 *     (n - 1) / block_size of them, so that the last token is always computed;
 *     each matched block gains one reference (leaving the free list if it was
 *     there). *n_cached = matched blocks * block_size tokens, already in the
 *     cache: append token_ids[*n_cached..n) with append_tokens.
 *   append_tokens: append_slots that also records the n token ids
 *     (token_ids: n int32, host) and registers blocks as they fill; a block
 *     whose entry already exists (an identical block elsewhere) is not
 *     registered, nor is anything after it in that sequence. Sequences that
 *     were ever appended with append_slots, and swapped-in sequences,
 *     register nothing.
 *   num_cached_blocks: registered blocks, in use or free. */
int pkv_seq_create_cached(pkv_alloc* a, const int32_t* token_ids, int32_t n, int64_t* seq_id,
                          int32_t* n_cached);
int pkv_seq_append_tokens(pkv_alloc* a, int64_t seq, const int32_t* token_ids, int32_t n,
                          int32_t* slots_out, int32_t* cow_pair_out, int32_t* n_cow);
int pkv_num_cached_blocks(pkv_alloc* a, int32_t* out);

/* ------------------------------------------------------------------------
 * Device status block (4 int32 in device memory, owned by the caller):
 *   [0] first error code (0, PKV_ETIMEOUT or PKV_EDEVICE), [1] detail (the
 *   offending index or wait site), [2] kernel id, [3] count of events.
 * ---------------------------------------------------------------------- */
int pkv_status_reset(int32_t* dev_status, void* stream);
/* Synchronises `stream`, reads the block and returns PKV_OK, PKV_ETIMEOUT or
 * PKV_EDEVICE (pkv_last_error() gives the detail). Does not clear it. */
int pkv_check_status(const int32_t* dev_status, void* stream);
/* Debug knob for tests: when nonzero, the next kernels treat their first
 * pipeline wait as expired (they record PKV_ETIMEOUT, let their own copies in
 * flight land, and return). Also sets the wait limit in nanoseconds when
 * timeout_ns > 0 (default 2e9). */
int pkv_debug_set_wait(int32_t force_timeout, uint64_t timeout_ns);

/* ------------------------------------------------------------------------
 * kv_append — "Batching, Scheduling, and Paging", section PagedAttention:
 * each new token's key and value rows are written into the slot the block
 * table assigned to it.
 *   k_new, v_new : bf16 [T][Hkv][D] (device)
 *   slot_mapping : int32 [T] (device); -1 skips the token; a slot outside
 *                  [0, num_blocks * block_size) is skipped and recorded as
 *                  PKV_EDEVICE in dev_status.
 *   k_cache, v_cache : the pools (device), written in place.
 * Bit-exact copy. Slots must be distinct (two tokens in one slot race).
 * ---------------------------------------------------------------------- */
int pkv_kv_append(const void* k_new, const void* v_new, const int32_t* slot_mapping, int32_t T,
                  void* k_cache, void* v_cache, int32_t num_blocks, int32_t Hkv, int32_t D,
                  int32_t block_size, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * block_copy — "Batching, Scheduling, and Paging", section Block sharing:
 * copy-on-write duplicates a whole physical block (keys and values).
 *   pairs : int32 [n][2] (device), (src, dst) block ids. No dst may appear
 *           twice or also be a src in the same call (they run in parallel).
 *           An id outside [0, num_blocks) skips the pair (PKV_EDEVICE).
 * Run it before the kv_append that writes into the copies, on one stream.
 * ---------------------------------------------------------------------- */
int pkv_block_copy(void* k_cache, void* v_cache, const int32_t* pairs, int32_t n,
                   int32_t num_blocks, int32_t Hkv, int32_t D, int32_t block_size,
                   int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * swap_blocks — copies whole blocks (keys and values) between the pools and
 * a contiguous buffer, for swapping a preempted request out and back in
 * ("Batching, Scheduling, and Paging", section PagedAttention).
 *   blocks       : int32 [n] (device), block ids in the pool; an id outside
 *                  [0, num_blocks) skips that slot (PKV_EDEVICE).
 *   k_buf, v_buf : bf16 [n][Hkv][block_size][D] each: device memory or
 *                  pinned host memory (the GPU reads or writes it over the
 *                  CPU-GPU link); pageable host memory is refused (PKV_EINVAL).
 *   to_buffer    : 1 copies pool -> buffer (swap-out), 0 buffer -> pool.
 * Bit-exact. The listed blocks must be distinct.
 * ---------------------------------------------------------------------- */
int pkv_swap_blocks(void* k_cache, void* v_cache, const int32_t* blocks, int32_t n,
                    int32_t num_blocks, int32_t Hkv, int32_t D, int32_t block_size, void* k_buf,
                    void* v_buf, int32_t to_buffer, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * paged_attention_decode — one query token per sequence ("Deep Dive:
 * continuous batching", section Selective batching; "Batching, Scheduling,
 * and Paging", section PagedAttention):
 *   out[s][h] = softmax_j(scale * q[s][h] . K_s[j]) V_s[j],  j = 0 .. L_s - 1
 * where K_s[j] = k_cache[bt_s[j / B]][h / G][j % B] and L_s = context_lens[s]
 * (the query's own token is already in the cache and is included).
 *   out          : bf16 [S][Hq][D] (device, written)
 *   q            : bf16 [S][Hq][D] (device)
 *   block_tables : int32 [S][max_blocks_per_seq] (device); entries past
 *                  ceil(L_s / B) are never read.
 *   context_lens : int32 [S] (device), each in [1, max_context_len].
 *   max_context_len : an upper bound of context_lens (host value); it sizes
 *                  the split into partitions and the workspace.
 *   partition_size : tokens per split-K partition (multiple of 16, >= 16), or
 *                  0 for the library default (1024). Long contexts are split
 *                  into partitions whose partial softmax states are merged by
 *                  a second kernel; the split depends only on positions, so
 *                  results do not depend on physical placement.
 *   workspace    : device scratch of pkv_decode_workspace_bytes() bytes.
 * Arithmetic: bf16 inputs, fp32 scores and accumulation, probabilities
 * entering the P.V product as two bf16 parts (hi + lo, ~2^-17 relative),
 * output rounded to bf16.
 * ---------------------------------------------------------------------- */
int pkv_decode_workspace_bytes(int32_t S, int32_t Hq, int32_t D, int32_t max_context_len,
                               int32_t partition_size, size_t* out);
int pkv_paged_attention_decode(void* out, const void* q, const void* k_cache,
                               const void* v_cache, const int32_t* block_tables,
                               int32_t max_blocks_per_seq, const int32_t* context_lens,
                               int32_t max_context_len, int32_t S, int32_t Hq, int32_t Hkv,
                               int32_t D, int32_t block_size, int32_t num_blocks, float scale,
                               int32_t partition_size, void* workspace, size_t workspace_bytes,
                               int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * paged_attention_decode_shared — the same decode for a batch in which
 * groups of sequences share their first tokens' physical blocks (parallel
 * samples of one prompt: "Batching, Scheduling, and Paging", section Block
 * sharing). The shared prefix of a group is read once for up to 16 / (Hq /
 * Hkv) members at a time (their query heads fill one 16-row MMA operand),
 * instead of once per member; each member's remaining tokens are decoded
 * as usual and the partial results merged. Results equal those of
 * pkv_paged_attention_decode up to floating-point rounding.
 *   group_start   : int32 [n_groups + 1] (device), members of group g are
 *                   group_members[group_start[g] .. group_start[g+1]).
 *   group_members : int32 (device), sequence indices; a sequence belongs to
 *                   at most one group; sequences in no group are decoded
 *                   alone.
 *   group_shared  : int32 [n_groups] (device): the number of leading tokens
 *                   whose block-table entries are identical for every member
 *                   (the caller's guarantee; the kernel reads the first
 *                   member's table for them). It is cut to whole 16-token
 *                   tiles and to the shortest member.
 *   workspace     : pkv_decode_shared_workspace_bytes() bytes.
 * Other arguments as in pkv_paged_attention_decode. Bad group entries
 * (indices outside 0..S-1, decreasing starts) are skipped and recorded
 * (PKV_EDEVICE).
 * ---------------------------------------------------------------------- */
int pkv_decode_shared_workspace_bytes(int32_t S, int32_t Hq, int32_t D,
                                      int32_t max_context_len, int32_t partition_size,
                                      size_t* out);
int pkv_paged_attention_decode_shared(void* out, const void* q, const void* k_cache,
                                      const void* v_cache, const int32_t* block_tables,
                                      int32_t max_blocks_per_seq, const int32_t* context_lens,
                                      int32_t max_context_len, const int32_t* group_start,
                                      const int32_t* group_members, const int32_t* group_shared,
                                      int32_t n_groups, int32_t S, int32_t Hq, int32_t Hkv,
                                      int32_t D, int32_t block_size, int32_t num_blocks,
                                      float scale, int32_t partition_size, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * paged_attention_decode_noalloc — the same decode as above, for callers that
 * cannot provide device scratch memory (a plugin handed only its inputs and
 * outputs, an engine whose KV pool already holds all free HBM, a decode loop
 * that must not call cudaMalloc because it can synchronise the device). The
 * pages have no counterpart: this is an interface convenience of the library.
 *   - Scratch: a fixed array of PKV_DECODE_NOALLOC_SCRATCH_BYTES inside the
 *     library, held on every GPU that loads the library until the process
 *     exits. A batch whose pkv_decode_workspace_bytes() exceeds it is rejected
 *     with PKV_EINVAL (a larger partition_size needs less).
 *   - Allocates nothing. The first call on a device looks up the array's
 *     device address for that device (once, with it current); make that first
 *     call before any stream capture. The address is kept for the life of the
 *     process: it does not survive cudaDeviceReset (the module is loaded
 *     again and the array may move), so do not call this entry point on a
 *     device after resetting it.
 *   - All calls share the one array, which keeps the last call's contents;
 *     every call rewrites what it reads first. Calls that overlap on the GPU
 *     (other streams, other host threads) race on it: serialise them.
 *   Arguments, layouts and results are those of pkv_paged_attention_decode.
 * ---------------------------------------------------------------------- */
#define PKV_DECODE_NOALLOC_SCRATCH_BYTES (64u << 20)
int pkv_paged_attention_decode_noalloc(void* out, const void* q, const void* k_cache,
                                       const void* v_cache, const int32_t* block_tables,
                                       int32_t max_blocks_per_seq, const int32_t* context_lens,
                                       int32_t max_context_len, int32_t S, int32_t Hq,
                                       int32_t Hkv, int32_t D, int32_t block_size,
                                       int32_t num_blocks, float scale, int32_t partition_size,
                                       int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * paged_attention_prefill — a chunk of a prompt attending causally over its
 * own cached blocks ("Deep Dive: continuous batching", section The
 * prefill/decode mix; the chunk's keys and values are appended first).
 * Sequence s owns query rows cu_q_lens[s] .. cu_q_lens[s+1]-1 (c_s rows);
 * they are its last c_s tokens, so row i sits at position L_s - c_s + i and
 *   out[row][h] = softmax_j(scale * q[row][h] . K_s[j]) V_s[j],
 *                 j = 0 .. L_s - c_s + i.
 *   out, q       : bf16 [total_q][Hq][D] (device)
 *   cu_q_lens    : int32 [S + 1] (device), cu_q_lens[0] = 0, nondecreasing,
 *                  cu_q_lens[S] = total_q, each c_s <= L_s and <= max_q_len.
 *   context_lens : int32 [S] (device), after the chunk was appended.
 *   workspace    : pkv_prefill_workspace_bytes() bytes of device scratch.
 * QK^T and PV run on the tcgen05 tensor cores (bf16 operands, fp32
 * accumulation in tensor memory); probabilities enter the PV product as two
 * bf16 parts (hi + lo, ~2^-17 relative).
 * ---------------------------------------------------------------------- */
int pkv_prefill_workspace_bytes(int32_t S, int32_t total_q, int32_t Hq, int32_t D,
                                size_t* out);
int pkv_paged_attention_prefill(void* out, const void* q, const int32_t* cu_q_lens,
                                const int32_t* context_lens, const void* k_cache,
                                const void* v_cache, const int32_t* block_tables,
                                int32_t max_blocks_per_seq, int32_t S, int32_t total_q,
                                int32_t max_q_len, int32_t max_context_len, int32_t Hq,
                                int32_t Hkv, int32_t D, int32_t block_size, int32_t num_blocks,
                                float scale, void* workspace, size_t workspace_bytes,
                                int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * FP8 (e4m3) pages. The continuous-batching page (section "Two orthogonal
 * fixes, one serving engine") counts FP8 arithmetic among the kernel-level
 * optimisations that stack with paging; the storage format below is this
 * library's. A page keeps one byte per element and one fp32 scale per token
 * row, so appending a token never touches the rest of its page:
 *   k_codes, v_codes   : uint8 [num_blocks][Hkv][block_size][D] (device),
 *                        e4m3 codes (1 sign, 4 exponent bits biased by 7,
 *                        3 mantissa bits; 0x7F / 0xFF are NaN; max 448).
 *   k_scales, v_scales : fp32 [num_blocks][Hkv][block_size] (device).
 *   element value = e4m3(code) * scale of its row.
 * kv_append_fp8 quantises each new (token, head) row of k_new / v_new (bf16
 * [T][Hkv][D]) with amax = its largest magnitude: scale = amax / 448 and
 * code = e4m3(x * (448 / amax)), both quotients and the product rounded to
 * fp32, the code rounded to nearest even and saturated; a zero row gets
 * scale 0. Slots as in pkv_kv_append (-1 skips; out-of-pool recorded).
 * paged_attention_decode_fp8 is pkv_paged_attention_decode over such pages
 * (same arguments otherwise, same workspace size): codes are widened to fp16
 * on chip, q is rounded to fp16 (exact for 2^-14 <= |q| <= 65504), key
 * scales multiply the scores, value scales the probabilities, and the
 * scaled probabilities enter the P.V product as two fp16 parts.
 * All arrays 16-byte aligned.
 * ---------------------------------------------------------------------- */
int pkv_kv_append_fp8(const void* k_new, const void* v_new, const int32_t* slot_mapping,
                      int32_t T, void* k_codes, void* v_codes, float* k_scales,
                      float* v_scales, int32_t num_blocks, int32_t Hkv, int32_t D,
                      int32_t block_size, int32_t* dev_status, void* stream);
int pkv_paged_attention_decode_fp8(void* out, const void* q, const void* k_codes,
                                   const void* v_codes, const float* k_scales,
                                   const float* v_scales, const int32_t* block_tables,
                                   int32_t max_blocks_per_seq, const int32_t* context_lens,
                                   int32_t max_context_len, int32_t S, int32_t Hq, int32_t Hkv,
                                   int32_t D, int32_t block_size, int32_t num_blocks,
                                   float scale, int32_t partition_size, void* workspace,
                                   size_t workspace_bytes, int32_t* dev_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
