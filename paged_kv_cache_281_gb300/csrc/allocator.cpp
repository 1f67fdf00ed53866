// Host block allocator with reference counts and copy-on-write.
//
// "Batching, Scheduling, and Paging" (datasystem.school, module 4):
//   section PagedAttention — the block table lives on the CPU; a block is
//     allocated only when the previous one fills and freed when the request
//     completes;
//   section Block sharing — forked samples reference the same physical blocks,
//     the first divergent write copies (copy-on-write) and reference counts
//     keep a shared block alive until its last user finishes.
//
// Data structures: a ring buffer holding the free list (first in, first out),
// one int32 count per block, and a hash map from sequence id to its block
// list and token count. Every operation checks its preconditions before it
// mutates anything, so a failed call leaves the allocator unchanged.
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "internal.h"

struct pkv_alloc {
  int32_t num_blocks = 0;
  int32_t block_size = 0;
  // free list as a ring buffer of capacity num_blocks
  std::vector<int32_t> ring;
  int32_t head = 0;
  int32_t count = 0;
  std::vector<int32_t> refcount;
  struct Seq {
    std::vector<int32_t> blocks;
    int32_t len = 0;
    bool swapped = false;  // blocks handed back; contents kept by the caller
  };
  std::unordered_map<int64_t, Seq> seqs;
  int64_t next_id = 0;

  int32_t pop_free() {
    int32_t b = ring[head];
    head = (head + 1) % num_blocks;
    --count;
    refcount[b] = 1;
    return b;
  }
  void push_free(int32_t b) {
    ring[(head + count) % num_blocks] = b;
    ++count;
  }
  Seq* find(int64_t id) {
    auto it = seqs.find(id);
    return it == seqs.end() ? nullptr : &it->second;
  }
};

using pkv::fail;
using pkv::ok;

extern "C" int pkv_alloc_create(int32_t num_blocks, int32_t block_size, const int32_t* free_order,
                                pkv_alloc** out) {
  PKV_REQUIRE(out != nullptr, "pkv_alloc_create: out is NULL");
  *out = nullptr;
  PKV_REQUIRE(num_blocks > 0, "pkv_alloc_create: num_blocks must be > 0 (got %d)", num_blocks);
  PKV_REQUIRE(block_size > 0, "pkv_alloc_create: block_size must be > 0 (got %d)", block_size);
  PKV_REQUIRE((int64_t)num_blocks * block_size < (int64_t(1) << 31),
              "pkv_alloc_create: num_blocks * block_size must fit int32 slots");
  pkv_alloc* a = new (std::nothrow) pkv_alloc();
  if (!a) return fail(PKV_ENOMEM, "pkv_alloc_create: out of host memory");
  a->num_blocks = num_blocks;
  a->block_size = block_size;
  a->ring.resize(num_blocks);
  a->refcount.assign(num_blocks, 0);
  if (free_order) {
    std::vector<char> seen(num_blocks, 0);
    for (int32_t i = 0; i < num_blocks; ++i) {
      int32_t b = free_order[i];
      if (b < 0 || b >= num_blocks || seen[b]) {
        delete a;
        return fail(PKV_EINVAL, "pkv_alloc_create: free_order is not a permutation (entry %d = %d)",
                    i, b);
      }
      seen[b] = 1;
      a->ring[i] = b;
    }
  } else {
    for (int32_t i = 0; i < num_blocks; ++i) a->ring[i] = i;
  }
  a->count = num_blocks;
  *out = a;
  return ok();
}

extern "C" int pkv_alloc_destroy(pkv_alloc* a) {
  delete a;
  return ok();
}

extern "C" int pkv_seq_create(pkv_alloc* a, int64_t* seq_id) {
  PKV_REQUIRE(a && seq_id, "pkv_seq_create: NULL argument");
  int64_t id = a->next_id++;
  a->seqs.emplace(id, pkv_alloc::Seq{});
  *seq_id = id;
  return ok();
}

extern "C" int pkv_seq_fork(pkv_alloc* a, int64_t parent, int64_t* child) {
  PKV_REQUIRE(a && child, "pkv_seq_fork: NULL argument");
  pkv_alloc::Seq* p = a->find(parent);
  PKV_REQUIRE(p, "pkv_seq_fork: unknown sequence %lld", (long long)parent);
  PKV_REQUIRE(!p->swapped, "pkv_seq_fork: sequence %lld is swapped out", (long long)parent);
  pkv_alloc::Seq copy = *p;
  for (int32_t b : copy.blocks) ++a->refcount[b];
  int64_t id = a->next_id++;
  a->seqs.emplace(id, std::move(copy));
  *child = id;
  return ok();
}

extern "C" int pkv_seq_append_slots(pkv_alloc* a, int64_t seq, int32_t n, int32_t* slots_out,
                                    int32_t* cow_pair_out, int32_t* n_cow) {
  PKV_REQUIRE(a && n_cow, "pkv_seq_append_slots: NULL argument");
  PKV_REQUIRE(n >= 0, "pkv_seq_append_slots: n must be >= 0 (got %d)", n);
  PKV_REQUIRE(n == 0 || slots_out, "pkv_seq_append_slots: slots_out is NULL");
  pkv_alloc::Seq* s = a->find(seq);
  PKV_REQUIRE(s, "pkv_seq_append_slots: unknown sequence %lld", (long long)seq);
  PKV_REQUIRE(!s->swapped, "pkv_seq_append_slots: sequence %lld is swapped out", (long long)seq);
  *n_cow = 0;
  if (n == 0) return ok();
  const int32_t B = a->block_size;
  const int64_t new_len = (int64_t)s->len + n;
  // Blocks needed: the ones that open past the current table, plus one copy
  // when the first new token lands in a shared, partially filled last block.
  const bool partial = (s->len % B) != 0;
  const bool cow = partial && a->refcount[s->blocks.back()] > 1;
  const int64_t need = (new_len + B - 1) / B - (int64_t)s->blocks.size() + (cow ? 1 : 0);
  if (need > a->count)
    return fail(PKV_ENOMEM, "pkv_seq_append_slots: sequence %lld needs %lld blocks, %d free",
                (long long)seq, (long long)need, a->count);
  if (cow) {
    PKV_REQUIRE(cow_pair_out, "pkv_seq_append_slots: cow_pair_out is NULL but a copy is needed");
    int32_t& last = s->blocks.back();
    int32_t fresh = a->pop_free();
    --a->refcount[last];
    cow_pair_out[0] = last;
    cow_pair_out[1] = fresh;
    *n_cow = 1;
    last = fresh;
  }
  for (int32_t i = 0; i < n; ++i) {
    int32_t pos = s->len + i;
    int32_t j = pos / B;
    if (j == (int32_t)s->blocks.size()) s->blocks.push_back(a->pop_free());
    slots_out[i] = s->blocks[j] * B + pos % B;
  }
  s->len = (int32_t)new_len;
  return ok();
}

extern "C" int pkv_seq_free(pkv_alloc* a, int64_t seq) {
  PKV_REQUIRE(a, "pkv_seq_free: NULL allocator");
  auto it = a->seqs.find(seq);
  PKV_REQUIRE(it != a->seqs.end(), "pkv_seq_free: unknown sequence %lld", (long long)seq);
  for (int32_t b : it->second.blocks)
    if (--a->refcount[b] == 0) a->push_free(b);
  a->seqs.erase(it);
  return ok();
}

extern "C" int pkv_seq_len(pkv_alloc* a, int64_t seq, int32_t* len) {
  PKV_REQUIRE(a && len, "pkv_seq_len: NULL argument");
  pkv_alloc::Seq* s = a->find(seq);
  PKV_REQUIRE(s, "pkv_seq_len: unknown sequence %lld", (long long)seq);
  *len = s->len;
  return ok();
}

extern "C" int pkv_seq_block_table(pkv_alloc* a, int64_t seq, int32_t* out, int32_t cap,
                                   int32_t* n) {
  PKV_REQUIRE(a && n, "pkv_seq_block_table: NULL argument");
  PKV_REQUIRE(cap >= 0 && (cap == 0 || out), "pkv_seq_block_table: bad output buffer");
  pkv_alloc::Seq* s = a->find(seq);
  PKV_REQUIRE(s, "pkv_seq_block_table: unknown sequence %lld", (long long)seq);
  int32_t len = (int32_t)s->blocks.size();
  int32_t m = len < cap ? len : cap;
  if (m) std::memcpy(out, s->blocks.data(), sizeof(int32_t) * m);
  *n = len;
  return ok();
}

extern "C" int pkv_block_refcount(pkv_alloc* a, int32_t block, int32_t* out) {
  PKV_REQUIRE(a && out, "pkv_block_refcount: NULL argument");
  PKV_REQUIRE(block >= 0 && block < a->num_blocks, "pkv_block_refcount: block %d out of range",
              block);
  *out = a->refcount[block];
  return ok();
}

extern "C" int pkv_num_free_blocks(pkv_alloc* a, int32_t* out) {
  PKV_REQUIRE(a && out, "pkv_num_free_blocks: NULL argument");
  *out = a->count;
  return ok();
}

extern "C" int pkv_build_block_tables(pkv_alloc* a, const int64_t* seqs, int32_t n,
                                      int32_t* tables_out, int32_t max_blocks_per_seq,
                                      int32_t* lens_out) {
  PKV_REQUIRE(a, "pkv_build_block_tables: NULL allocator");
  PKV_REQUIRE(n >= 0 && max_blocks_per_seq > 0, "pkv_build_block_tables: bad sizes");
  PKV_REQUIRE(n == 0 || (seqs && tables_out && lens_out), "pkv_build_block_tables: NULL array");
  for (int32_t i = 0; i < n; ++i) {
    pkv_alloc::Seq* s = a->find(seqs[i]);
    PKV_REQUIRE(s, "pkv_build_block_tables: unknown sequence %lld", (long long)seqs[i]);
    PKV_REQUIRE(!s->swapped, "pkv_build_block_tables: sequence %lld is swapped out",
                (long long)seqs[i]);
    PKV_REQUIRE((int32_t)s->blocks.size() <= max_blocks_per_seq,
                "pkv_build_block_tables: sequence %lld has %zu blocks > %d", (long long)seqs[i],
                s->blocks.size(), max_blocks_per_seq);
  }
  for (int32_t i = 0; i < n; ++i) {
    pkv_alloc::Seq* s = a->find(seqs[i]);
    int32_t* row = tables_out + (int64_t)i * max_blocks_per_seq;
    int32_t m = (int32_t)s->blocks.size();
    if (m) std::memcpy(row, s->blocks.data(), sizeof(int32_t) * m);
    for (int32_t j = m; j < max_blocks_per_seq; ++j) row[j] = 0;
    lens_out[i] = s->len;
  }
  return ok();
}

// Preemption ("Batching, Scheduling, and Paging", section PagedAttention: when
// HBM runs out a request is evicted, swapped to CPU memory or recomputed).
extern "C" int pkv_seq_swap_out(pkv_alloc* a, int64_t seq, int32_t* blocks_out, int32_t cap,
                                int32_t* n) {
  PKV_REQUIRE(a && n, "pkv_seq_swap_out: NULL argument");
  pkv_alloc::Seq* s = a->find(seq);
  PKV_REQUIRE(s, "pkv_seq_swap_out: unknown sequence %lld", (long long)seq);
  PKV_REQUIRE(!s->swapped, "pkv_seq_swap_out: sequence %lld is already swapped out",
              (long long)seq);
  const int32_t m = (int32_t)s->blocks.size();
  PKV_REQUIRE(cap >= m && (m == 0 || blocks_out),
              "pkv_seq_swap_out: blocks_out holds %d entries, %d needed", cap, m);
  for (int32_t i = 0; i < m; ++i) {
    const int32_t b = s->blocks[i];
    blocks_out[i] = b;
    if (--a->refcount[b] == 0) a->push_free(b);
  }
  s->blocks.clear();
  s->swapped = true;
  *n = m;
  return ok();
}

extern "C" int pkv_seq_swap_in(pkv_alloc* a, int64_t seq, int32_t* blocks_out, int32_t cap,
                               int32_t* n) {
  PKV_REQUIRE(a && n, "pkv_seq_swap_in: NULL argument");
  pkv_alloc::Seq* s = a->find(seq);
  PKV_REQUIRE(s, "pkv_seq_swap_in: unknown sequence %lld", (long long)seq);
  PKV_REQUIRE(s->swapped, "pkv_seq_swap_in: sequence %lld is not swapped out", (long long)seq);
  const int32_t m = (s->len + a->block_size - 1) / a->block_size;
  PKV_REQUIRE(cap >= m && (m == 0 || blocks_out),
              "pkv_seq_swap_in: blocks_out holds %d entries, %d needed", cap, m);
  if (m > a->count)
    return fail(PKV_ENOMEM, "pkv_seq_swap_in: sequence %lld needs %d blocks, %d free",
                (long long)seq, m, a->count);
  for (int32_t i = 0; i < m; ++i) {
    const int32_t b = a->pop_free();
    s->blocks.push_back(b);
    blocks_out[i] = b;
  }
  s->swapped = false;
  *n = m;
  return ok();
}
