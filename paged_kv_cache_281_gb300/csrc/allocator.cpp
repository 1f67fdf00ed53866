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
// Data structures: a doubly linked free list (first in, first out), one
// int32 count per block, a hash map from sequence id to its block list and
// token count, and the prefix-cache index of full blocks. Every operation checks its preconditions before it
// mutates anything, so a failed call leaves the allocator unchanged.
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "internal.h"

struct pkv_alloc {
  int32_t num_blocks = 0;
  int32_t block_size = 0;
  // free list, first in first out, as a doubly linked list over block ids so
  // that a cached block can leave it from the middle when a lookup revives it
  std::vector<int32_t> next, prev;
  std::vector<char> on_free;
  int32_t head = -1, tail = -1;
  int32_t count = 0;
  std::vector<int32_t> refcount;
  struct Seq {
    std::vector<int32_t> blocks;
    int32_t len = 0;
    bool swapped = false;  // blocks handed back; contents kept by the caller
    bool tracked = true;   // token ids known for every position (prefix cache)
    std::vector<int32_t> tokens;
    int32_t reg_upto = 0;  // leading blocks that are registered, chained
    uint64_t mark = 0;     // the last iteration_prepare call that listed it
  };
  std::unordered_map<int64_t, Seq> seqs;
  int64_t next_id = 0;
  uint64_t epoch = 0;               // iteration_prepare calls so far
  std::vector<Seq*> batch;          // the current call's sequences, in work order

  // Prefix cache: a full block is registered under (the registered block
  // before it, or -1, and its B token ids). Registered blocks keep their
  // entry after their last user leaves and can be revived by a lookup until
  // the free list hands them out again.
  struct Entry {
    bool registered = false;
    int32_t parent = -1;
    std::vector<int32_t> tokens;
    std::vector<int32_t> children;
  };
  std::vector<Entry> entry;
  std::unordered_map<uint64_t, std::vector<int32_t>> index;
  int32_t num_registered = 0;

  static uint64_t key_of(int32_t parent, const int32_t* tok, int32_t B) {
    // FNV-1a over the parent id and the token ids; entries are compared in
    // full, so collisions only cost a longer bucket
    uint64_t h = 1469598103934665603ull;
    auto mix = [&h](uint32_t x) {
      for (int i = 0; i < 4; ++i) {
        h ^= (x >> (8 * i)) & 0xffu;
        h *= 1099511628211ull;
      }
    };
    mix((uint32_t)parent);
    for (int32_t i = 0; i < B; ++i) mix((uint32_t)tok[i]);
    return h;
  }
  int32_t lookup(int32_t parent, const int32_t* tok) const {
    auto it = index.find(key_of(parent, tok, block_size));
    if (it == index.end()) return -1;
    for (int32_t c : it->second) {
      const Entry& e = entry[c];
      if (e.parent == parent && std::memcmp(e.tokens.data(), tok, sizeof(int32_t) * block_size) == 0)
        return c;
    }
    return -1;
  }
  void register_block(int32_t b, int32_t parent, const int32_t* tok) {
    Entry& e = entry[b];
    e.registered = true;
    e.parent = parent;
    e.tokens.assign(tok, tok + block_size);
    index[key_of(parent, tok, block_size)].push_back(b);
    if (parent >= 0) entry[parent].children.push_back(b);
    ++num_registered;
  }
  // Drops b's entry and, below it, its descendants' (all of them are free
  // whenever b is: a user of a block also uses the block before it).
  void unregister(int32_t b) {
    std::vector<int32_t> stack{b};
    const int32_t root_parent = entry[b].parent;
    if (root_parent >= 0) {
      auto& ch = entry[root_parent].children;
      for (size_t i = 0; i < ch.size(); ++i)
        if (ch[i] == b) {
          ch[i] = ch.back();
          ch.pop_back();
          break;
        }
    }
    while (!stack.empty()) {
      int32_t x = stack.back();
      stack.pop_back();
      Entry& e = entry[x];
      auto it = index.find(key_of(e.parent, e.tokens.data(), block_size));
      auto& bucket = it->second;
      for (size_t i = 0; i < bucket.size(); ++i)
        if (bucket[i] == x) {
          bucket[i] = bucket.back();
          bucket.pop_back();
          break;
        }
      if (bucket.empty()) index.erase(it);
      for (int32_t c : e.children) stack.push_back(c);
      e = Entry{};
      --num_registered;
    }
  }

  void unlink(int32_t b) {
    if (prev[b] >= 0) next[prev[b]] = next[b]; else head = next[b];
    if (next[b] >= 0) prev[next[b]] = prev[b]; else tail = prev[b];
    prev[b] = next[b] = -1;
    on_free[b] = 0;
    --count;
  }
  int32_t pop_free() {
    int32_t b = head;
    unlink(b);
    if (entry[b].registered) unregister(b);  // handed out again: its contents will change
    refcount[b] = 1;
    return b;
  }
  void push_free(int32_t b) {
    prev[b] = tail;
    next[b] = -1;
    if (tail >= 0) next[tail] = b; else head = b;
    tail = b;
    on_free[b] = 1;
    ++count;
  }
  // A reference to a block found by a lookup (revived from the free list if
  // nobody holds it).
  void take_cached(int32_t b) {
    if (refcount[b] == 0) unlink(b);
    ++refcount[b];
  }
  // Registers the blocks of a tracked sequence that have become full, in
  // order; an identical block registered elsewhere ends the chain (the
  // sequence's later blocks then stay unregistered).
  void register_full_blocks(Seq& s) {
    const int32_t B = block_size;
    const int32_t full = s.len / B;
    while (s.tracked && s.reg_upto < full) {
      const int32_t j = s.reg_upto;
      const int32_t parent = j == 0 ? -1 : s.blocks[j - 1];
      const int32_t* tok = s.tokens.data() + (int64_t)j * B;
      if (lookup(parent, tok) >= 0) {
        s.tracked = false;
        s.tokens.clear();
        break;
      }
      register_block(s.blocks[j], parent, tok);
      ++s.reg_upto;
    }
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
  a->next.assign(num_blocks, -1);
  a->prev.assign(num_blocks, -1);
  a->on_free.assign(num_blocks, 0);
  a->refcount.assign(num_blocks, 0);
  a->entry.resize(num_blocks);
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
    }
    for (int32_t i = 0; i < num_blocks; ++i) a->push_free(free_order[i]);
  } else {
    for (int32_t i = 0; i < num_blocks; ++i) a->push_free(i);
  }
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

extern "C" int pkv_seq_create_many(pkv_alloc* a, int32_t n, int64_t* seq_ids) {
  PKV_REQUIRE(a && n >= 0 && (n == 0 || seq_ids), "pkv_seq_create_many: bad arguments");
  for (int32_t i = 0; i < n; ++i) {
    const int64_t id = a->next_id++;
    a->seqs.emplace(id, pkv_alloc::Seq{});
    seq_ids[i] = id;
  }
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

namespace {

// Reserves slots for n new tokens of a sequence; token_ids (nullable) are
// recorded for the prefix cache.
int append_seq(pkv_alloc* a, pkv_alloc::Seq* s, int64_t seq, int32_t n,
               const int32_t* token_ids, int32_t* slots_out, int32_t* cow_pair_out,
               int32_t* n_cow, const char* who);

int append_impl(pkv_alloc* a, int64_t seq, int32_t n, const int32_t* token_ids,
                int32_t* slots_out, int32_t* cow_pair_out, int32_t* n_cow, const char* who) {
  PKV_REQUIRE(a && n_cow, "%s: NULL argument", who);
  pkv_alloc::Seq* s = a->find(seq);
  PKV_REQUIRE(s, "%s: unknown sequence %lld", who, (long long)seq);
  return append_seq(a, s, seq, n, token_ids, slots_out, cow_pair_out, n_cow, who);
}

// append_impl on a sequence already looked up
int append_seq(pkv_alloc* a, pkv_alloc::Seq* s, int64_t seq, int32_t n,
               const int32_t* token_ids, int32_t* slots_out, int32_t* cow_pair_out,
               int32_t* n_cow, const char* who) {
  PKV_REQUIRE(n >= 0, "%s: n must be >= 0 (got %d)", who, n);
  PKV_REQUIRE(n == 0 || slots_out, "%s: slots_out is NULL", who);
  PKV_REQUIRE(!s->swapped, "%s: sequence %lld is swapped out", who, (long long)seq);
  *n_cow = 0;
  if (n == 0) return ok();
  const int32_t B = a->block_size;
  const int64_t new_len = (int64_t)s->len + n;
  PKV_REQUIRE(new_len < (int64_t(1) << 31), "%s: sequence length overflows int32", who);
  // Blocks needed: the ones that open past the current table, plus one copy
  // when the first new token lands in a shared, partially filled last block.
  const bool partial = (s->len % B) != 0;
  const bool cow = partial && a->refcount[s->blocks.back()] > 1;
  const int64_t need = (new_len + B - 1) / B - (int64_t)s->blocks.size() + (cow ? 1 : 0);
  if (need > a->count)
    return fail(PKV_ENOMEM, "%s: sequence %lld needs %lld blocks, %d free", who,
                (long long)seq, (long long)need, a->count);
  PKV_REQUIRE(!cow || cow_pair_out, "%s: cow_pair_out is NULL but a copy is needed", who);
  if (cow) {
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
  if (s->tracked && token_ids) {
    s->tokens.insert(s->tokens.end(), token_ids, token_ids + n);
    a->register_full_blocks(*s);
  } else {
    s->tracked = false;
    s->tokens.clear();
  }
  return ok();
}

}  // namespace

extern "C" int pkv_seq_append_slots(pkv_alloc* a, int64_t seq, int32_t n, int32_t* slots_out,
                                    int32_t* cow_pair_out, int32_t* n_cow) {
  return append_impl(a, seq, n, nullptr, slots_out, cow_pair_out, n_cow, "pkv_seq_append_slots");
}

// Prefix caching ("Batching, Scheduling, and Paging", section Block sharing:
// identical prefixes of different requests can share blocks; "Paging the KV
// Cache": a system prompt common to many requests occupies one set of pages).
extern "C" int pkv_seq_append_tokens(pkv_alloc* a, int64_t seq, const int32_t* token_ids,
                                     int32_t n, int32_t* slots_out, int32_t* cow_pair_out,
                                     int32_t* n_cow) {
  PKV_REQUIRE(n == 0 || token_ids, "pkv_seq_append_tokens: token_ids is NULL");
  return append_impl(a, seq, n, token_ids, slots_out, cow_pair_out, n_cow,
                     "pkv_seq_append_tokens");
}

extern "C" int pkv_seq_create_cached(pkv_alloc* a, const int32_t* token_ids, int32_t n,
                                     int64_t* seq_id, int32_t* n_cached) {
  PKV_REQUIRE(a && seq_id && n_cached, "pkv_seq_create_cached: NULL argument");
  PKV_REQUIRE(n >= 0 && (n == 0 || token_ids), "pkv_seq_create_cached: bad token array");
  const int32_t B = a->block_size;
  pkv_alloc::Seq s;
  // at most the full blocks before the last token: that token is always computed
  const int32_t max_full = n > 0 ? (n - 1) / B : 0;
  int32_t parent = -1;
  for (int32_t j = 0; j < max_full; ++j) {
    const int32_t b = a->lookup(parent, token_ids + (int64_t)j * B);
    if (b < 0) break;
    a->take_cached(b);
    s.blocks.push_back(b);
    parent = b;
  }
  s.len = (int32_t)s.blocks.size() * B;
  s.reg_upto = (int32_t)s.blocks.size();
  s.tokens.assign(token_ids, token_ids + s.len);
  int64_t id = a->next_id++;
  a->seqs.emplace(id, std::move(s));
  *seq_id = id;
  *n_cached = (int32_t)(a->seqs[id].len);
  return ok();
}

extern "C" int pkv_num_cached_blocks(pkv_alloc* a, int32_t* out) {
  PKV_REQUIRE(a && out, "pkv_num_cached_blocks: NULL argument");
  *out = a->num_registered;
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

extern "C" int pkv_seq_free_many(pkv_alloc* a, const int64_t* seqs, int32_t n) {
  const char* who = "pkv_seq_free_many";
  PKV_REQUIRE(a && n >= 0 && (n == 0 || seqs), "%s: bad arguments", who);
  // every id known and listed once, else nothing is freed
  const uint64_t ep = ++a->epoch;
  for (int32_t i = 0; i < n; ++i) {
    pkv_alloc::Seq* s = a->find(seqs[i]);
    PKV_REQUIRE(s, "%s: unknown sequence %lld", who, (long long)seqs[i]);
    PKV_REQUIRE(s->mark != ep, "%s: sequence %lld appears twice", who, (long long)seqs[i]);
    s->mark = ep;
  }
  for (int32_t i = 0; i < n; ++i) {
    auto it = a->seqs.find(seqs[i]);
    for (int32_t b : it->second.blocks)
      if (--a->refcount[b] == 0) a->push_free(b);
    a->seqs.erase(it);
  }
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
  s->tracked = false;  // fresh blocks are not registered
  s->tokens.clear();
  s->reg_upto = 0;
  *n = m;
  return ok();
}

// ---------------------------------------------------------------------------
// One iteration's host work in one call ("Batching, Scheduling, and Paging",
// section Continuous batching: the batch is rebuilt every iteration, and the
// CPU-side work per iteration is the overhead to keep small; "Deep Dive:
// continuous batching", section Iteration-level scheduling). The appends keep
// the per-sequence rules of append_impl; the batch is all or nothing: a
// dry run over the whole list (including the refcounts that earlier copies
// in the same batch release) decides before anything changes.

namespace {

constexpr int64_t kMetaAlign = 64;  // bytes; every section starts on a line

int64_t align_up(int64_t x) { return (x + kMetaAlign - 1) / kMetaAlign * kMetaAlign; }

int layout_impl(int32_t n_prefill, int32_t n_decode, int64_t n_tokens,
                int32_t max_blocks_per_seq, pkv_iteration_layout* L, const char* who) {
  PKV_REQUIRE(L, "%s: layout is NULL", who);
  PKV_REQUIRE(n_prefill >= 0 && n_decode >= 0 && n_tokens >= 0 && max_blocks_per_seq > 0,
              "%s: bad sizes", who);
  const int64_t n = (int64_t)n_prefill + n_decode;
  const int64_t W = max_blocks_per_seq;
  int64_t off = 0;
  std::memset(L, 0, sizeof(*L));
  L->slot_mapping = off;   off = align_up(off + 4 * n_tokens);
  L->cu_q_lens = off;      off = align_up(off + 4 * ((int64_t)n_prefill + 1));
  L->prefill_lens = off;   off = align_up(off + 4 * (int64_t)n_prefill);
  L->prefill_tables = off; off = align_up(off + 4 * (int64_t)n_prefill * W);
  L->decode_lens = off;    off = align_up(off + 4 * (int64_t)n_decode);
  L->decode_tables = off;  off = align_up(off + 4 * (int64_t)n_decode * W);
  L->cow_pairs = off;      off = align_up(off + 8 * n);
  L->total_bytes = off;
  L->table_width = max_blocks_per_seq;
  return PKV_OK;
}

}  // namespace

extern "C" int pkv_iteration_layout_bytes(int32_t n_prefill, int32_t n_decode,
                                          int32_t n_tokens, int32_t max_blocks_per_seq,
                                          pkv_iteration_layout* layout) {
  if (int rc = layout_impl(n_prefill, n_decode, n_tokens, max_blocks_per_seq, layout,
                           "pkv_iteration_layout_bytes"))
    return rc;
  return ok();
}

extern "C" int pkv_iteration_prepare(pkv_alloc* a, const int64_t* seqs, const int32_t* counts,
                                     int32_t n_prefill, int32_t n_decode,
                                     int32_t max_blocks_per_seq, void* buf, size_t buf_bytes,
                                     pkv_iteration_layout* layout, int32_t* n_fit) {
  const char* who = "pkv_iteration_prepare";
  PKV_REQUIRE(a && layout && n_fit, "%s: NULL argument", who);
  PKV_REQUIRE(n_prefill >= 0 && n_decode >= 0, "%s: bad sizes", who);
  const int32_t n = n_prefill + n_decode;
  PKV_REQUIRE(n == 0 || (seqs && counts), "%s: NULL array", who);
  PKV_REQUIRE(buf, "%s: buf is NULL", who);
  const int32_t B = a->block_size;
  // validate every work and dry-run the block needs, in order
  int64_t n_tokens = 0, need = 0;
  int32_t fit = n, width = 1;  // the longest table after the appends
  std::unordered_map<int32_t, int32_t> released;  // refs dropped by earlier copies
  // a sequence listed twice carries this call's mark already
  const uint64_t ep = ++a->epoch;
  a->batch.resize((size_t)n);
  for (int32_t i = 0; i < n; ++i) {
    pkv_alloc::Seq* s = a->find(seqs[i]);
    PKV_REQUIRE(s, "%s: unknown sequence %lld (work %d)", who, (long long)seqs[i], i);
    PKV_REQUIRE(!s->swapped, "%s: sequence %lld is swapped out", who, (long long)seqs[i]);
    PKV_REQUIRE(s->mark != ep, "%s: sequence %lld appears twice", who, (long long)seqs[i]);
    s->mark = ep;
    a->batch[i] = s;
    const int32_t c = counts[i];
    PKV_REQUIRE(i < n_prefill ? c >= 1 : c == 1,
                "%s: work %d: a prefill chunk needs >= 1 token and a decode exactly 1 (got %d)",
                who, i, c);
    const int64_t new_len = (int64_t)s->len + c;
    PKV_REQUIRE(new_len < (int64_t(1) << 31), "%s: sequence length overflows int32", who);
    PKV_REQUIRE((new_len + B - 1) / B <= max_blocks_per_seq,
                "%s: sequence %lld would need %lld blocks > max_blocks_per_seq %d", who,
                (long long)seqs[i], (long long)((new_len + B - 1) / B), max_blocks_per_seq);
    bool cow = false;
    if (s->len % B != 0) {
      const int32_t last = s->blocks.back();
      auto it = released.find(last);
      const int32_t refs = a->refcount[last] - (it == released.end() ? 0 : it->second);
      if (refs > 1) {
        cow = true;
        ++released[last];
      }
    }
    need += (new_len + B - 1) / B - (int64_t)s->blocks.size() + (cow ? 1 : 0);
    if ((new_len + B - 1) / B > width) width = (int32_t)((new_len + B - 1) / B);
    if (need > a->count && fit == n) fit = i;
    n_tokens += c;
  }
  PKV_REQUIRE(n_tokens < (int64_t(1) << 31), "%s: too many tokens", who);
  // tables are as wide as the batch's longest one (at most max_blocks_per_seq),
  // so the buffer a caller sized with pkv_iteration_layout_bytes always fits
  if (int rc = layout_impl(n_prefill, n_decode, n_tokens, width, layout, who)) return rc;
  PKV_REQUIRE(buf_bytes >= (size_t)layout->total_bytes, "%s: buf has %zu bytes, needs %lld", who,
              buf_bytes, (long long)layout->total_bytes);
  *n_fit = fit;
  if (fit < n)
    return fail(PKV_ENOMEM,
                "%s: the batch needs %lld free blocks, %d free; the first %d works fit", who,
                (long long)need, a->count, fit);
  // apply: cannot fail any more
  uint8_t* base = static_cast<uint8_t*>(buf);
  int32_t* slots = reinterpret_cast<int32_t*>(base + layout->slot_mapping);
  int32_t* cu = reinterpret_cast<int32_t*>(base + layout->cu_q_lens);
  int32_t* pairs = reinterpret_cast<int32_t*>(base + layout->cow_pairs);
  int32_t n_cow = 0, max_q = 0;
  cu[0] = 0;
  for (int32_t i = 0; i < n; ++i) {
    int32_t got_cow = 0;
    append_seq(a, a->batch[i], seqs[i], counts[i], nullptr, slots, pairs + 2 * n_cow, &got_cow,
               who);
    slots += counts[i];
    n_cow += got_cow;
    if (i < n_prefill) {
      cu[i + 1] = cu[i] + counts[i];
      if (counts[i] > max_q) max_q = counts[i];
    }
  }
  const int64_t W = width;
  int32_t max_len[2] = {0, 0};
  for (int32_t part = 0; part < 2; ++part) {
    const int32_t first = part == 0 ? 0 : n_prefill;
    const int32_t count = part == 0 ? n_prefill : n_decode;
    int32_t* lens = reinterpret_cast<int32_t*>(
        base + (part == 0 ? layout->prefill_lens : layout->decode_lens));
    int32_t* tables = reinterpret_cast<int32_t*>(
        base + (part == 0 ? layout->prefill_tables : layout->decode_tables));
    for (int32_t k = 0; k < count; ++k) {
      const pkv_alloc::Seq* s = a->batch[first + k];
      int32_t* row = tables + k * W;
      const int32_t m = (int32_t)s->blocks.size();
      // (entries past the last block stay as they were: no kernel reads them)
      if (m) std::memcpy(row, s->blocks.data(), sizeof(int32_t) * m);
      lens[k] = s->len;
      if (s->len > max_len[part]) max_len[part] = s->len;
    }
  }
  layout->n_tokens = (int32_t)n_tokens;
  layout->n_cow = n_cow;
  layout->max_q_len = max_q;
  layout->max_prefill_len = max_len[0];
  layout->max_decode_len = max_len[1];
  return ok();
}
