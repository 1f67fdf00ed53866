"""Reference model of the block table and its CPU-side allocator.

Follows "Batching, Scheduling, and Paging" (datasystem.school, module 4):

* section *PagedAttention*: each sequence's KV cache is split into fixed-size
  blocks stored non-contiguously; a per-sequence block table maps logical
  block ``j`` to a physical block; the CPU allocates a new block only when the
  previous one fills and frees blocks when the request completes;
* section *Block sharing*: parallel samples point at the same physical blocks;
  the first divergent write triggers copy-on-write, and reference counts keep
  a shared block alive until its last user finishes.

Readings where the page is silent:

* free blocks are handed out first-in first-out; the initial order is the
  caller's permutation, and a block whose count drops to zero joins the tail;
* copy-on-write applies only to a *partially filled* shared last block that
  receives a new token: the writer gets a fresh block, a ``(src, dst)`` copy
  pair is emitted and the source's count drops by one, so with four sharers
  the first three writers copy and the fourth writes in place; full shared
  blocks are never written and never copied;
* a slot is ``physical_block * block_size + offset``;
* an append that cannot get all the blocks it needs fails as a whole and
  changes nothing;
* eviction when memory runs out (same page, section PagedAttention: swap the
  request to CPU memory or discard and recompute it): swapping out hands the
  sequence's blocks back in table order (each loses one reference) and keeps
  its length; swapping in takes fresh blocks for all its tokens, first in
  first out, all or nothing. Recomputing is freeing and starting again;
* prefix caching (section *Block sharing*: identical prefixes of different
  requests can share blocks; "Paging the KV Cache": one set of pages for a
  system prompt that many concurrent requests share): a full block whose
  token ids are known is registered under the whole token prefix it ends
  (at most one block per prefix); a new request starts with the registered
  blocks of its longest registered full-block prefix, leaving at least its
  last token to compute; a registered block stays registered after its last
  user leaves, and loses its entry (with every entry that extends its prefix)
  when the free list hands it out again. A sequence stops registering at the
  first block whose prefix is already registered elsewhere, or once it has
  been appended without token ids or swapped in.

TEST INFRASTRUCTURE ONLY (see the package docstring).
"""

from __future__ import annotations

from collections import deque


class OutOfBlocks(Exception):
    """No free block for an append; the allocator state is unchanged."""


class BlockAllocator:
    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        if free_order is None:
            free_order = range(num_blocks)
        order = [int(b) for b in free_order]
        assert sorted(order) == list(range(num_blocks)), "free_order must be a permutation"
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free = deque(order)
        self.refcount = [0] * num_blocks
        self.seqs: dict[int, dict] = {}
        self._next_id = 0
        self.registry: dict[tuple, int] = {}     # token prefix -> block that ends it
        self.prefix_of: dict[int, tuple] = {}    # block -> its registered prefix

    # -- sequences ---------------------------------------------------------
    def create(self) -> int:
        sid = self._next_id
        self._next_id += 1
        self.seqs[sid] = {"blocks": [], "len": 0, "swapped": False, "tokens": [],
                          "registered": 0}
        return sid

    def create_cached(self, tokens) -> tuple[int, int]:
        """A sequence starting with the registered blocks of ``tokens``'s
        longest registered full-block prefix; returns ``(sid, cached tokens)``."""
        tokens = [int(t) for t in tokens]
        B = self.block_size
        sid = self.create()
        seq = self.seqs[sid]
        j = 0
        while j < (len(tokens) - 1) // B and tuple(tokens[:(j + 1) * B]) in self.registry:
            b = self.registry[tuple(tokens[:(j + 1) * B])]
            if self.refcount[b] == 0:
                self.free.remove(b)
            self.refcount[b] += 1
            seq["blocks"].append(b)
            j += 1
        seq["len"] = j * B
        seq["tokens"] = tokens[:j * B]
        seq["registered"] = j
        return sid, j * B

    def append_tokens(self, sid: int, tokens):
        """``append_slots`` recording the token ids; full blocks get registered."""
        tokens = [int(t) for t in tokens]
        slots, pairs = self.append_slots(sid, len(tokens), _keep_tokens=True)
        seq = self.seqs[sid]
        if seq["tokens"] is None:
            return slots, pairs
        seq["tokens"] += tokens
        B = self.block_size
        while seq["registered"] < seq["len"] // B:
            j = seq["registered"]
            key = tuple(seq["tokens"][:(j + 1) * B])
            if key in self.registry:
                seq["tokens"] = None          # an identical block is registered elsewhere
                break
            self.registry[key] = seq["blocks"][j]
            self.prefix_of[seq["blocks"][j]] = key
            seq["registered"] += 1
        return slots, pairs

    def num_cached(self) -> int:
        return len(self.registry)

    def fork(self, parent: int) -> int:
        """A new sequence that shares every block of ``parent`` (Block sharing)."""
        src = self.seqs[parent]
        sid = self._next_id
        self._next_id += 1
        assert not src["swapped"], "cannot fork a swapped-out sequence"
        self.seqs[sid] = {"blocks": list(src["blocks"]), "len": src["len"], "swapped": False,
                          "tokens": None if src["tokens"] is None else list(src["tokens"]),
                          "registered": src["registered"]}
        for b in src["blocks"]:
            self.refcount[b] += 1
        return sid

    def free_seq(self, sid: int) -> None:
        """Drop the sequence; a block returns to the free list at count zero."""
        seq = self.seqs.pop(sid)
        for b in seq["blocks"]:
            self.refcount[b] -= 1
            if self.refcount[b] == 0:
                self.free.append(b)

    def _take(self) -> int:
        b = self.free.popleft()
        self.refcount[b] = 1
        if b in self.prefix_of:
            # handed out again: drop its entry and every entry extending its prefix
            p = self.prefix_of[b]
            for key in [k for k in self.registry if k[:len(p)] == p]:
                del self.prefix_of[self.registry.pop(key)]
        return b

    def blocks_needed(self, sid: int, n: int) -> int:
        seq = self.seqs[sid]
        B = self.block_size
        L = seq["len"]
        need = -(-(L + n) // B) - len(seq["blocks"])
        if n > 0 and L % B != 0 and self.refcount[seq["blocks"][-1]] > 1:
            need += 1
        return need

    def swap_out(self, sid: int) -> list[int]:
        """Give the sequence's blocks back (table order); it keeps its length."""
        seq = self.seqs[sid]
        assert not seq["swapped"]
        blocks = list(seq["blocks"])
        for b in blocks:
            self.refcount[b] -= 1
            if self.refcount[b] == 0:
                self.free.append(b)
        seq["blocks"] = []
        seq["swapped"] = True
        return blocks

    def swap_in(self, sid: int) -> list[int]:
        """Fresh blocks for all of a swapped-out sequence's tokens."""
        seq = self.seqs[sid]
        assert seq["swapped"]
        need = -(-seq["len"] // self.block_size)
        if need > len(self.free):
            raise OutOfBlocks(f"sequence {sid} needs {need} blocks, {len(self.free)} free")
        seq["blocks"] = [self._take() for _ in range(need)]
        seq["swapped"] = False
        seq["tokens"], seq["registered"] = None, 0   # fresh blocks are not registered
        return list(seq["blocks"])

    def append_slots(self, sid: int, n: int, _keep_tokens: bool = False):
        """Reserve slots for ``n`` new tokens; return ``(slots, cow_pairs)``."""
        assert not self.seqs[sid]["swapped"], "append to a swapped-out sequence"
        if self.blocks_needed(sid, n) > len(self.free):
            raise OutOfBlocks(f"sequence {sid} needs {self.blocks_needed(sid, n)} blocks, "
                              f"{len(self.free)} free")
        seq = self.seqs[sid]
        B = self.block_size
        slots, pairs = [], []
        for pos in range(seq["len"], seq["len"] + n):
            j, off = divmod(pos, B)
            if j == len(seq["blocks"]):
                # previous block is full (or there is none): allocate on fill
                seq["blocks"].append(self._take())
            elif self.refcount[seq["blocks"][j]] > 1:
                # first divergent write into a shared partial block
                old = seq["blocks"][j]
                new = self._take()
                self.refcount[old] -= 1
                seq["blocks"][j] = new
                pairs.append((old, new))
            slots.append(seq["blocks"][j] * B + off)
        seq["len"] += n
        if n > 0 and not _keep_tokens:
            seq["tokens"] = None                  # token ids unknown from here on
        return slots, pairs

    # -- queries -----------------------------------------------------------
    def block_table(self, sid: int) -> list[int]:
        return list(self.seqs[sid]["blocks"])

    def seq_len(self, sid: int) -> int:
        return self.seqs[sid]["len"]

    def num_free(self) -> int:
        return len(self.free)

    def check_invariants(self) -> None:
        """Counts equal table references; free + referenced = all blocks."""
        refs = [0] * self.num_blocks
        for seq in self.seqs.values():
            if seq["swapped"]:
                assert not seq["blocks"]
                continue
            assert len(seq["blocks"]) == -(-seq["len"] // self.block_size)
            for b in seq["blocks"]:
                refs[b] += 1
        assert refs == self.refcount
        free = set(self.free)
        assert len(free) == len(self.free)
        for b in range(self.num_blocks):
            assert (b in free) == (refs[b] == 0)
        # the prefix cache: one block per prefix, chains closed under shortening
        assert {b: k for k, b in self.registry.items()} == self.prefix_of
        for key, b in self.registry.items():
            assert len(key) % self.block_size == 0 and len(key) > 0
            if len(key) > self.block_size:
                assert key[:-self.block_size] in self.registry
        for seq in self.seqs.values():
            if seq["tokens"] is not None and not seq["swapped"]:
                assert len(seq["tokens"]) == seq["len"]
                for j in range(seq["registered"]):
                    key = tuple(seq["tokens"][:(j + 1) * self.block_size])
                    assert self.registry.get(key) == seq["blocks"][j]
