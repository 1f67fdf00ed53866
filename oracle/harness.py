"""Builds the oracle's view of a workload: its own allocator, pools and outputs.

TEST INFRASTRUCTURE ONLY, like the rest of this package: everything here
runs the CPU oracle on the seeded workload inputs (``workloads``), and
nothing reads a value produced by the library. The tests, the smoke check
and the benchmark's CPU-baseline leg use it.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from oracle import attention, cache, paging
from workloads import BF16_NAN
from workloads.schedule import OutOfBlocks, iteration_inputs


@dataclass
class OracleDecodeState:
    alloc: paging.BlockAllocator
    seq_ids: list
    k_cache: np.ndarray
    v_cache: np.ndarray
    tables: list                  # list of per-sequence block lists
    slots: list                   # per-sequence slot lists (all tokens)

    def padded_tables(self, width: int | None = None) -> np.ndarray:
        width = width or max(1, max(len(t) for t in self.tables))
        out = np.zeros((len(self.tables), width), dtype=np.int32)
        for s, t in enumerate(self.tables):
            out[s, :len(t)] = t
        return out


def empty_pools(num_blocks, Hkv, B, D, poison=True):
    fill = BF16_NAN if poison else np.uint16(0)
    k = np.full((num_blocks, Hkv, B, D), fill, dtype=np.uint16)
    v = np.full((num_blocks, Hkv, B, D), fill, dtype=np.uint16)
    return k, v


def build_decode_state(w, poison=True, include_last=True) -> OracleDecodeState:
    """Allocate every sequence's blocks through the oracle allocator and write
    its tokens (all of them, or all but the last when ``include_last`` is
    False) into NaN-poisoned pools."""
    alloc = paging.BlockAllocator(w.num_blocks, w.block_size, w.free_order)
    k_cache, v_cache = empty_pools(w.num_blocks, w.Hkv, w.block_size, w.D, poison)
    cu = w.cu_lens
    seq_ids, tables, slots = [], [], []
    for s in range(w.S):
        sid = alloc.create()
        sl, pairs = alloc.append_slots(sid, int(w.context_lens[s]))
        assert not pairs
        seq_ids.append(sid)
        tables.append(alloc.block_table(sid))
        slots.append(sl)
        n = len(sl) if include_last else len(sl) - 1
        cache.append(k_cache, v_cache, w.k[cu[s]:cu[s] + n], w.v[cu[s]:cu[s] + n],
                     sl[:n], w.block_size)
    return OracleDecodeState(alloc, seq_ids, k_cache, v_cache, tables, slots)


def decode_reference(w, st: OracleDecodeState, seqs=None) -> np.ndarray:
    return attention.decode(w.q, st.k_cache, st.v_cache, st.tables, w.context_lens,
                            w.block_size, w.scale, seqs=seqs)


@dataclass
class OracleSharedPrefixState:
    alloc: paging.BlockAllocator
    sample_ids: list              # [n_prompts * n_samples] sequence ids
    k_cache: np.ndarray
    v_cache: np.ndarray
    prefix_slots: list            # per prompt
    tail_slots: list              # per sample
    cow_pairs: list               # all (src, dst) pairs, in append order
    tables: list


def build_shared_prefix_state(w, poison=True) -> OracleSharedPrefixState:
    """The build order of a shared-prefix workload, on the oracle side."""
    alloc = paging.BlockAllocator(w.num_blocks, w.block_size, w.free_order)
    k_cache, v_cache = empty_pools(w.num_blocks, w.Hkv, w.block_size, w.D, poison)
    sample_ids, prefix_slots = [], []
    for p in range(w.n_prompts):
        sid = alloc.create()
        sl, pairs = alloc.append_slots(sid, w.prefix_len)
        assert not pairs
        prefix_slots.append(sl)
        cache.append(k_cache, v_cache, w.prefix_k[p], w.prefix_v[p], sl, w.block_size)
        sample_ids.append(sid)
        for _ in range(w.n_samples - 1):
            sample_ids.append(alloc.fork(sid))
    tail_slots, cow_pairs = [], []
    for i, sid in enumerate(sample_ids):
        sl, pairs = alloc.append_slots(sid, int(w.tails.reshape(-1)[i]))
        tail_slots.append(sl)
        cow_pairs.extend(pairs)
    # copy-on-write copies run before any tail token is written
    cache.block_copy(k_cache, v_cache, cow_pairs)
    cu = w.cu_tails
    for i in range(len(sample_ids)):
        cache.append(k_cache, v_cache, w.tail_k[cu[i]:cu[i + 1]], w.tail_v[cu[i]:cu[i + 1]],
                     tail_slots[i], w.block_size)
    tables = [alloc.block_table(sid) for sid in sample_ids]
    return OracleSharedPrefixState(alloc, sample_ids, k_cache, v_cache, prefix_slots,
                                   tail_slots, cow_pairs, tables)


def bf16_tolerance_ok(gpu: np.ndarray, ref: np.ndarray, atol=2e-3, rtol=1e-2) -> np.ndarray:
    """Elementwise ``|gpu - ref| <= atol + rtol * |ref|``."""
    return np.abs(gpu - ref) <= atol + rtol * np.abs(ref)


class OracleTrace:
    """The continuous-batching trace on the oracle side: the oracle's
    allocator model, its own pools and fp64 attention for chosen sequences."""

    def __init__(self, cfg, poison=True):
        self.cfg = cfg
        self.alloc = paging.BlockAllocator(cfg.num_blocks, cfg.block_size)
        self.k_cache, self.v_cache = empty_pools(cfg.num_blocks, cfg.Hkv, cfg.block_size,
                                                 cfg.D, poison)
        self.sid = {}
        self.scale = 1.0 / np.sqrt(cfg.D)

    def step(self, itr):
        """Reserve slots and write this iteration's tokens; returns the slots."""
        for rid in itr.admitted:
            self.sid[rid] = self.alloc.create()
        slots = []
        for wk in itr.work:
            sl, pairs = self.alloc.append_slots(self.sid[wk.rid], wk.n)
            assert not pairs
            slots.extend(sl)
        cache.append(self.k_cache, self.v_cache, itr.k, itr.v, slots, self.cfg.block_size)
        return np.asarray(slots, dtype=np.int32)

    def prefill(self, itr, which):
        """fp64 outputs of the prefill works with indices ``which``: {index: [n, Hq, D]}."""
        out = {}
        pre = itr.prefill
        row0 = np.concatenate([[0], np.cumsum([wk.n for wk in pre])])
        for i in which:
            wk = pre[i]
            sid = self.sid[wk.rid]
            L = self.alloc.seq_len(sid)
            cu = np.array([0, wk.n])
            out[i] = attention.prefill(itr.q[row0[i]:row0[i] + wk.n], cu, [L], self.k_cache,
                                       self.v_cache, [self.alloc.block_table(sid)],
                                       self.cfg.block_size, self.scale)
        return out

    def decode(self, itr, which):
        """fp64 outputs of the decode works with indices ``which``: {index: [Hq, D]}."""
        out = {}
        n_pre = sum(wk.n for wk in itr.prefill)
        dec = itr.decode
        for i in which:
            sid = self.sid[dec[i].rid]
            L = self.alloc.seq_len(sid)
            out[i] = attention.decode(itr.q[n_pre + i:n_pre + i + 1], self.k_cache, self.v_cache,
                                      [self.alloc.block_table(sid)], [L], self.cfg.block_size,
                                      self.scale)[0]
        return out

    def finish(self, itr):
        for rid in itr.finished:
            self.alloc.free_seq(self.sid.pop(rid))


# ---------------------------------------------------------------- preemption


class OracleAllocator:
    """Adapter over oracle.paging.BlockAllocator."""

    def __init__(self, num_blocks, block_size):
        self.paging = paging
        self.a = paging.BlockAllocator(num_blocks, block_size)

    def create(self):
        return self.a.create()

    def append(self, sid, n):
        try:
            slots, pairs = self.a.append_slots(sid, n)
        except self.paging.OutOfBlocks as e:
            raise OutOfBlocks(str(e)) from None
        assert not pairs
        return slots

    def free(self, sid):
        self.a.free_seq(sid)

    def create_cached(self, tokens):
        return self.a.create_cached(tokens)

    def append_tokens(self, sid, tokens):
        try:
            slots, pairs = self.a.append_tokens(sid, tokens)
        except self.paging.OutOfBlocks as e:
            raise OutOfBlocks(str(e)) from None
        assert not pairs
        return slots

    def num_cached(self):
        return self.a.num_cached()

    def swap_out(self, sid):
        return self.a.swap_out(sid)

    def swap_in(self, sid):
        try:
            return self.a.swap_in(sid)
        except self.paging.OutOfBlocks as e:
            raise OutOfBlocks(str(e)) from None

    def table(self, sid):
        return self.a.block_table(sid)

    def num_free(self):
        return self.a.num_free()


class OracleRunner:
    """Replays the same events with the CPU oracle."""

    def __init__(self, cfg, num_blocks):
        self.cfg = cfg
        self.k_cache, self.v_cache = empty_pools(num_blocks, cfg.Hkv, cfg.block_size, cfg.D)
        self.saved = {}
        self.scale = 1.0 / np.sqrt(cfg.D)

    def run(self, ev, values):
        cfg = self.cfg
        shape = (cfg.Hkv, cfg.block_size, cfg.D)
        for kind, rid, blocks in ev.ops:
            if kind == "swap_out":
                kb = np.empty((len(blocks),) + shape, np.uint16)
                vb = np.empty_like(kb)
                cache.swap_blocks(self.k_cache, self.v_cache, blocks, kb, vb, 0)
                self.saved[rid] = (kb, vb)
            else:
                kb, vb = self.saved.pop(rid)
                cache.swap_blocks(self.k_cache, self.v_cache, blocks, kb, vb, 1)
        pre, dec, q, k, v, slots, meta = iteration_inputs(cfg, ev, values)
        cache.append(self.k_cache, self.v_cache, k, v, slots, cfg.block_size)
        return pre, dec, q, meta

    def prefill(self, ev, pre, q, meta, i):
        tables, lens = meta["prefill"]
        a, b = int(meta["cu"][i]), int(meta["cu"][i + 1])
        return attention.prefill(q[a:b], np.array([0, b - a]), [int(lens[i])], self.k_cache,
                                 self.v_cache, [tables[i]], self.cfg.block_size, self.scale)

    def decode(self, ev, q, meta, i):
        tables, lens = meta["decode"]
        n_pre = int(meta["cu"][-1])
        return attention.decode(q[n_pre + i:n_pre + i + 1], self.k_cache, self.v_cache,
                                [tables[i]], [int(lens[i])], self.cfg.block_size, self.scale)[0]
