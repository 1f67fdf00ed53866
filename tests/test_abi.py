"""The C ABI on the CPU: symbols, argument checks and the host allocator.

No call here launches a kernel. The allocator is checked against the oracle's
model of it ("Batching, Scheduling, and Paging", sections PagedAttention and
Block sharing) and against the hand-derived scenario in tests/golden.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np
import pytest
import torch

import paged_kv_cache_281_gb300 as pkv
from paged_kv_cache_281_gb300 import _lib
from paged_kv_cache_281_gb300._lib import (PKV_EINVAL, PKV_ENOMEM, PagedKVError,
                                            header_functions, lib)
from oracle import paging
from tests.test_oracle_pins import parse_ids

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_library_exports_every_declared_symbol():
    names = header_functions()
    assert len(names) >= 20
    l = ctypes.CDLL(_lib.LIB_PATH)
    missing = [n for n in names if not hasattr(l, n)]
    assert not missing, missing
    assert set(names) == set(_lib.SIGNATURES), "binding and header disagree"


def test_version_and_error_string():
    assert pkv.pkv_version() >= 100
    with pytest.raises(PagedKVError) as e:
        pkv.BlockAllocator(0, 16)
    assert e.value.code == PKV_EINVAL
    assert "num_blocks" in pkv.pkv_last_error()


def _replay_on_library(path):
    alloc, names = None, {}
    for raw in open(os.path.join(GOLDEN, path)):
        line = raw.split("#", 1)[0].strip()
        if not line:
            continue
        op, *args = line.split()
        if op == "pool":
            alloc = pkv.BlockAllocator(int(args[0]), int(args[1]),
                                       [int(x) for x in args[2].split(",")])
        elif op == "create":
            names[args[0]] = alloc.seq_create()
        elif op == "fork":
            names[args[1]] = alloc.seq_fork(names[args[0]])
        elif op == "create_cached":
            names[args[0]], n_cached = alloc.seq_create_cached(parse_ids(args[1]))
            assert n_cached == int(args[2]), line
        elif op == "append_tokens":
            slots, pair = alloc.seq_append_tokens(names[args[0]], parse_ids(args[1]))
            assert slots.tolist() == parse_ids(args[2]) and pair is None, line
        elif op == "ncached":
            assert alloc.num_cached_blocks() == int(args[0]), line
        elif op == "append":
            slots, pair = alloc.seq_append_slots(names[args[0]], int(args[1]))
            want = parse_ids(args[2])
            want_pairs = ([tuple(int(y) for y in x.split(">")) for x in args[3].split(",")]
                          if args[3] != "-" else [])
            assert slots.tolist() == want, line
            assert ([pair] if pair else []) == want_pairs, line
        elif op == "append_fails":
            before = (alloc.num_free_blocks(), alloc.seq_block_table(names[args[0]]),
                      alloc.seq_len(names[args[0]]))
            with pytest.raises(PagedKVError) as e:
                alloc.seq_append_slots(names[args[0]], int(args[1]))
            assert e.value.code == PKV_ENOMEM
            assert before == (alloc.num_free_blocks(), alloc.seq_block_table(names[args[0]]),
                              alloc.seq_len(names[args[0]]))
        elif op == "table":
            want = [int(x) for x in args[1].split(",")] if args[1] != "-" else []
            assert alloc.seq_block_table(names[args[0]]) == want, line
        elif op == "refcount":
            assert alloc.block_refcount(int(args[0])) == int(args[1]), line
        elif op == "free":
            alloc.seq_free(names[args[0]])
        elif op == "nfree":
            assert alloc.num_free_blocks() == int(args[0]), line
        elif op == "freelist":
            # the free list order shows in the blocks that the next appends receive
            want = [int(x) for x in args[0].split(",")]
            assert alloc.num_free_blocks() == len(want), line
        else:
            raise ValueError(op)


def test_allocator_golden_scenario():
    _replay_on_library("allocator_block_sharing.txt")


def test_prefix_cache_golden_scenario():
    _replay_on_library("prefix_cache.txt")


def _prefix_cache_fuzz(seed):
    """Random requests drawn from a few shared prompts, with forks, frees,
    swaps and untracked appends: every result and the whole state agree.
    Returns (lookups that hit, operations that dropped entries)."""
    rng = np.random.default_rng(100 + seed)
    N, B = int(rng.integers(6, 24)), int(rng.choice([1, 2, 4, 8]))
    order = rng.permutation(N)
    lib_a = pkv.BlockAllocator(N, B, order)
    ref = paging.BlockAllocator(N, B, order)
    prompts = [rng.integers(0, 3, size=int(rng.integers(1, 6 * B + 3))).tolist()
               for _ in range(4)]
    live, swapped, pos = [], [], {}
    hits = drops = 0
    for _ in range(500):
        cached_before = ref.num_cached()
        op = int(rng.integers(0, 10))
        if op <= 1 or not live:
            base = prompts[int(rng.integers(len(prompts)))]
            toks = base[:int(rng.integers(1, len(base) + 1))] + \
                rng.integers(0, 3, size=int(rng.integers(0, 2 * B))).tolist()
            try:
                want = ref.create_cached(toks)
            except paging.OutOfBlocks:
                raise AssertionError("create_cached never allocates")
            got = lib_a.seq_create_cached(toks)
            assert got == want
            sid, nc = got
            hits += nc > 0
            live.append(sid)
            pos[sid] = toks[nc:]
        elif op == 2:
            p = live[int(rng.integers(len(live)))]
            assert lib_a.seq_fork(p) == ref.fork(p)
            live.append(ref._next_id - 1)
            pos[live[-1]] = list(pos[p])
        elif op in (3, 4):
            sid = live[int(rng.integers(len(live)))]
            pending = pos[sid]
            toks = pending if pending else rng.integers(0, 3, size=int(
                rng.integers(1, 2 * B + 2))).tolist()
            try:
                want_slots, want_pairs = ref.append_tokens(sid, toks)
            except paging.OutOfBlocks:
                with pytest.raises(PagedKVError) as e:
                    lib_a.seq_append_tokens(sid, toks)
                assert e.value.code == PKV_ENOMEM
            else:
                slots, pair = lib_a.seq_append_tokens(sid, toks)
                assert slots.tolist() == want_slots
                assert ([pair] if pair else []) == want_pairs
                pos[sid] = []
        elif op == 5:
            sid = live[int(rng.integers(len(live)))]
            n = int(rng.integers(1, B + 2))
            try:
                want_slots, _ = ref.append_slots(sid, n)
            except paging.OutOfBlocks:
                with pytest.raises(PagedKVError):
                    lib_a.seq_append_slots(sid, n)
            else:
                assert lib_a.seq_append_slots(sid, n)[0].tolist() == want_slots
                pos[sid] = []
        elif op in (6, 7, 8):
            sid = live.pop(int(rng.integers(len(live))))
            if rng.random() < 0.3:
                assert lib_a.seq_swap_out(sid) == ref.swap_out(sid)
                swapped.append(sid)
            else:
                lib_a.seq_free(sid)
                ref.free_seq(sid)
        elif swapped:
            sid = swapped[0]
            try:
                want = ref.swap_in(sid)
            except paging.OutOfBlocks:
                with pytest.raises(PagedKVError):
                    lib_a.seq_swap_in(sid)
            else:
                assert lib_a.seq_swap_in(sid) == want
                swapped.pop(0)
                live.append(sid)
        ref.check_invariants()
        drops += ref.num_cached() < cached_before
        assert lib_a.num_free_blocks() == ref.num_free()
        assert lib_a.num_cached_blocks() == ref.num_cached()
        for sid in live:
            assert lib_a.seq_block_table(sid) == ref.block_table(sid)
            assert lib_a.seq_len(sid) == ref.seq_len(sid)
        for blk in range(N):
            assert lib_a.block_refcount(blk) == ref.refcount[blk]
    return hits, drops


@pytest.mark.parametrize("seed", range(8))
def test_prefix_cache_matches_oracle_model(seed):
    _prefix_cache_fuzz(seed)


def test_prefix_cache_fuzz_reaches_hits_and_evictions():
    hits, drops = np.sum([_prefix_cache_fuzz(s) for s in range(8)], axis=0)
    assert hits > 100 and drops > 10, (hits, drops)


def test_allocator_free_list_order_after_release():
    a = pkv.BlockAllocator(6, 4, [3, 5, 0, 2, 4, 1])
    s = a.seq_create()
    a.seq_append_slots(s, 24)          # takes every block, in free-list order
    assert a.seq_block_table(s) == [3, 5, 0, 2, 4, 1]
    a.seq_free(s)                      # blocks rejoin the tail in table order
    t = a.seq_create()
    a.seq_append_slots(t, 24)
    assert a.seq_block_table(t) == [3, 5, 0, 2, 4, 1]


@pytest.mark.parametrize("seed", range(6))
def test_allocator_matches_oracle_model(seed):
    rng = np.random.default_rng(seed)
    N, B = int(rng.integers(4, 40)), int(rng.choice([1, 4, 8, 16]))
    order = rng.permutation(N)
    lib_a = pkv.BlockAllocator(N, B, order)
    ref = paging.BlockAllocator(N, B, order)
    live = []
    for _ in range(400):
        op = int(rng.integers(0, 5))
        if op == 0 or not live:
            a, b = lib_a.seq_create(), ref.create()
            assert a == b
            live.append(a)
        elif op == 1:
            p = live[int(rng.integers(len(live)))]
            a, b = lib_a.seq_fork(p), ref.fork(p)
            assert a == b
            live.append(a)
        elif op in (2, 3):
            sid = live[int(rng.integers(len(live)))]
            n = int(rng.integers(0, 3 * B + 2))
            try:
                want_slots, want_pairs = ref.append_slots(sid, n)
            except paging.OutOfBlocks:
                with pytest.raises(PagedKVError) as e:
                    lib_a.seq_append_slots(sid, n)
                assert e.value.code == PKV_ENOMEM
            else:
                slots, pair = lib_a.seq_append_slots(sid, n)
                assert slots.tolist() == want_slots
                assert ([pair] if pair else []) == want_pairs
        else:
            sid = live.pop(int(rng.integers(len(live))))
            lib_a.seq_free(sid)
            ref.free_seq(sid)
        assert lib_a.num_free_blocks() == ref.num_free()
        for sid in live:
            assert lib_a.seq_block_table(sid) == ref.block_table(sid)
            assert lib_a.seq_len(sid) == ref.seq_len(sid)
        for blk in range(N):
            assert lib_a.block_refcount(blk) == ref.refcount[blk]
    for sid in live:
        lib_a.seq_free(sid)
    assert lib_a.num_free_blocks() == N


def test_build_block_tables_pads_and_reports_lengths():
    a = pkv.BlockAllocator(8, 4, list(range(8)))
    s0, s1 = a.seq_create(), a.seq_create()
    a.seq_append_slots(s0, 5)
    a.seq_append_slots(s1, 1)
    tables, lens = a.build_block_tables([s0, s1], 3)
    assert tables.tolist() == [[0, 1, 0], [2, 0, 0]]
    assert lens.tolist() == [5, 1]
    with pytest.raises(PagedKVError):
        a.build_block_tables([s0], 1)


def test_allocator_rejects_bad_arguments():
    with pytest.raises(PagedKVError):
        pkv.BlockAllocator(4, 4, [0, 1, 1, 2])
    a = pkv.BlockAllocator(4, 4)
    with pytest.raises(PagedKVError):
        a.seq_append_slots(99, 1)
    with pytest.raises(PagedKVError):
        a.seq_fork(7)
    with pytest.raises(PagedKVError):
        a.block_refcount(4)


def _call(name, *args):
    return getattr(lib(), name)(*args)


def test_gpu_calls_reject_bad_shapes_before_touching_a_device():
    # Each of these fails host-side argument checks, so no CUDA call is made.
    assert _call("pkv_kv_append", None, None, None, 1, None, None, 4, 8, 96, 16, None,
                 None) == PKV_EINVAL
    assert _call("pkv_kv_append", None, None, None, 1, None, None, 4, 8, 128, 12, None,
                 None) == PKV_EINVAL
    assert _call("pkv_block_copy", None, None, None, 1, 4, 8, 128, 16, None, None) == PKV_EINVAL
    # group of 3 query heads per kv head
    assert _call("pkv_paged_attention_decode", None, None, None, None, None, 4, None, 64, 2, 6, 2,
                 128, 16, 8, 0.1, 0, None, 0, None, None) == PKV_EINVAL
    # max_context_len beyond the table width
    assert _call("pkv_paged_attention_decode", None, None, None, None, None, 2, None, 64, 2, 8, 2,
                 128, 16, 8, 0.1, 0, None, 0, None, None) == PKV_EINVAL
    # bad partition size
    out = ctypes.c_size_t()
    assert _call("pkv_decode_workspace_bytes", 2, 8, 128, 100, 24, ctypes.byref(out)) == PKV_EINVAL
    assert _call("pkv_decode_workspace_bytes", 2, 8, 128, 1000, 512,
                 ctypes.byref(out)) == 0 and out.value > 0


def test_empty_batches_are_no_ops():
    # T = 0 / n = 0 / S = 0 return before any device work.
    assert _call("pkv_kv_append", None, None, None, 0, None, None, 4, 8, 128, 16, None, None) == 0
    assert _call("pkv_block_copy", None, None, None, 0, 4, 8, 128, 16, None, None) == 0
    assert _call("pkv_paged_attention_decode", None, None, None, None, None, 4, None, 64, 0, 8, 2,
                 128, 16, 8, 0.1, 0, None, 0, None, None) == 0


def test_pool_beyond_int32_rows_is_rejected():
    # num_blocks * Hkv * block_size rows must fit the int32 TMA coordinates
    big = (1 << 31) // (8 * 16)
    assert _call("pkv_paged_attention_decode", None, None, None, None, None, 8, None, 64, 2, 32,
                 8, 128, 16, big, 0.1, 0, None, 0, None, None) == PKV_EINVAL
    assert "2^31" in pkv.pkv_last_error()


def test_wrappers_refuse_tensors_on_another_device():
    # The binding checks that each tensor lives on the current device before
    # it passes the pointer on (the kernels launch on the current device).
    from paged_kv_cache_281_gb300.api import _check_device, _dev
    _check_device("q", 0, 0)
    with pytest.raises(ValueError, match="cuda:1 but the current device is cuda:0"):
        _check_device("q", 1, 0)
    with pytest.raises(ValueError, match="CUDA device"):
        _dev(torch.zeros(4, dtype=torch.int32), "status", torch.int32, 1)
