"""pkv_iteration_prepare against the oracle's allocator model (CPU only).

One call per iteration reserves every work's slots and writes the slot
mapping, cu_q_lens, context lengths, block tables and copy-on-write
pairs into one host buffer ("Batching, Scheduling, and Paging", section
Continuous batching: the per-iteration CPU work is the overhead to keep
small). Each work must get exactly what the per-sequence rules give it
(section PagedAttention: a block only when the last one fills; section Block
sharing: copy-on-write of a shared, partially filled last block), applied in
the order of the list; the oracle's model applies the same appends one by
one. A batch that does not fit changes nothing and reports how many leading
works would fit.
"""

from __future__ import annotations

import copy

import numpy as np
import pytest

import paged_kv_cache_281_gb300 as pkv
from oracle import paging
from paged_kv_cache_281_gb300._lib import PKV_EINVAL, PKV_ENOMEM, PagedKVError


def _section(buf, layout, name, count, shape=None):
    off = getattr(layout, name)
    a = buf[off:off + 4 * count].view(np.int32)
    return a.reshape(shape) if shape else a


def _tables_equal(got, want, lens, B):
    """Row i holds the first ceil(lens[i] / B) entries of the oracle's table;
    the entries after them are left unwritten (nothing reads them)."""
    assert got.shape == want.shape
    return all(np.array_equal(g[:-(-int(n) // B)], w[:-(-int(n) // B)])
               for g, w, n in zip(got, want, lens))


def _oracle_batch(ora, ids, counts, n_prefill):
    """The same works through the oracle model, one append at a time; the
    tables are as wide as the batch's longest one."""
    slots, pairs = [], []
    for sid, c in zip(ids, counts):
        s, p = ora.append_slots(sid, int(c))
        slots.extend(s)
        pairs.extend(p)
    W = max([1] + [len(ora.block_table(sid)) for sid in ids])
    tables = np.zeros((len(ids), W), np.int32)
    for i, sid in enumerate(ids):
        t = ora.block_table(sid)
        tables[i, :len(t)] = t
    lens = np.array([ora.seq_len(sid) for sid in ids], np.int32)
    cu = np.concatenate([[0], np.cumsum(counts[:n_prefill])]).astype(np.int32)
    return np.array(slots, np.int32), pairs, tables, lens, cu


def _scenario(seed):
    rng = np.random.default_rng(0x281 + 300 + seed)
    N, B, W = 160, 16, 40
    order = rng.permutation(N).astype(np.int32)
    lib = pkv.BlockAllocator(N, B, order)
    ora = paging.BlockAllocator(N, B, order.tolist())
    lib_ids, ora_ids = [], []
    # prompts, some forked so that partially filled last blocks are shared
    for _ in range(12):
        a, b = lib.seq_create(), ora.create()
        n = int(rng.integers(1, 60))
        lib.seq_append_slots(a, n)
        ora.append_slots(b, n)
        lib_ids.append(a), ora_ids.append(b)
        for _ in range(int(rng.integers(0, 3))):
            lib_ids.append(lib.seq_fork(a)), ora_ids.append(ora.fork(b))
    buf = np.zeros(1 << 20, np.uint8)
    enomem = 0
    for step in range(40):
        # retire sequences about to outgrow the table width, and a random one
        # now and then, so the pool keeps moving
        # (the library's batched calls, the oracle's one by one)
        gone = []
        for k in reversed(range(len(lib_ids))):
            if (ora.seq_len(ora_ids[k]) > (W - 8) * B
                    or (rng.random() < 0.05 and len(lib_ids) > 4)):
                gone.append(lib_ids.pop(k))
                ora.free_seq(ora_ids.pop(k))
        lib.seq_free_many(gone)
        if len(lib_ids) < 6:
            k = 6 - len(lib_ids)
            lib_ids.extend(int(x) for x in lib.seq_create_many(k))
            ora_ids.extend(ora.create() for _ in range(k))
        live = rng.permutation(len(lib_ids))[:int(rng.integers(1, len(lib_ids) + 1))]
        n_prefill = int(rng.integers(0, len(live) + 1))
        counts = np.array([int(rng.integers(1, 120)) if i < n_prefill else 1
                           for i in range(len(live))], np.int32)
        lids = [lib_ids[i] for i in live]
        oids = [ora_ids[i] for i in live]
        snap = copy.deepcopy(ora)
        try:
            want = _oracle_batch(ora, oids, counts, n_prefill)
            fits = True
        except paging.OutOfBlocks:
            ora = snap
            fits = False
        if not fits:
            # the oracle's one-by-one appends give the index of the first miss
            probe = copy.deepcopy(ora)
            first_miss = 0
            for sid, c in zip(oids, counts):
                try:
                    probe.append_slots(sid, int(c))
                except paging.OutOfBlocks:
                    break
                first_miss += 1
            free_before = lib.num_free_blocks()
            with pytest.raises(PagedKVError) as e:
                lib.iteration_prepare(lids, counts, n_prefill, W, buf)
            assert e.value.code == PKV_ENOMEM and e.value.n_fit == first_miss
            assert lib.num_free_blocks() == free_before == ora.num_free()
            enomem += 1
        else:
            L = lib.iteration_prepare(lids, counts, n_prefill, W, buf)
            slots, pairs, tables, lens, cu = want
            assert L.n_tokens == len(slots) and L.n_cow == len(pairs)
            Wt = tables.shape[1]
            assert L.table_width == Wt <= W
            assert np.array_equal(_section(buf, L, "slot_mapping", len(slots)), slots)
            assert np.array_equal(_section(buf, L, "cu_q_lens", n_prefill + 1), cu)
            np_ = n_prefill
            assert np.array_equal(_section(buf, L, "prefill_lens", np_), lens[:np_])
            assert _tables_equal(_section(buf, L, "prefill_tables", np_ * Wt, (np_, Wt)),
                                 tables[:np_], lens[:np_], B)
            nd = len(lids) - np_
            assert np.array_equal(_section(buf, L, "decode_lens", nd), lens[np_:])
            assert _tables_equal(_section(buf, L, "decode_tables", nd * Wt, (nd, Wt)),
                                 tables[np_:], lens[np_:], B)
            got_pairs = _section(buf, L, "cow_pairs", 2 * len(pairs), (len(pairs), 2))
            assert [tuple(p) for p in got_pairs.tolist()] == [tuple(p) for p in pairs]
            assert L.max_q_len == (int(counts[:np_].max()) if np_ else 0)
            assert L.max_prefill_len == (int(lens[:np_].max()) if np_ else 0)
            assert L.max_decode_len == (int(lens[np_:].max()) if nd else 0)
            assert lib.num_free_blocks() == ora.num_free()
    ora.check_invariants()
    return enomem


def test_iteration_prepare_matches_oracle_model():
    # every batch equals the oracle model's one-by-one appends; some do not fit
    assert sum(_scenario(seed) for seed in range(6)) >= 3


def test_out_of_blocks_counts_the_copies_earlier_works_release():
    # three sharers of a half-full block: the first two copy it, the third
    # (by then its only user) writes in place, as one-by-one appends would
    lib, ora = pkv.BlockAllocator(10, 16), paging.BlockAllocator(10, 16)
    a, b = lib.seq_create(), ora.create()
    lib.seq_append_slots(a, 24), ora.append_slots(b, 24)
    la, oa = [a, lib.seq_fork(a), lib.seq_fork(a)], [b, ora.fork(b), ora.fork(b)]
    n3, o3 = lib.seq_create(), ora.create()
    buf = np.zeros(1 << 14, np.uint8)
    # 7 blocks for the prompt, then one copy each for the first two sharers:
    # 9 needed, 8 free; the first two works fit
    with pytest.raises(PagedKVError) as e:
        lib.iteration_prepare([n3] + la, [112, 1, 1, 1], 1, 8, buf)
    assert e.value.code == PKV_ENOMEM and e.value.n_fit == 2
    assert lib.num_free_blocks() == 8 and lib.block_refcount(lib.seq_block_table(a)[1]) == 3
    # a shorter prompt fits: 6 + 2 copies = 8
    L = lib.iteration_prepare([n3] + la, [96, 1, 1, 1], 1, 8, buf)
    slots, pairs, tables, lens, cu = _oracle_batch(ora, [o3] + oa, np.array([96, 1, 1, 1]), 1)
    assert L.n_cow == 2 and len(pairs) == 2 and L.table_width == 6
    assert np.array_equal(_section(buf, L, "slot_mapping", 99), slots)
    got = _section(buf, L, "cow_pairs", 4, (2, 2)).tolist()
    assert [tuple(p) for p in got] == [tuple(p) for p in pairs]
    assert _tables_equal(_section(buf, L, "decode_tables", 18, (3, 6)), tables[1:], lens[1:], 16)
    assert lib.num_free_blocks() == ora.num_free() == 0


def test_iteration_prepare_rejects_bad_batches_unchanged():
    a = pkv.BlockAllocator(64, 16)
    s0, s1 = a.seq_create(), a.seq_create()
    a.seq_append_slots(s0, 20)
    buf = np.zeros(1 << 16, np.uint8)
    free = a.num_free_blocks()
    bad = [
        ([s0, s0], [1, 1], 0),            # a sequence twice
        ([s0, 99], [1, 1], 0),            # unknown sequence
        ([s0, s1], [0, 1], 1),            # empty prompt chunk
        ([s0, s1], [3, 2], 1),            # a decode of two tokens
        ([s1], [16 * 8 + 1], 1),          # longer than max_blocks_per_seq (8)
    ]
    for ids, counts, n_prefill in bad:
        with pytest.raises(PagedKVError) as e:
            a.iteration_prepare(ids, counts, n_prefill, 8, buf)
        assert e.value.code == PKV_EINVAL
        assert a.num_free_blocks() == free and a.seq_len(s0) == 20 and a.seq_len(s1) == 0
    with pytest.raises(PagedKVError) as e:            # buffer too small
        a.iteration_prepare([s0], [1], 0, 8, np.zeros(64, np.uint8))
    assert e.value.code == PKV_EINVAL and a.seq_len(s0) == 20
    L = a.iteration_prepare([], [], 0, 8, buf)            # an empty iteration is fine
    assert L.n_tokens == 0 and L.total_bytes > 0


def test_layout_sections_are_aligned_and_sized():
    L = pkv.iteration_layout_bytes(3, 5, 77, 10)
    assert L.table_width == 10
    offs = [L.slot_mapping, L.cu_q_lens, L.prefill_lens, L.prefill_tables, L.decode_lens,
            L.decode_tables, L.cow_pairs]
    assert all(o % 64 == 0 for o in offs) and offs == sorted(offs)
    assert L.cu_q_lens >= 4 * 77 and L.prefill_tables >= L.prefill_lens + 4 * 3
    assert L.decode_lens >= L.prefill_tables + 4 * 3 * 10
    assert L.total_bytes >= L.cow_pairs + 8 * 8


def test_iteration_run_checks_before_any_launch():
    # an iteration without tokens or copies launches nothing; bad sizes and a
    # missing layout are refused before any CUDA call
    import ctypes
    from paged_kv_cache_281_gb300._lib import IterationLayout, lib
    empty = IterationLayout()
    args = lambda meta, lay, npre, ndec: (meta, lay, npre, ndec, None, None, None, None, None,
                                          None, 64, 8, 2, 128, 16, ctypes.c_float(0.1), 0, None,
                                          0, None, 0, None, None)
    assert lib().pkv_iteration_run(*args(None, ctypes.byref(empty), 0, 0)) == 0
    assert lib().pkv_iteration_run(*args(None, None, 0, 0)) == PKV_EINVAL
    assert lib().pkv_iteration_run(*args(None, ctypes.byref(empty), -1, 0)) == PKV_EINVAL
    one = IterationLayout()
    one.n_tokens = 1
    assert lib().pkv_iteration_run(*args(None, ctypes.byref(one), 0, 1)) == PKV_EINVAL  # meta NULL
    junk = ctypes.create_string_buffer(64)
    assert lib().pkv_iteration_run(*args(junk, ctypes.byref(one), 0, 1)) == PKV_EINVAL  # width 0


def test_batched_create_and_free():
    lib = pkv.BlockAllocator(32, 16)
    ids = [int(x) for x in lib.seq_create_many(3)]
    assert ids == [0, 1, 2]
    for sid in ids:
        lib.seq_append_slots(sid, 20)          # two blocks each
    assert lib.num_free_blocks() == 26
    # a repeated or unknown id: an error, and nothing freed
    with pytest.raises(pkv.PagedKVError):
        lib.seq_free_many([ids[0], ids[0]])
    with pytest.raises(pkv.PagedKVError):
        lib.seq_free_many([ids[1], 99])
    assert lib.num_free_blocks() == 26
    lib.seq_free_many(ids[:2])
    assert lib.num_free_blocks() == 30
    lib.seq_free_many([])
    assert lib.seq_create_many(0).shape == (0,)
    assert int(lib.seq_create_many(1)[0]) == 3  # ids are never reused


def test_table_rows_past_the_last_block_are_left_as_they_were():
    # each row holds the sequence's blocks; the rest of the row keeps whatever
    # the buffer held (no kernel reads it), so the prepare writes no more than
    # the blocks themselves
    lib = pkv.BlockAllocator(64, 16)
    ids = [int(x) for x in lib.seq_create_many(3)]
    buf = np.full(1 << 16, 0x5A, np.uint8)
    L = lib.iteration_prepare(ids, [40, 100, 1], 2, 16, buf)
    sentinel = np.frombuffer(bytes([0x5A] * 4), np.int32)[0]
    W = int(L.table_width)
    assert W == 7                                   # ceil(100 / 16) is the longest
    for name, first, count in (("prefill_tables", 0, 2), ("decode_tables", 2, 1)):
        off = getattr(L, name)
        rows = buf[off:off + 4 * count * W].view(np.int32).reshape(count, W)
        for r, sid in enumerate(ids[first:first + count]):
            table = lib.seq_block_table(sid)
            assert list(rows[r, :len(table)]) == table
            assert np.all(rows[r, len(table):] == sentinel)
