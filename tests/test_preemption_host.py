"""Preemption on the host: the library's allocator against the oracle's model.

"Batching, Scheduling, and Paging" (section PagedAttention): when HBM runs
out, a request is swapped to CPU memory or discarded and recomputed. The same
scheduler drives both allocators through a trace on an undersized pool; every
decision (swap lists, slots, completions) must be identical.
"""

from __future__ import annotations

import pytest

import paged_kv_cache_281_gb300 as pkv
from oracle import paging
from oracle.harness import OracleAllocator
from workloads.schedule import LibraryAllocator, run_schedule, small_trace_config


@pytest.mark.parametrize("mode", ["swap", "recompute"])
def test_preempting_schedule_matches_oracle_model(mode):
    cfg = small_trace_config(iterations=80)
    num_blocks = 120
    lib_events, lib_sched = run_schedule(cfg, num_blocks, mode, LibraryAllocator)
    ref_events, ref_sched = run_schedule(cfg, num_blocks, mode, OracleAllocator)
    assert [(e.ops, e.work, e.finished) for e in lib_events] == \
           [(e.ops, e.work, e.finished) for e in ref_events]
    assert sum(e.preempted for e in lib_events) > 5          # the pool really is short
    assert lib_sched.alloc.num_free() == ref_sched.alloc.num_free()
    ref_sched.alloc.a.check_invariants()


def test_swap_out_and_in_semantics():
    a = pkv.BlockAllocator(8, 4, list(range(8)))
    s, t = a.seq_create(), a.seq_create()
    a.seq_append_slots(s, 9)                      # blocks 0, 1, 2
    u = a.seq_fork(s)
    a.seq_append_slots(t, 4)                      # block 3
    assert a.seq_swap_out(s) == [0, 1, 2]         # still referenced by the fork
    assert a.num_free_blocks() == 4
    assert a.seq_len(s) == 9 and a.seq_block_table(s) == []
    with pytest.raises(pkv.PagedKVError):
        a.seq_append_slots(s, 1)                  # swapped out: no appends
    with pytest.raises(pkv.PagedKVError):
        a.build_block_tables([s], 4)
    a.seq_free(u)                                 # the last users of 0, 1, 2 leave
    assert a.num_free_blocks() == 7
    assert a.seq_swap_in(s) == [4, 5, 6]          # fresh blocks, first in first out
    a.seq_append_slots(s, 1)
    assert a.seq_block_table(s) == [4, 5, 6]
    a.seq_swap_out(t)
    with pytest.raises(pkv.PagedKVError) as e:
        big = a.seq_create()
        a.seq_append_slots(big, 32)               # needs 8 blocks, 5 free
    assert e.value.code == -2


def test_swap_in_is_all_or_nothing():
    a = pkv.BlockAllocator(4, 4, list(range(4)))
    ref = paging.BlockAllocator(4, 4, list(range(4)))
    s = a.seq_create(); rs = ref.create()
    a.seq_append_slots(s, 12); ref.append_slots(rs, 12)
    assert a.seq_swap_out(s) == ref.swap_out(rs) == [0, 1, 2]
    t = a.seq_create(); rt = ref.create()
    a.seq_append_slots(t, 8); ref.append_slots(rt, 8)   # takes 3, 0
    before = a.num_free_blocks()
    with pytest.raises(pkv.PagedKVError) as e:
        a.seq_swap_in(s)
    assert e.value.code == -2 and a.num_free_blocks() == before
    with pytest.raises(paging.OutOfBlocks):
        ref.swap_in(rs)
    a.seq_free(t); ref.free_seq(rt)
    assert a.seq_swap_in(s) == ref.swap_in(rs)
