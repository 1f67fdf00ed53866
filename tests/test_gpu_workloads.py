"""The shared-prefix and continuous-batching workloads end to end on the GPU.

Shared prefix ("Batching, Scheduling, and Paging", section Block sharing):
64 prompts x 4 samples share their prompt's prefix blocks through refcounts;
with a 1032-token prefix the half-full last shared block is copied on the
first divergent append. The library's allocator must make the same choices as
the oracle's model, the pools must match byte for byte, decode must match the
oracle, and a shared prefix must decode bit-identically to duplicated copies.

Trace ("Deep Dive: continuous batching", sections Iteration-level scheduling
and The prefill/decode mix): 200 iterations that admit, chunk-prefill, decode
and retire requests, each iteration running kv_append, chunked paged prefill
and paged decode over all active sequences (one iteration in three through
the separate calls, one through pkv_iteration_run, one through
pkv_iteration_step). Checking every iteration in full
would take the oracle about eight minutes of one host core (about 2.3 s per
iteration), so every 10th iteration is checked in full and a seeded 1/8 of
the prefill requests and of the decode sequences of every other iteration.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

from workloads.device import (DeviceTrace, bf16_bits, bf16_to_f64, decode_shared_prefix,
                               run_decode, setup_decode, setup_shared_prefix, to_dev_bf16)
from oracle.harness import OracleTrace, build_shared_prefix_state
from tests.test_gpu_decode import assert_close
from oracle import attention
from workloads import TraceConfig, config4, generator, make_decode_workload, trace_iterations

import paged_kv_cache_281_gb300 as pkv

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("variant", ["a", "b"])
def test_shared_prefix(variant):
    w = config4(variant)
    d = setup_shared_prefix(w)
    out = bf16_to_f64(decode_shared_prefix(w, d))
    pkv.pkv_check_status(d.status)
    st = build_shared_prefix_state(w)
    # same allocator decisions: slots, copy pairs, tables
    assert [list(s) for s in d.prefix_slots] == st.prefix_slots
    assert [list(s) for s in d.tail_slots] == st.tail_slots
    assert d.cow_pairs == st.cow_pairs
    assert (len(d.cow_pairs) > 0) == (variant == "b")
    assert [list(r[:len(t)]) for r, t in zip(d.tables, st.tables)] == st.tables
    # byte-identical pools after prefix append, copy-on-write and tail append
    assert np.array_equal(bf16_bits(d.k_cache), st.k_cache)
    assert np.array_equal(bf16_bits(d.v_cache), st.v_cache)
    # prefix blocks really are shared (refcount = samples) and not duplicated
    first = d.tables[0][0]
    assert d.alloc.block_refcount(int(first)) == w.n_samples
    ref = attention.decode(w.q, st.k_cache, st.v_cache, st.tables, w.context_lens, w.block_size,
                           w.scale)
    assert_close(out, ref, w.name)


def test_shared_prefix_equals_duplicated_copies_bit_exact():
    w = config4("b", n_prompts=8)
    d = setup_shared_prefix(w)
    shared = bf16_bits(decode_shared_prefix(w, d, partition_size=128))
    dup = make_decode_workload("dup", w.context_lens, w.Hq, w.Hkv, w.D, w.block_size, seed=1)
    ks, vs = [], []
    cu = w.cu_tails
    for i in range(w.S):
        p = i // w.n_samples
        ks.append(np.concatenate([w.prefix_k[p], w.tail_k[cu[i]:cu[i + 1]]]))
        vs.append(np.concatenate([w.prefix_v[p], w.tail_v[cu[i]:cu[i + 1]]]))
    dup.k, dup.v, dup.q = np.concatenate(ks), np.concatenate(vs), w.q
    dd = setup_decode(dup, partition_size=128)
    assert np.array_equal(shared, bf16_bits(run_decode(dup, dd)))


def seeded_eighth(rng, n):
    """A seeded ceil(n / 8) of range(n), sorted."""
    return sorted(rng.choice(n, -(-n // 8), replace=False).tolist()) if n else []


def test_continuous_batching_trace():
    cfg = TraceConfig()
    gpu, ora = DeviceTrace(cfg), OracleTrace(cfg)
    rng = generator(cfg.seed, 77)
    checked_pre = checked_dec = 0
    for itr in trace_iterations(cfg):
        slots = ora.step(itr)
        if itr.index % 3 == 2:
            # every third iteration through pkv_iteration_step (allocator work,
            # metadata copy and launches in one call)
            pre_out, dec_out, meta = gpu.step(itr, to_dev_bf16(itr.q), to_dev_bf16(itr.k),
                                              to_dev_bf16(itr.v))
        else:
            meta = gpu.host_metadata(itr)
            # the others alternate between the separate calls and pkv_iteration_run
            pre_out, dec_out = gpu.run_iteration(itr, meta, fused=itr.index % 3 == 1)
        got_slots = gpu.host_section(meta, "slot_mapping", itr.num_tokens)
        assert np.array_equal(got_slots, slots), f"iteration {itr.index}: slots differ"
        full = itr.index % 10 == 0
        n_pre, n_dec = len(itr.prefill), len(itr.decode)
        pick_pre = range(n_pre) if full else seeded_eighth(rng, n_pre)
        pick_dec = range(n_dec) if full else seeded_eighth(rng, n_dec)
        if pick_pre:
            got = bf16_to_f64(pre_out)
            row0 = np.concatenate([[0], np.cumsum([wk.n for wk in itr.prefill])])
            for i, ref in ora.prefill(itr, pick_pre).items():
                assert_close(got[row0[i]:row0[i + 1]], ref, f"iteration {itr.index} prefill {i}")
                checked_pre += 1
        if pick_dec:
            got = bf16_to_f64(dec_out)
            for i, ref in ora.decode(itr, pick_dec).items():
                assert_close(got[i], ref, f"iteration {itr.index} decode {i}")
                checked_dec += 1
        if pre_out is not None:
            assert torch.isfinite(pre_out.float()).all()
        if dec_out is not None:
            assert torch.isfinite(dec_out.float()).all()
        gpu.finish(itr)
        ora.finish(itr)
    pkv.pkv_check_status(gpu.status)
    assert gpu.alloc.num_free_blocks() == ora.alloc.num_free()
    assert checked_pre > 100 and checked_dec > 9000
