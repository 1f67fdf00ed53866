"""Preemption end to end on the GPU: swap-out/in and recompute against the oracle.

"Batching, Scheduling, and Paging" (section PagedAttention): when HBM runs
out a request is evicted — swapped to CPU memory or discarded and recomputed.
A continuous-batching trace runs on a pool far smaller than its worst case;
the library's allocator and pkv_swap_blocks (over pinned host memory) carry
the evictions, and every iteration's attention is compared with the oracle
replaying the same decisions (every 5th iteration in full, the others on a
seeded sample). Swapping must also restore the cache bit for bit.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import paged_kv_cache_281_gb300 as pkv
from workloads.device import bf16_bits, bf16_to_f64
from oracle.harness import OracleAllocator, OracleRunner
from workloads.device import GpuRunner
from workloads.schedule import LibraryAllocator, TokenValues, run_schedule, small_trace_config
from tests.test_gpu_decode import assert_close
from workloads import generator

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", ["swap", "recompute"])
def test_undersized_pool_trace(mode):
    cfg = small_trace_config(iterations=60)
    num_blocks = 120
    gpu_events, _ = run_schedule(cfg, num_blocks, mode, LibraryAllocator)
    ref_events, _ = run_schedule(cfg, num_blocks, mode, OracleAllocator)
    assert [(e.ops, e.work) for e in gpu_events] == [(e.ops, e.work) for e in ref_events]
    assert sum(e.preempted for e in gpu_events) > 5
    values = TokenValues(cfg)
    gpu, ora = GpuRunner(cfg, num_blocks), OracleRunner(cfg, num_blocks)
    rng = generator(cfg.seed, 99)
    checked = 0
    for ev in gpu_events:
        pre, dec, pre_out, dec_out = gpu.run(ev, values)
        _, _, q, meta = ora.run(ev, values)
        full = ev.index % 5 == 0
        pick_pre = range(len(pre)) if full else ([int(rng.integers(len(pre)))] if pre else [])
        pick_dec = range(len(dec)) if full else ([int(rng.integers(len(dec)))] if dec else [])
        if pre:
            got = bf16_to_f64(pre_out)
            for i in pick_pre:
                a, b = int(meta["cu"][i]), int(meta["cu"][i + 1])
                assert_close(got[a:b], ora.prefill(ev, pre, q, meta, i),
                             f"{mode} iteration {ev.index} prefill {i}")
                checked += 1
        if dec:
            got = bf16_to_f64(dec_out)
            for i in pick_dec:
                assert_close(got[i], ora.decode(ev, q, meta, i),
                             f"{mode} iteration {ev.index} decode {i}")
                checked += 1
    pkv.pkv_check_status(gpu.status)
    assert checked > 100
    if mode == "swap":
        assert gpu.swap_bytes > 0
    # both pools start from the same poison and see the same writes and swaps
    assert np.array_equal(bf16_bits(gpu.k_cache), ora.k_cache)
    assert np.array_equal(bf16_bits(gpu.v_cache), ora.v_cache)


def test_swap_round_trip_bit_exact_through_pinned_host():
    from workloads.device import poisoned_pools
    from workloads import normal_bf16
    N, Hkv, B, D = 64, 8, 16, 128
    kc, vc = poisoned_pools(N, Hkv, B, D)
    kc.view(torch.int16).copy_(torch.from_numpy(normal_bf16((N, Hkv, B, D), 71).view(np.int16)))
    vc.view(torch.int16).copy_(torch.from_numpy(normal_bf16((N, Hkv, B, D), 72).view(np.int16)))
    before_k, before_v = bf16_bits(kc), bf16_bits(vc)
    src = [5, 17, 3, 40]
    dst = [60, 2, 33, 9]
    kb = torch.empty((4, Hkv, B, D), dtype=torch.bfloat16).pin_memory()
    vb = torch.empty_like(kb).pin_memory()
    st = pkv.new_status()
    pkv.pkv_swap_blocks(kc, vc, torch.tensor(src, dtype=torch.int32, device="cuda"), kb, vb, True,
                        status=st)
    torch.cuda.synchronize()
    assert np.array_equal(kb.view(torch.int16).numpy().view(np.uint16), before_k[src])
    pkv.pkv_swap_blocks(kc, vc, torch.tensor(dst, dtype=torch.int32, device="cuda"), kb, vb,
                        False, status=st)
    pkv.pkv_check_status(st)
    after_k, after_v = bf16_bits(kc), bf16_bits(vc)
    assert np.array_equal(after_k[dst], before_k[src])
    assert np.array_equal(after_v[dst], before_v[src])
    keep = [b for b in range(N) if b not in dst]
    assert np.array_equal(after_k[keep], before_k[keep])


def test_swap_refuses_pageable_host_memory():
    from workloads.device import poisoned_pools
    kc, vc = poisoned_pools(8, 2, 16, 64)
    kb = torch.empty((1, 2, 16, 64), dtype=torch.bfloat16)      # pageable
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.pkv_swap_blocks(kc, vc, torch.tensor([1], dtype=torch.int32, device="cuda"), kb,
                            kb.clone(), True)
    assert e.value.code == -1
