"""Prefix caching on the GPU: shared system-prompt blocks against the oracle
and against the same requests computed without caching.

"Paging the KV Cache" (lecture 6): a system prompt shared by many requests
can occupy one set of pages referenced by all of them. Requests in three
waves share a 200-token system prompt; with the cache, every request after
the first starts from the prompt's 12 full registered blocks (192 tokens) and
prefills only the rest, including after the blocks' earlier users have all
finished. Attention outputs must match the oracle replaying the same
decisions, and decode outputs must equal, bit for bit, those of the run that
recomputes every prompt (the same values in other blocks).
"""

from __future__ import annotations

import numpy as np
import pytest

import paged_kv_cache_281_gb300 as pkv
from workloads.device import bf16_to_f64
from tests.prefix_cache import PrefixConfig, PrefixValues, prefix_schedule
from oracle.harness import OracleAllocator, OracleRunner
from workloads.device import GpuRunner
from workloads.schedule import LibraryAllocator
from tests.test_gpu_decode import assert_close

pytestmark = pytest.mark.gpu


def test_shared_system_prompt_with_and_without_cache():
    cfg = PrefixConfig()
    lib_alloc = LibraryAllocator(cfg.num_blocks, cfg.block_size)
    ev_c, hits = prefix_schedule(cfg, lib_alloc, cached=True)
    ev_o, hits_o = prefix_schedule(cfg, OracleAllocator(cfg.num_blocks, cfg.block_size),
                                   cached=True)
    ev_u, _ = prefix_schedule(cfg, LibraryAllocator(cfg.num_blocks, cfg.block_size),
                              cached=False)
    assert [(e.work, e.tables) for e in ev_c] == [(e.work, e.tables) for e in ev_o]
    full = cfg.system_len // cfg.block_size * cfg.block_size
    assert hits == hits_o and hits[0] == 0
    assert all(h == full for r, h in hits.items() if r > 0)

    values = PrefixValues(cfg)
    gpu_c, gpu_u = GpuRunner(cfg, cfg.num_blocks), GpuRunner(cfg, cfg.num_blocks)
    ora = OracleRunner(cfg, cfg.num_blocks)
    checked = exact_prefill = 0
    for ec, eu in zip(ev_c, ev_u):
        pre_c, dec_c, pre_out_c, dec_out_c = gpu_c.run(ec, values)
        pre_u, dec_u, pre_out_u, dec_out_u = gpu_u.run(eu, values)
        _, _, q, meta = ora.run(ec, values)
        if pre_c:
            got = bf16_to_f64(pre_out_c)
            got_u = bf16_to_f64(pre_out_u)
            cu_u = np.concatenate([[0], np.cumsum([w[3] for w in pre_u])])
            for i, w in enumerate(pre_c):
                a, b = int(meta["cu"][i]), int(meta["cu"][i + 1])
                assert_close(got[a:b], ora.prefill(ec, pre_c, q, meta, i),
                             f"iteration {ec.index} request {w[0]} prefill")
                # the uncached run's chunk ends with the same positions
                j = [x[0] for x in pre_u].index(w[0])
                rows_u = got_u[cu_u[j + 1] - (b - a):cu_u[j + 1]]
                assert_close(got[a:b], rows_u, f"request {w[0]}: cached vs recomputed prompt")
                exact_prefill += int(np.array_equal(got[a:b], rows_u))
                checked += 1
        if dec_c:
            got = bf16_to_f64(dec_out_c)
            assert [w[0] for w in dec_c] == [w[0] for w in dec_u]
            assert np.array_equal(got, bf16_to_f64(dec_out_u)), \
                f"iteration {ec.index}: decode differs between cached and recomputed prompts"
            for i in range(len(dec_c)):
                assert_close(got[i], ora.decode(ec, q, meta, i),
                             f"iteration {ec.index} decode {i}")
                checked += 1
    pkv.pkv_check_status(gpu_c.status)
    pkv.pkv_check_status(gpu_u.status)
    assert checked > 50
    print(f"prefill chunks bit-identical to the recomputed run: {exact_prefill}")
    # the cached run holds the system prompt once per wave instead of once per request
    assert lib_alloc.num_cached() >= full // cfg.block_size
