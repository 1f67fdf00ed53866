"""Decode and prefill steps captured in a CUDA graph and replayed.

Every launch of the library is stream-ordered (no host synchronisation, no
allocation, tensor maps passed by value), so a caller can capture a step of
the continuous-batching loop ("Deep Dive: continuous batching", section
Iteration-level scheduling: the same kernels run every iteration) once and
replay it to save the per-launch host cost. The replayed step must give the
eager step's output bit for bit: a decode step on a batch with one partition
per sequence (plan, decode) and one with several (plan, decode, combine), and
a prefill launch of each kind (one CTA per item; plan and persistent grid).
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import paged_kv_cache_281_gb300 as pkv
from workloads import config1, make_decode_workload, normal_bf16
from workloads.device import (bf16_bits, bf16_to_f64, decode_step, poisoned_pools,
                              setup_decode, to_dev_bf16)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", ["tiny", "ragged"])
def test_decode_step_replays_from_a_cuda_graph(case):
    if case == "tiny":
        w = config1()
    else:
        w = make_decode_workload("graph_ragged", (100, 3000, 17, 1025, 2048), Hq=32, Hkv=8,
                                 D=128, block_size=16, seed=3301)
    d = setup_decode(w, append_last=False)
    decode_step(w, d)
    torch.cuda.synchronize()
    pkv.pkv_check_status(d.status)
    want = bf16_bits(d.out).copy()

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        decode_step(w, d)  # warm-up on the capturing stream's side
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        decode_step(w, d)
    d.out.fill_(float("nan"))
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    pkv.pkv_check_status(d.status)
    assert np.array_equal(bf16_bits(d.out), want)


@pytest.mark.parametrize("case", ["one CTA per item", "persistent grid"])
def test_prefill_replays_from_a_cuda_graph(case):
    # a small launch runs one CTA per work item; a large one a plan kernel and
    # a persistent grid chained by programmatic dependent launch
    if case == "one CTA per item":
        lens, chunks = (300, 129, 40), [300, 33, 40]
    else:
        lens, chunks = (1024,) * 16, [1024] * 16
    w = make_decode_workload("graph_prefill", lens, Hq=32, Hkv=8, D=128, block_size=16,
                             seed=3302)
    d = setup_decode(w)
    cu = torch.from_numpy(np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)).cuda()
    T = int(sum(chunks))
    q = to_dev_bf16(normal_bf16((T, w.Hq, w.D), 3303))
    out = torch.full_like(q, float("nan"))
    ws = torch.empty(pkv.pkv_prefill_workspace_bytes(w.S, T, w.Hq, w.D), dtype=torch.uint8,
                     device="cuda")

    def prefill():
        pkv.pkv_paged_attention_prefill(out, q, cu, d.context_lens, d.k_cache, d.v_cache,
                                        d.block_tables, max(chunks), w.max_context_len, w.scale,
                                        ws, status=d.status)

    prefill()
    torch.cuda.synchronize()
    pkv.pkv_check_status(d.status)
    want = bf16_bits(out).copy()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        prefill()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        prefill()
    out.fill_(float("nan"))
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    pkv.pkv_check_status(d.status)
    assert np.array_equal(bf16_bits(out), want)


def test_iteration_run_replays_from_a_cuda_graph():
    # prompt chunks and decodes in one pkv_iteration_run: the prefill runs on
    # the library's second stream, forked from the captured stream after the
    # append and joined back into it, so the capture holds both branches
    N, B, Hq, Hkv, D, W = 200, 16, 16, 4, 128, 24
    lib = pkv.BlockAllocator(N, B)
    kc, vc = poisoned_pools(N, Hkv, B, D)
    seqs = [lib.seq_create() for _ in range(6)]
    buf = torch.empty(1 << 20, dtype=torch.uint8).pin_memory()
    status = pkv.new_status()
    scale = 1.0 / np.sqrt(D)

    def iteration(works, n_prefill, seed):
        counts = [c for _, c in works]
        T = sum(counts)
        q = to_dev_bf16(normal_bf16((T, Hq, D), seed))
        k = to_dev_bf16(normal_bf16((T, Hkv, D), seed + 1))
        v = to_dev_bf16(normal_bf16((T, Hkv, D), seed + 2))
        L = lib.iteration_prepare([seqs[i] for i, _ in works], counts, n_prefill, W, buf)
        meta = buf[:L.total_bytes].cuda()
        out = torch.full((T, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        dws = torch.empty(pkv.pkv_decode_workspace_bytes(len(works), Hq, D, W * B),
                          dtype=torch.uint8, device="cuda")
        pws = torch.empty(pkv.pkv_prefill_workspace_bytes(max(1, n_prefill), T, Hq, D),
                          dtype=torch.uint8, device="cuda")

        def run():
            pkv.pkv_iteration_run(meta, L, n_prefill, len(works) - n_prefill, q, k, v, out, kc,
                                  vc, scale, dws, pws, status=status)
        return run, out

    run0, _ = iteration(list(enumerate((40, 77, 130, 16, 300, 9))), 6, 9400)
    run0()
    # two prompt chunks beside four decodes (appending the same tokens to the
    # same slots again leaves the pools as they were)
    run1, out = iteration([(0, 21), (4, 50), (1, 1), (2, 1), (3, 1), (5, 1)], 2, 9500)
    run1()
    torch.cuda.synchronize()
    pkv.pkv_check_status(status)
    want = bf16_bits(out).copy()
    assert np.isfinite(bf16_to_f64(out)).all()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run1()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run1()
    out.fill_(float("nan"))
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    pkv.pkv_check_status(status)
    assert np.array_equal(bf16_bits(out), want)
