"""A decode step captured in a CUDA graph and replayed.

Every launch of the library is stream-ordered (no host synchronisation, no
allocation, tensor maps passed by value), so a caller can capture a step of
the continuous-batching loop ("Deep Dive: continuous batching", section
Iteration-level scheduling: the same kernels run every iteration) once and
replay it to save the per-launch host cost. The replayed step must give the
eager step's output bit for bit, on a batch with one partition per sequence
(plan, decode) and one with several (plan, decode, combine).
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import paged_kv_cache_281_gb300 as pkv
from workloads import config1, make_decode_workload
from workloads.device import bf16_bits, decode_step, setup_decode

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
