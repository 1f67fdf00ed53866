"""The decode entry point that allocates nothing, checked against the regular one.

``pkv_paged_attention_decode_noalloc`` serves callers that cannot give the
library device scratch memory (a plugin handed only its inputs and outputs, an
engine whose KV pool already holds every free byte of HBM, a loop that must not
call cudaMalloc). Its split-K scratch is a fixed array inside the library. This
file runs last so that a failure here leaves every other test already run; it
also passes on its own in a fresh process.
"""

from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_281_gb300 as pkv
from paged_kv_cache_281_gb300._lib import PKV_EINVAL, lib
from workloads.device import bf16_to_f64, run_decode, setup_decode
from oracle.harness import bf16_tolerance_ok
from workloads import config3, make_decode_workload

pytestmark = pytest.mark.gpu


def _noalloc(w, d, out):
    pkv.pkv_paged_attention_decode_noalloc(out, d.q, d.k_cache, d.v_cache, d.block_tables,
                                           d.context_lens, d.max_context_len, w.scale,
                                           partition_size=d.partition_size, status=d.status)
    return out


@pytest.mark.parametrize("which", ["llama3_8b_gqa", "ragged_small"])
def test_noalloc_matches_workspace_decode_twice(which):
    if which == "llama3_8b_gqa":
        w = config3()
    else:
        w = make_decode_workload("ragged_small", (1, 17, 513, 2049, 100), Hq=16, Hkv=4, D=128,
                                 block_size=16, seed=4242)
    d = setup_decode(w)
    ref = bf16_to_f64(run_decode(w, d, out=torch.empty_like(d.out)))
    for call in range(2):                         # the array keeps the last call's contents
        out = torch.full_like(d.out, float("nan"))
        got = bf16_to_f64(_noalloc(w, d, out))
        pkv.pkv_check_status(d.status)
        assert np.isfinite(got).all(), f"call {call}: non-finite output"
        ok = bf16_tolerance_ok(got, ref)
        assert ok.all(), f"call {call}: {(~ok).sum()} elements outside tolerance"


def test_noalloc_rejects_batches_beyond_its_scratch():
    # 4096 sequences of up to 8192 tokens need far more partial-state scratch
    # than the built-in array holds; the call must refuse before touching the GPU.
    need = pkv.pkv_decode_workspace_bytes(4096, 64, 128, 8192, 16)
    assert need > pkv.NOALLOC_SCRATCH_BYTES
    rc = lib().pkv_paged_attention_decode_noalloc(
        None, None, None, None, None, 512, None, 8192, 4096, 64, 8, 128, 16, 100000,
        ctypes.c_float(0.1), 16, None, None)
    assert rc == PKV_EINVAL
    assert "scratch" in pkv.pkv_last_error()
