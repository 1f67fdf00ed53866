"""The decode entry point that allocates nothing, checked against the regular one.

``pkv_paged_attention_decode_noalloc`` serves callers that cannot give the
library device scratch memory (a plugin handed only its inputs and outputs, an
engine whose KV pool already holds every free byte of HBM, a loop that must not
call cudaMalloc). Its split-K scratch is a fixed array inside the library. It
runs the same plan, partition and combine kernels with the same split as
``pkv_paged_attention_decode``, so the two must agree bit for bit; the ragged
batch is also compared with the fp64 oracle. This file runs last so that a
failure here leaves every other test already run; it also passes on its own in
a fresh process.
"""

from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_281_gb300 as pkv
from oracle.harness import bf16_tolerance_ok, build_decode_state, decode_reference
from paged_kv_cache_281_gb300._lib import PKV_EINVAL, lib
from workloads import config3, make_decode_workload
from workloads.device import bf16_bits, bf16_to_f64, run_decode, setup_decode

pytestmark = pytest.mark.gpu


def _noalloc(w, d, out, partition_size=None):
    ps = d.partition_size if partition_size is None else partition_size
    pkv.pkv_paged_attention_decode_noalloc(out, d.q, d.k_cache, d.v_cache, d.block_tables,
                                           d.context_lens, d.max_context_len, w.scale,
                                           partition_size=ps, status=d.status)
    return out


def _ragged():
    return make_decode_workload("ragged_small", (1, 17, 513, 2049, 100), Hq=16, Hkv=4, D=128,
                                block_size=16, seed=4242)


def test_noalloc_bit_equal_across_interleaved_shapes():
    # Calls that use the shared array differently follow one another: many
    # partitions over 256 sequences, then 5 sequences with a 16-token split (a
    # different item list, partition count and partial-state layout), then the
    # first batch again. Anything read from the previous call's leftovers
    # (items, ticket, partial states) would change bits.
    big, small = config3(), _ragged()
    d_big, d_small = setup_decode(big), setup_decode(small, partition_size=16)
    ref_big = bf16_bits(run_decode(big, d_big, out=torch.empty_like(d_big.out)))
    ref_small = bf16_bits(run_decode(small, d_small, out=torch.empty_like(d_small.out)))
    for call, (w, d, ref) in enumerate([(big, d_big, ref_big), (small, d_small, ref_small),
                                        (big, d_big, ref_big), (small, d_small, ref_small)]):
        out = torch.full_like(d.out, float("nan"))
        got = bf16_bits(_noalloc(w, d, out))
        pkv.pkv_check_status(d.status)
        assert np.array_equal(got, ref), (
            f"call {call} ({w.name}): {int((got != ref).sum())} elements differ from the "
            "workspace decode")


def test_noalloc_ragged_matches_oracle_twice():
    w = _ragged()
    d = setup_decode(w)
    ref = decode_reference(w, build_decode_state(w))
    for call in range(2):                         # the array keeps the last call's contents
        out = torch.full_like(d.out, float("nan"))
        got = bf16_to_f64(_noalloc(w, d, out))
        pkv.pkv_check_status(d.status)
        assert np.isfinite(got).all(), f"call {call}: non-finite output"
        ok = bf16_tolerance_ok(got, ref)
        assert ok.all(), f"call {call}: {(~ok).sum()} elements outside tolerance"


def test_noalloc_empty_batch_is_a_no_op():
    w = _ragged()
    d = setup_decode(w)
    e = lambda t: t[:0]
    empty_out = torch.empty(0, w.Hq, w.D, dtype=torch.bfloat16, device="cuda")
    pkv.pkv_paged_attention_decode_noalloc(empty_out, e(d.q), d.k_cache, d.v_cache,
                                           e(d.block_tables), e(d.context_lens),
                                           d.max_context_len, w.scale, status=d.status)
    pkv.pkv_check_status(d.status)
    # a real call right after still matches the workspace decode bit for bit
    ref = bf16_bits(run_decode(w, d, out=torch.empty_like(d.out)))
    got = bf16_bits(_noalloc(w, d, torch.full_like(d.out, float("nan"))))
    pkv.pkv_check_status(d.status)
    assert np.array_equal(got, ref)


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
