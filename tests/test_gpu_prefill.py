"""paged_attention_prefill on the GPU against the fp64 oracle.

A prompt chunk attends causally over its own cached blocks ("Deep Dive:
continuous batching", sections Selective batching and The prefill/decode mix):
row i of a chunk of c tokens sits at position L - c + i and sees keys
0 .. L - c + i. Tolerance |gpu - ref| <= 2e-3 + 1e-2 |ref|.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import paged_kv_cache_281_gb300 as pkv
from oracle import attention
from workloads.device import bf16_to_f64, run_decode, setup_decode, to_dev_bf16
from oracle.harness import build_decode_state
from tests.test_gpu_decode import assert_close
from workloads import make_decode_workload, normal_bf16

pytestmark = pytest.mark.gpu


def run_prefill(w, d, chunks, q_bits, status=None):
    cu = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    q = to_dev_bf16(q_bits)
    out = torch.full_like(q, float("nan"))
    ws = torch.empty(pkv.pkv_prefill_workspace_bytes(w.S, int(cu[-1]), w.Hq, w.D),
                     dtype=torch.uint8, device="cuda")
    pkv.pkv_paged_attention_prefill(out, q, torch.from_numpy(cu).cuda(), d.context_lens,
                                    d.k_cache, d.v_cache, d.block_tables,
                                    max(chunks) if len(chunks) else 0, w.max_context_len,
                                    w.scale, ws, status=d.status if status is None else status)
    return out, cu


def check_prefill(w, chunks, seed=0):
    d = setup_decode(w)
    q_bits = normal_bf16((int(sum(chunks)), w.Hq, w.D), 5000 + seed)
    out, cu = run_prefill(w, d, chunks, q_bits)
    pkv.pkv_check_status(d.status)
    st = build_decode_state(w)
    ref = attention.prefill(q_bits, cu, w.context_lens, st.k_cache, st.v_cache, st.tables,
                            w.block_size, w.scale)
    got = bf16_to_f64(out)
    rows = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in range(w.S)]).astype(np.int64)
    assert_close(got[rows], ref[rows], w.name)
    return got, ref, d


# (context length, chunk length) pairs: single tokens, whole prompts, chunks
# after a prefix, tile and page boundaries, a ragged tail.
CASES = ((1, 1), (17, 17), (130, 33), (300, 300), (257, 129), (64, 1), (700, 212))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("B", [8, 16, 32])
def test_shapes(D, G, B):
    lens = [L for L, _ in CASES]
    chunks = [c for _, c in CASES]
    w = make_decode_workload(f"prefill_D{D}_G{G}_B{B}", lens, Hq=2 * G, Hkv=2, D=D, block_size=B,
                             seed=3000 + D + 10 * G + B)
    check_prefill(w, chunks, seed=G + B)


def test_single_key_returns_v():
    # one visible key: the output row is that key's value row (up to bf16 of V)
    w = make_decode_workload("prefill_one", (1, 1), Hq=8, Hkv=2, D=128, block_size=16, seed=3099)
    got, _, _ = check_prefill(w, [1, 1], seed=3)
    G = w.Hq // w.Hkv
    for s in range(w.S):
        for h in range(w.Hq):
            want = attention.widen_bf16(w.v[s, h // G])
            assert np.array_equal(got[s, h], want)


def test_seventy_b_shape_chunks():
    # 64 query / 8 kv heads, D=128: chunks of up to 512 after prefixes up to 512
    lens = (512, 1024, 37, 900, 530)
    chunks = [512, 512, 37, 388, 18]
    w = make_decode_workload("prefill_70b", lens, Hq=64, Hkv=8, D=128, block_size=16, seed=3100)
    check_prefill(w, chunks, seed=1)


def test_sequences_without_queries():
    w = make_decode_workload("prefill_gaps", (40, 90, 33), Hq=8, Hkv=2, D=128, block_size=16,
                             seed=3101)
    check_prefill(w, [0, 90, 0], seed=2)


def test_last_row_equals_decode():
    w = make_decode_workload("prefill_vs_decode", (77, 513, 1200), Hq=32, Hkv=8, D=128,
                             block_size=16, seed=3102)
    d = setup_decode(w)
    chunks = [20, 300, 128]
    q_bits = normal_bf16((sum(chunks), w.Hq, w.D), 5100)
    cu = np.cumsum(chunks)
    for s in range(w.S):
        q_bits[cu[s] - 1] = w.q[s]     # the chunk's last query is the decode query
    out, _ = run_prefill(w, d, chunks, q_bits)
    dec = bf16_to_f64(run_decode(w, d))
    got = bf16_to_f64(out)[cu - 1]
    assert_close(got, dec, "last prefill row vs decode")


def test_bad_table_entry_is_reported():
    w = make_decode_workload("prefill_bad", (200,), Hq=8, Hkv=2, D=128, block_size=16, seed=3103)
    d = setup_decode(w)
    d.block_tables[0, 3] = w.num_blocks + 11
    run_prefill(w, d, [200], normal_bf16((200, 8, 128), 5200))
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.pkv_check_status(d.status)
    assert e.value.code == -5


def test_forced_timeout_reports_and_recovers():
    w = make_decode_workload("prefill_timeout", (300, 140), Hq=8, Hkv=2, D=128, block_size=16,
                             seed=3104)
    d = setup_decode(w)
    q_bits = normal_bf16((440, 8, 128), 5300)
    try:
        pkv.pkv_debug_set_wait(True)
        run_prefill(w, d, [300, 140], q_bits)
        with pytest.raises(pkv.PagedKVError) as e:
            pkv.pkv_check_status(d.status)
        assert e.value.code == -4
    finally:
        pkv.pkv_debug_set_wait(False)
    pkv.pkv_status_reset(d.status)
    check_prefill(w, [300, 140], seed=9)


def test_long_prefix_chunks():
    # chunks after a long cached prefix: up to 128 key tiles per query tile
    w = make_decode_workload("prefill_long", (8192, 4096, 2000), Hq=16, Hkv=2, D=128,
                             block_size=16, seed=3200)
    check_prefill(w, [512, 1, 700], seed=11)


# Launches with at least four work items per resident CTA run on the
# persistent grid (plan + ticket); these two cover its one- and two-tile forms.
def check_prefill_sampled(w, chunks, seqs, seed):
    d = setup_decode(w)
    q_bits = normal_bf16((int(sum(chunks)), w.Hq, w.D), 5000 + seed)
    out, cu = run_prefill(w, d, chunks, q_bits)
    pkv.pkv_check_status(d.status)
    st = build_decode_state(w)
    ref = attention.prefill(q_bits, cu, w.context_lens, st.k_cache, st.v_cache, st.tables,
                            w.block_size, w.scale, seqs=seqs)
    got = bf16_to_f64(out)
    rows = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in seqs]).astype(np.int64)
    assert_close(got[rows], ref[rows], w.name)
    return d, q_bits, cu


@pytest.mark.parametrize("D,B", [(128, 16), (128, 8), (64, 32)])
def test_persistent_grid_long_chunks(D, B):
    # 16 fresh 600-token prompts, 32/8 heads: ~2,500 items of one Q tile; a
    # key tile holds 64 / B pages, one load each
    lens = [600] * 16
    w = make_decode_workload(f"prefill_persistent_1_D{D}_B{B}", lens, Hq=32, Hkv=8, D=D,
                             block_size=B, seed=3300 + D + B)
    check_prefill_sampled(w, lens, [0, 5, 15], seed=21)


def test_persistent_grid_short_chunks_after_long_prefixes():
    # 64 chunks of 40 tokens after ~2,000 cached tokens, 64/8 heads
    lens = [2000 + 7 * i for i in range(64)]
    w = make_decode_workload("prefill_persistent_2", lens, Hq=64, Hkv=8, D=128, block_size=16,
                             seed=3301)
    check_prefill_sampled(w, [40] * 64, [0, 31, 63], seed=22)


def test_persistent_grid_many_sequences():
    # 1,100 sequences (two chunks of the plan's 1,024 threads), ragged chunks
    # after ragged prefixes, enough items for the persistent grid
    rng = np.random.default_rng(3170)
    lens = rng.integers(1, 201, size=1100)
    chunks = [int(rng.integers(1, L + 1)) for L in lens]
    w = make_decode_workload("prefill_many", tuple(int(x) for x in lens), Hq=8, Hkv=2, D=64,
                             block_size=16, seed=3171)
    check_prefill(w, chunks, seed=71)


def test_persistent_grid_timeout_and_bad_entry():
    lens = [600] * 16
    w = make_decode_workload("prefill_persistent_err", lens, Hq=32, Hkv=8, D=128,
                             block_size=16, seed=3302)
    d = setup_decode(w)
    q_bits = normal_bf16((sum(lens), w.Hq, w.D), 5400)
    try:
        pkv.pkv_debug_set_wait(True)
        run_prefill(w, d, lens, q_bits)
        with pytest.raises(pkv.PagedKVError) as e:
            pkv.pkv_check_status(d.status)
        assert e.value.code == -4
    finally:
        pkv.pkv_debug_set_wait(False)
    pkv.pkv_status_reset(d.status)
    d.block_tables[3, 5] = w.num_blocks + 1
    run_prefill(w, d, lens, q_bits)
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.pkv_check_status(d.status)
    assert e.value.code == -5
