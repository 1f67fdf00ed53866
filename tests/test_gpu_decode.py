"""paged_attention_decode on the GPU against the fp64 oracle.

Definition ("Deep Dive: continuous batching", section Selective batching):
softmax(Q K^T / sqrt(d_k)) V per request over its own tokens, here gathered
through each request's block table ("Batching, Scheduling, and Paging",
section PagedAttention). Tolerance for bf16 inputs with fp32 accumulation:
|gpu - ref| <= 2e-3 + 1e-2 |ref| elementwise. Pools are NaN-poisoned outside
the cached tokens, so any read past a sequence end or into a free block shows
up as a non-finite output.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import paged_kv_cache_281_gb300 as pkv
from workloads.device import bf16_bits, bf16_to_f64, decode_step, run_decode, setup_decode
from oracle.harness import bf16_tolerance_ok, build_decode_state, decode_reference
from workloads import config1, config2, config3, make_decode_workload

pytestmark = pytest.mark.gpu


def assert_close(gpu, ref, what=""):
    assert np.isfinite(gpu).all(), f"{what}: non-finite output"
    ok = bf16_tolerance_ok(gpu, ref)
    if not ok.all():
        idx = np.argwhere(~ok)[:5]
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} outside tolerance, "
                             f"first {idx.tolist()}: gpu {gpu[tuple(idx[0])]} ref "
                             f"{ref[tuple(idx[0])]}")


def check_against_oracle(w, partition_size=0, seqs=None):
    d = setup_decode(w, partition_size=partition_size, append_last=False)
    out = bf16_to_f64(decode_step(w, d))
    pkv.pkv_check_status(d.status)
    st = build_decode_state(w)
    # the library's allocator placed the blocks exactly like the oracle's model
    assert [list(r[:len(t)]) for r, t in zip(d.tables, st.tables)] == st.tables
    # the pools after the append are byte-identical to the oracle's pools
    assert np.array_equal(bf16_bits(d.k_cache), st.k_cache)
    assert np.array_equal(bf16_bits(d.v_cache), st.v_cache)
    ref = decode_reference(w, st, seqs=seqs)
    sel = list(range(w.S)) if seqs is None else list(seqs)
    assert_close(out[sel], ref[sel], w.name)
    return out, d


def test_config1_tiny():
    check_against_oracle(config1())


RAGGED = (1, 2, 15, 16, 17, 31, 33, 64, 65, 129, 300, 515, 700)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("B", [8, 16, 32])
def test_shapes_ragged(D, G, B):
    w = make_decode_workload(f"ragged_D{D}_G{G}_B{B}", RAGGED, Hq=2 * G, Hkv=2, D=D,
                             block_size=B, seed=1000 + D + 10 * G + B)
    check_against_oracle(w, partition_size=128)


@pytest.mark.parametrize("partition", [16, 48, 256, 2048, 0])
def test_partition_sizes_agree(partition):
    w = make_decode_workload("parts", (1, 16, 17, 511, 512, 513, 1500, 2049), Hq=32, Hkv=8,
                             D=128, block_size=16, seed=1100)
    check_against_oracle(w, partition_size=partition)


def test_more_sequences_than_plan_threads():
    # 1,100 sequences: the plan lists full partitions and tails over two
    # chunks of its 1,024 threads
    lens = np.random.default_rng(1150).integers(1, 601, size=1100)
    w = make_decode_workload("many_seqs", tuple(int(x) for x in lens), Hq=4, Hkv=2, D=64,
                             block_size=16, seed=1151)
    check_against_oracle(w, partition_size=256)


def test_split_independence_within_tolerance():
    w = make_decode_workload("split", (900, 2000, 37), Hq=32, Hkv=8, D=128, block_size=16,
                             seed=1101)
    d = setup_decode(w, partition_size=16)
    a = bf16_to_f64(run_decode(w, d, out=torch.empty_like(d.out), partition_size=16))
    b = bf16_to_f64(run_decode(w, d, out=torch.empty_like(d.out), partition_size=1024))
    assert_close(a, b, "partition 16 vs 1024")


def test_single_key_returns_v_exactly():
    w = make_decode_workload("one", (1, 1, 1, 1), Hq=8, Hkv=2, D=128, block_size=16, seed=1102)
    d = setup_decode(w)
    out = bf16_bits(run_decode(w, d))
    G = w.Hq // w.Hkv
    for s in range(w.S):
        for h in range(w.Hq):
            assert np.array_equal(out[s, h], w.v[s, h // G])


def test_placement_does_not_change_a_bit():
    w1 = make_decode_workload("place", (5, 77, 300, 1025), Hq=16, Hkv=4, D=128, block_size=16,
                              seed=1103)
    w2 = make_decode_workload("place", (5, 77, 300, 1025), Hq=16, Hkv=4, D=128, block_size=16,
                              seed=1103)
    w2.free_order = w2.free_order[::-1].copy()
    d1, d2 = setup_decode(w1, partition_size=64), setup_decode(w2, partition_size=64)
    assert not np.array_equal(d1.tables, d2.tables)
    assert np.array_equal(bf16_bits(run_decode(w1, d1)), bf16_bits(run_decode(w2, d2)))


def test_deterministic_across_runs():
    w = make_decode_workload("det", (2000, 3, 700), Hq=32, Hkv=8, D=128, block_size=16,
                             seed=1104)
    d = setup_decode(w, partition_size=128)
    a = bf16_bits(run_decode(w, d, out=torch.empty_like(d.out)))
    b = bf16_bits(run_decode(w, d, out=torch.empty_like(d.out)))
    assert np.array_equal(a, b)


def test_config2_llama2_7b_full():
    # every one of the 64 sequences, in the launch configuration the
    # benchmark times (default partition size)
    check_against_oracle(config2())


def test_config3_llama3_8b_full():
    # all 256 sequences of the full-size launch (the oracle takes seconds)
    out, _ = check_against_oracle(config3())
    assert np.isfinite(out).all()


def test_bad_table_entry_is_skipped_and_reported():
    w = make_decode_workload("bad", (40, 40), Hq=8, Hkv=2, D=128, block_size=16, seed=1105)
    d = setup_decode(w)
    bt = d.block_tables.clone()
    bt[1, 1] = w.num_blocks + 3
    pkv.pkv_paged_attention_decode(d.out, d.q, d.k_cache, d.v_cache, bt, d.context_lens,
                                   d.max_context_len, w.scale, d.workspace, status=d.status)
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.pkv_check_status(d.status)
    assert e.value.code == -5
    # sequence 0 is untouched by the bad entry of sequence 1
    st = build_decode_state(w)
    ref = decode_reference(w, st, seqs=[0])
    assert_close(bf16_to_f64(d.out)[0], ref[0], "good sequence")


def test_forced_timeout_reports_and_recovers():
    w = make_decode_workload("timeout", (300, 20), Hq=8, Hkv=2, D=128, block_size=16, seed=1106)
    d = setup_decode(w, partition_size=64)
    try:
        pkv.pkv_debug_set_wait(True)
        run_decode(w, d)
        with pytest.raises(pkv.PagedKVError) as e:
            pkv.pkv_check_status(d.status)
        assert e.value.code == -4
    finally:
        pkv.pkv_debug_set_wait(False)
    pkv.pkv_status_reset(d.status)
    out = bf16_to_f64(run_decode(w, d))
    pkv.pkv_check_status(d.status)
    assert_close(out, decode_reference(w, build_decode_state(w)), "after recovery")


def test_rejects_small_workspace():
    w = make_decode_workload("ws", (600,), Hq=8, Hkv=2, D=128, block_size=16, seed=1107)
    d = setup_decode(w)
    with pytest.raises(pkv.PagedKVError):
        pkv.pkv_paged_attention_decode(d.out, d.q, d.k_cache, d.v_cache, d.block_tables,
                                       d.context_lens, d.max_context_len, w.scale,
                                       d.workspace[:256], partition_size=16)


@pytest.mark.parametrize("B", [8, 16, 32])
def test_maximum_context_length(B):
    # the longest context the workloads produce (the 8192-token clip), next to
    # a one-token sequence and one just past a partition boundary, with the
    # largest GQA group
    w = make_decode_workload(f"max_len_B{B}", (8192, 1, 4097), Hq=16, Hkv=2, D=128,
                             block_size=B, seed=1300 + B)
    check_against_oracle(w)
