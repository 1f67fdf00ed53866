"""Shared-prefix decode on the GPU against the oracle.

"Batching, Scheduling, and Paging" (section Block sharing): parallel samples
of a prompt point at the same physical blocks for the prompt. The group path
reads a group's shared blocks once for up to 16 / (Hq/Hkv) samples; the
result must be the attention definition for every sample (the oracle, which
knows nothing of groups), within |gpu - ref| <= 2e-3 + 1e-2 |ref|, and agree
with the ordinary decode of the same batch.
"""

from __future__ import annotations

import numpy as np
import pytest

import paged_kv_cache_281_gb300 as pkv
from oracle import attention
from workloads.device import (bf16_to_f64, decode_shared_grouped, decode_shared_prefix,
                               setup_shared_prefix, shared_groups)
from oracle.harness import build_shared_prefix_state
from tests.test_gpu_decode import assert_close
from workloads import config4, make_shared_prefix_workload

pytestmark = pytest.mark.gpu


def reference(w):
    st = build_shared_prefix_state(w)
    return attention.decode(w.q, st.k_cache, st.v_cache, st.tables, w.context_lens, w.block_size,
                            w.scale)


@pytest.mark.parametrize("variant", ["a", "b"])
def test_config4_grouped(variant):
    w = config4(variant)
    d = setup_shared_prefix(w)
    groups = shared_groups(w, d)
    assert np.all(groups[2] == 1024)          # 64 whole shared blocks in both variants
    out = bf16_to_f64(decode_shared_grouped(w, d, groups))
    pkv.pkv_check_status(d.status)
    assert_close(out, reference(w), w.name)
    plain = bf16_to_f64(decode_shared_prefix(w, d))
    assert_close(out, plain, "grouped vs ordinary decode")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("B", [8, 16, 32])
def test_shapes(D, G, B):
    # 5 samples: several member chunks when 16 / G < 5; prefix not a multiple
    # of 16; tails from 0
    w = make_shared_prefix_workload(f"grouped_D{D}_G{G}_B{B}", n_prompts=3, n_samples=5,
                                    prefix=150, tail_max=70, Hq=2 * G, Hkv=2, D=D, block_size=B,
                                    seed=7000 + D + 10 * G + B)
    d = setup_shared_prefix(w)
    out = bf16_to_f64(decode_shared_grouped(w, d))
    pkv.pkv_check_status(d.status)
    assert_close(out, reference(w), w.name)


@pytest.mark.parametrize("partition_size", [16, 64, 1024])
def test_partitions_and_groups_of_all_sizes(partition_size):
    w = make_shared_prefix_workload("grouped_sizes", n_prompts=4, n_samples=17, prefix=300,
                                    tail_max=200, Hq=8, Hkv=8, D=128, block_size=16, seed=7100)
    d = setup_shared_prefix(w)
    out = bf16_to_f64(decode_shared_grouped(w, d, partition_size=partition_size))
    pkv.pkv_check_status(d.status)
    assert_close(out, reference(w), f"partition {partition_size}")


def test_edge_groups():
    w = make_shared_prefix_workload("grouped_edges", n_prompts=4, n_samples=4, prefix=96,
                                    tail_max=40, Hq=16, Hkv=4, D=128, block_size=16, seed=7200)
    d = setup_shared_prefix(w)
    ref = reference(w)
    start, members, sh = shared_groups(w, d)
    # group 1 shares nothing, group 2 is a single sample (of prompt 2, whose
    # other samples are in no group), prompt 3 is in no group
    sh = sh.copy()
    sh[1] = 0
    start = np.array([0, 4, 8, 9], dtype=np.int32)
    members = members[:9]
    sh = sh[:3]
    out = bf16_to_f64(decode_shared_grouped(w, d, (start, members, sh)))
    pkv.pkv_check_status(d.status)
    assert_close(out, ref, "edge groups")


def test_members_without_private_tokens():
    # every sample's context is exactly the shared prefix: the group items
    # write the final output themselves
    w = make_shared_prefix_workload("grouped_no_tails", n_prompts=2, n_samples=4, prefix=512,
                                    tail_max=0, Hq=32, Hkv=8, D=128, block_size=16, seed=7300)
    d = setup_shared_prefix(w)
    # the claimed shared length exceeds every member's context: cut to it
    out = bf16_to_f64(decode_shared_grouped(w, d, shared_groups(w, d, shared=10_000)))
    pkv.pkv_check_status(d.status)
    assert_close(out, reference(w), "no tails")


def test_bad_group_entry_is_reported_then_recovers():
    w = make_shared_prefix_workload("grouped_bad", n_prompts=2, n_samples=4, prefix=200,
                                    tail_max=30, Hq=16, Hkv=4, D=128, block_size=16, seed=7400)
    d = setup_shared_prefix(w)
    start, members, sh = shared_groups(w, d)
    bad = members.copy()
    bad[2] = w.S + 3
    decode_shared_grouped(w, d, (start, bad, sh))
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.pkv_check_status(d.status)
    assert e.value.code == -5
    pkv.pkv_status_reset(d.status)
    try:
        pkv.pkv_debug_set_wait(True)
        decode_shared_grouped(w, d)
        with pytest.raises(pkv.PagedKVError) as e:
            pkv.pkv_check_status(d.status)
        assert e.value.code == -4
    finally:
        pkv.pkv_debug_set_wait(False)
    pkv.pkv_status_reset(d.status)
    out = bf16_to_f64(decode_shared_grouped(w, d))
    pkv.pkv_check_status(d.status)
    assert_close(out, reference(w), "after recovery")


def test_long_shared_prefix_many_partitions():
    # 4 x 2000-token prefixes shared by 6 samples each, tails up to 3000 tokens
    # (contexts up to 5000): several shared and private partitions per member
    w = make_shared_prefix_workload("grouped_long", n_prompts=4, n_samples=6, prefix=2000,
                                    tail_max=3000, Hq=32, Hkv=8, D=128, block_size=16,
                                    seed=7500)
    d = setup_shared_prefix(w)
    out = bf16_to_f64(decode_shared_grouped(w, d, partition_size=512))
    pkv.pkv_check_status(d.status)
    assert_close(out, reference(w), "long shared prefixes")


def test_forced_timeout_reports_and_recovers():
    # every wait gives up at once: each team of warps leaves its item after
    # its loads in flight have landed, the status says PKV_ETIMEOUT, and the
    # next call (waits restored) is correct
    w = make_shared_prefix_workload("grouped_timeout", n_prompts=3, n_samples=5, prefix=300,
                                    tail_max=200, Hq=8, Hkv=2, D=128, block_size=16, seed=7190)
    d = setup_shared_prefix(w)
    try:
        pkv.pkv_debug_set_wait(True)
        decode_shared_grouped(w, d)
        with pytest.raises(pkv.PagedKVError) as e:
            pkv.pkv_check_status(d.status)
        assert e.value.code == -4
    finally:
        pkv.pkv_debug_set_wait(False)
    pkv.pkv_status_reset(d.status)
    out = bf16_to_f64(decode_shared_grouped(w, d))
    pkv.pkv_check_status(d.status)
    assert_close(out, reference(w), "after recovery")
