"""kv_append and block_copy on the GPU against the oracle: bit-exact.

"Batching, Scheduling, and Paging": section PagedAttention (each new token's
K/V goes to the slot its block table assigned) and section Block sharing
(copy-on-write duplicates a whole block). Pools start NaN-poisoned, so every
byte the kernels must leave alone is checked too.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import paged_kv_cache_281_gb300 as pkv
from oracle import cache
from workloads.device import bf16_bits, poisoned_pools, to_dev_bf16
from oracle.harness import empty_pools
from workloads import generator, normal_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("Hkv,D,B", [(8, 128, 16), (1, 64, 8), (32, 128, 32), (2, 64, 16)])
def test_kv_append_bit_exact(Hkv, D, B):
    N = 37
    g = generator(900, Hkv, D, B)
    T = 3 * B + 5
    slots = g.permutation(N * B)[:T].astype(np.int32)
    slots[::7] = -1                        # padding tokens are skipped
    k_new = normal_bf16((T, Hkv, D), 901, Hkv)
    v_new = normal_bf16((T, Hkv, D), 902, Hkv)
    kc, vc = empty_pools(N, Hkv, B, D)
    cache.append(kc, vc, k_new, v_new, slots, B)
    dk, dv = poisoned_pools(N, Hkv, B, D)
    st = pkv.new_status()
    pkv.pkv_kv_append(to_dev_bf16(k_new), to_dev_bf16(v_new), torch.from_numpy(slots).cuda(),
                      dk, dv, status=st)
    pkv.pkv_check_status(st)
    assert np.array_equal(bf16_bits(dk), kc)
    assert np.array_equal(bf16_bits(dv), vc)


def test_kv_append_large_batch_bit_exact():
    # a prefill-sized append: thousands of tokens, grid-stride loop wraps
    N, Hkv, D, B = 2048, 8, 128, 16
    T = 20000
    slots = generator(903).permutation(N * B)[:T].astype(np.int32)
    k_new = normal_bf16((T, Hkv, D), 904)
    v_new = normal_bf16((T, Hkv, D), 905)
    kc, vc = empty_pools(N, Hkv, B, D)
    cache.append(kc, vc, k_new, v_new, slots, B)
    dk, dv = poisoned_pools(N, Hkv, B, D)
    pkv.pkv_kv_append(to_dev_bf16(k_new), to_dev_bf16(v_new), torch.from_numpy(slots).cuda(),
                      dk, dv)
    assert np.array_equal(bf16_bits(dk), kc)
    assert np.array_equal(bf16_bits(dv), vc)


def test_kv_append_out_of_range_slot_is_skipped_and_reported():
    N, Hkv, D, B = 4, 2, 64, 16
    slots = np.array([3, N * B + 7, 5], dtype=np.int32)
    k_new = normal_bf16((3, Hkv, D), 906)
    kc, vc = empty_pools(N, Hkv, B, D)
    cache.append(kc, vc, k_new, k_new, [3, -1, 5], B)
    dk, dv = poisoned_pools(N, Hkv, B, D)
    st = pkv.new_status()
    pkv.pkv_kv_append(to_dev_bf16(k_new), to_dev_bf16(k_new), torch.from_numpy(slots).cuda(),
                      dk, dv, status=st)
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.pkv_check_status(st)
    assert e.value.code == -5
    assert np.array_equal(bf16_bits(dk), kc)


def test_kv_append_empty_batch():
    dk, dv = poisoned_pools(4, 2, 16, 64)
    before = bf16_bits(dk)
    e = torch.empty(0, 2, 64, dtype=torch.bfloat16, device="cuda")
    pkv.pkv_kv_append(e, e, torch.empty(0, dtype=torch.int32, device="cuda"), dk, dv)
    assert np.array_equal(bf16_bits(dk), before)


@pytest.mark.parametrize("Hkv,D,B", [(8, 128, 16), (1, 64, 8), (4, 128, 32)])
def test_block_copy_bit_exact(Hkv, D, B):
    N = 64
    g = generator(910, Hkv, D, B)
    kc = normal_bf16((N, Hkv, B, D), 911, Hkv)
    vc = normal_bf16((N, Hkv, B, D), 912, Hkv)
    perm = g.permutation(N)
    pairs = np.stack([perm[:20], perm[20:40]], axis=1).astype(np.int32)  # dst never a src
    dk, dv = to_dev_bf16(kc), to_dev_bf16(vc)
    cache.block_copy(kc, vc, pairs)
    st = pkv.new_status()
    pkv.pkv_block_copy(dk, dv, torch.from_numpy(pairs).cuda(), status=st)
    pkv.pkv_check_status(st)
    assert np.array_equal(bf16_bits(dk), kc)
    assert np.array_equal(bf16_bits(dv), vc)


def test_block_copy_bad_id_is_skipped_and_reported():
    N, Hkv, D, B = 8, 2, 64, 16
    kc = normal_bf16((N, Hkv, B, D), 913)
    dk, dv = to_dev_bf16(kc), to_dev_bf16(kc)
    pairs = torch.tensor([[1, 2], [3, N + 4], [-2, 5]], dtype=torch.int32, device="cuda")
    st = pkv.new_status()
    pkv.pkv_block_copy(dk, dv, pairs, status=st)
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.pkv_check_status(st)
    assert e.value.code == -5
    want = kc.copy()
    cache.block_copy(want, want.copy(), [(1, 2)])
    assert np.array_equal(bf16_bits(dk), want)
