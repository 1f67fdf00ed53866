"""FP8 (e4m3) pages on the GPU against the oracle.

kv_append_fp8 must produce the oracle's codes and scales bit for bit (the
quantiser's decisions are integer results of fp32 arithmetic that both sides
perform in the same precision). Decode over the pages is compared with the
oracle's attention over the dequantised pages, element by element, within
|gpu - ref| <= 2e-3 + 1e-2 |ref|.
"""

from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import paged_kv_cache_281_gb300 as pkv
from oracle import fp8 as ofp8
from workloads.device import bf16_to_f64, to_dev_bf16
from tests.test_gpu_decode import assert_close
from workloads import generator, make_decode_workload, normal_bf16

pytestmark = pytest.mark.gpu


def codes_np(t):
    return t.cpu().numpy()


def build_fp8(w, poison=True):
    """Device and oracle FP8 pools holding every token of the workload, placed
    by the workload's block permutation."""
    N, Hkv, B, D = w.num_blocks, w.Hkv, w.block_size, w.D
    k8, v8, ks, vs = pkv.new_fp8_pools(N, Hkv, B, D)
    if poison:  # codes 0x7F are NaN: any read of a slot past the end shows up
        k8.fill_(0x7F), v8.fill_(0x7F), ks.fill_(float("nan")), vs.fill_(float("nan"))
    ok8, ov8 = codes_np(k8).copy(), codes_np(v8).copy()
    oks, ovs = ks.cpu().numpy().copy(), vs.cpu().numpy().copy()
    alloc = pkv.BlockAllocator(N, B, w.free_order)
    seqs, slots = [], []
    for L in w.context_lens:
        sid = alloc.seq_create()
        sl, _ = alloc.seq_append_slots(sid, int(L))
        seqs.append(sid)
        slots.append(sl)
    maxB = max(1, max(math.ceil(int(L) / B) for L in w.context_lens))
    tables, lens = alloc.build_block_tables(seqs, maxB)
    slot_all = np.concatenate(slots).astype(np.int32)
    st = pkv.new_status()
    pkv.pkv_kv_append_fp8(to_dev_bf16(w.k), to_dev_bf16(w.v), torch.from_numpy(slot_all).cuda(),
                          k8, v8, ks, vs, status=st)
    pkv.pkv_check_status(st)
    ofp8.append(ok8, ov8, oks, ovs, w.k, w.v, slot_all, B)
    return (k8, v8, ks, vs), (ok8, ov8, oks, ovs), tables, lens, st


def run_decode_fp8(w, dev_pools, tables, lens, partition_size=0, status=None):
    k8, v8, ks, vs = dev_pools
    out = torch.full((w.S, w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(pkv.pkv_decode_workspace_bytes(w.S, w.Hq, w.D, w.max_context_len,
                                                    partition_size),
                     dtype=torch.uint8, device="cuda")
    pkv.pkv_paged_attention_decode_fp8(out, to_dev_bf16(w.q), k8, v8, ks, vs,
                                       torch.from_numpy(tables).cuda(),
                                       torch.from_numpy(lens).cuda(), w.max_context_len, w.scale,
                                       ws, partition_size=partition_size, status=status)
    return out


def check(w, partition_size=0):
    dev, ora, tables, lens, st = build_fp8(w)
    assert np.array_equal(codes_np(dev[0]), ora[0]), "key codes differ"
    assert np.array_equal(codes_np(dev[1]), ora[1]), "value codes differ"
    assert np.array_equal(dev[2].cpu().numpy(), ora[2], equal_nan=True), "key scales differ"
    assert np.array_equal(dev[3].cpu().numpy(), ora[3], equal_nan=True), "value scales differ"
    out = run_decode_fp8(w, dev, tables, lens, partition_size, status=st)
    pkv.pkv_check_status(st)
    ref = ofp8.decode(w.q, ora[0], ora[1], ora[2], ora[3], tables, lens, w.block_size, w.scale)
    assert_close(bf16_to_f64(out), ref, w.name)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("B", [8, 16, 32])
def test_shapes(D, G, B):
    lens = (1, 2, 17, 64, 300, 1500, 33)
    w = make_decode_workload(f"fp8_D{D}_G{G}_B{B}", lens, Hq=2 * G, Hkv=2, D=D, block_size=B,
                             seed=6000 + D + 10 * G + B)
    check(w)


@pytest.mark.parametrize("partition_size", [16, 256, 1024])
def test_llama3_shape_partitions(partition_size):
    g = generator(0x281, 61)
    lens = np.clip(np.round(np.exp(np.log(1024) + 0.8 * g.standard_normal(48))), 16, 8192)
    w = make_decode_workload("fp8_llama3", lens.astype(int), Hq=32, Hkv=8, D=128, block_size=16,
                             seed=6100)
    check(w, partition_size)


def test_quantiser_edge_rows():
    # zero rows, single large values, tiny values, -0 and values that saturate
    T, Hkv, D, B = 6, 2, 128, 16
    k = normal_bf16((T, Hkv, D), 6200)
    v = normal_bf16((T, Hkv, D), 6201)
    k[0] = 0
    v[0, 1] = 0x8000                         # -0.0 everywhere in one row
    k[1, 0, :] = 0
    k[1, 0, 7] = 0x4780                      # 65536: one nonzero value
    k[2] = (k[2] & 0x807F) | 0x0800          # tiny magnitudes (~1e-34)
    v[3, :, 5] = 0x7F00                      # 1.7e38: dominates its row
    k8, v8, ks, vs = pkv.new_fp8_pools(4, Hkv, B, D)
    slots = np.array([0, 1, 17, 33, 2, -1], dtype=np.int32)
    pkv.pkv_kv_append_fp8(to_dev_bf16(k), to_dev_bf16(v), torch.from_numpy(slots).cuda(), k8, v8,
                          ks, vs)
    torch.cuda.synchronize()
    ok8, ov8 = np.zeros((4, Hkv, B, D), np.uint8), np.zeros((4, Hkv, B, D), np.uint8)
    oks, ovs = np.zeros((4, Hkv, B), np.float32), np.zeros((4, Hkv, B), np.float32)
    ofp8.append(ok8, ov8, oks, ovs, k, v, slots, B)
    assert np.array_equal(codes_np(k8), ok8)
    assert np.array_equal(codes_np(v8), ov8)
    assert np.array_equal(ks.cpu().numpy(), oks)
    assert np.array_equal(vs.cpu().numpy(), ovs)


def test_every_code_round_trips_through_the_kernel():
    # rows whose values are all 256 codes' values (NaN codes replaced) scaled
    # so that amax = 448: the kernel must reproduce each code exactly
    D, B = 128, 16
    vals = ofp8.e4m3_decode(np.arange(256, dtype=np.uint8))
    vals[np.isnan(vals)] = 0.0
    rows = vals.reshape(2, 128)
    rows[:, 0] = 448.0
    bits = (rows.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)  # exact in bf16
    k = bits.reshape(2, 1, D)
    k8, v8, ks, vs = pkv.new_fp8_pools(1, 1, B, D)
    pkv.pkv_kv_append_fp8(to_dev_bf16(k), to_dev_bf16(k), torch.tensor([0, 1], dtype=torch.int32,
                                                                       device="cuda"),
                          k8, v8, ks, vs)
    torch.cuda.synchronize()
    got = codes_np(k8)[0, 0, :2].reshape(-1)
    want = ofp8.e4m3_encode(rows.reshape(-1).astype(np.float32))
    assert np.array_equal(got, want)
    assert ks.cpu().numpy()[0, 0, 0] == 1.0


def test_bad_table_entry_and_timeout_are_reported():
    w = make_decode_workload("fp8_bad", (200, 50), Hq=8, Hkv=2, D=128, block_size=16, seed=6300)
    dev, ora, tables, lens, st = build_fp8(w)
    bad = tables.copy()
    bad[0, 3] = w.num_blocks + 5
    run_decode_fp8(w, dev, bad, lens, status=st)
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.pkv_check_status(st)
    assert e.value.code == -5
    pkv.pkv_status_reset(st)
    try:
        pkv.pkv_debug_set_wait(True)
        run_decode_fp8(w, dev, tables, lens, status=st)
        with pytest.raises(pkv.PagedKVError) as e:
            pkv.pkv_check_status(st)
        assert e.value.code == -4
    finally:
        pkv.pkv_debug_set_wait(False)
    pkv.pkv_status_reset(st)
    out = run_decode_fp8(w, dev, tables, lens, status=st)
    pkv.pkv_check_status(st)
    ref = ofp8.decode(w.q, ora[0], ora[1], ora[2], ora[3], tables, lens, w.block_size, w.scale)
    assert_close(bf16_to_f64(out), ref, "after recovery")


def test_fp8_close_to_bf16_decode():
    # the quantisation error itself: fp8 decode stays near the bf16 result
    from workloads.device import run_decode, setup_decode
    w = make_decode_workload("fp8_vs_bf16", (700, 1300, 90), Hq=32, Hkv=8, D=128, block_size=16,
                             seed=6400)
    dev, ora, tables, lens, st = build_fp8(w)
    out8 = bf16_to_f64(run_decode_fp8(w, dev, tables, lens, status=st))
    d = setup_decode(w)
    out16 = bf16_to_f64(run_decode(w, d))
    assert np.max(np.abs(out8 - out16)) < 0.05


@pytest.mark.parametrize("B", [16, 32])
def test_maximum_context_length(B):
    # the longest context the configurations use (8192 tokens), next to tiny ones
    w = make_decode_workload(f"fp8_max_B{B}", (8192, 1, 4097, 8191), Hq=64, Hkv=8, D=128,
                             block_size=B, seed=6500 + B)
    check(w)
