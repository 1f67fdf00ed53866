"""One iteration through the two per-iteration calls, against the oracle.

``pkv_iteration_prepare`` reserves every work's slots and writes the
iteration's metadata into one host buffer; one copy takes it to the device;
``pkv_iteration_run`` launches the copy-on-write copies, the appends, the
prefill of the prompt chunks and the decode of the running sequences from
it ("Deep Dive: continuous batching", sections Iteration-level scheduling and
The prefill/decode mix; "Batching, Scheduling, and Paging", sections
PagedAttention and Block sharing). Prompts are forked into samples so that
half-full shared blocks are copied on their first divergent write. The
oracle applies the same appends one by one with its own allocator model,
copies, writes and attends; pools must match bit for bit, attention within
|gpu - ref| <= 2e-3 + 1e-2 |ref|.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import paged_kv_cache_281_gb300 as pkv
from oracle import attention, cache, paging
from oracle.harness import empty_pools
from tests.test_gpu_decode import assert_close
from workloads import normal_bf16
from workloads.device import bf16_bits, bf16_to_f64, poisoned_pools, to_dev_bf16

pytestmark = pytest.mark.gpu

N, B, Hq, Hkv, D, W = 200, 16, 16, 4, 128, 24


class Sides:
    def __init__(self):
        self.lib = pkv.BlockAllocator(N, B)
        self.ora = paging.BlockAllocator(N, B)
        self.kc, self.vc = poisoned_pools(N, Hkv, B, D)
        self.ok, self.ov = empty_pools(N, Hkv, B, D)
        self.status = pkv.new_status()
        self.ids = []            # (library id, oracle id) per sequence
        self.buf = torch.empty(1 << 20, dtype=torch.uint8).pin_memory()
        self.scale = 1.0 / np.sqrt(D)

    def new(self):
        self.ids.append((self.lib.seq_create(), self.ora.create()))
        return len(self.ids) - 1

    def fork(self, i):
        a, b = self.ids[i]
        self.ids.append((self.lib.seq_fork(a), self.ora.fork(b)))
        return len(self.ids) - 1

    def iteration(self, works, seed):
        """``works``: [(sequence index, token count)], prompt chunks first
        (count > 1 or a first token), then decodes (count 1)."""
        n_prefill = sum(1 for _, c, kind in works if kind == "prefill")
        counts = [c for _, c, _ in works]
        T = sum(counts)
        q = normal_bf16((T, Hq, D), seed)
        k = normal_bf16((T, Hkv, D), seed + 1)
        v = normal_bf16((T, Hkv, D), seed + 2)
        # library: one prepare, one copy, one run
        L = self.lib.iteration_prepare([self.ids[i][0] for i, _, _ in works], counts, n_prefill,
                                       W, self.buf)
        meta = self.buf[:L.total_bytes].cuda()
        out = torch.full((T, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        dws = torch.empty(pkv.pkv_decode_workspace_bytes(max(1, len(works)), Hq, D, W * B),
                          dtype=torch.uint8, device="cuda")
        pws = torch.empty(pkv.pkv_prefill_workspace_bytes(max(1, n_prefill), T, Hq, D),
                          dtype=torch.uint8, device="cuda")
        pkv.pkv_iteration_run(meta, L, n_prefill, len(works) - n_prefill, to_dev_bf16(q),
                              to_dev_bf16(k), to_dev_bf16(v), out, self.kc, self.vc, self.scale,
                              dws, pws, status=self.status)
        pkv.pkv_check_status(self.status)
        # oracle: the same appends one by one, copies first, then the writes
        slots, pairs = [], []
        for i, c, _ in works:
            s, p = self.ora.append_slots(self.ids[i][1], c)
            slots.extend(s)
            pairs.extend(p)
        assert L.n_cow == len(pairs)
        got_slots = self.buf[L.slot_mapping:L.slot_mapping + 4 * T].numpy().view(np.int32)
        assert np.array_equal(got_slots, slots)
        cache.block_copy(self.ok, self.ov, pairs)
        cache.append(self.ok, self.ov, k, v, slots, B)
        assert np.array_equal(bf16_bits(self.kc), self.ok)
        assert np.array_equal(bf16_bits(self.vc), self.ov)
        got = bf16_to_f64(out)
        row = 0
        for i, c, kind in works:
            sid = self.ids[i][1]
            table, length = [self.ora.block_table(sid)], [self.ora.seq_len(sid)]
            if kind == "prefill":
                ref = attention.prefill(q[row:row + c], [0, c], length, self.ok, self.ov, table,
                                        B, self.scale)
            else:
                ref = attention.decode(q[row:row + 1], self.ok, self.ov, table, length, B,
                                       self.scale)
            assert_close(got[row:row + c], ref, f"sequence {i} ({kind})")
            row += c
        return L


def test_iteration_with_forks_and_copy_on_write():
    sd = Sides()
    prompts = [sd.new() for _ in range(4)]
    # iteration 0: four prompts prefilled (lengths 40, 77, 130, 16)
    sd.iteration([(p, c, "prefill") for p, c in zip(prompts, (40, 77, 130, 16))], 9100)
    # two more samples per prompt share its blocks, half-full last ones included
    samples = [s for p in prompts for s in (p, sd.fork(p), sd.fork(p))]
    # iteration 1: every sample decodes one token; the first two sharers of a
    # half-full block copy it, the last writes in place
    L = sd.iteration([(s, 1, "decode") for s in samples], 9200)
    assert L.n_cow == 6
    # iteration 2: prompt chunks for some samples, decodes for the others
    works = [(samples[0], 21, "prefill"), (samples[4], 5, "prefill"), (samples[10], 33, "prefill")]
    works += [(s, 1, "decode") for s in samples if s not in (samples[0], samples[4], samples[10])]
    sd.iteration(works, 9300)
    assert sd.lib.num_free_blocks() == sd.ora.num_free()


def test_iteration_run_equals_separate_calls_bit_for_bit():
    # pkv_iteration_run runs the prefill on a second stream beside the decode;
    # the outputs and the pools must be exactly those of the same calls made
    # one after another on one stream from the same metadata
    lib = pkv.BlockAllocator(N, B)
    kc, vc = poisoned_pools(N, Hkv, B, D)
    seqs = [lib.seq_create() for _ in range(6)]
    buf = torch.empty(1 << 20, dtype=torch.uint8).pin_memory()
    status = pkv.new_status()
    scale = 1.0 / np.sqrt(D)

    def batch(works, n_prefill, seed):
        counts = [c for _, c in works]
        T = sum(counts)
        q = to_dev_bf16(normal_bf16((T, Hq, D), seed))
        k = to_dev_bf16(normal_bf16((T, Hkv, D), seed + 1))
        v = to_dev_bf16(normal_bf16((T, Hkv, D), seed + 2))
        L = lib.iteration_prepare([seqs[i] for i, _ in works], counts, n_prefill, W, buf)
        return L, buf[:L.total_bytes].cuda(), q, k, v, T

    def workspaces(n, n_prefill, T):
        return (torch.empty(pkv.pkv_decode_workspace_bytes(n, Hq, D, W * B), dtype=torch.uint8,
                            device="cuda"),
                torch.empty(pkv.pkv_prefill_workspace_bytes(max(1, n_prefill), T, Hq, D),
                            dtype=torch.uint8, device="cuda"))

    L0, meta0, q0, k0, v0, T0 = batch(list(enumerate((40, 77, 130, 16, 300, 9))), 6, 9600)
    dws, pws = workspaces(6, 6, T0)
    out0 = torch.empty(T0, Hq, D, dtype=torch.bfloat16, device="cuda")
    pkv.pkv_iteration_run(meta0, L0, 6, 0, q0, k0, v0, out0, kc, vc, scale, dws, pws,
                          status=status)
    # a mixed iteration: two prompt chunks, four decodes
    works, n_pre = [(0, 21), (4, 50), (1, 1), (2, 1), (3, 1), (5, 1)], 2
    L1, meta1, q1, k1, v1, T1 = batch(works, n_pre, 9700)
    kc2, vc2 = kc.clone(), vc.clone()
    dws, pws = workspaces(len(works), n_pre, T1)
    out_run = torch.full((T1, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    pkv.pkv_iteration_run(meta1, L1, n_pre, len(works) - n_pre, q1, k1, v1, out_run, kc, vc,
                          scale, dws, pws, status=status)
    # the same work through the separate calls, serially, on the copies
    sec = lambda name, count: meta1[getattr(L1, name):getattr(L1, name) + 4 * count].view(
        torch.int32)
    Wt, n_dec, rows = int(L1.table_width), len(works) - n_pre, 21 + 50
    out_sep = torch.full_like(out_run, float("nan"))
    pkv.pkv_kv_append(k1, v1, sec("slot_mapping", T1), kc2, vc2, status=status)
    pkv.pkv_paged_attention_prefill(out_sep[:rows], q1[:rows], sec("cu_q_lens", n_pre + 1),
                                    sec("prefill_lens", n_pre), kc2, vc2,
                                    sec("prefill_tables", n_pre * Wt).view(n_pre, Wt),
                                    int(L1.max_q_len), int(L1.max_prefill_len), scale, pws,
                                    status=status)
    pkv.pkv_paged_attention_decode(out_sep[rows:], q1[rows:], kc2, vc2,
                                   sec("decode_tables", n_dec * Wt).view(n_dec, Wt),
                                   sec("decode_lens", n_dec), int(L1.max_decode_len), scale, dws,
                                   status=status)
    torch.cuda.synchronize()
    pkv.pkv_check_status(status)
    assert L1.n_cow == 0
    assert np.array_equal(bf16_bits(out_run), bf16_bits(out_sep))
    assert np.isfinite(bf16_to_f64(out_run)).all()
    assert np.array_equal(bf16_bits(kc), bf16_bits(kc2))
    assert np.array_equal(bf16_bits(vc), bf16_bits(vc2))


def test_step_function_and_bound_stepper_agree():
    # pkv_iteration_step through the plain wrapper and through an
    # IterationStepper (its fixed arguments checked once) on twin allocators
    # and pools: the same slots, outputs and pools, bit for bit
    sides = []
    for _ in range(2):
        lib = pkv.BlockAllocator(N, B)
        kc, vc = poisoned_pools(N, Hkv, B, D)
        sides.append((lib, kc, vc, [int(x) for x in lib.seq_create_many(6)],
                      torch.empty(1 << 20, dtype=torch.uint8).pin_memory(),
                      torch.empty(1 << 20, dtype=torch.uint8, device="cuda")))
    status = pkv.new_status()
    scale = 1.0 / np.sqrt(D)
    dws = torch.empty(pkv.pkv_decode_workspace_bytes(6, Hq, D, W * B), dtype=torch.uint8,
                      device="cuda")
    pws = torch.empty(pkv.pkv_prefill_workspace_bytes(6, 1024, Hq, D), dtype=torch.uint8,
                      device="cuda")
    lib1, kc1, vc1, ids1, hb1, db1 = sides[1]
    stepper = pkv.IterationStepper(lib1, W, db1, kc1, vc1, scale, dws, pws, status=status)
    outs = [[], []]
    batches = [(list(enumerate((40, 77, 130, 16, 300, 9))), 6),
               ([(0, 21), (4, 50), (1, 1), (2, 1), (3, 1), (5, 1)], 2)]
    for it, (works, n_pre) in enumerate(batches):
        counts = np.array([c for _, c in works], np.int32)
        T = int(counts.sum())
        q = to_dev_bf16(normal_bf16((T, Hq, D), 9800 + 10 * it))
        k = to_dev_bf16(normal_bf16((T, Hkv, D), 9801 + 10 * it))
        v = to_dev_bf16(normal_bf16((T, Hkv, D), 9802 + 10 * it))
        for side, (lib, kc, vc, ids, hb, db) in enumerate(sides):
            out = torch.full((T, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
            seqs = [ids[i] for i, _ in works]
            if side == 0:
                L = pkv.pkv_iteration_step(lib, seqs, counts, n_pre, W, hb, db, q, k, v, out, kc,
                                           vc, scale, dws, pws, status=status)
            else:
                L = stepper(seqs, counts, n_pre, hb, q, k, v, out)
            torch.cuda.synchronize()
            outs[side].append((bf16_bits(out).copy(),
                               hb[L.slot_mapping:L.slot_mapping + 4 * T].numpy().view(np.int32)
                               .copy()))
    pkv.pkv_check_status(status)
    for (o0, s0), (o1, s1) in zip(*outs):
        assert np.array_equal(s0, s1)
        assert np.array_equal(o0, o1)
    assert np.array_equal(bf16_bits(sides[0][1]), bf16_bits(sides[1][1]))
    assert np.array_equal(bf16_bits(sides[0][2]), bf16_bits(sides[1][2]))
