"""Pins the CPU oracle to facts that do not come from the oracle itself.

Each ``pin_*`` function checks the oracle against one of:

* brute force on tiny inputs: pure-Python loops over contiguous keys/values,
  with no paging, no max subtraction and its own bf16 decoding;
* torch's fp64 ``scaled_dot_product_attention`` on CPU (an independent
  implementation of ``softmax(Q K^T / sqrt(d_k)) V``, "Deep Dive: continuous
  batching", section *Selective batching*);
* closed forms (a single key, a zero query, equal keys, equal values, two
  keys, one dominant score);
* invariants fixed by "Batching, Scheduling, and Paging" (sections
  *PagedAttention* and *Block sharing*): physical placement does not matter,
  a shared block equals duplicated copies, copy-on-write leaves the other
  sharers alone, allocation happens only when a block fills, and counts keep
  shared blocks alive;
* a hand-derived allocator scenario stored under ``tests/golden``.

``test_planted_mistakes_are_caught`` plants plausible mistakes in the oracle
(on the CPU) and checks that at least one pin fails for each.
"""

from __future__ import annotations

import math
import os
import struct

import numpy as np
import pytest

from oracle import attention, cache, fp8, paging
from oracle.harness import build_decode_state, build_shared_prefix_state, empty_pools
from workloads import config1, config4, make_decode_workload, normal_bf16

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers

def bits_to_float(b: int) -> float:
    return struct.unpack("<f", struct.pack("<I", int(b) << 16))[0]


def brute_attention(q, keys, values, scale):
    """Plain loops: weights exp(scale q.k) normalised, no max subtraction."""
    ws = [math.exp(scale * sum(a * b for a, b in zip(q, k))) for k in keys]
    tot = sum(ws)
    return [sum(w * v[d] for w, v in zip(ws, values)) / tot for d in range(len(values[0]))]


def logical_rows(arr_bits, start, n, head):
    return [[bits_to_float(x) for x in arr_bits[start + j, head]] for j in range(n)]


def tiny_gqa_workload(seed=7, lens=(1, 5, 9, 14), Hq=4, Hkv=2, D=8, B=4):
    return make_decode_workload("tiny_gqa", lens, Hq=Hq, Hkv=Hkv, D=D, block_size=B,
                                seed=seed, num_blocks=16)


def decode_oracle(w, st):
    return attention.decode(w.q, st.k_cache, st.v_cache, st.tables, w.context_lens,
                            w.block_size, w.scale)


# ---------------------------------------------------------------- pins

def pin_widen_bf16():
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x8000, 0x3FC0, 0x7F7F, 0x0001], np.uint16)
    want = [1.0, -2.0, 0.0, -0.0, 1.5, 3.3895313892515355e38, 9.183549615799121e-41]
    got = attention.widen_bf16(bits)
    assert list(got) == want


def pin_decode_brute_force():
    w = tiny_gqa_workload()
    st = build_decode_state(w)
    out = decode_oracle(w, st)
    G = w.Hq // w.Hkv
    cu = w.cu_lens
    for s in range(w.S):
        L = int(w.context_lens[s])
        for h in range(w.Hq):
            q = [bits_to_float(x) for x in w.q[s, h]]
            ref = brute_attention(q, logical_rows(w.k, cu[s], L, h // G),
                                  logical_rows(w.v, cu[s], L, h // G), w.scale)
            assert np.max(np.abs(out[s, h] - ref)) <= 1e-12


def pin_prefill_brute_force():
    w = tiny_gqa_workload(seed=8, lens=(3, 6, 11))
    st = build_decode_state(w)
    chunks = [1, 6, 4]
    cu_q = np.concatenate([[0], np.cumsum(chunks)])
    cu = w.cu_lens
    q_bits = normal_bf16((sum(chunks), w.Hq, w.D), 77)
    out = attention.prefill(q_bits, cu_q, w.context_lens, st.k_cache, st.v_cache, st.tables,
                            w.block_size, w.scale)
    G = w.Hq // w.Hkv
    for s in range(w.S):
        L, c = int(w.context_lens[s]), chunks[s]
        for i in range(c):
            pos = L - c + i
            for h in range(w.Hq):
                q = [bits_to_float(x) for x in q_bits[cu_q[s] + i, h]]
                ref = brute_attention(q, logical_rows(w.k, cu[s], pos + 1, h // G),
                                      logical_rows(w.v, cu[s], pos + 1, h // G), w.scale)
                assert np.max(np.abs(out[cu_q[s] + i, h] - ref)) <= 1e-12


def _torch_reference(q, K, V, scale, mask):
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    return F.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(K), torch.from_numpy(V),
        attn_mask=torch.from_numpy(mask), scale=scale).numpy()


def pin_decode_torch_sdpa():
    w = config1()
    st = build_decode_state(w)
    out = decode_oracle(w, st)
    cu = w.cu_lens
    for s in range(w.S):
        L = int(w.context_lens[s])
        q = attention.widen_bf16(w.q[s])[:, None, :]                      # [H, 1, D]
        K = attention.widen_bf16(w.k[cu[s]:cu[s] + L]).transpose(1, 0, 2)  # [H, L, D]
        V = attention.widen_bf16(w.v[cu[s]:cu[s] + L]).transpose(1, 0, 2)
        ref = _torch_reference(q, K, V, w.scale, np.ones((1, L), bool))[:, 0, :]
        assert np.max(np.abs(out[s] - ref)) <= 1e-12


def pin_prefill_torch_sdpa():
    w = make_decode_workload("p", (40, 23), Hq=4, Hkv=1, D=16, block_size=8, seed=11)
    st = build_decode_state(w)
    chunks = [17, 23]
    cu_q = np.concatenate([[0], np.cumsum(chunks)])
    q_bits = normal_bf16((sum(chunks), w.Hq, w.D), 99)
    out = attention.prefill(q_bits, cu_q, w.context_lens, st.k_cache, st.v_cache, st.tables,
                            w.block_size, w.scale)
    cu = w.cu_lens
    for s in range(w.S):
        L, c = int(w.context_lens[s]), chunks[s]
        q = attention.widen_bf16(q_bits[cu_q[s]:cu_q[s + 1]]).transpose(1, 0, 2)
        K = np.repeat(attention.widen_bf16(w.k[cu[s]:cu[s] + L]).transpose(1, 0, 2), 4, axis=0)
        V = np.repeat(attention.widen_bf16(w.v[cu[s]:cu[s] + L]).transpose(1, 0, 2), 4, axis=0)
        mask = np.arange(L)[None, :] <= (L - c + np.arange(c))[:, None]
        ref = _torch_reference(q, K, V, w.scale, mask).transpose(1, 0, 2)
        assert np.max(np.abs(out[cu_q[s]:cu_q[s + 1]] - ref)) <= 1e-12


def pin_single_key_returns_v():
    w = make_decode_workload("one", (1, 1, 1), Hq=4, Hkv=2, D=16, block_size=16, seed=3)
    st = build_decode_state(w)
    out = decode_oracle(w, st)
    G = w.Hq // w.Hkv
    for s in range(w.S):
        for h in range(w.Hq):
            want = [bits_to_float(x) for x in w.v[s, h // G]]
            assert list(out[s, h]) == want


def pin_closed_forms():
    rng = np.random.default_rng(5)
    D, L = 8, 13
    K = rng.standard_normal((L, D))
    V = rng.standard_normal((L, D))
    # zero query: uniform weights, the mean of the values
    out = attention.attend(np.zeros((1, D)), K, V, 0.3, [L])[0]
    assert np.allclose(out, V.mean(axis=0), rtol=0, atol=1e-13)
    # equal keys: uniform weights again
    Ke = np.tile(K[:1], (L, 1))
    out = attention.attend(rng.standard_normal((1, D)), Ke, V, 0.3, [L])[0]
    assert np.allclose(out, V.mean(axis=0), rtol=0, atol=1e-13)
    # equal values: the value itself
    Ve = np.tile(V[:1], (L, 1))
    out = attention.attend(rng.standard_normal((1, D)), K, Ve, 0.3, [L])[0]
    assert np.allclose(out, V[0], rtol=0, atol=1e-13)
    # one dominant score: the one-hot row (other weights below e^-700)
    q = np.zeros((1, D)); q[0, 0] = 1.0
    Kd = np.zeros((L, D)); Kd[5, 0] = 1000.0
    out = attention.attend(q, Kd, V, 1.0, [L])[0]
    assert np.array_equal(out, V[5])
    # two keys: weights are the logistic function of the score difference
    q = np.array([[1.0, 2.0]])
    K2 = np.array([[0.5, -1.0], [2.0, 0.25]])
    V2 = np.array([[3.0, -1.0], [-2.0, 4.0]])
    scale = 1 / math.sqrt(2)
    d = scale * ((1.0 * 2.0 + 2.0 * 0.25) - (1.0 * 0.5 + 2.0 * -1.0))
    w1 = 1.0 / (1.0 + math.exp(-d))
    want = (1 - w1) * V2[0] + w1 * V2[1]
    out = attention.attend(q, K2, V2, scale, [2])[0]
    assert np.max(np.abs(out - want)) <= 1e-15
    # the causal limit: a row limited to one key returns that key's value
    out = attention.attend(rng.standard_normal((2, D)), K, V, 0.3, [1, L])
    assert np.array_equal(out[0], V[0])


def pin_placement_invariance():
    w1 = tiny_gqa_workload(seed=21)
    w2 = tiny_gqa_workload(seed=21)
    w2.free_order = w2.free_order[::-1].copy()
    o1 = decode_oracle(w1, build_decode_state(w1))
    st2 = build_decode_state(w2)
    o2 = decode_oracle(w2, st2)
    assert build_decode_state(w1).tables != st2.tables
    assert np.array_equal(o1, o2)


def _small_shared(variant):
    return config4(variant, n_prompts=2, n_samples=4, tail_max=20)


def pin_shared_equals_duplicated():
    for variant in ("a", "b"):
        w = _small_shared(variant)
        st = build_shared_prefix_state(w)
        out = attention.decode(w.q, st.k_cache, st.v_cache, st.tables, w.context_lens,
                               w.block_size, w.scale)
        # the same tokens written into private, duplicated blocks
        lens = w.context_lens
        dup = make_decode_workload("dup", lens, w.Hq, w.Hkv, w.D, w.block_size, seed=0)
        ks, vs = [], []
        cu = w.cu_tails
        for i in range(w.S):
            p = i // w.n_samples
            ks.append(np.concatenate([w.prefix_k[p], w.tail_k[cu[i]:cu[i + 1]]]))
            vs.append(np.concatenate([w.prefix_v[p], w.tail_v[cu[i]:cu[i + 1]]]))
        dup.k, dup.v, dup.q = np.concatenate(ks), np.concatenate(vs), w.q
        ref = decode_oracle(dup, build_decode_state(dup))
        assert np.array_equal(out, ref)
        # sharing really happened: prefix blocks are referenced by all samples
        first = st.tables[0][0]
        assert all(t[0] == first for t in st.tables[:w.n_samples])


def pin_cow_isolation():
    w = _small_shared("b")                 # 1032-token prefix: last shared block half full
    alloc = paging.BlockAllocator(w.num_blocks, w.block_size, w.free_order)
    sid = alloc.create()
    alloc.append_slots(sid, w.prefix_len)
    kids = [alloc.fork(sid) for _ in range(3)]
    shared_last = alloc.block_table(sid)[-1]
    before = alloc.block_table(kids[1])
    slots, pairs = alloc.append_slots(kids[0], 1)
    # the writer got a private copy of the partial block; the others did not move
    assert pairs == [(shared_last, alloc.block_table(kids[0])[-1])]
    assert alloc.block_table(kids[1]) == before
    assert alloc.refcount[shared_last] == 3
    # bytes: every copy and the source still hold the shared prefix tokens
    st = build_shared_prefix_state(w)
    idx, off = divmod(w.prefix_len, w.block_size)
    n_copies = 0
    for p in range(w.n_prompts):
        src = st.prefix_slots[p][-1] // w.block_size
        for j in range(w.n_samples):
            blk = st.tables[p * w.n_samples + j][idx]
            n_copies += blk != src
            for kc, pref in ((st.k_cache, w.prefix_k), (st.v_cache, w.prefix_v)):
                assert np.array_equal(kc[blk, :, :off],
                                      pref[p, idx * w.block_size:].transpose(1, 0, 2))
    assert n_copies == len(st.cow_pairs) > 0
    # every other sharer still decodes exactly as if it had been alone
    pin_shared_equals_duplicated()


def pin_decode_equals_last_prefill_row():
    w = tiny_gqa_workload(seed=31, lens=(7, 12, 20))
    st = build_decode_state(w)
    dec = decode_oracle(w, st)
    chunks = [3, 12, 5]
    cu_q = np.concatenate([[0], np.cumsum(chunks)])
    q_bits = normal_bf16((sum(chunks), w.Hq, w.D), 5)
    for s in range(w.S):
        q_bits[cu_q[s + 1] - 1] = w.q[s]
    pre = attention.prefill(q_bits, cu_q, w.context_lens, st.k_cache, st.v_cache, st.tables,
                            w.block_size, w.scale)
    for s in range(w.S):
        assert np.max(np.abs(pre[cu_q[s + 1] - 1] - dec[s])) <= 1e-13


def pin_append_gather_roundtrip():
    w = tiny_gqa_workload(seed=41, lens=(4, 9, 17, 2))
    st = build_decode_state(w)
    cu = w.cu_lens
    for s in range(w.S):
        L = int(w.context_lens[s])
        assert np.array_equal(cache.gather(st.k_cache, st.tables[s], L, w.block_size),
                              w.k[cu[s]:cu[s] + L])
        assert np.array_equal(cache.gather(st.v_cache, st.tables[s], L, w.block_size),
                              w.v[cu[s]:cu[s] + L])
    # slot -1 is skipped
    k2, v2 = st.k_cache.copy(), st.v_cache.copy()
    cache.append(k2, v2, w.k[:1], w.v[:1], [-1], w.block_size)
    assert np.array_equal(k2, st.k_cache)


def pin_poisoned_slots_unread():
    w = config1()
    st = build_decode_state(w, poison=True)
    assert np.isnan(attention.widen_bf16(st.k_cache)).any()
    assert np.isfinite(decode_oracle(w, st)).all()


def parse_ids(spec):
    """A golden-file id list: comma items, each an id or an inclusive range a..b."""
    if spec == "-":
        return []
    out = []
    for item in spec.split(","):
        if ".." in item:
            a, b = item.split("..")
            out.extend(range(int(a), int(b) + 1))
        else:
            out.append(int(item))
    return out


def _run_allocator_script(path):
    """Replays ``tests/golden/<path>``; see that file for the format."""
    alloc = None
    names = {}
    for raw in open(os.path.join(GOLDEN, path)):
        line = raw.split("#", 1)[0].strip()
        if not line:
            continue
        op, *args = line.split()
        if op == "pool":
            n, bs = int(args[0]), int(args[1])
            order = [int(x) for x in args[2].split(",")]
            alloc = paging.BlockAllocator(n, bs, order)
        elif op == "create":
            names[args[0]] = alloc.create()
        elif op == "fork":
            names[args[1]] = alloc.fork(names[args[0]])
        elif op == "create_cached":
            names[args[0]], n_cached = alloc.create_cached(parse_ids(args[1]))
            assert n_cached == int(args[2]), (line, n_cached)
        elif op == "append_tokens":
            slots, pairs = alloc.append_tokens(names[args[0]], parse_ids(args[1]))
            assert slots == parse_ids(args[2]), (line, slots)
            assert pairs == [] and args[3] == "-", line
        elif op == "ncached":
            assert alloc.num_cached() == int(args[0]), (line, alloc.num_cached())
        elif op == "append":
            slots, pairs = alloc.append_slots(names[args[0]], int(args[1]))
            exp_slots = parse_ids(args[2])
            exp_pairs = ([tuple(int(y) for y in x.split(">")) for x in args[3].split(",")]
                         if args[3] != "-" else [])
            assert slots == exp_slots, (line, slots)
            assert pairs == exp_pairs, (line, pairs)
        elif op == "append_fails":
            snap = (list(alloc.free), list(alloc.refcount), alloc.block_table(names[args[0]]))
            with pytest.raises(paging.OutOfBlocks):
                alloc.append_slots(names[args[0]], int(args[1]))
            assert snap == (list(alloc.free), list(alloc.refcount),
                            alloc.block_table(names[args[0]]))
        elif op == "table":
            want = [int(x) for x in args[1].split(",")] if args[1] != "-" else []
            assert alloc.block_table(names[args[0]]) == want, line
        elif op == "refcount":
            assert alloc.refcount[int(args[0])] == int(args[1]), line
        elif op == "free":
            alloc.free_seq(names[args[0]])
        elif op == "nfree":
            assert alloc.num_free() == int(args[0]), line
        elif op == "freelist":
            assert list(alloc.free) == [int(x) for x in args[0].split(",")], line
        else:
            raise ValueError(op)
        alloc.check_invariants()


def pin_allocator_golden():
    _run_allocator_script("allocator_block_sharing.txt")


def pin_prefix_cache_golden():
    _run_allocator_script("prefix_cache.txt")


def pin_allocator_fuzz():
    rng = np.random.default_rng(1234)
    for trial in range(30):
        N, B = int(rng.integers(1, 24)), int(rng.choice([1, 2, 4, 16]))
        alloc = paging.BlockAllocator(N, B, rng.permutation(N))
        live = []
        for _ in range(200):
            op = rng.integers(0, 4)
            if op == 0 or not live:
                live.append(alloc.create())
            elif op == 1:
                live.append(alloc.fork(live[rng.integers(len(live))]))
            elif op == 2:
                sid = live[rng.integers(len(live))]
                try:
                    alloc.append_slots(sid, int(rng.integers(0, 2 * B + 2)))
                except paging.OutOfBlocks:
                    pass
            else:
                alloc.free_seq(live.pop(rng.integers(len(live))))
            alloc.check_invariants()
        for sid in live:
            alloc.free_seq(sid)
        assert alloc.num_free() == N


def pin_swap_round_trip():
    """Evicting a request to host memory and bringing it back ("Batching,
    Scheduling, and Paging", section PagedAttention) restores its tokens in
    whatever blocks it gets back; blocks a fork still uses stay allocated."""
    N, B, Hkv, D, L = 12, 4, 2, 8, 10
    alloc = paging.BlockAllocator(N, B, list(range(N)))
    kc, vc = empty_pools(N, Hkv, B, D)
    k, v = normal_bf16((L, Hkv, D), 901), normal_bf16((L, Hkv, D), 902)
    q = normal_bf16((1, 2 * Hkv, D), 903)
    s = alloc.create()
    slots, _ = alloc.append_slots(s, L)
    cache.append(kc, vc, k, v, slots, B)
    before = attention.decode(q, kc, vc, [alloc.block_table(s)], [L], B, 0.3)
    f = alloc.fork(s)
    out_blocks = alloc.swap_out(s)
    alloc.check_invariants()
    assert out_blocks == [0, 1, 2] and alloc.num_free() == N - 3   # the fork holds them
    kb, vb = np.zeros((3, Hkv, B, D), np.uint16), np.zeros((3, Hkv, B, D), np.uint16)
    cache.swap_blocks(kc, vc, out_blocks, kb, vb, 0)
    alloc.free_seq(f)
    assert alloc.num_free() == N
    # another request takes (and overwrites) every free block but two
    t = alloc.create()
    t_slots, _ = alloc.append_slots(t, 4 * B * 2 + 2 * B)
    cache.append(kc, vc, normal_bf16((len(t_slots), Hkv, D), 904),
                 normal_bf16((len(t_slots), Hkv, D), 905), t_slots, B)
    alloc.free_seq(t)
    in_blocks = alloc.swap_in(s)
    alloc.check_invariants()
    assert len(in_blocks) == -(-L // B) and in_blocks != out_blocks
    assert alloc.seq_len(s) == L and alloc.block_table(s) == in_blocks
    cache.swap_blocks(kc, vc, in_blocks, kb, vb, 1)
    assert np.array_equal(cache.gather(kc, in_blocks, L, B), k)
    assert np.array_equal(cache.gather(vc, in_blocks, L, B), v)
    after = attention.decode(q, kc, vc, [in_blocks], [L], B, 0.3)
    assert np.array_equal(after, before)


def pin_e4m3_against_torch():
    """torch's float8_e4m3fn conversion (an independent implementation of the
    same format, round to nearest even) agrees code for code inside the range
    where it does not turn to NaN, and value for value on all 256 codes."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(81)
    x = np.concatenate([
        (rng.standard_normal(100000) * 40).astype(np.float32),
        (rng.standard_normal(20000) * 0.01).astype(np.float32),
        # exact midpoints between neighbouring codes, where ties decide
        ((fp8.e4m3_decode(np.arange(0, 126)) + fp8.e4m3_decode(np.arange(1, 127))) / 2
         ).astype(np.float32),
        np.float32([0.0, -0.0, 448.0, -448.0, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10]),
    ])
    x = x[np.abs(x) < 464]
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.e4m3_encode(x), want)
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = fp8.e4m3_decode(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[~np.isnan(got)], ref[~np.isnan(ref)])


def pin_e4m3_closed_forms():
    """Round trip of every finite code, saturation, and hand-worked ties."""
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(fp8.e4m3_encode(fp8.e4m3_decode(codes).astype(np.float32)), codes)
    assert fp8.e4m3_encode(np.float32([1000.0, -1e9, 449.0])).tolist() == [0x7E, 0xFE, 0x7E]
    assert fp8.e4m3_decode(np.uint8([0x7E, 0x38, 0x01, 0x08, 0x3A])).tolist() == \
        [448.0, 1.0, 2.0 ** -9, 2.0 ** -6, 1.25]
    # 1 + 1/16 lies halfway between 1 (mantissa 000) and 1.125 (001): even wins
    # 1 + 3/16 lies halfway between 1.125 (001) and 1.25 (010): even wins
    assert fp8.e4m3_encode(np.float32([1.0625, 1.1875, -1.0625])).tolist() == [0x38, 0x3A, 0xB8]


def pin_fp8_quantize_rows():
    """Zero rows, single-value rows and the relative error bound of e4m3."""
    D = 64
    rows = np.zeros((3, D), dtype=np.uint16)
    one = attention.widen_bf16(np.uint16([0x3FC0]))[0]            # 1.5
    rows[1, 5] = 0x3FC0
    rows[2] = normal_bf16((D,), 82)
    codes, scales = fp8.quantize_rows(rows)
    assert scales[0] == 0 and not codes[0].any()
    assert codes[1, 5] == 0x7E and np.count_nonzero(codes[1]) == 1
    assert scales[1] == np.float32(one) / np.float32(448.0)
    x = attention.widen_bf16(rows[2])
    deq = fp8.e4m3_decode(codes[2]) * float(scales[2])
    amax = np.max(np.abs(x))
    # normal codes: half a mantissa step (2^-4 relative); subnormals: 2^-10 of amax
    assert np.all(np.abs(deq - x) <= np.maximum(np.abs(x) * 2.0 ** -4, amax * 2.0 ** -10) * 1.001)


def pin_fp8_decode_exact_values():
    """K/V rows that e4m3 represents exactly (codes times a power of two, each
    row reaching +-448 times it): the fp8 path equals the bf16 oracle."""
    rng = np.random.default_rng(83)
    w = tiny_gqa_workload(seed=84, lens=(5, 17, 33))
    for arr in (w.k, w.v):
        codes = rng.integers(0, 0x7E, size=arr.shape).astype(np.uint8)
        codes[..., 0] = 0x7E
        codes |= (rng.integers(0, 2, size=arr.shape) * 0x80).astype(np.uint8)
        vals = fp8.e4m3_decode(codes) * 2.0 ** -6
        arr[...] = (vals.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    st = build_decode_state(w)
    ref = attention.decode(w.q, st.k_cache, st.v_cache, st.tables, w.context_lens, w.block_size,
                           w.scale)
    N, Hkv, B, D = st.k_cache.shape
    k8, v8 = np.zeros((N, Hkv, B, D), np.uint8), np.zeros((N, Hkv, B, D), np.uint8)
    ks, vs = np.zeros((N, Hkv, B), np.float32), np.zeros((N, Hkv, B), np.float32)
    slots = np.concatenate([[st.tables[s][j // B] * B + j % B for j in range(w.context_lens[s])]
                            for s in range(w.S)])
    fp8.append(k8, v8, ks, vs, w.k, w.v, slots, B)
    got = fp8.decode(w.q, k8, v8, ks, vs, st.tables, w.context_lens, B, w.scale)
    assert np.array_equal(got, ref)


PINS = [pin_widen_bf16, pin_decode_brute_force, pin_prefill_brute_force,
        pin_decode_torch_sdpa, pin_prefill_torch_sdpa, pin_single_key_returns_v,
        pin_closed_forms, pin_placement_invariance, pin_shared_equals_duplicated,
        pin_cow_isolation, pin_decode_equals_last_prefill_row, pin_append_gather_roundtrip,
        pin_poisoned_slots_unread, pin_allocator_golden, pin_allocator_fuzz,
        pin_swap_round_trip, pin_prefix_cache_golden, pin_e4m3_against_torch,
        pin_e4m3_closed_forms, pin_fp8_quantize_rows, pin_fp8_decode_exact_values]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


# ---------------------------------------------------------------- planted mistakes

def _mut_attend_no_scale(q, K, V, scale, limits):
    return _ORIG["attend"](q, K, V, 1.0, limits)


def _mut_attend_kv_swapped(q, K, V, scale, limits):
    return _ORIG["attend"](q, V, K, scale, limits)


def _mut_attend_off_by_one(q, K, V, scale, limits):
    return _ORIG["attend"](q, K, V, scale, np.minimum(np.asarray(limits) + 1, K.shape[0]))


def _mut_attend_unnormalised(q, K, V, scale, limits):
    out = _ORIG["attend"](q, K, V, scale, limits)
    return out * 1.0001


def _mut_attend_sign(q, K, V, scale, limits):
    return _ORIG["attend"](q, K, V, -scale, limits)


def _mut_attend_drop_last_key(q, K, V, scale, limits):
    lim = np.asarray(limits)
    return _ORIG["attend"](q, K, V, scale, np.maximum(lim - 1, 1))


def _mut_gather_offset_shift(cache_, block_table, length, block_size):
    out = np.empty((length, cache_.shape[1], cache_.shape[3]), dtype=cache_.dtype)
    for j in range(length):
        out[j] = cache_[int(block_table[j // block_size]), :, (j + 1) % block_size, :]
    return out


def _mut_gather_first_block(cache_, block_table, length, block_size):
    out = np.empty((length, cache_.shape[1], cache_.shape[3]), dtype=cache_.dtype)
    for j in range(length):
        out[j] = cache_[int(block_table[0]), :, j % block_size, :]
    return out


def _mut_widen(bits):
    return _ORIG["widen"](bits) * (1 + 2.0 ** -7)


def _mut_group_all_on_first(Hq, Hkv):
    return Hq


def _mut_append_no_cow(self, sid, n, _keep_tokens=False):
    seq = self.seqs[sid]
    B = self.block_size
    slots = []
    for pos in range(seq["len"], seq["len"] + n):
        j, off = divmod(pos, B)
        if j == len(seq["blocks"]):
            seq["blocks"].append(self._take())
        slots.append(seq["blocks"][j] * B + off)
    seq["len"] += n
    if n > 0 and not _keep_tokens:
        seq["tokens"] = None
    return slots, []


def _mut_free_lifo(self, sid):
    seq = self.seqs.pop(sid)
    for b in seq["blocks"]:
        self.refcount[b] -= 1
        if self.refcount[b] == 0:
            self.free.appendleft(b)


def _mut_swap_direction(k_cache, v_cache, blocks, k_buf, v_buf, direction):
    _ORIG["swap_blocks"](k_cache, v_cache, blocks, k_buf, v_buf, 1 - direction)


def _mut_swap_out_ignores_sharing(self, sid):
    seq = self.seqs[sid]
    blocks = list(seq["blocks"])
    for b in blocks:
        self.refcount[b] = 0
        self.free.append(b)
    seq["blocks"] = []
    seq["swapped"] = True
    return blocks


def _mut_swap_in_one_short(self, sid):
    seq = self.seqs[sid]
    need = max(-(-seq["len"] // self.block_size) - 1, 0)
    seq["blocks"] = [self._take() for _ in range(need)]
    seq["swapped"] = False
    return list(seq["blocks"])


def _mut_take_keeps_descendants(self):
    b = self.free.popleft()
    self.refcount[b] = 1
    if b in self.prefix_of:
        del self.registry[self.prefix_of.pop(b)]      # extensions wrongly kept
    return b


def _mut_cached_whole_prompt(self, tokens):
    tokens = [int(t) for t in tokens]
    B = self.block_size
    sid = self.create()
    seq = self.seqs[sid]
    j = 0
    while j < len(tokens) // B and tuple(tokens[:(j + 1) * B]) in self.registry:
        b = self.registry[tuple(tokens[:(j + 1) * B])]
        if self.refcount[b] == 0:
            self.free.remove(b)
        self.refcount[b] += 1
        seq["blocks"].append(b)
        j += 1
    seq["len"], seq["tokens"], seq["registered"] = j * B, tokens[:j * B], j
    return sid, j * B


def _mut_e4m3_ties_away(x):
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    vals = fp8.e4m3_decode(np.arange(0, 127))
    a = np.minimum(np.abs(x), 448.0)
    hi = np.minimum(np.searchsorted(vals, a, side="left"), 126)
    lo = np.maximum(hi - 1, 0)
    idx = np.where(vals[hi] - a <= a - vals[lo], hi, lo)     # ties go up
    out = idx.astype(np.uint8)
    return np.where(np.signbit(x), out | 0x80, out).astype(np.uint8)


def _mut_e4m3_bias8(codes):
    return _ORIG["e4m3_decode"](codes) / 2.0


def _mut_quantize_max_240(bits):
    x = attention.widen_bf16(bits).astype(np.float32)
    amax = np.max(np.abs(x), axis=-1).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        inv = np.where(amax > 0, np.float32(240.0) / amax, np.float32(0)).astype(np.float32)
        scale = (amax / np.float32(240.0)).astype(np.float32)
    return fp8.e4m3_encode((x * inv[..., None]).astype(np.float32)), scale


def _mut_dequant_no_scale(codes, scales, table, length, block_size):
    return _ORIG["dequantize_seq"](codes, np.ones_like(scales), table, length, block_size)


_ORIG = {"attend": attention.attend, "e4m3_decode": fp8.e4m3_decode,
         "dequantize_seq": fp8.dequantize_seq, "swap_blocks": cache.swap_blocks, "widen": attention.widen_bf16,
         "group": attention._group}

MUTATIONS = {
    "no_scale": (attention, "attend", _mut_attend_no_scale),
    "kv_swapped": (attention, "attend", _mut_attend_kv_swapped),
    "causal_off_by_one": (attention, "attend", _mut_attend_off_by_one),
    "unnormalised": (attention, "attend", _mut_attend_unnormalised),
    "score_sign": (attention, "attend", _mut_attend_sign),
    "drop_last_key": (attention, "attend", _mut_attend_drop_last_key),
    "gather_offset_shift": (attention, "gather", _mut_gather_offset_shift),
    "gather_first_block": (attention, "gather", _mut_gather_first_block),
    "widen_wrong": (attention, "widen_bf16", _mut_widen),
    "gqa_all_heads_on_kv0": (attention, "_group", _mut_group_all_on_first),
    "no_copy_on_write": (paging.BlockAllocator, "append_slots", _mut_append_no_cow),
    "free_list_lifo": (paging.BlockAllocator, "free_seq", _mut_free_lifo),
    "swap_direction": (cache, "swap_blocks", _mut_swap_direction),
    "swap_out_ignores_sharing": (paging.BlockAllocator, "swap_out",
                                 _mut_swap_out_ignores_sharing),
    "swap_in_one_short": (paging.BlockAllocator, "swap_in", _mut_swap_in_one_short),
    "prefix_cache_keeps_extensions": (paging.BlockAllocator, "_take",
                                      _mut_take_keeps_descendants),
    "prefix_cache_whole_prompt": (paging.BlockAllocator, "create_cached",
                                  _mut_cached_whole_prompt),
    "e4m3_ties_away_from_zero": (fp8, "e4m3_encode", _mut_e4m3_ties_away),
    "e4m3_exponent_bias_8": (fp8, "e4m3_decode", _mut_e4m3_bias8),
    "fp8_quantise_to_240": (fp8, "quantize_rows", _mut_quantize_max_240),
    "fp8_scales_ignored": (fp8, "dequantize_seq", _mut_dequant_no_scale),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistakes_are_caught(name, monkeypatch):
    target, attr, repl = MUTATIONS[name]
    monkeypatch.setattr(target, attr, repl)
    failed = []
    for pin in PINS:
        try:
            pin()
        except (AssertionError, IndexError, ValueError, KeyError, paging.OutOfBlocks):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {name}"
