"""Sets a workload up on the GPU through the library's own API.

The library's allocator hands out the blocks, ``pkv_kv_append`` writes the
tokens into NaN-poisoned pools, and the decode/prefill calls run on them.
Used by the benchmark, the tests and the smoke check; nothing here computes
attention, and nothing here touches the oracle.
"""

from __future__ import annotations

import time
from dataclasses import dataclass

import numpy as np
import torch

import paged_kv_cache_281_gb300 as pkv
from workloads import BF16_NAN
from workloads.schedule import iteration_inputs


def to_dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def poisoned_pools(N, Hkv, B, D, device="cuda", poison=True):
    fill = int(np.int16(np.uint16(BF16_NAN).view(np.int16))) if poison else 0
    k = torch.full((N, Hkv, B, D), fill, dtype=torch.int16, device=device).view(torch.bfloat16)
    v = torch.full((N, Hkv, B, D), fill, dtype=torch.int16, device=device).view(torch.bfloat16)
    return k, v


@dataclass
class DeviceDecode:
    alloc: pkv.BlockAllocator
    seqs: list
    tables: np.ndarray            # host int32 [S, maxB]
    slots: np.ndarray             # host int32 [sum L], packed by sequence
    last_slots: np.ndarray        # host int32 [S], slot of each sequence's newest token
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    q: torch.Tensor
    block_tables: torch.Tensor
    context_lens: torch.Tensor
    k_last: torch.Tensor          # [S, Hkv, D] newest tokens (appended by the step)
    v_last: torch.Tensor
    last_slot_mapping: torch.Tensor
    out: torch.Tensor
    workspace: torch.Tensor
    status: torch.Tensor
    max_context_len: int
    partition_size: int


def setup_decode(w, partition_size=0, poison=True, append_last=True, device="cuda",
                 max_blocks_per_seq=None) -> DeviceDecode:
    """Allocates every sequence's blocks and writes its tokens (all but the
    newest one unless ``append_last``)."""
    alloc = pkv.BlockAllocator(w.num_blocks, w.block_size, w.free_order)
    seqs, slots = [], []
    for s in range(w.S):
        sid = alloc.seq_create()
        sl, pair = alloc.seq_append_slots(sid, int(w.context_lens[s]))
        assert pair is None
        seqs.append(sid)
        slots.append(sl)
    maxB = max_blocks_per_seq or w.max_blocks_per_seq
    tables, lens = alloc.build_block_tables(seqs, maxB)
    assert np.array_equal(lens, w.context_lens)
    slots_all = np.concatenate(slots).astype(np.int32)
    k_cache, v_cache = poisoned_pools(w.num_blocks, w.Hkv, w.block_size, w.D, device, poison)
    cu = w.cu_lens
    last_idx = cu[1:] - 1
    write = slots_all.copy()
    if not append_last:
        write[last_idx] = -1
    status = pkv.new_status(device)
    pkv.pkv_kv_append(to_dev_bf16(w.k, device), to_dev_bf16(w.v, device),
                      torch.from_numpy(write).to(device), k_cache, v_cache, status=status)
    ws_bytes = pkv.pkv_decode_workspace_bytes(w.S, w.Hq, w.D, w.max_context_len, partition_size)
    return DeviceDecode(
        alloc=alloc, seqs=seqs, tables=tables, slots=slots_all,
        last_slots=slots_all[last_idx], k_cache=k_cache, v_cache=v_cache,
        q=to_dev_bf16(w.q, device), block_tables=torch.from_numpy(tables).to(device),
        context_lens=torch.from_numpy(lens).to(device),
        k_last=to_dev_bf16(w.k[last_idx], device), v_last=to_dev_bf16(w.v[last_idx], device),
        last_slot_mapping=torch.from_numpy(slots_all[last_idx].copy()).to(device),
        out=torch.empty(w.S, w.Hq, w.D, dtype=torch.bfloat16, device=device),
        workspace=torch.empty(ws_bytes, dtype=torch.uint8, device=device),
        status=status, max_context_len=w.max_context_len, partition_size=partition_size)


def run_decode(w, d: DeviceDecode, out=None, partition_size=None, stream=None) -> torch.Tensor:
    out = d.out if out is None else out
    ps = d.partition_size if partition_size is None else partition_size
    ws = d.workspace
    need = pkv.pkv_decode_workspace_bytes(w.S, w.Hq, w.D, d.max_context_len, ps)
    if ws.numel() < need:
        ws = torch.empty(need, dtype=torch.uint8, device=out.device)
    pkv.pkv_paged_attention_decode(out, d.q, d.k_cache, d.v_cache, d.block_tables,
                                   d.context_lens, d.max_context_len, w.scale, ws,
                                   partition_size=ps, status=d.status, stream=stream)
    return out


def decode_step(w, d: DeviceDecode, stream=None) -> torch.Tensor:
    """One decode step: append each sequence's newest token, then attend."""
    pkv.pkv_kv_append(d.k_last, d.v_last, d.last_slot_mapping, d.k_cache, d.v_cache,
                      status=d.status, stream=stream)
    return run_decode(w, d, stream=stream)


# ---------------------------------------------------------------- shared prefix

@dataclass
class DeviceSharedPrefix:
    alloc: pkv.BlockAllocator
    sample_ids: list
    prefix_slots: list
    tail_slots: list
    cow_pairs: list
    tables: np.ndarray
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    q: torch.Tensor
    block_tables: torch.Tensor
    context_lens: torch.Tensor
    status: torch.Tensor
    max_context_len: int


def setup_shared_prefix(w, device="cuda") -> DeviceSharedPrefix:
    """The shared-prefix build order through the library: prefixes appended,
    samples forked, tails reserved (copy-on-write pairs collected), copies
    made, then tails written."""
    alloc = pkv.BlockAllocator(w.num_blocks, w.block_size, w.free_order)
    sample_ids, prefix_slots = [], []
    for _ in range(w.n_prompts):
        sid = alloc.seq_create()
        sl, pair = alloc.seq_append_slots(sid, w.prefix_len)
        assert pair is None
        prefix_slots.append(sl)
        sample_ids.append(sid)
        for _ in range(w.n_samples - 1):
            sample_ids.append(alloc.seq_fork(sid))
    tail_slots, pairs = [], []
    for i, sid in enumerate(sample_ids):
        sl, pair = alloc.seq_append_slots(sid, int(w.tails.reshape(-1)[i]))
        tail_slots.append(sl)
        if pair is not None:
            pairs.append(pair)
    k_cache, v_cache = poisoned_pools(w.num_blocks, w.Hkv, w.block_size, w.D, device)
    status = pkv.new_status(device)
    pkv.pkv_kv_append(to_dev_bf16(w.prefix_k.reshape(-1, w.Hkv, w.D), device),
                      to_dev_bf16(w.prefix_v.reshape(-1, w.Hkv, w.D), device),
                      torch.from_numpy(np.concatenate(prefix_slots).astype(np.int32)).to(device),
                      k_cache, v_cache, status=status)
    if pairs:
        pkv.pkv_block_copy(k_cache, v_cache,
                           torch.tensor(pairs, dtype=torch.int32, device=device), status=status)
    tails = np.concatenate(tail_slots).astype(np.int32)
    if tails.size:
        pkv.pkv_kv_append(to_dev_bf16(w.tail_k, device), to_dev_bf16(w.tail_v, device),
                          torch.from_numpy(tails).to(device), k_cache, v_cache, status=status)
    lens = w.context_lens
    maxB = -(-int(lens.max()) // w.block_size)
    tables, got_lens = alloc.build_block_tables(sample_ids, maxB)
    assert np.array_equal(got_lens, lens)
    return DeviceSharedPrefix(alloc, sample_ids, prefix_slots, tail_slots, pairs, tables,
                              k_cache, v_cache, to_dev_bf16(w.q, device),
                              torch.from_numpy(tables).to(device),
                              torch.from_numpy(got_lens).to(device), status, int(lens.max()))


def decode_shared_prefix(w, d: DeviceSharedPrefix, partition_size=0) -> torch.Tensor:
    out = torch.empty(w.S, w.Hq, w.D, dtype=torch.bfloat16, device=d.q.device)
    ws = torch.empty(pkv.pkv_decode_workspace_bytes(w.S, w.Hq, w.D, d.max_context_len,
                                                    partition_size),
                     dtype=torch.uint8, device=d.q.device)
    pkv.pkv_paged_attention_decode(out, d.q, d.k_cache, d.v_cache, d.block_tables,
                                   d.context_lens, d.max_context_len, w.scale, ws,
                                   partition_size=partition_size, status=d.status)
    return out


def shared_groups(w, d: DeviceSharedPrefix, shared=None):
    """Group arrays for pkv_paged_attention_decode_shared: one group per
    prompt (its samples), sharing the leading block-table entries that are
    identical for all of them (``shared`` overrides the token count)."""
    B, n = w.block_size, w.n_samples
    start = np.arange(0, w.S + 1, n, dtype=np.int32)
    members = np.arange(w.S, dtype=np.int32)
    sh = []
    for p in range(w.n_prompts):
        rows = d.tables[p * n:(p + 1) * n]
        lens = w.context_lens[p * n:(p + 1) * n]
        nb = min(-(-int(L) // B) for L in lens)
        same = 0
        while same < nb and np.all(rows[:, same] == rows[0, same]):
            same += 1
        sh.append(same * B if shared is None else shared)
    return start, members, np.asarray(sh, dtype=np.int32)


def decode_shared_grouped(w, d: DeviceSharedPrefix, groups=None, partition_size=0):
    """Shared-prefix decode of the workload through the group path."""
    dev = d.q.device
    start, members, sh = groups if groups is not None else shared_groups(w, d)
    out = torch.full((w.S, w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(pkv.pkv_decode_shared_workspace_bytes(w.S, w.Hq, w.D, d.max_context_len,
                                                           partition_size),
                     dtype=torch.uint8, device=dev)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    pkv.pkv_paged_attention_decode_shared(out, d.q, d.k_cache, d.v_cache, d.block_tables,
                                          d.context_lens, d.max_context_len, t(start),
                                          t(members), t(sh), w.scale, ws,
                                          partition_size=partition_size, status=d.status)
    return out


# ---------------------------------------------------------------- trace

class DeviceTrace:
    """Runs the continuous-batching trace through the library. Per iteration
    one call (``pkv_iteration_prepare``) reserves every work's slots (new
    blocks only when the last one fills) and writes the slot mapping, prompt
    offsets, context lengths and block tables into a pinned staging buffer;
    one host-to-device copy uploads it; ``kv_append`` writes every new
    token, prefill attends for the prompt chunks and decode for the running
    sequences; finished requests free their blocks."""

    RING = 4  # pinned staging buffers the host may fill ahead of the GPU

    def __init__(self, cfg, device="cuda", partition_size=0):
        self.cfg = cfg
        self.device = device
        self.partition_size = partition_size  # decode split-K partition (0: the default)
        self.alloc = pkv.BlockAllocator(cfg.num_blocks, cfg.block_size)
        self.k_cache, self.v_cache = poisoned_pools(cfg.num_blocks, cfg.Hkv, cfg.block_size,
                                                    cfg.D, device)
        self.status = pkv.new_status(device)
        self.sid = {}
        self.sid_arr = np.full(1024, -1, dtype=np.int64)  # the same map, by request id
        self.max_blocks = -(-(cfg.prompt_max + cfg.out_cap) // cfg.block_size)
        self.scale = 1.0 / np.sqrt(cfg.D)
        self.ws = torch.empty(pkv.pkv_decode_workspace_bytes(
            cfg.max_running, cfg.Hq, cfg.D, cfg.prompt_max + cfg.out_cap, partition_size),
            dtype=torch.uint8, device=device)
        # prefill work items: at most every running request's whole chunk
        self.pws = torch.empty(pkv.pkv_prefill_workspace_bytes(
            cfg.max_running, cfg.max_running * cfg.chunk, cfg.Hq, cfg.D),
            dtype=torch.uint8, device=device)
        cap = pkv.iteration_layout_bytes(cfg.max_running, cfg.max_running,
                                         cfg.max_running * cfg.chunk, self.max_blocks).total_bytes
        self.staging = [torch.empty(cap, dtype=torch.uint8).pin_memory()
                        for _ in range(self.RING)]
        self.staged = [None] * self.RING   # event after the last upload from each buffer
        self.events = [torch.cuda.Event() for _ in range(self.RING)]  # reused by step()
        self.next = 0
        self.wait_s = 0.0                   # host time spent waiting for a free buffer
        self.lib_s = 0.0                    # host time inside the library's per-iteration calls
        self.dev_meta = None                # device copy of the metadata (pkv_iteration_step)
        self.stepper = None                 # pkv_iteration_step bound to the above

    def admit(self, rids):
        """New sequences for the admitted requests ``rids`` (one library call)."""
        if not len(rids):
            return
        sids = self.alloc.seq_create_many(len(rids))
        top = max(rids)
        if top >= self.sid_arr.shape[0]:
            grow = max(top + 1, 2 * self.sid_arr.shape[0]) - self.sid_arr.shape[0]
            self.sid_arr = np.concatenate([self.sid_arr, np.full(grow, -1, dtype=np.int64)])
        self.sid_arr[list(rids)] = sids
        self.sid.update(zip(rids, sids.tolist()))

    def host_metadata(self, itr):
        """The iteration's host side: new sequences for admitted requests,
        then one library call for every work's slots and the metadata."""
        self.admit(itr.admitted)
        k = self.next
        self.next = (k + 1) % self.RING
        if self.staged[k] is not None:
            w0 = time.perf_counter()
            self.staged[k].synchronize()    # its previous upload has left the buffer
            self.wait_s += time.perf_counter() - w0
            self.staged[k] = None
        rids, counts, n_pre, _ = itr.arrays()
        t0 = time.perf_counter()
        layout = self.alloc.iteration_prepare(self.sid_arr[rids], counts, n_pre, self.max_blocks,
                                              self.staging[k])
        self.lib_s += time.perf_counter() - t0
        return {"staging": k, "layout": layout, "n_prefill": n_pre,
                "n_decode": counts.shape[0] - n_pre}

    def host_section(self, meta, name, count):
        """A host view of one section of the staged metadata (int32)."""
        off = getattr(meta["layout"], name)
        return self.staging[meta["staging"]][off:off + 4 * count].numpy().view(np.int32)

    def upload_meta(self, meta, stream=None):
        """One host-to-device copy of the staged metadata; returns the device
        buffer and the launch arguments read from the layout."""
        L, k = meta["layout"], meta["staging"]
        stream = stream or torch.cuda.current_stream()
        n = int(L.total_bytes)
        buf = torch.empty(n, dtype=torch.uint8, device=self.device)
        with torch.cuda.stream(stream):
            buf.copy_(self.staging[k][:n], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(stream)
        self.staged[k] = ev
        W = int(L.table_width)
        sec = lambda name, count: buf[getattr(L, name):getattr(L, name) + 4 * count].view(
            torch.int32)
        npre, ndec = meta["n_prefill"], meta["n_decode"]
        up = {"meta": buf, "n_pre": 0, "layout_meta": meta}
        if L.n_tokens:
            up["slots"] = sec("slot_mapping", L.n_tokens)
        if npre:
            up["pre"] = (sec("cu_q_lens", npre + 1), sec("prefill_lens", npre),
                         sec("prefill_tables", npre * W).view(npre, W), int(L.max_q_len),
                         int(L.max_prefill_len))
        if ndec:
            up["dec"] = (sec("decode_lens", ndec), sec("decode_tables", ndec * W).view(ndec, W),
                         int(L.max_decode_len), ndec)
        return up

    def upload(self, itr, meta, stream=None):
        """Host -> device copies of one iteration's metadata and token values."""
        dev = self.device
        up = self.upload_meta(meta, stream)
        up["q"] = to_dev_bf16(np.ascontiguousarray(itr.q), dev)
        up["n_pre"] = sum(w.n for w in itr.prefill)
        if itr.num_tokens:
            up["k"] = to_dev_bf16(np.ascontiguousarray(itr.k), dev)
            up["v"] = to_dev_bf16(np.ascontiguousarray(itr.v), dev)
        return up

    def launch(self, up, stream=None, events=None):
        """The GPU part of one iteration: kv_append, prefill, decode. With
        ``events`` (four CUDA events) the boundaries are recorded on ``stream``."""
        cfg, dev = self.cfg, self.device
        rec = (lambda i: events[i].record(stream)) if events else (lambda i: None)
        rec(0)
        if "slots" in up:
            pkv.pkv_kv_append(up["k"], up["v"], up["slots"], self.k_cache, self.v_cache,
                              status=self.status, stream=stream)
        rec(1)
        pre_out = dec_out = None
        n_pre = up["n_pre"]
        if "pre" in up:
            cu, lens, tables, max_q, max_ctx = up["pre"]
            pre_out = torch.empty(n_pre, cfg.Hq, cfg.D, dtype=torch.bfloat16, device=dev)
            pkv.pkv_paged_attention_prefill(pre_out, up["q"][:n_pre], cu, lens, self.k_cache,
                                            self.v_cache, tables, max_q, max_ctx, self.scale,
                                            self.pws, status=self.status, stream=stream)
        rec(2)
        if "dec" in up:
            lens, tables, max_ctx, n = up["dec"]
            dec_out = torch.empty(n, cfg.Hq, cfg.D, dtype=torch.bfloat16, device=dev)
            pkv.pkv_paged_attention_decode(dec_out, up["q"][n_pre:], self.k_cache, self.v_cache,
                                           tables, lens, max_ctx, self.scale, self.ws,
                                           partition_size=self.partition_size,
                                           status=self.status, stream=stream)
        rec(3)
        return pre_out, dec_out

    def launch_fused(self, up, stream=None):
        """The same GPU work through one library call (pkv_iteration_run):
        copies, appends, prefill and decode from the uploaded metadata."""
        cfg = self.cfg
        meta = up["layout_meta"]
        out = torch.empty(up["q"].shape[0], cfg.Hq, cfg.D, dtype=torch.bfloat16,
                          device=self.device)
        k, v = (up["k"], up["v"]) if "k" in up else (up["q"][:0, :cfg.Hkv],) * 2
        t0 = time.perf_counter()
        pkv.pkv_iteration_run(up["meta"], meta["layout"], meta["n_prefill"], meta["n_decode"],
                              up["q"], k, v, out, self.k_cache, self.v_cache,
                              self.scale, self.ws, self.pws, partition_size=self.partition_size,
                              status=self.status, stream=stream)
        self.lib_s += time.perf_counter() - t0
        n_pre = up["n_pre"]
        return out[:n_pre], out[n_pre:]

    def step(self, itr, q, k, v, stream=None):
        """One iteration through pkv_iteration_step (the allocator work, the
        metadata copy and the launches in one library call), with the token
        values already on the device. Returns (prefill_out, decode_out, meta);
        ``host_section(meta, ...)`` reads the staged metadata."""
        cfg = self.cfg
        self.admit(itr.admitted)
        kk = self.next
        self.next = (kk + 1) % self.RING
        if self.staged[kk] is not None:
            w0 = time.perf_counter()
            self.staged[kk].synchronize()    # its previous copy has left the buffer
            self.wait_s += time.perf_counter() - w0
        rids, counts, n_pre, rows = itr.arrays()
        ids = self.sid_arr[rids]
        stream = stream or torch.cuda.current_stream()
        if self.stepper is None:
            # the call bound once to the allocator, pools, device metadata
            # buffer and workspaces (their checks done here, not per iteration)
            self.dev_meta = torch.empty(self.staging[0].numel(), dtype=torch.uint8,
                                        device=self.device)
            self.stepper = pkv.IterationStepper(self.alloc, self.max_blocks, self.dev_meta,
                                                self.k_cache, self.v_cache, self.scale, self.ws,
                                                self.pws, partition_size=self.partition_size,
                                                status=self.status)
        out = torch.empty(q.shape[0], cfg.Hq, cfg.D, dtype=torch.bfloat16, device=self.device)
        t0 = time.perf_counter()
        layout = self.stepper(ids, counts, n_pre, self.staging[kk], q, k, v, out, stream=stream)
        self.lib_s += time.perf_counter() - t0
        ev = self.events[kk]
        ev.record(stream)
        self.staged[kk] = ev
        n = counts.shape[0]
        meta = {"staging": kk, "layout": layout, "n_prefill": n_pre, "n_decode": n - n_pre}
        return (out[:rows] if n_pre else None), (out[rows:] if n > n_pre else None), meta

    def run_iteration(self, itr, meta, stream=None, fused=False):
        """Upload and run one iteration, through the separate calls or through
        pkv_iteration_run; returns (prefill_out, decode_out)."""
        up = self.upload(itr, meta, stream)
        if fused:
            pre, dec = self.launch_fused(up, stream=stream)
            return (pre if meta["n_prefill"] else None), (dec if meta["n_decode"] else None)
        return self.launch(up, stream=stream)

    def finish(self, itr):
        """Frees the sequences of the requests that completed (one library call)."""
        if len(itr.finished):
            self.alloc.seq_free_many([self.sid.pop(rid) for rid in itr.finished])


# ---------------------------------------------------------------- preemption

class GpuRunner:
    """Replays scheduler events with the library on the GPU."""

    def __init__(self, cfg, num_blocks, device="cuda"):
        import torch
        import paged_kv_cache_281_gb300 as pkv
        self.torch, self.pkv, self.cfg, self.dev = torch, pkv, cfg, device
        self.k_cache, self.v_cache = poisoned_pools(num_blocks, cfg.Hkv, cfg.block_size, cfg.D,
                                                    device)
        self.status = pkv.new_status(device)
        self.saved = {}
        self.swap_bytes = 0
        self.scale = 1.0 / np.sqrt(cfg.D)
        self.ws = torch.empty(pkv.pkv_decode_workspace_bytes(
            cfg.max_running, cfg.Hq, cfg.D, cfg.prompt_max + cfg.out_cap + cfg.chunk),
            dtype=torch.uint8, device=device)
        self.pws = None  # prefill work items, sized per call

    def run(self, ev, values):
        torch, pkv, cfg, dev = self.torch, self.pkv, self.cfg, self.dev
        shape = (cfg.Hkv, cfg.block_size, cfg.D)
        for kind, rid, blocks in ev.ops:
            bl = torch.tensor(blocks, dtype=torch.int32, device=dev)
            if kind == "swap_out":
                kb = torch.empty((len(blocks),) + shape, dtype=torch.bfloat16).pin_memory()
                vb = torch.empty_like(kb).pin_memory()
                pkv.pkv_swap_blocks(self.k_cache, self.v_cache, bl, kb, vb, True,
                                    status=self.status)
                self.saved[rid] = (kb, vb)
            else:
                kb, vb = self.saved.pop(rid)
                pkv.pkv_swap_blocks(self.k_cache, self.v_cache, bl, kb, vb, False,
                                    status=self.status)
            self.swap_bytes += 2 * kb.numel() * 2
        pre, dec, q, k, v, slots, meta = iteration_inputs(cfg, ev, values)
        pre_out = dec_out = None
        if len(slots):
            pkv.pkv_kv_append(to_dev_bf16(k, dev), to_dev_bf16(v, dev),
                              torch.from_numpy(slots).to(dev), self.k_cache, self.v_cache,
                              status=self.status)
        qd = to_dev_bf16(q, dev)
        n_pre = int(meta["cu"][-1])
        if pre:
            tables, lens = meta["prefill"]
            need = pkv.pkv_prefill_workspace_bytes(len(pre), n_pre, cfg.Hq, cfg.D)
            if self.pws is None or self.pws.numel() < need:
                self.pws = torch.empty(need, dtype=torch.uint8, device=dev)
            pre_out = torch.empty(n_pre, cfg.Hq, cfg.D, dtype=torch.bfloat16, device=dev)
            pkv.pkv_paged_attention_prefill(
                pre_out, qd[:n_pre], torch.from_numpy(meta["cu"]).to(dev),
                torch.from_numpy(lens).to(dev), self.k_cache, self.v_cache,
                torch.from_numpy(tables).to(dev), int(np.diff(meta["cu"]).max()),
                int(lens.max()), self.scale, self.pws, status=self.status)
        if dec:
            tables, lens = meta["decode"]
            dec_out = torch.empty(len(dec), cfg.Hq, cfg.D, dtype=torch.bfloat16, device=dev)
            pkv.pkv_paged_attention_decode(
                dec_out, qd[n_pre:], self.k_cache, self.v_cache, torch.from_numpy(tables).to(dev),
                torch.from_numpy(lens).to(dev), int(lens.max()), self.scale, self.ws,
                status=self.status)
        torch.cuda.synchronize()  # the pinned swap buffers of swap-ins may be released now
        return pre, dec, pre_out, dec_out
