"""Iteration-level scheduling with a pool too small for the worst case.

"Batching, Scheduling, and Paging" (section PagedAttention): when HBM runs
out, a request is evicted — swapped to CPU memory, or discarded and
recomputed later. This scheduler runs a continuous-batching trace against an
undersized pool and evicts the most recently admitted running request when an
append cannot get its blocks, in one of two modes:

* ``swap``: the victim's blocks are copied out and handed back; it resumes
  (first in, first out, before new admissions) when its blocks fit again;
* ``recompute``: the victim's blocks are freed and it re-enters the queue; on
  resumption it re-prefills every token it had cached, with the same values.

The scheduler only decides; an allocator adapter (``LibraryAllocator`` here
over the library's allocator, or the oracle's model of it) answers the block
requests, and two executors (``workloads.device.GpuRunner`` on the GPU, the
oracle's runner on the CPU) replay the resulting events. It draws the
arrivals from the trace's seeded streams and computes no attention.
"""

from __future__ import annotations

from collections import deque
from dataclasses import dataclass, field

import numpy as np

from workloads import TraceConfig, generator, normal_bf16_from


class OutOfBlocks(Exception):
    pass


class LibraryAllocator:
    """Adapter over paged_kv_cache_281_gb300.BlockAllocator."""

    def __init__(self, num_blocks, block_size):
        import paged_kv_cache_281_gb300 as pkv
        from paged_kv_cache_281_gb300._lib import PKV_ENOMEM
        self.pkv, self.enomem = pkv, PKV_ENOMEM
        self.a = pkv.BlockAllocator(num_blocks, block_size)

    def _guard(self, fn, *args):
        try:
            return fn(*args)
        except self.pkv.PagedKVError as e:
            if e.code == self.enomem:
                raise OutOfBlocks(str(e)) from None
            raise

    def create(self):
        return self.a.seq_create()

    def append(self, sid, n):
        slots, pair = self._guard(self.a.seq_append_slots, sid, n)
        assert pair is None
        return [int(x) for x in slots]

    def free(self, sid):
        self.a.seq_free(sid)

    def create_cached(self, tokens):
        return self.a.seq_create_cached(tokens)

    def append_tokens(self, sid, tokens):
        slots, pair = self._guard(self.a.seq_append_tokens, sid, tokens)
        assert pair is None
        return [int(x) for x in slots]

    def num_cached(self):
        return self.a.num_cached_blocks()

    def swap_out(self, sid):
        return self.a.seq_swap_out(sid)

    def swap_in(self, sid):
        return self._guard(self.a.seq_swap_in, sid)

    def table(self, sid):
        return self.a.seq_block_table(sid)

    def num_free(self):
        return self.a.num_free_blocks()


class TokenValues:
    """Per-request q/k/v values drawn in position order and kept, so that a
    recomputed request re-appends exactly the values it had."""

    def __init__(self, cfg: TraceConfig):
        self.cfg = cfg
        self.W = (cfg.Hq + 2 * cfg.Hkv) * cfg.D
        self.rows: dict[int, np.ndarray] = {}
        self.gens: dict[int, np.random.Generator] = {}

    def get(self, rid, start, n):
        have = self.rows.get(rid, np.zeros((0, self.W), np.uint16))
        if start + n > have.shape[0]:
            g = self.gens.setdefault(rid, generator(self.cfg.seed, 1, rid))
            more = normal_bf16_from(g, (start + n - have.shape[0], self.W))
            have = np.concatenate([have, more])
            self.rows[rid] = have
        return have[start:start + n]


@dataclass
class Req:
    rid: int
    prompt: int
    out: int
    sid: int = -1
    pos: int = 0              # tokens in the cache
    prefill_to: int = 0       # tokens to (re-)prefill before decoding
    generated: int = 0
    state: str = "waiting"    # waiting | running | swapped


@dataclass
class Event:
    """What one iteration did, in the order the host decided it."""

    index: int
    ops: list = field(default_factory=list)      # ("swap_in"|"swap_out", rid, blocks)
    work: list = field(default_factory=list)     # (rid, sid, start, n, kind, slots)
    tables: dict = field(default_factory=dict)   # rid -> block table after this step's appends
    finished: list = field(default_factory=list)
    preempted: int = 0


class PreemptingScheduler:
    """``watermark`` blocks are kept free at admission (new requests wait
    rather than take the last blocks the running ones will grow into)."""

    def __init__(self, cfg: TraceConfig, num_blocks: int, mode: str, alloc, watermark: int = 0):
        assert mode in ("swap", "recompute")
        self.cfg, self.mode, self.alloc = cfg, mode, alloc
        self.num_blocks = num_blocks
        self.watermark = watermark
        self.g = generator(cfg.seed, 0)
        self.waiting: deque = deque()
        self.swapped: deque = deque()
        self.running: list[Req] = []
        self.next_rid = 0

    def _evict(self, victim: Req, ev: Event):
        self.running.remove(victim)
        ev.preempted += 1
        if self.mode == "swap":
            blocks = self.alloc.swap_out(victim.sid)
            ev.ops.append(("swap_out", victim.rid, blocks))
            victim.state = "swapped"
            self.swapped.append(victim)
        else:
            self.alloc.free(victim.sid)
            victim.prefill_to = max(victim.prompt, victim.pos)
            victim.pos = 0
            victim.sid = -1
            victim.state = "waiting"
            self.waiting.appendleft(victim)

    def step(self, it: int) -> Event:
        cfg, B = self.cfg, self.cfg.block_size
        ev = Event(index=it)
        for _ in range(int(self.g.poisson(cfg.arrival_rate))):
            prompt = int(self.g.integers(cfg.prompt_min, cfg.prompt_max, endpoint=True))
            out = int(min(cfg.out_cap, self.g.geometric(1.0 / cfg.out_mean)))
            self.waiting.append(Req(self.next_rid, prompt, out, prefill_to=prompt))
            self.next_rid += 1
        # resume swapped requests first, then admit queued ones
        while self.swapped and len(self.running) < cfg.max_running:
            r = self.swapped[0]
            try:
                blocks = self.alloc.swap_in(r.sid)
            except OutOfBlocks:
                break
            self.swapped.popleft()
            ev.ops.append(("swap_in", r.rid, blocks))
            r.state = "running"
            self.running.append(r)
        while (self.waiting and not self.swapped and len(self.running) < cfg.max_running
               and self.alloc.num_free() - self.watermark
               >= -(-min(cfg.chunk, self.waiting[0].prefill_to) // B)):
            r = self.waiting.popleft()
            r.sid = self.alloc.create()
            r.state = "running"
            self.running.append(r)
        # one step of work per running request, evicting the newest on shortage
        i = 0
        while i < len(self.running):
            r = self.running[i]
            if r.pos < r.prefill_to:
                n, kind = min(cfg.chunk, r.prefill_to - r.pos), "prefill"
            else:
                n, kind = 1, "decode"
            while True:
                try:
                    slots = self.alloc.append(r.sid, n)
                    break
                except OutOfBlocks:
                    victim = self.running[-1]
                    self._evict(victim, ev)
                    if victim is r:
                        slots = None
                        break
            if slots is None:
                continue  # r itself was evicted; the list shrank
            ev.work.append((r.rid, r.sid, r.pos, n, kind, slots))
            r.pos += n
            if kind == "prefill":
                if r.pos == r.prefill_to and r.generated == 0:
                    r.generated = 1
            else:
                r.generated += 1
            i += 1
        ev.tables = {w[0]: self.alloc.table(w[1]) for w in ev.work}
        for r in list(self.running):
            if r.generated >= r.out:
                self.alloc.free(r.sid)
                self.running.remove(r)
                ev.finished.append(r.rid)
        return ev


def small_trace_config(iterations=60) -> TraceConfig:
    """A trace small enough to keep every request's values and check often."""
    return TraceConfig(iterations=iterations, arrival_rate=4.0, prompt_min=16, prompt_max=200,
                       chunk=128, out_mean=40.0, out_cap=160, max_running=48, Hq=16, Hkv=4, D=128,
                       block_size=16, seed=0x281 + 50)


def run_schedule(cfg, num_blocks, mode, alloc_factory, watermark=0):
    """All events of the trace for one allocator."""
    sched = PreemptingScheduler(cfg, num_blocks, mode, alloc_factory(num_blocks, cfg.block_size),
                                watermark)
    return [sched.step(it) for it in range(cfg.iterations)], sched


def iteration_inputs(cfg, ev: Event, values: TokenValues):
    """Per-token q/k/v of an iteration (prefill rows first, then decode rows),
    the slots, and the prefill/decode metadata."""
    pre = [w for w in ev.work if w[4] == "prefill"]
    dec = [w for w in ev.work if w[4] == "decode"]
    order = pre + dec
    rows = [values.get(w[0], w[2], w[3]) for w in order]
    W = values.W
    vals = np.concatenate(rows) if rows else np.zeros((0, W), np.uint16)
    T = vals.shape[0]
    qd, kd = cfg.Hq * cfg.D, cfg.Hkv * cfg.D
    q = np.ascontiguousarray(vals[:, :qd]).reshape(T, cfg.Hq, cfg.D)
    k = np.ascontiguousarray(vals[:, qd:qd + kd]).reshape(T, cfg.Hkv, cfg.D)
    v = np.ascontiguousarray(vals[:, qd + kd:]).reshape(T, cfg.Hkv, cfg.D)
    slots = np.asarray([s for w in order for s in w[5]], dtype=np.int32)
    width = max([len(ev.tables[w[0]]) for w in order] + [1])
    meta = {}
    for name, ws in (("prefill", pre), ("decode", dec)):
        tables = np.zeros((len(ws), width), dtype=np.int32)
        for i, w in enumerate(ws):
            t = ev.tables[w[0]]
            tables[i, :len(t)] = t
        lens = np.asarray([w[2] + w[3] for w in ws], dtype=np.int32)
        meta[name] = (tables, lens)
    meta["cu"] = np.concatenate([[0], np.cumsum([w[3] for w in pre])]).astype(np.int32)
    return pre, dec, q, k, v, slots, meta
