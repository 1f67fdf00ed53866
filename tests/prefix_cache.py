"""Requests that share a system prompt, with and without prefix caching.

"Paging the KV Cache" (lecture 6): a system prompt shared by many concurrent
requests can occupy one set of pages referenced by all of them; "Batching,
Scheduling, and Paging" (section Block sharing) calls sharing identical
prefixes across requests the seed of prefix caching. Every request is the
same system prompt followed by its own question, then a few decode steps.
With caching, a request starts from the registered blocks of the prompt's
full blocks and prefills only the rest; without, it prefills everything.
The K/V (and query) values of a position inside the system prompt depend only
on the position, so a cached block holds exactly what the request would have
computed. Test infrastructure; the executors are
``workloads.device.GpuRunner`` and ``oracle.harness.OracleRunner``.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from workloads.schedule import Event
from workloads import generator, normal_bf16_from


@dataclass
class PrefixConfig:
    Hq: int = 16
    Hkv: int = 4
    D: int = 128
    block_size: int = 16
    system_len: int = 200
    question_min: int = 1
    question_max: int = 40
    waves: tuple = ((0, 6), (2, 6), (9, 5))      # (iteration, requests admitted)
    decode_steps: int = 4
    iterations: int = 14
    num_blocks: int = 400
    seed: int = 0x281 + 60
    # sizes the executors need
    max_running: int = 64
    chunk: int = 0

    @property
    def prompt_max(self):
        return self.system_len + self.question_max

    @property
    def out_cap(self):
        return self.decode_steps + 1


class PrefixValues:
    """Per-position values: a system-prompt position's row depends only on the
    position; a request's later rows on the request and position."""

    def __init__(self, cfg: PrefixConfig):
        self.cfg = cfg
        self.W = (cfg.Hq + 2 * cfg.Hkv) * cfg.D
        self.system = normal_bf16_from(generator(cfg.seed, 7), (cfg.system_len, self.W))
        self.own: dict[int, np.ndarray] = {}
        self.gens: dict[int, np.random.Generator] = {}

    def get(self, rid, start, n):
        P = self.cfg.system_len
        rows = []
        if start < P:
            rows.append(self.system[start:min(start + n, P)])
        end = start + n
        if end > P:
            a = max(start, P) - P
            have = self.own.get(rid, np.zeros((0, self.W), np.uint16))
            if end - P > have.shape[0]:
                g = self.gens.setdefault(rid, generator(self.cfg.seed, 8, rid))
                have = np.concatenate([have, normal_bf16_from(g, (end - P - have.shape[0],
                                                                  self.W))])
                self.own[rid] = have
            rows.append(have[a:end - P])
        return np.concatenate(rows)


def prefix_schedule(cfg: PrefixConfig, alloc, cached: bool):
    """The events of the workload: per iteration the admitted requests' prompts
    (from the first uncached token when ``cached``), one decode token for every
    earlier request, and completions. Returns (events, cached tokens per request)."""
    g = generator(cfg.seed, 9)
    system = g.integers(0, 32000, size=cfg.system_len).tolist()
    arrivals = {it: n for it, n in cfg.waves}
    running = {}          # rid -> [sid, pos, decodes left]
    hits = {}
    next_rid = 0
    events = []
    for it in range(cfg.iterations):
        ev = Event(index=it)
        for r in list(running):
            sid, pos, left = running[r]
            slots = alloc.append_tokens(sid, [int(g.integers(0, 32000))])
            ev.work.append((r, sid, pos, 1, "decode", slots))
            running[r] = [sid, pos + 1, left - 1]
        for _ in range(arrivals.get(it, 0)):
            q = int(g.integers(cfg.question_min, cfg.question_max, endpoint=True))
            tokens = system + g.integers(0, 32000, size=q).tolist()
            if cached:
                sid, n_cached = alloc.create_cached(tokens)
            else:
                sid, n_cached = alloc.create(), 0
            slots = alloc.append_tokens(sid, tokens[n_cached:])
            ev.work.insert(sum(1 for w in ev.work if w[4] == "prefill"),
                           (next_rid, sid, n_cached, len(tokens) - n_cached, "prefill", slots))
            running[next_rid] = [sid, len(tokens), cfg.decode_steps]
            hits[next_rid] = n_cached
            next_rid += 1
        ev.tables = {w[0]: alloc.table(w[1]) for w in ev.work}
        for r in list(running):
            if running[r][2] == 0:
                alloc.free(running[r][0])
                ev.finished.append(r)
                del running[r]
        events.append(ev)
    return events, hits
