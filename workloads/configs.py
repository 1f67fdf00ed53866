"""Synthetic workloads shaped like the pages' serving scenarios.

Each workload is a *logical* description: sequence lengths, the seeded order
in which physical blocks are handed out, and the bf16 values of every token's
query, key and value.  Which physical block a token lands in is decided by a
block allocator (the library's, or the oracle's model of it); this module
decides nothing about paging and computes no attention.

Named workloads (seed ``0x281 + index``):

1. ``tiny``            — 4 sequences, cached lengths {5,17,33,64}, 8/8 heads,
                         D=64, B=16, a 64-block pool handed out in a seeded
                         random order; one token appended per sequence, then
                         one decode step.
2. ``llama2_7b_mha``   — 64 sequences, 32/32 heads, D=128, lengths U[128,2048].
3. ``llama3_8b_gqa``   — 256 sequences, 32/8 heads, D=128, lengths log-normal
                         (median 1024, sigma 0.8) clipped to [16, 8192].
4. ``shared_prefix``   — 64 prompts x 4 samples sharing a 1024-token prefix
                         (variant ``a``) or 1032 tokens (variant ``b``, whose last
                         shared block is half full), tails U[0, 512].
5. ``trace``           — 200 iterations of iteration-level scheduling: Poisson(8)
                         arrivals, prompts U[32,1024] in chunks of <=512,
                         outputs Geometric(1/256) capped at 1536, <=256 running,
                         64/8 heads, D=128.

Lengths in configs 2 and 3 are the lengths the decode step attends over: they
include the token appended in that step.
"""

from __future__ import annotations

import math
from collections import deque
from dataclasses import dataclass, field

import numpy as np

from .rng import generator, normal_bf16_from

SEED_BASE = 0x281


def pool_blocks(lengths, block_size: int, slack: float = 1.1) -> int:
    """Pool size rule: the blocks the lengths need, plus 10% free."""
    need = sum(-(-int(n) // block_size) for n in lengths)
    return int(math.ceil(slack * need))


@dataclass
class DecodeWorkload:
    """A decode step over a ragged batch.

    ``context_lens[s]`` counts the tokens sequence ``s`` attends over, the
    newly appended one included.  ``k``/``v`` hold every token of every
    sequence, packed by ``cu_lens`` (``k[cu_lens[s] + j]`` is token ``j`` of
    sequence ``s``), as bf16 bits of shape ``[sum(L), Hkv, D]``.  The last
    token of each sequence is the one appended by the step itself.
    """

    name: str
    S: int
    Hq: int
    Hkv: int
    D: int
    block_size: int
    num_blocks: int
    context_lens: np.ndarray      # int32 [S]
    free_order: np.ndarray        # int32 [num_blocks], a permutation
    q: np.ndarray                 # uint16 [S, Hq, D]
    k: np.ndarray                 # uint16 [sum L, Hkv, D]
    v: np.ndarray                 # uint16 [sum L, Hkv, D]
    scale: float
    seed: int = 0

    @property
    def cu_lens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.context_lens, dtype=np.int64)])

    @property
    def total_tokens(self) -> int:
        return int(self.context_lens.sum())

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.S else 0

    @property
    def max_blocks_per_seq(self) -> int:
        return max(1, -(-self.max_context_len // self.block_size))

    def kv_bytes(self) -> int:
        """Bytes of K and V the decode step must read once (algorithmic)."""
        return self.total_tokens * 2 * self.Hkv * self.D * 2


def make_decode_workload(name: str, context_lens, Hq: int, Hkv: int, D: int,
                         block_size: int, seed: int, num_blocks: int | None = None,
                         slack: float = 1.1) -> DecodeWorkload:
    lens = np.asarray(context_lens, dtype=np.int32)
    S = int(lens.shape[0])
    if num_blocks is None:
        num_blocks = max(1, pool_blocks(lens, block_size, slack))
    g = generator(seed, 1)
    free_order = g.permutation(num_blocks).astype(np.int32)
    total = int(lens.sum())
    q = normal_bf16_from(generator(seed, 2), (S, Hq, D))
    k = normal_bf16_from(generator(seed, 3), (total, Hkv, D))
    v = normal_bf16_from(generator(seed, 4), (total, Hkv, D))
    return DecodeWorkload(name=name, S=S, Hq=Hq, Hkv=Hkv, D=D, block_size=block_size,
                          num_blocks=int(num_blocks), context_lens=lens,
                          free_order=free_order, q=q, k=k, v=v,
                          scale=1.0 / math.sqrt(D), seed=seed)


def lognormal_lengths(g: np.random.Generator, n: int, median: float, sigma: float,
                      lo: int, hi: int) -> np.ndarray:
    """round(exp(ln(median) + sigma*z)), clipped to [lo, hi]."""
    z = g.standard_normal(n)
    return np.clip(np.rint(np.exp(math.log(median) + sigma * z)), lo, hi).astype(np.int32)


def config1() -> DecodeWorkload:
    seed = SEED_BASE + 1
    cached = np.array([5, 17, 33, 64], dtype=np.int32)
    return make_decode_workload("tiny", cached + 1, Hq=8, Hkv=8, D=64, block_size=16,
                                seed=seed, num_blocks=64)


def config2(S: int = 64) -> DecodeWorkload:
    seed = SEED_BASE + 2
    lens = generator(seed, 0).integers(128, 2048, size=S, endpoint=True).astype(np.int32)
    return make_decode_workload("llama2_7b_mha", lens, Hq=32, Hkv=32, D=128,
                                block_size=16, seed=seed)


def config3_lengths(S: int = 256) -> np.ndarray:
    return lognormal_lengths(generator(SEED_BASE + 3, 0), S, 1024.0, 0.8, 16, 8192)


def config3(S: int = 256) -> DecodeWorkload:
    seed = SEED_BASE + 3
    return make_decode_workload("llama3_8b_gqa", config3_lengths(S), Hq=32, Hkv=8, D=128,
                                block_size=16, seed=seed)


# --------------------------------------------------------------------------
# Config 4: parallel sampling over a shared prompt prefix.


@dataclass
class SharedPrefixWorkload:
    """``n_prompts`` prompts, each with a prefix shared by ``n_samples`` samples.

    Build order (both the library harness and the oracle follow it):
    for each prompt, create a sequence and append the prefix; fork it
    ``n_samples - 1`` times (sample 0 is the original sequence); then, prompt
    by prompt and sample by sample, append each sample's tail.  The decode
    query of sample ``(p, j)`` attends its ``prefix_len + tails[p, j]`` tokens.
    """

    name: str
    n_prompts: int
    n_samples: int
    prefix_len: int
    tails: np.ndarray             # int32 [n_prompts, n_samples]
    Hq: int
    Hkv: int
    D: int
    block_size: int
    num_blocks: int
    free_order: np.ndarray        # int32 [num_blocks]
    prefix_k: np.ndarray          # uint16 [n_prompts, prefix_len, Hkv, D]
    prefix_v: np.ndarray
    tail_k: np.ndarray            # uint16 [sum tails, Hkv, D], packed sample-major
    tail_v: np.ndarray
    q: np.ndarray                 # uint16 [n_prompts * n_samples, Hq, D]
    scale: float

    @property
    def S(self) -> int:
        return self.n_prompts * self.n_samples

    @property
    def context_lens(self) -> np.ndarray:
        return (self.prefix_len + self.tails.reshape(-1)).astype(np.int32)

    @property
    def cu_tails(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.tails.reshape(-1), dtype=np.int64)])

    def logical_kv_bytes(self) -> int:
        return int(self.context_lens.sum()) * 2 * self.Hkv * self.D * 2

    def unique_kv_bytes(self) -> int:
        """Bytes of distinct cached tokens: each prefix once, each tail once."""
        toks = self.n_prompts * self.prefix_len + int(self.tails.sum())
        return toks * 2 * self.Hkv * self.D * 2


def make_shared_prefix_workload(name: str, n_prompts: int, n_samples: int, prefix: int,
                                tail_max: int, Hq: int, Hkv: int, D: int, block_size: int,
                                seed: int, tail_min: int = 0) -> SharedPrefixWorkload:
    B = block_size
    tails = generator(seed, 0).integers(tail_min, tail_max, size=(n_prompts, n_samples),
                                        endpoint=True).astype(np.int32)
    # Every sample may own a copy of the last shared block plus its tail blocks.
    per_prompt = -(-prefix // B)
    need = n_prompts * per_prompt + sum(
        -(-(prefix + int(t)) // B) - prefix // B for t in tails.reshape(-1))
    num_blocks = int(math.ceil(1.1 * need))
    free_order = generator(seed, 1).permutation(num_blocks).astype(np.int32)
    total_tail = int(tails.sum())
    return SharedPrefixWorkload(
        name=name, n_prompts=n_prompts, n_samples=n_samples,
        prefix_len=prefix, tails=tails, Hq=Hq, Hkv=Hkv, D=D, block_size=B,
        num_blocks=num_blocks, free_order=free_order,
        prefix_k=normal_bf16_from(generator(seed, 2), (n_prompts, prefix, Hkv, D)),
        prefix_v=normal_bf16_from(generator(seed, 3), (n_prompts, prefix, Hkv, D)),
        tail_k=normal_bf16_from(generator(seed, 4), (total_tail, Hkv, D)),
        tail_v=normal_bf16_from(generator(seed, 5), (total_tail, Hkv, D)),
        q=normal_bf16_from(generator(seed, 6), (n_prompts * n_samples, Hq, D)),
        scale=1.0 / math.sqrt(D))


def config4(variant: str = "a", n_prompts: int = 64, n_samples: int = 4,
            tail_max: int = 512) -> SharedPrefixWorkload:
    prefix = {"a": 1024, "b": 1032}[variant]
    w = make_shared_prefix_workload(f"shared_prefix_{variant}", n_prompts, n_samples, prefix,
                                    tail_max, Hq=32, Hkv=8, D=128, block_size=16,
                                    seed=SEED_BASE + 4)
    return w


# --------------------------------------------------------------------------
# Config 5: an iteration-level scheduling trace.


@dataclass
class TraceConfig:
    iterations: int = 200
    arrival_rate: float = 8.0
    prompt_min: int = 32
    prompt_max: int = 1024
    chunk: int = 512
    out_mean: float = 256.0
    out_cap: int = 1536
    max_running: int = 256
    Hq: int = 64
    Hkv: int = 8
    D: int = 128
    block_size: int = 16
    seed: int = SEED_BASE + 5

    @property
    def num_blocks(self) -> int:
        """Worst case: every running request at full prompt + output length."""
        return self.max_running * (-(-(self.prompt_max + self.out_cap) // self.block_size))


@dataclass
class Work:
    """Tokens ``start .. start+n-1`` of request ``rid`` processed this iteration."""

    rid: int
    start: int
    n: int
    kind: str                     # "prefill" or "decode"


@dataclass
class Iteration:
    index: int
    admitted: list[int]           # requests that joined the running set now
    work: list[Work]              # prefill chunks first, then decode tokens
    finished: list[int]           # requests that complete with this iteration
    # per-token values of this iteration, packed in ``work`` order
    q: np.ndarray = field(default=None)   # uint16 [T, Hq, D]
    k: np.ndarray = field(default=None)   # uint16 [T, Hkv, D]
    v: np.ndarray = field(default=None)
    _arrays: tuple = field(default=None, repr=False)

    def arrays(self):
        """(request ids int64 [n], token counts int32 [n], prefill works,
        prefill rows) of ``work`` in order, as the scheduler hands them to
        the engine (computed once)."""
        if self._arrays is None:
            n_pre = sum(1 for w in self.work if w.kind == "prefill")
            self._arrays = (np.array([w.rid for w in self.work], dtype=np.int64),
                            np.array([w.n for w in self.work], dtype=np.int32), n_pre,
                            sum(w.n for w in self.work[:n_pre]))
        return self._arrays

    @property
    def prefill(self) -> list[Work]:
        return [w for w in self.work if w.kind == "prefill"]

    @property
    def decode(self) -> list[Work]:
        return [w for w in self.work if w.kind == "decode"]

    @property
    def num_tokens(self) -> int:
        return sum(w.n for w in self.work)


def trace_iterations(cfg: TraceConfig, with_values: bool = True):
    """Yield the iterations of the continuous-batching trace.

    Each iteration admits queued requests first-come-first-served while fewer
    than ``max_running`` run, gives each running request either its next
    prompt chunk (at most ``chunk`` tokens) or, once its prompt is cached, one
    decode token, and retires requests that have produced ``out_len`` tokens.
    The last prompt chunk yields a request's first output token, so a request
    runs ``out_len - 1`` decode iterations.
    """
    g = generator(cfg.seed, 0)
    W = (cfg.Hq + 2 * cfg.Hkv) * cfg.D
    queue: deque = deque()
    running: dict[int, dict] = {}
    next_rid = 0
    p_geo = 1.0 / cfg.out_mean
    for it in range(cfg.iterations):
        for _ in range(int(g.poisson(cfg.arrival_rate))):
            prompt = int(g.integers(cfg.prompt_min, cfg.prompt_max, endpoint=True))
            out = int(min(cfg.out_cap, g.geometric(p_geo)))
            queue.append((next_rid, prompt, out))
            next_rid += 1
        admitted = []
        while queue and len(running) < cfg.max_running:
            rid, prompt, out = queue.popleft()
            running[rid] = {"prompt": prompt, "out": out, "pos": 0, "generated": 0,
                            "gen": generator(cfg.seed, 1, rid) if with_values else None}
            admitted.append(rid)
        prefill, decode, finished = [], [], []
        for rid, st in running.items():
            if st["pos"] < st["prompt"]:
                n = min(cfg.chunk, st["prompt"] - st["pos"])
                prefill.append(Work(rid, st["pos"], n, "prefill"))
                st["pos"] += n
                if st["pos"] == st["prompt"]:
                    st["generated"] = 1
            else:
                decode.append(Work(rid, st["pos"], 1, "decode"))
                st["pos"] += 1
                st["generated"] += 1
            if st["generated"] >= st["out"]:
                finished.append(rid)
        work = prefill + decode
        itr = Iteration(index=it, admitted=admitted, work=work, finished=finished)
        if with_values:
            T = itr.num_tokens
            vals = np.empty((T, W), dtype=np.uint16)
            o = 0
            for w in work:
                vals[o:o + w.n] = normal_bf16_from(running[w.rid]["gen"], (w.n, W))
                o += w.n
            qd = cfg.Hq * cfg.D
            kd = cfg.Hkv * cfg.D
            itr.q = vals[:, :qd].reshape(T, cfg.Hq, cfg.D)
            itr.k = vals[:, qd:qd + kd].reshape(T, cfg.Hkv, cfg.D)
            itr.v = vals[:, qd + kd:].reshape(T, cfg.Hkv, cfg.D)
        for rid in finished:
            del running[rid]
        yield itr
