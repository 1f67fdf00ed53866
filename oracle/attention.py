"""Reference attention over paged K/V, in fp64.

"Deep Dive: continuous batching" (worksonmygpu.com), section *Selective
batching*: attention computes ``softmax(Q K^T / sqrt(d_k)) V`` for each token
over its own request's prior tokens only, request by request.  Here each
request's keys and values are first rebuilt as contiguous arrays from the
paged cache through its block table ("Batching, Scheduling, and Paging",
section *PagedAttention*), then the definition is evaluated directly:
scores, subtraction of the row maximum, exponentials, normalisation, and the
weighted sum of values.

Readings where the pages are silent:

* the scale is a parameter; the workloads pass ``1/sqrt(D)``;
* a decode query is the sequence's newest token, whose key and value are
  already in the cache, so it attends to all ``context_len`` tokens, itself
  included;
* a prefill chunk of ``c`` queries is the last ``c`` tokens of its sequence:
  query ``i`` sits at position ``L - c + i`` and attends to keys
  ``0 .. L - c + i`` (causal);
* query head ``h`` reads key/value head ``h // (Hq / Hkv)`` (grouped heads).

Inputs are bf16 bit patterns widened exactly to float64; outputs are float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).
"""

from __future__ import annotations

import numpy as np

from .cache import gather


def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> exact float64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float, limits) -> np.ndarray:
    """``softmax(scale * q K^T) V`` where row ``i`` sees keys ``0 .. limits[i]-1``.

    ``q``: [n, D], ``K``/``V``: [L, D], all float64.  Returns [n, D].
    """
    limits = np.asarray(limits, dtype=np.int64)
    n, L = q.shape[0], K.shape[0]
    visible = np.arange(L)[None, :] < limits[:, None]
    scores = np.where(visible, scale * (q @ K.T), -np.inf)
    m = scores.max(axis=1, keepdims=True)
    w = np.where(visible, np.exp(scores - m), 0.0)
    return (w @ V) / w.sum(axis=1, keepdims=True)


def _group(Hq: int, Hkv: int) -> int:
    assert Hq % Hkv == 0, "query heads must be a multiple of key/value heads"
    return Hq // Hkv


def decode(q_bits, k_cache, v_cache, block_tables, context_lens, block_size: int,
           scale: float, seqs=None) -> np.ndarray:
    """One query per sequence at position ``L-1`` attending keys ``0 .. L-1``.

    ``q_bits``: [S, Hq, D] bf16 bits; caches: [N, Hkv, B, D] bf16 bits.
    ``seqs`` restricts the work to a subset of sequences (others stay NaN).
    """
    S, Hq, D = q_bits.shape
    Hkv = k_cache.shape[1]
    G = _group(Hq, Hkv)
    out = np.full((S, Hq, D), np.nan)
    for s in (range(S) if seqs is None else seqs):
        L = int(context_lens[s])
        K = widen_bf16(gather(k_cache, block_tables[s], L, block_size))
        V = widen_bf16(gather(v_cache, block_tables[s], L, block_size))
        q = widen_bf16(q_bits[s])
        for h in range(Hq):
            out[s, h] = attend(q[h][None, :], K[:, h // G], V[:, h // G], scale, [L])[0]
    return out


def prefill(q_bits, cu_q_lens, context_lens, k_cache, v_cache, block_tables,
            block_size: int, scale: float, seqs=None) -> np.ndarray:
    """Causal attention for prompt chunks packed by ``cu_q_lens``.

    Sequence ``s`` owns query rows ``cu_q_lens[s] .. cu_q_lens[s+1]-1``; its
    ``c`` queries are its last ``c`` tokens out of ``context_lens[s]``.
    """
    Tq, Hq, D = q_bits.shape
    Hkv = k_cache.shape[1]
    G = _group(Hq, Hkv)
    out = np.full((Tq, Hq, D), np.nan)
    S = len(context_lens)
    for s in (range(S) if seqs is None else seqs):
        a, b = int(cu_q_lens[s]), int(cu_q_lens[s + 1])
        c, L = b - a, int(context_lens[s])
        if c == 0:
            continue
        assert c <= L, "a chunk cannot be longer than its context"
        K = widen_bf16(gather(k_cache, block_tables[s], L, block_size))
        V = widen_bf16(gather(v_cache, block_tables[s], L, block_size))
        q = widen_bf16(q_bits[a:b])
        limits = L - c + np.arange(c) + 1
        for h in range(Hq):
            out[a:b, h] = attend(q[:, h], K[:, h // G], V[:, h // G], scale, limits)
    return out
