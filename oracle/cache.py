"""Reference cache operations on the paged layout, element by element.

Layout (a reading: the pages fix no layout): the key pool and the value pool
are separate arrays of bf16 bit patterns shaped ``[num_blocks, Hkv, B, D]``;
token ``j`` of a sequence with block table ``bt`` lives in physical block
``bt[j // B]`` at offset ``j % B`` ("Batching, Scheduling, and Paging",
section *PagedAttention*: the block table maps logical to physical blocks).

TEST INFRASTRUCTURE ONLY (see the package docstring).
"""

from __future__ import annotations

import numpy as np


def append(k_cache: np.ndarray, v_cache: np.ndarray, k_new: np.ndarray, v_new: np.ndarray,
           slot_mapping, block_size: int) -> None:
    """Write token ``t``'s key/value rows into slot ``slot_mapping[t]``; -1 skips."""
    for t, slot in enumerate(slot_mapping):
        slot = int(slot)
        if slot < 0:
            continue
        blk, off = divmod(slot, block_size)
        k_cache[blk, :, off, :] = k_new[t]
        v_cache[blk, :, off, :] = v_new[t]


def block_copy(k_cache: np.ndarray, v_cache: np.ndarray, pairs) -> None:
    """Copy whole physical blocks ``src -> dst`` for each pair, in order."""
    for src, dst in pairs:
        k_cache[int(dst)] = k_cache[int(src)]
        v_cache[int(dst)] = v_cache[int(src)]


def gather(cache: np.ndarray, block_table, length: int, block_size: int) -> np.ndarray:
    """A sequence's first ``length`` tokens as a contiguous ``[length, Hkv, D]`` array."""
    out = np.empty((length,) + (cache.shape[1], cache.shape[3]), dtype=cache.dtype)
    for j in range(length):
        out[j] = cache[int(block_table[j // block_size]), :, j % block_size, :]
    return out


def swap_blocks(k_cache: np.ndarray, v_cache: np.ndarray, blocks, k_buf: np.ndarray,
                v_buf: np.ndarray, direction: int) -> None:
    """Whole-block copies between the pools and a contiguous buffer.

    ``direction`` 0: buffer slot ``i`` receives block ``blocks[i]`` (swap-out);
    1: block ``blocks[i]`` receives buffer slot ``i`` (swap-in).
    """
    for i, b in enumerate(blocks):
        b = int(b)
        if direction == 0:
            k_buf[i] = k_cache[b]
            v_buf[i] = v_cache[b]
        else:
            k_cache[b] = k_buf[i]
            v_cache[b] = v_buf[i]
