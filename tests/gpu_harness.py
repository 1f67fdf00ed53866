"""Sets a workload up on the GPU through the library's own API.

The library's allocator hands out the blocks, ``pkv_kv_append`` writes the
tokens into NaN-poisoned pools, and the decode/prefill calls run on them.
Nothing here computes attention.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

import paged_kv_cache_281_gb300 as pkv
from workloads import BF16_NAN


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
