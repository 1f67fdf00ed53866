"""Python binding of the C ABI: argument marshalling only.

Each function carries the name of the C call it wraps and passes tensor data
pointers, sizes and the current CUDA stream straight through; every step of
the computation runs in the library's kernels. Shapes are read from the
tensors:

* ``k_cache``/``v_cache``: bf16 ``[num_blocks, Hkv, block_size, D]``
* ``q``/``out`` (decode): bf16 ``[S, Hq, D]``; (prefill): ``[total_q, Hq, D]``
* ``block_tables``: int32 ``[S, max_blocks_per_seq]``; ``context_lens``: int32 ``[S]``
* ``slot_mapping``: int32 ``[T]``; ``pairs``: int32 ``[n, 2]``
* ``status``: int32 ``[4]`` on the device (optional)
"""

from __future__ import annotations

import ctypes

import numpy as np
import torch

from ._lib import IterationLayout, PagedKVError, check, lib

__all__ = [
    "IterationStepper",
    "PagedKVError", "pkv_version", "pkv_last_error", "BlockAllocator",
    "pkv_kv_append", "pkv_block_copy", "pkv_swap_blocks", "pkv_decode_workspace_bytes",
    "pkv_paged_attention_decode", "pkv_paged_attention_decode_noalloc",
    "NOALLOC_SCRATCH_BYTES", "pkv_prefill_workspace_bytes",
    "pkv_paged_attention_prefill", "pkv_status_reset", "pkv_check_status",
    "pkv_debug_set_wait", "new_status", "new_fp8_pools", "pkv_kv_append_fp8",
    "pkv_paged_attention_decode_fp8", "pkv_decode_shared_workspace_bytes",
    "pkv_paged_attention_decode_shared", "IterationLayout", "iteration_layout_bytes",
    "pkv_iteration_run", "pkv_iteration_step",
]


def pkv_version() -> int:
    return lib().pkv_version()


def pkv_last_error() -> str:
    return lib().pkv_last_error().decode()


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check_device(name: str, index: int, current: int) -> None:
    # The library launches on the current device and builds its tile maps
    # over the pointers it is given; a tensor on another GPU would be read
    # through the wrong device's address space, so refuse it here.
    if index != current:
        raise ValueError(f"{name} lives on cuda:{index} but the current device is "
                         f"cuda:{current}; call under torch.cuda.device({index})")


def _dev(t: torch.Tensor, name: str, dtype: torch.dtype, ndim: int | None = None,
         cur: int | None = None):
    """Checks one tensor argument; ``cur`` is the current device (queried when
    not given, so a call with many tensors can query it once)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must live on a CUDA device")
    _check_device(name, t.device.index, torch.cuda.current_device() if cur is None else cur)
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got shape {tuple(t.shape)}")
    return t


def new_status(device=None) -> torch.Tensor:
    """A zeroed device status block (4 int32)."""
    return torch.zeros(4, dtype=torch.int32, device=device or "cuda")


# ---------------------------------------------------------------- allocator

class BlockAllocator:
    """The library's host block allocator (``pkv_alloc_*`` / ``pkv_seq_*``)."""

    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        self._h = ctypes.c_void_p()
        order = None
        if free_order is not None:
            self._order = np.ascontiguousarray(free_order, dtype=np.int32)
            order = self._order.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        check(lib().pkv_alloc_create(int(num_blocks), int(block_size), order,
                                     ctypes.byref(self._h)))
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)

    def close(self) -> None:
        if self._h:
            lib().pkv_alloc_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def seq_create(self) -> int:
        out = ctypes.c_int64()
        check(lib().pkv_seq_create(self._h, ctypes.byref(out)))
        return out.value

    def seq_fork(self, parent: int) -> int:
        out = ctypes.c_int64()
        check(lib().pkv_seq_fork(self._h, int(parent), ctypes.byref(out)))
        return out.value

    def seq_append_slots(self, seq: int, n: int):
        """Returns ``(slots int32[n], (src, dst) or None)``."""
        slots = np.empty(max(int(n), 1), dtype=np.int32)
        pair = np.zeros(2, dtype=np.int32)
        ncow = ctypes.c_int32()
        check(lib().pkv_seq_append_slots(
            self._h, int(seq), int(n), slots.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
            pair.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), ctypes.byref(ncow)))
        return slots[:int(n)], ((int(pair[0]), int(pair[1])) if ncow.value else None)

    def seq_append_tokens(self, seq: int, token_ids):
        """``seq_append_slots`` that also records the token ids for the prefix cache."""
        ids = np.ascontiguousarray(token_ids, dtype=np.int32)
        n = int(ids.shape[0])
        slots = np.empty(max(n, 1), dtype=np.int32)
        pair = np.zeros(2, dtype=np.int32)
        ncow = ctypes.c_int32()
        check(lib().pkv_seq_append_tokens(
            self._h, int(seq), ids.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), n,
            slots.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
            pair.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), ctypes.byref(ncow)))
        return slots[:n], ((int(pair[0]), int(pair[1])) if ncow.value else None)

    def seq_create_cached(self, token_ids):
        """A new sequence starting with the cached blocks of ``token_ids``'s
        prefix; returns ``(seq, n_cached)``."""
        ids = np.ascontiguousarray(token_ids, dtype=np.int32)
        sid, nc = ctypes.c_int64(), ctypes.c_int32()
        check(lib().pkv_seq_create_cached(self._h, ids.ctypes.data_as(
            ctypes.POINTER(ctypes.c_int32)), int(ids.shape[0]), ctypes.byref(sid),
            ctypes.byref(nc)))
        return sid.value, nc.value

    def num_cached_blocks(self) -> int:
        out = ctypes.c_int32()
        check(lib().pkv_num_cached_blocks(self._h, ctypes.byref(out)))
        return out.value

    def seq_free(self, seq: int) -> None:
        check(lib().pkv_seq_free(self._h, int(seq)))

    def seq_create_many(self, n: int) -> np.ndarray:
        """``pkv_seq_create_many``: ``n`` new sequences' ids (int64)."""
        out = np.empty(int(n), dtype=np.int64)
        check(lib().pkv_seq_create_many(self._h, int(n), out.ctypes.data))
        return out

    def seq_free_many(self, seqs) -> None:
        """``pkv_seq_free_many``: frees every listed sequence, or none."""
        ids = np.ascontiguousarray(seqs, dtype=np.int64)
        check(lib().pkv_seq_free_many(self._h, ids.ctypes.data, int(ids.shape[0])))

    def seq_len(self, seq: int) -> int:
        out = ctypes.c_int32()
        check(lib().pkv_seq_len(self._h, int(seq), ctypes.byref(out)))
        return out.value

    def seq_block_table(self, seq: int) -> list[int]:
        n = ctypes.c_int32()
        check(lib().pkv_seq_block_table(self._h, int(seq), None, 0, ctypes.byref(n)))
        buf = np.empty(max(n.value, 1), dtype=np.int32)
        check(lib().pkv_seq_block_table(self._h, int(seq),
                                        buf.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                        n.value, ctypes.byref(n)))
        return buf[:n.value].tolist()

    def _blocks_call(self, fn, seq: int) -> list[int]:
        cap = max(1, self.num_blocks)
        buf = np.empty(cap, dtype=np.int32)
        n = ctypes.c_int32()
        check(fn(self._h, int(seq), buf.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), cap,
                 ctypes.byref(n)))
        return buf[:n.value].tolist()

    def seq_swap_out(self, seq: int) -> list[int]:
        """Give the sequence's blocks back (table order); it keeps its length."""
        return self._blocks_call(lib().pkv_seq_swap_out, seq)

    def seq_swap_in(self, seq: int) -> list[int]:
        """Fresh blocks for a swapped-out sequence (PagedKVError PKV_ENOMEM if short)."""
        return self._blocks_call(lib().pkv_seq_swap_in, seq)

    def block_refcount(self, block: int) -> int:
        out = ctypes.c_int32()
        check(lib().pkv_block_refcount(self._h, int(block), ctypes.byref(out)))
        return out.value

    def num_free_blocks(self) -> int:
        out = ctypes.c_int32()
        check(lib().pkv_num_free_blocks(self._h, ctypes.byref(out)))
        return out.value

    def build_block_tables(self, seqs, max_blocks_per_seq: int):
        """Padded int32 ``[n, max_blocks_per_seq]`` tables and ``[n]`` lengths (host)."""
        ids = np.ascontiguousarray(seqs, dtype=np.int64)
        n = ids.shape[0]
        tables = np.empty((max(n, 1), int(max_blocks_per_seq)), dtype=np.int32)
        lens = np.empty(max(n, 1), dtype=np.int32)
        check(lib().pkv_build_block_tables(
            self._h, ids.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), n,
            tables.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), int(max_blocks_per_seq),
            lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))))
        return tables[:n], lens[:n]

    def iteration_prepare(self, seqs, counts, n_prefill: int, max_blocks_per_seq: int, buf):
        """``pkv_iteration_prepare``: every work's appends and the iteration's
        metadata in one call. ``seqs``/``counts`` list the prompt chunks first
        (``n_prefill`` of them), then the decodes (count 1). ``buf`` is a
        host buffer (a numpy array or a CPU, e.g. pinned, torch tensor) of at
        least ``iteration_layout_bytes(...).total_bytes`` bytes. Returns the
        layout; raises PagedKVError (PKV_ENOMEM, nothing changed) with
        ``n_fit`` set to the number of leading works that would fit."""
        ids = np.ascontiguousarray(seqs, dtype=np.int64)
        cnt = np.ascontiguousarray(counts, dtype=np.int32)
        n = int(ids.shape[0])
        if cnt.shape[0] != n or not 0 <= n_prefill <= n:
            raise ValueError("seqs and counts must have the same length >= n_prefill")
        if isinstance(buf, torch.Tensor):
            if buf.is_cuda or not buf.is_contiguous():
                raise ValueError("buf must be contiguous host memory")
            addr, nbytes = buf.data_ptr(), buf.numel() * buf.element_size()
        else:
            if not buf.flags["C_CONTIGUOUS"] or not buf.flags["WRITEABLE"]:
                raise ValueError("buf must be a writable contiguous array")
            addr, nbytes = buf.ctypes.data, buf.nbytes
        layout, fit = IterationLayout(), ctypes.c_int32()
        rc = lib().pkv_iteration_prepare(
            self._h, ids.ctypes.data, cnt.ctypes.data, int(n_prefill),
            n - int(n_prefill), int(max_blocks_per_seq), addr, nbytes, ctypes.byref(layout),
            ctypes.byref(fit))
        if rc != 0:
            err = PagedKVError(rc, pkv_last_error())
            err.n_fit = fit.value
            raise err
        return layout


def pkv_iteration_run(meta, layout, n_prefill: int, n_decode: int, q, k_new, v_new, out, k_cache, v_cache, scale: float, decode_ws, prefill_ws,
                      partition_size: int = 0, status=None, stream=None) -> None:
    """``pkv_iteration_run``: the iteration's copies, appends, prefill and
    decode from one device copy (``meta``, uint8) of the buffer
    ``iteration_prepare`` filled; ``layout`` is what it returned (its
    ``table_width`` is the block tables' row length)."""
    cur = torch.cuda.current_device()
    N, Hkv, B, D = _pool_shape(k_cache, v_cache, cur)
    _dev(meta, "meta", torch.uint8, 1, cur)
    for name, t in (("q", q), ("out", out), ("k_new", k_new), ("v_new", v_new)):
        _dev(t, name, torch.bfloat16, 3, cur)
    _dev(decode_ws, "decode_ws", torch.uint8, 1, cur)
    _dev(prefill_ws, "prefill_ws", torch.uint8, 1, cur)
    T, Hq = int(layout.n_tokens), int(q.shape[1])
    if meta.numel() < layout.total_bytes:
        raise ValueError("meta is shorter than the layout")
    if q.shape != (T, Hq, D) or out.shape != q.shape or k_new.shape != (T, Hkv, D) or \
            v_new.shape != k_new.shape:
        raise ValueError(f"q/out must be [{T}, Hq, {D}] and k_new/v_new [{T}, {Hkv}, {D}]")
    check(lib().pkv_iteration_run(
        meta.data_ptr(), ctypes.byref(layout), int(n_prefill), int(n_decode), q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
        out.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), N, Hq, Hkv, D, B, float(scale),
        int(partition_size), decode_ws.data_ptr(), int(decode_ws.numel()), prefill_ws.data_ptr(),
        int(prefill_ws.numel()), _ptr(status), _stream(stream)))


def pkv_iteration_step(alloc: BlockAllocator, seqs, counts, n_prefill: int,
                       max_blocks_per_seq: int, host_buf, dev_buf, q, k_new, v_new, out, k_cache,
                       v_cache, scale: float, decode_ws, prefill_ws, partition_size: int = 0,
                       status=None, stream=None):
    """``pkv_iteration_step``: ``iteration_prepare`` into ``host_buf`` (a
    pinned CPU uint8 tensor), one asynchronous copy to ``dev_buf`` (a device
    uint8 tensor) and ``pkv_iteration_run``, in one call. Do not reuse
    ``host_buf`` before the copy has completed. Returns the layout; raises
    PagedKVError (PKV_ENOMEM, nothing changed) with ``n_fit`` set."""
    cur = torch.cuda.current_device()
    N, Hkv, B, D = _pool_shape(k_cache, v_cache, cur)
    _dev(dev_buf, "dev_buf", torch.uint8, 1, cur)
    for name, t in (("q", q), ("out", out), ("k_new", k_new), ("v_new", v_new)):
        _dev(t, name, torch.bfloat16, 3, cur)
    _dev(decode_ws, "decode_ws", torch.uint8, 1, cur)
    _dev(prefill_ws, "prefill_ws", torch.uint8, 1, cur)
    if host_buf.is_cuda or host_buf.dtype != torch.uint8 or not host_buf.is_contiguous():
        raise ValueError("host_buf must be a contiguous CPU uint8 tensor (pinned)")
    ids = np.ascontiguousarray(seqs, dtype=np.int64)
    cnt = np.ascontiguousarray(counts, dtype=np.int32)
    n = int(ids.shape[0])
    T, Hq = int(cnt.sum()), int(q.shape[1])
    if cnt.shape[0] != n or not 0 <= n_prefill <= n:
        raise ValueError("seqs and counts must have the same length >= n_prefill")
    if q.shape != (T, Hq, D) or out.shape != q.shape or k_new.shape != (T, Hkv, D) or \
            v_new.shape != k_new.shape:
        raise ValueError(f"q/out must be [{T}, Hq, {D}] and k_new/v_new [{T}, {Hkv}, {D}]")
    layout, fit = IterationLayout(), ctypes.c_int32()
    rc = lib().pkv_iteration_step(
        alloc._h, ids.ctypes.data, cnt.ctypes.data, int(n_prefill), n - int(n_prefill),
        int(max_blocks_per_seq), host_buf.data_ptr(), int(host_buf.numel()),
        dev_buf.data_ptr(), int(dev_buf.numel()), q.data_ptr(), k_new.data_ptr(),
        v_new.data_ptr(), out.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), N, Hq, Hkv, D,
        B, float(scale), int(partition_size), decode_ws.data_ptr(), int(decode_ws.numel()),
        prefill_ws.data_ptr(), int(prefill_ws.numel()), _ptr(status), _stream(stream),
        ctypes.byref(layout), ctypes.byref(fit))
    if rc != 0:
        err = PagedKVError(rc, pkv_last_error())
        err.n_fit = fit.value
        raise err
    return layout


class IterationStepper:
    """``pkv_iteration_step`` bound to one allocator, its pools, the device
    copy of the metadata, the workspaces and the status block: their checks
    are done once, here, and each call checks only that iteration's own
    arguments (ids, counts, the pinned staging buffer, q, k_new, v_new,
    out). The bound tensors are kept alive by the stepper; calls must be made
    with the same current device."""

    def __init__(self, alloc: BlockAllocator, max_blocks_per_seq: int, dev_buf, k_cache, v_cache,
                 scale: float, decode_ws, prefill_ws, partition_size: int = 0, status=None):
        cur = torch.cuda.current_device()
        self._cur = cur
        N, Hkv, B, D = _pool_shape(k_cache, v_cache, cur)
        _dev(dev_buf, "dev_buf", torch.uint8, 1, cur)
        _dev(decode_ws, "decode_ws", torch.uint8, 1, cur)
        _dev(prefill_ws, "prefill_ws", torch.uint8, 1, cur)
        if status is not None:
            _dev(status, "status", torch.int32, 1, cur)
        self._keep = (alloc, dev_buf, k_cache, v_cache, decode_ws, prefill_ws, status)
        self._Hkv, self._D = Hkv, D
        self._head = (alloc._h,)
        self._fixed = (int(max_blocks_per_seq), dev_buf.data_ptr(), int(dev_buf.numel()))
        self._pools = (k_cache.data_ptr(), v_cache.data_ptr(), N)
        self._tail = (B, float(scale), int(partition_size), decode_ws.data_ptr(),
                      int(decode_ws.numel()), prefill_ws.data_ptr(), int(prefill_ws.numel()),
                      _ptr(status))

    def __call__(self, seqs, counts, n_prefill: int, host_buf, q, k_new, v_new, out,
                 stream=None):
        """One iteration (see ``pkv_iteration_step``); returns the layout."""
        cur = self._cur
        if torch.cuda.current_device() != cur:
            raise ValueError(f"the stepper is bound to cuda:{cur}; call it under "
                             f"torch.cuda.device({cur})")
        for name, t in (("q", q), ("out", out), ("k_new", k_new), ("v_new", v_new)):
            _dev(t, name, torch.bfloat16, 3, cur)
        if host_buf.is_cuda or host_buf.dtype != torch.uint8 or not host_buf.is_contiguous():
            raise ValueError("host_buf must be a contiguous CPU uint8 tensor (pinned)")
        ids = np.ascontiguousarray(seqs, dtype=np.int64)
        cnt = np.ascontiguousarray(counts, dtype=np.int32)
        n = int(ids.shape[0])
        Hkv, D = self._Hkv, self._D
        T, Hq = int(cnt.sum()), int(q.shape[1])
        if cnt.shape[0] != n or not 0 <= n_prefill <= n:
            raise ValueError("seqs and counts must have the same length >= n_prefill")
        if q.shape != (T, Hq, D) or out.shape != q.shape or k_new.shape != (T, Hkv, D) or \
                v_new.shape != k_new.shape:
            raise ValueError(f"q/out must be [{T}, Hq, {D}] and k_new/v_new [{T}, {Hkv}, {D}]")
        layout, fit = IterationLayout(), ctypes.c_int32()
        rc = lib().pkv_iteration_step(
            *self._head, ids.ctypes.data, cnt.ctypes.data, int(n_prefill), n - int(n_prefill),
            self._fixed[0], host_buf.data_ptr(), int(host_buf.numel()), self._fixed[1],
            self._fixed[2], q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), out.data_ptr(),
            *self._pools, Hq, Hkv, D, *self._tail, _stream(stream), ctypes.byref(layout),
            ctypes.byref(fit))
        if rc != 0:
            err = PagedKVError(rc, pkv_last_error())
            err.n_fit = fit.value
            raise err
        return layout


def iteration_layout_bytes(n_prefill: int, n_decode: int, n_tokens: int,
                           max_blocks_per_seq: int) -> IterationLayout:
    """``pkv_iteration_layout_bytes``: offsets and size of one iteration's
    metadata buffer."""
    layout = IterationLayout()
    check(lib().pkv_iteration_layout_bytes(int(n_prefill), int(n_decode), int(n_tokens),
                                           int(max_blocks_per_seq), ctypes.byref(layout)))
    return layout


# ---------------------------------------------------------------- GPU calls

def _pool_shape(k_cache: torch.Tensor, v_cache: torch.Tensor, cur: int | None = None):
    _dev(k_cache, "k_cache", torch.bfloat16, 4, cur)
    _dev(v_cache, "v_cache", torch.bfloat16, 4, cur)
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache must have the same shape")
    return tuple(int(x) for x in k_cache.shape)  # N, Hkv, B, D


def pkv_status_reset(status: torch.Tensor, stream=None) -> None:
    _dev(status, "status", torch.int32, 1)
    check(lib().pkv_status_reset(status.data_ptr(), _stream(stream)))


def pkv_check_status(status: torch.Tensor, stream=None) -> None:
    """Raises PagedKVError (PKV_ETIMEOUT / PKV_EDEVICE) if a kernel recorded one."""
    _dev(status, "status", torch.int32, 1)
    check(lib().pkv_check_status(status.data_ptr(), _stream(stream)))


def pkv_debug_set_wait(force_timeout: bool, timeout_ns: int = 0) -> None:
    check(lib().pkv_debug_set_wait(1 if force_timeout else 0, int(timeout_ns)))


def pkv_kv_append(k_new, v_new, slot_mapping, k_cache, v_cache, status=None, stream=None) -> None:
    cur = torch.cuda.current_device()
    N, Hkv, B, D = _pool_shape(k_cache, v_cache, cur)
    _dev(k_new, "k_new", torch.bfloat16, 3, cur)
    _dev(v_new, "v_new", torch.bfloat16, 3, cur)
    _dev(slot_mapping, "slot_mapping", torch.int32, 1, cur)
    T = int(slot_mapping.shape[0])
    if k_new.shape != (T, Hkv, D) or v_new.shape != (T, Hkv, D):
        raise ValueError(f"k_new/v_new must be [{T}, {Hkv}, {D}]")
    check(lib().pkv_kv_append(k_new.data_ptr(), v_new.data_ptr(), slot_mapping.data_ptr(), T,
                              k_cache.data_ptr(), v_cache.data_ptr(), N, Hkv, D, B,
                              _ptr(status), _stream(stream)))


def pkv_block_copy(k_cache, v_cache, pairs, status=None, stream=None) -> None:
    cur = torch.cuda.current_device()
    N, Hkv, B, D = _pool_shape(k_cache, v_cache, cur)
    _dev(pairs, "pairs", torch.int32, 2, cur)
    if pairs.shape[1] != 2:
        raise ValueError("pairs must be [n, 2]")
    check(lib().pkv_block_copy(k_cache.data_ptr(), v_cache.data_ptr(), pairs.data_ptr(),
                               int(pairs.shape[0]), N, Hkv, D, B, _ptr(status), _stream(stream)))


def pkv_swap_blocks(k_cache, v_cache, blocks, k_buf, v_buf, to_buffer: bool, status=None,
                    stream=None) -> None:
    """Copy whole blocks between the pools and ``k_buf``/``v_buf`` (device or
    pinned host tensors shaped ``[n, Hkv, B, D]``)."""
    N, Hkv, B, D = _pool_shape(k_cache, v_cache)
    _dev(blocks, "blocks", torch.int32, 1)
    n = int(blocks.shape[0])
    for name, t in (("k_buf", k_buf), ("v_buf", v_buf)):
        if t.dtype != torch.bfloat16 or not t.is_contiguous() or t.shape != (n, Hkv, B, D):
            raise ValueError(f"{name} must be a contiguous bf16 [{n}, {Hkv}, {B}, {D}] tensor")
    check(lib().pkv_swap_blocks(k_cache.data_ptr(), v_cache.data_ptr(), blocks.data_ptr(), n, N,
                                Hkv, D, B, k_buf.data_ptr(), v_buf.data_ptr(),
                                1 if to_buffer else 0, _ptr(status), _stream(stream)))


def pkv_decode_workspace_bytes(S: int, Hq: int, D: int, max_context_len: int,
                               partition_size: int = 0) -> int:
    out = ctypes.c_size_t()
    check(lib().pkv_decode_workspace_bytes(int(S), int(Hq), int(D), int(max_context_len),
                                           int(partition_size), ctypes.byref(out)))
    return out.value


def pkv_paged_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens,
                               max_context_len: int, scale: float, workspace,
                               partition_size: int = 0, status=None, stream=None) -> None:
    cur = torch.cuda.current_device()
    N, Hkv, B, D = _pool_shape(k_cache, v_cache, cur)
    _dev(q, "q", torch.bfloat16, 3, cur)
    _dev(out, "out", torch.bfloat16, 3, cur)
    _dev(block_tables, "block_tables", torch.int32, 2, cur)
    _dev(context_lens, "context_lens", torch.int32, 1, cur)
    _dev(workspace, "workspace", torch.uint8, 1, cur)
    S, Hq = int(q.shape[0]), int(q.shape[1])
    if q.shape[2] != D or out.shape != q.shape:
        raise ValueError("q/out must be [S, Hq, D] with the pools' D")
    if block_tables.shape[0] != S or context_lens.shape[0] != S:
        raise ValueError("block_tables/context_lens must have S rows")
    check(lib().pkv_paged_attention_decode(
        out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        block_tables.data_ptr(), int(block_tables.shape[1]), context_lens.data_ptr(),
        int(max_context_len), S, Hq, Hkv, D, B, N, float(scale), int(partition_size),
        workspace.data_ptr(), int(workspace.numel()), _ptr(status), _stream(stream)))


# ---------------------------------------------------------------- shared prefixes

def pkv_decode_shared_workspace_bytes(S: int, Hq: int, D: int, max_context_len: int,
                                      partition_size: int = 0) -> int:
    out = ctypes.c_size_t()
    check(lib().pkv_decode_shared_workspace_bytes(int(S), int(Hq), int(D), int(max_context_len),
                                                  int(partition_size), ctypes.byref(out)))
    return out.value


def pkv_paged_attention_decode_shared(out, q, k_cache, v_cache, block_tables, context_lens,
                                      max_context_len: int, group_start, group_members,
                                      group_shared, scale: float, workspace,
                                      partition_size: int = 0, status=None, stream=None) -> None:
    """Decode where groups of sequences share their first tokens' blocks: each
    group's shared prefix is read once for several members."""
    N, Hkv, B, D = _pool_shape(k_cache, v_cache)
    _dev(q, "q", torch.bfloat16, 3)
    _dev(out, "out", torch.bfloat16, 3)
    _dev(block_tables, "block_tables", torch.int32, 2)
    _dev(context_lens, "context_lens", torch.int32, 1)
    _dev(workspace, "workspace", torch.uint8, 1)
    for name, t in (("group_start", group_start), ("group_members", group_members),
                    ("group_shared", group_shared)):
        _dev(t, name, torch.int32, 1)
    n_groups = int(group_shared.shape[0])
    if group_start.shape[0] != n_groups + 1:
        raise ValueError("group_start must have n_groups + 1 entries")
    S, Hq = int(q.shape[0]), int(q.shape[1])
    if q.shape[2] != D or out.shape != q.shape:
        raise ValueError("q/out must be [S, Hq, D] with the pools' D")
    if block_tables.shape[0] != S or context_lens.shape[0] != S:
        raise ValueError("block_tables/context_lens must have S rows")
    check(lib().pkv_paged_attention_decode_shared(
        out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        block_tables.data_ptr(), int(block_tables.shape[1]), context_lens.data_ptr(),
        int(max_context_len), group_start.data_ptr(), group_members.data_ptr(),
        group_shared.data_ptr(), n_groups, S, Hq, Hkv, D, B, N, float(scale),
        int(partition_size), workspace.data_ptr(), int(workspace.numel()), _ptr(status),
        _stream(stream)))


# ---------------------------------------------------------------- FP8 pages

def _fp8_pools(k_codes, v_codes, k_scales, v_scales):
    _dev(k_codes, "k_codes", torch.uint8, 4)
    _dev(v_codes, "v_codes", torch.uint8, 4)
    _dev(k_scales, "k_scales", torch.float32, 3)
    _dev(v_scales, "v_scales", torch.float32, 3)
    if k_codes.shape != v_codes.shape or k_scales.shape != v_scales.shape or \
            tuple(k_scales.shape) != tuple(k_codes.shape[:3]):
        raise ValueError("codes must be [N, Hkv, B, D] and scales [N, Hkv, B], K and V alike")
    return tuple(int(x) for x in k_codes.shape)  # N, Hkv, B, D


def new_fp8_pools(num_blocks: int, Hkv: int, block_size: int, D: int, device=None):
    """Zeroed FP8 pools: (k_codes, v_codes, k_scales, v_scales)."""
    dev = device or "cuda"
    codes = [torch.zeros((num_blocks, Hkv, block_size, D), dtype=torch.uint8, device=dev)
             for _ in range(2)]
    scales = [torch.zeros((num_blocks, Hkv, block_size), dtype=torch.float32, device=dev)
              for _ in range(2)]
    return codes[0], codes[1], scales[0], scales[1]


def pkv_kv_append_fp8(k_new, v_new, slot_mapping, k_codes, v_codes, k_scales, v_scales,
                      status=None, stream=None) -> None:
    N, Hkv, B, D = _fp8_pools(k_codes, v_codes, k_scales, v_scales)
    _dev(k_new, "k_new", torch.bfloat16, 3)
    _dev(v_new, "v_new", torch.bfloat16, 3)
    _dev(slot_mapping, "slot_mapping", torch.int32, 1)
    T = int(slot_mapping.shape[0])
    if k_new.shape != (T, Hkv, D) or v_new.shape != (T, Hkv, D):
        raise ValueError(f"k_new/v_new must be [{T}, {Hkv}, {D}]")
    check(lib().pkv_kv_append_fp8(k_new.data_ptr(), v_new.data_ptr(), slot_mapping.data_ptr(), T,
                                  k_codes.data_ptr(), v_codes.data_ptr(), k_scales.data_ptr(),
                                  v_scales.data_ptr(), N, Hkv, D, B, _ptr(status),
                                  _stream(stream)))


def pkv_paged_attention_decode_fp8(out, q, k_codes, v_codes, k_scales, v_scales, block_tables,
                                   context_lens, max_context_len: int, scale: float, workspace,
                                   partition_size: int = 0, status=None, stream=None) -> None:
    N, Hkv, B, D = _fp8_pools(k_codes, v_codes, k_scales, v_scales)
    _dev(q, "q", torch.bfloat16, 3)
    _dev(out, "out", torch.bfloat16, 3)
    _dev(block_tables, "block_tables", torch.int32, 2)
    _dev(context_lens, "context_lens", torch.int32, 1)
    _dev(workspace, "workspace", torch.uint8, 1)
    S, Hq = int(q.shape[0]), int(q.shape[1])
    if q.shape[2] != D or out.shape != q.shape:
        raise ValueError("q/out must be [S, Hq, D] with the pools' D")
    if block_tables.shape[0] != S or context_lens.shape[0] != S:
        raise ValueError("block_tables/context_lens must have S rows")
    check(lib().pkv_paged_attention_decode_fp8(
        out.data_ptr(), q.data_ptr(), k_codes.data_ptr(), v_codes.data_ptr(), k_scales.data_ptr(),
        v_scales.data_ptr(), block_tables.data_ptr(), int(block_tables.shape[1]),
        context_lens.data_ptr(), int(max_context_len), S, Hq, Hkv, D, B, N, float(scale),
        int(partition_size), workspace.data_ptr(), int(workspace.numel()), _ptr(status),
        _stream(stream)))


NOALLOC_SCRATCH_BYTES = 64 << 20  # PKV_DECODE_NOALLOC_SCRATCH_BYTES


def pkv_paged_attention_decode_noalloc(out, q, k_cache, v_cache, block_tables, context_lens,
                                       max_context_len: int, scale: float, partition_size: int = 0,
                                       status=None, stream=None) -> None:
    """Decode for callers that cannot supply device scratch: the library uses a
    fixed internal array of NOALLOC_SCRATCH_BYTES instead, shared by all calls
    (serialise overlapping calls). Allocates no memory."""
    N, Hkv, B, D = _pool_shape(k_cache, v_cache)
    _dev(q, "q", torch.bfloat16, 3)
    _dev(out, "out", torch.bfloat16, 3)
    _dev(block_tables, "block_tables", torch.int32, 2)
    _dev(context_lens, "context_lens", torch.int32, 1)
    S, Hq = int(q.shape[0]), int(q.shape[1])
    if q.shape[2] != D or out.shape != q.shape:
        raise ValueError("q/out must be [S, Hq, D] with the pools' D")
    if block_tables.shape[0] != S or context_lens.shape[0] != S:
        raise ValueError("block_tables/context_lens must have S rows")
    check(lib().pkv_paged_attention_decode_noalloc(
        out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        block_tables.data_ptr(), int(block_tables.shape[1]), context_lens.data_ptr(),
        int(max_context_len), S, Hq, Hkv, D, B, N, float(scale), int(partition_size),
        _ptr(status), _stream(stream)))


def pkv_prefill_workspace_bytes(S: int, total_q: int, Hq: int, D: int) -> int:
    out = ctypes.c_size_t()
    check(lib().pkv_prefill_workspace_bytes(int(S), int(total_q), int(Hq), int(D),
                                            ctypes.byref(out)))
    return out.value


def pkv_paged_attention_prefill(out, q, cu_q_lens, context_lens, k_cache, v_cache, block_tables,
                                max_q_len: int, max_context_len: int, scale: float, workspace,
                                status=None, stream=None) -> None:
    cur = torch.cuda.current_device()
    N, Hkv, B, D = _pool_shape(k_cache, v_cache, cur)
    _dev(q, "q", torch.bfloat16, 3, cur)
    _dev(out, "out", torch.bfloat16, 3, cur)
    _dev(cu_q_lens, "cu_q_lens", torch.int32, 1, cur)
    _dev(context_lens, "context_lens", torch.int32, 1, cur)
    _dev(block_tables, "block_tables", torch.int32, 2, cur)
    _dev(workspace, "workspace", torch.uint8, 1, cur)
    total_q, Hq = int(q.shape[0]), int(q.shape[1])
    S = int(context_lens.shape[0])
    if cu_q_lens.shape[0] != S + 1 or block_tables.shape[0] != S:
        raise ValueError("cu_q_lens must be [S+1] and block_tables [S, *]")
    if q.shape[2] != D or out.shape != q.shape:
        raise ValueError("q/out must be [total_q, Hq, D] with the pools' D")
    check(lib().pkv_paged_attention_prefill(
        out.data_ptr(), q.data_ptr(), cu_q_lens.data_ptr(), context_lens.data_ptr(),
        k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
        int(block_tables.shape[1]), S, total_q, int(max_q_len), int(max_context_len), Hq, Hkv,
        D, B, N, float(scale), workspace.data_ptr(), int(workspace.numel()), _ptr(status),
        _stream(stream)))
