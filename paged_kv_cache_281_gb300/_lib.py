"""ctypes declarations of the C ABI in ``include/pagedkv.h``.

Loading fails loudly when ``libpagedkv.so`` is missing: there is no fallback
implementation of any call.
"""

from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpagedkv.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "pagedkv.h")

PKV_OK, PKV_EINVAL, PKV_ENOMEM, PKV_ECUDA, PKV_ETIMEOUT, PKV_EDEVICE = 0, -1, -2, -3, -4, -5
STATUS_NAMES = {0: "PKV_OK", -1: "PKV_EINVAL", -2: "PKV_ENOMEM", -3: "PKV_ECUDA",
                -4: "PKV_ETIMEOUT", -5: "PKV_EDEVICE"}

i32, i64, u64, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float
vp, sz = ctypes.c_void_p, ctypes.c_size_t
P = ctypes.POINTER

class IterationLayout(ctypes.Structure):
    """``pkv_iteration_layout``: byte offsets of one iteration's metadata."""
    _fields_ = [(n, ctypes.c_int64) for n in (
        "slot_mapping", "cu_q_lens", "prefill_lens", "prefill_tables", "decode_lens",
        "decode_tables", "cow_pairs", "total_bytes")] + [(n, ctypes.c_int32) for n in (
        "n_tokens", "n_cow", "max_q_len", "max_prefill_len", "max_decode_len", "table_width")]


SIGNATURES = {
    "pkv_last_error": (ctypes.c_char_p, []),
    "pkv_version": (ctypes.c_int, []),
    "pkv_alloc_create": (ctypes.c_int, [i32, i32, P(i32), P(vp)]),
    "pkv_alloc_destroy": (ctypes.c_int, [vp]),
    "pkv_seq_create": (ctypes.c_int, [vp, P(i64)]),
    "pkv_seq_fork": (ctypes.c_int, [vp, i64, P(i64)]),
    "pkv_seq_append_slots": (ctypes.c_int, [vp, i64, i32, P(i32), P(i32), P(i32)]),
    "pkv_seq_free": (ctypes.c_int, [vp, i64]),
    # (per-iteration calls: host arrays passed as plain addresses, the
    # cheapest conversion ctypes offers)
    "pkv_seq_create_many": (ctypes.c_int, [vp, i32, vp]),
    "pkv_seq_free_many": (ctypes.c_int, [vp, vp, i32]),
    "pkv_seq_len": (ctypes.c_int, [vp, i64, P(i32)]),
    "pkv_seq_block_table": (ctypes.c_int, [vp, i64, P(i32), i32, P(i32)]),
    "pkv_block_refcount": (ctypes.c_int, [vp, i32, P(i32)]),
    "pkv_num_free_blocks": (ctypes.c_int, [vp, P(i32)]),
    "pkv_build_block_tables": (ctypes.c_int, [vp, P(i64), i32, P(i32), i32, P(i32)]),
    "pkv_iteration_layout_bytes": (ctypes.c_int, [i32, i32, i32, i32, P(IterationLayout)]),
    "pkv_iteration_prepare": (ctypes.c_int, [vp, vp, vp, i32, i32, i32, vp, sz,
                                             P(IterationLayout), P(i32)]),
    "pkv_iteration_run": (ctypes.c_int, [vp, P(IterationLayout), i32, i32, vp, vp, vp, vp,
                                         vp, vp, i32, i32, i32, i32, i32, f32, i32, vp, sz, vp,
                                         sz, vp, vp]),
    "pkv_iteration_step": (ctypes.c_int, [vp, vp, vp, i32, i32, i32, vp, sz, vp, sz, vp,
                                          vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32,
                                          vp, sz, vp, sz, vp, vp, P(IterationLayout), P(i32)]),
    "pkv_seq_swap_out": (ctypes.c_int, [vp, i64, P(i32), i32, P(i32)]),
    "pkv_seq_swap_in": (ctypes.c_int, [vp, i64, P(i32), i32, P(i32)]),
    "pkv_seq_create_cached": (ctypes.c_int, [vp, P(i32), i32, P(i64), P(i32)]),
    "pkv_seq_append_tokens": (ctypes.c_int, [vp, i64, P(i32), i32, P(i32), P(i32), P(i32)]),
    "pkv_num_cached_blocks": (ctypes.c_int, [vp, P(i32)]),
    "pkv_swap_blocks": (ctypes.c_int, [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, i32, vp, vp]),
    "pkv_status_reset": (ctypes.c_int, [vp, vp]),
    "pkv_check_status": (ctypes.c_int, [vp, vp]),
    "pkv_debug_set_wait": (ctypes.c_int, [i32, u64]),
    "pkv_kv_append": (ctypes.c_int, [vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, vp, vp]),
    "pkv_decode_shared_workspace_bytes": (ctypes.c_int, [i32, i32, i32, i32, i32, P(sz)]),
    "pkv_paged_attention_decode_shared": (ctypes.c_int, [vp, vp, vp, vp, vp, i32, vp, i32, vp, vp,
                                                         vp, i32, i32, i32, i32, i32, i32, i32,
                                                         f32, i32, vp, sz, vp, vp]),
    "pkv_kv_append_fp8": (ctypes.c_int, [vp, vp, vp, i32, vp, vp, vp, vp, i32, i32, i32, i32, vp,
                                         vp]),
    "pkv_paged_attention_decode_fp8": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, vp, i32, vp, i32,
                                                      i32, i32, i32, i32, i32, i32, f32, i32, vp,
                                                      sz, vp, vp]),
    "pkv_block_copy": (ctypes.c_int, [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp]),
    "pkv_decode_workspace_bytes": (ctypes.c_int, [i32, i32, i32, i32, i32, P(sz)]),
    "pkv_paged_attention_decode": (ctypes.c_int, [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32,
                                                  i32, i32, i32, f32, i32, vp, sz, vp, vp]),
    "pkv_paged_attention_decode_noalloc": (ctypes.c_int, [vp, vp, vp, vp, vp, i32, vp, i32, i32,
                                                          i32, i32, i32, i32, i32, f32, i32, vp,
                                                          vp]),
    "pkv_prefill_workspace_bytes": (ctypes.c_int, [i32, i32, i32, i32, P(sz)]),
    "pkv_paged_attention_prefill": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                                   i32, i32, i32, i32, i32, i32, f32, vp, sz, vp,
                                                   vp]),
}

_lib = None


class PagedKVError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {message}")
        self.code = code


def header_functions() -> list[str]:
    """Names of the functions ``include/pagedkv.h`` declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text)))


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is not built: run paged_kv_cache_281_gb300.build.build() "
                "(nvcc, sm_103a); there is no fallback implementation")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _lib = l
    return _lib


def check(code: int) -> None:
    if code != PKV_OK:
        raise PagedKVError(code, lib().pkv_last_error().decode())
