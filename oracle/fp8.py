"""FP8 (e4m3) KV pages: quantisation and attention over dequantised pages.

TEST INFRASTRUCTURE ONLY (see the package docstring).

"Two orthogonal fixes, one serving engine" (the continuous-batching page)
lists FP8 arithmetic among the kernel-level optimisations that stack with
paging; the pages fix no storage format. Readings taken here:

* each key and value row (one token, one kv head, D elements) is stored as D
  e4m3 codes plus one fp32 scale; the scales of a page sit in per-page scale
  arrays ``[num_blocks][Hkv][block_size]``, one per token row, so appending a
  token never rewrites the rest of its page;
* a row with largest magnitude ``amax`` gets ``scale = amax / 448`` and codes
  ``e4m3(x * (448 / amax))``, both quotients and the product rounded to fp32,
  the code rounded to nearest (ties to even) and saturated at +-448; a row of
  zeros gets scale 0 and codes 0;
* the value a code stands for is ``decode(code) * scale``, and attention is
  the definition of ``oracle.attention`` evaluated on those values.

e4m3 (sign, 4 exponent bits with bias 7, 3 mantissa bits): exponent field e >
0 gives (1 + m/8) 2^(e-7); e = 0 gives (m/8) 2^-6; the all-ones pattern
(e = 15, m = 7) is NaN and there is no infinity, so the largest finite value
is 1.75 * 2^8 = 448.
"""

from __future__ import annotations

import numpy as np

from .attention import _group, attend, widen_bf16

E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """Codes (uint8) -> float64 values from the bit fields."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = (1.0 + m / 8.0) * np.ldexp(1.0, e - 7)
    sub = (m / 8.0) * 2.0 ** -6
    val = np.where(e > 0, normal, sub)
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


def _finite_table():
    """The 127 non-negative finite values and their codes, ascending."""
    codes = np.arange(0, 127, dtype=np.uint8)
    return e4m3_decode(codes), codes


def e4m3_encode(x) -> np.ndarray:
    """float32 values -> e4m3 codes, round to nearest with ties to even (the
    even code is the one with mantissa bit 0), saturating at +-448; the sign
    bit is kept, also for values that round to zero."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)  # exact
    vals, codes = _finite_table()
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.searchsorted(vals, a, side="left")            # first value >= a
    hi = np.minimum(hi, len(vals) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - vals[lo], vals[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (codes[hi] % 2 == 0))
    idx = np.where(vals[hi] == a, hi, np.where(pick_hi, hi, lo))
    out = codes[idx].astype(np.uint8)
    return np.where(np.signbit(x), out | 0x80, out).astype(np.uint8)   # -0 keeps its sign


def quantize_rows(bits: np.ndarray):
    """bf16 rows ``[..., D]`` -> (codes uint8 ``[..., D]``, scales float32 ``[...]``)."""
    x = widen_bf16(bits).astype(np.float32)               # exact
    amax = np.max(np.abs(x), axis=-1).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        inv = np.where(amax > 0, np.float32(E4M3_MAX) / amax, np.float32(0)).astype(np.float32)
        scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    y = (x * inv[..., None]).astype(np.float32)
    return e4m3_encode(y), scale


def append(k8, v8, ks, vs, k_new_bits, v_new_bits, slot_mapping, block_size: int) -> None:
    """Quantise each new token's rows and write codes and scales into its slot;
    slot -1 skips."""
    kc, ksc = quantize_rows(k_new_bits)
    vc, vsc = quantize_rows(v_new_bits)
    for t, slot in enumerate(slot_mapping):
        slot = int(slot)
        if slot < 0:
            continue
        b, off = divmod(slot, block_size)
        k8[b, :, off, :] = kc[t]
        v8[b, :, off, :] = vc[t]
        ks[b, :, off] = ksc[t]
        vs[b, :, off] = vsc[t]


def dequantize_seq(codes, scales, table, length: int, block_size: int) -> np.ndarray:
    """A sequence's rows ``[length, Hkv, D]`` in float64 through its block table."""
    Hkv, D = codes.shape[1], codes.shape[3]
    out = np.empty((length, Hkv, D))
    for j in range(length):
        b, off = int(table[j // block_size]), j % block_size
        out[j] = e4m3_decode(codes[b, :, off, :]) * scales[b, :, off].astype(np.float64)[:, None]
    return out


def decode(q_bits, k8, v8, ks, vs, block_tables, context_lens, block_size: int, scale: float,
           seqs=None) -> np.ndarray:
    """One query per sequence at position L-1 over the dequantised pages."""
    S, Hq, D = q_bits.shape
    Hkv = k8.shape[1]
    G = _group(Hq, Hkv)
    q = widen_bf16(q_bits)
    out = np.zeros((S, Hq, D))
    for s in (range(S) if seqs is None else seqs):
        L = int(context_lens[s])
        K = dequantize_seq(k8, ks, block_tables[s], L, block_size)
        V = dequantize_seq(v8, vs, block_tables[s], L, block_size)
        for h in range(Hq):
            out[s, h] = attend(q[s, h][None, :], K[:, h // G], V[:, h // G], scale, [L])[0]
    return out
