"""fp8 (E4M3) KV cache: quantised cache write and dequantised read -- oracle only.

"paged-attention-impl-detail" (guijiagi.com), 实践建议 item 4: the KV cache
inside a block can be quantised on its own (与量化配合：块内KV Cache可以独立量化),
for more tokens per byte of memory.

Readings (the page fixes neither the format nor the scale granularity):

* Format: OCP FP8 E4M3 -- 1 sign bit, 4 exponent bits (bias 7), 3
  mantissa bits, no infinities, one NaN pattern per sign (S.1111.111);
  largest finite value 448 = 1.75 * 2^8, smallest normal 2^-6, subnormals
  m / 8 * 2^-6.
* Scale: one float32 scale per (token, kv head) row, kept inside the row's
  block, so a block's contents are quantised independently of every other
  block and a decode append never re-quantises earlier tokens.  The scale
  is amax / 448 over the row's head_dim values (1 when the row is all
  zeros), so the row uses the whole E4M3 range.
* Arithmetic: the row's values (fp16 / bf16, exact in float32) are divided
  by the scale in float32 with one correct rounding, then rounded to the
  nearest E4M3 value, ties to even, with magnitudes past 448 clamped to 448
  (saturating).  amax / 448 is one correctly rounded float32 division.
* Dequantised value = E4M3 value * scale, exact in float64.  Attention is
  the float64 decode attention of ``oracle.attention`` on those values.
* Scale array layout: ``[num_blocks, num_kv_heads, block_size]`` float32, so
  the scales of one (block, kv head) are contiguous.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use this module.
"""

from __future__ import annotations

from typing import Sequence

import numpy as np

from .paged_cache import split_slot

E4M3_MAX = 448.0
_BIAS = 7


def e4m3_to_float(code: int) -> float:
    """Value of one E4M3 code (float64), from the format's definition."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0xF and man == 0x7:
        return float("nan")
    if exp == 0:
        return sign * (man / 8.0) * 2.0 ** (1 - _BIAS)
    return sign * (1.0 + man / 8.0) * 2.0 ** (exp - _BIAS)


# every finite non-negative E4M3 value with its code, in increasing order
_POS = sorted((e4m3_to_float(c), c) for c in range(0x80) if c != 0x7F)
_POS_VALUES = np.array([v for v, _ in _POS])
_POS_CODES = np.array([c for _, c in _POS])


def float_to_e4m3(x: float) -> int:
    """Nearest E4M3 code to ``x``, ties to the even code, magnitudes past 448
    clamped to 448 (saturating).  ``x`` must not be NaN."""
    x = float(x)
    if x != x:
        raise ValueError("NaN has no saturating E4M3 rounding here")
    sign = 0x80 if (x < 0 or (x == 0 and np.signbit(x))) else 0
    a = min(abs(x), E4M3_MAX)
    i = int(np.searchsorted(_POS_VALUES, a))        # first value >= a
    if i < len(_POS_VALUES) and _POS_VALUES[i] == a:
        return sign | int(_POS_CODES[i])
    lo, hi = _POS_VALUES[i - 1], _POS_VALUES[i]
    if a - lo < hi - a:
        code = _POS_CODES[i - 1]
    elif hi - a < a - lo:
        code = _POS_CODES[i]
    else:                                           # tie: the code with an even mantissa
        code = _POS_CODES[i - 1] if _POS_CODES[i - 1] % 2 == 0 else _POS_CODES[i]
    return sign | int(code)


def float_to_e4m3_array(x: np.ndarray) -> np.ndarray:
    """``float_to_e4m3`` applied to every element of a float array (the same
    nearest / ties-to-even / saturating rule, vectorised with a sorted-table
    search; pinned against the scalar form)."""
    x = np.asarray(x, dtype=np.float64)
    if np.isnan(x).any():
        raise ValueError("NaN has no saturating E4M3 rounding here")
    sign = np.where(np.signbit(x), 0x80, 0).astype(np.uint8)
    a = np.minimum(np.abs(x), E4M3_MAX)
    n = len(_POS_VALUES)
    i = np.searchsorted(_POS_VALUES, a)             # first value >= a
    ic = np.minimum(i, n - 1)
    exact = _POS_VALUES[ic] == a
    lo_i = np.maximum(i - 1, 0)
    lo, hi = _POS_VALUES[lo_i], _POS_VALUES[ic]
    d_lo, d_hi = a - lo, hi - a
    lo_code, hi_code = _POS_CODES[lo_i], _POS_CODES[ic]
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo_code % 2 == 0))
    code = np.where(exact, _POS_CODES[ic], np.where(pick_lo, lo_code, hi_code))
    return (code.astype(np.uint8) | sign).astype(np.uint8)


def e4m3_to_float_array(codes: np.ndarray) -> np.ndarray:
    """``e4m3_to_float`` of every code (float64)."""
    table = np.array([e4m3_to_float(c) for c in range(256)], dtype=np.float64)
    return table[np.asarray(codes, dtype=np.uint8)]


def row_scale(row_f32: np.ndarray) -> np.float32:
    """amax / 448 in float32 (one correctly rounded division); 1 for a zero row."""
    amax = np.float32(np.max(np.abs(row_f32))) if row_f32.size else np.float32(0)
    if amax == 0:
        return np.float32(1.0)
    return np.float32(amax) / np.float32(E4M3_MAX)


def quantize_row(row_f32: np.ndarray):
    """One (token, kv head) row -> (uint8 codes, float32 scale)."""
    row_f32 = np.asarray(row_f32, dtype=np.float32)
    s = row_scale(row_f32)
    scaled = row_f32 / s                            # float32, correctly rounded
    codes = np.array([float_to_e4m3(v) for v in scaled], dtype=np.uint8)
    return codes, s


def dequantize_row(codes: np.ndarray, scale) -> np.ndarray:
    return np.array([e4m3_to_float(c) for c in codes], dtype=np.float64) * float(scale)


def quantize_rows(rows_f32: np.ndarray):
    """``quantize_row`` over the last axis of ``rows_f32`` ([..., D]):
    (uint8 codes [..., D], float32 scales [...]); the same float32 steps."""
    rows_f32 = np.asarray(rows_f32, dtype=np.float32)
    amax = np.max(np.abs(rows_f32), axis=-1).astype(np.float32)
    scale = np.where(amax == 0, np.float32(1.0), amax / np.float32(E4M3_MAX)).astype(np.float32)
    scaled = (rows_f32 / scale[..., None]).astype(np.float32)
    return float_to_e4m3_array(scaled), scale


def reshape_and_cache_fp8(k_f32: np.ndarray, v_f32: np.ndarray, k_codes: np.ndarray, v_codes: np.ndarray,
                          k_scales: np.ndarray, v_scales: np.ndarray, slot_mapping: Sequence[int]) -> None:
    """Quantised cache write (MiniPaged-Qwen §12 with the rows quantised):
    token t's row of kv head h goes to ``codes[slot // bs, slot % bs, h]``
    and its scale to ``scales[slot // bs, h, slot % bs]``; ``slot == -1`` is
    a padded token (nothing read or written).  Inputs are the rows as
    float32 (exact for fp16 / bf16)."""
    num_blocks, block_size, num_kv_heads, _ = k_codes.shape
    for t, slot in enumerate(slot_mapping):
        slot = int(slot)
        if slot == -1:
            continue
        if slot < 0 or slot >= num_blocks * block_size:
            raise ValueError(f"slot {slot} outside the pool")
        pb, off = split_slot(slot, block_size)
        for h in range(num_kv_heads):
            k_codes[pb, off, h], k_scales[pb, h, off] = quantize_row(k_f32[t, h])
            v_codes[pb, off, h], v_scales[pb, h, off] = quantize_row(v_f32[t, h])


def gather_dequantized(codes: np.ndarray, scales: np.ndarray, table: Sequence[int], seq_len: int) -> np.ndarray:
    """A sequence's logical rows ``[seq_len, Hkv, D]`` in float64, read
    through its table in table order (LLM-algo ch.22 TODO 4) and dequantised."""
    num_blocks, block_size, num_kv_heads, head_dim = codes.shape
    out = np.empty((seq_len, num_kv_heads, head_dim), dtype=np.float64)
    for pos in range(seq_len):
        pb = int(table[pos // block_size])
        if pb < 0 or pb >= num_blocks:
            raise ValueError(f"block {pb} outside the pool")
        off = pos % block_size
        for h in range(num_kv_heads):
            out[pos, h] = dequantize_row(codes[pb, off, h], scales[pb, h, off])
    return out
