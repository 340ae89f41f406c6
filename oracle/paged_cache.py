"""Address mapping, cache write (scatter) and logical gather -- oracle only.

Layout reading: each layer's key and value caches are arrays of shape
``[num_blocks, block_size, num_kv_heads, head_dim]``.  The pages print
several layouts (MiniPaged-Qwen §11 puts the head axis before the block
offset; the guijiagi "paged-attention-impl-detail" KVBlock keeps
``[block_size, n_kv_heads, head_dim]`` inside a block; LLM-algo ch.22's
ledger prints ``[layers, 2, kv_heads, block_size, head_dim]``).  We take the
block-major ``[NB, BS, Hkv, D]`` order; only ``cache_index`` knows it, so
the choice is isolated to one function.

Arrays hold raw storage elements: float32, float16, or bfloat16 kept as its
16-bit pattern in a uint16 array (numpy has no bfloat16).  Writes copy
elements, so they are bit-exact by construction; ``to_float64`` is the only
place that interprets the bits.
"""

from __future__ import annotations

from typing import Sequence, Tuple

import numpy as np


# -- address mapping ----------------------------------------------------------

def logical_block(pos: int, block_size: int) -> int:
    """MiniPaged-Qwen §3: logical block = floor(token_pos / block_size)."""
    return pos // block_size


def block_offset(pos: int, block_size: int) -> int:
    """MiniPaged-Qwen §3: block offset = token_pos mod block_size."""
    return pos % block_size


def slot_of(table: Sequence[int], pos: int, block_size: int) -> int:
    """MiniPaged-Qwen §3 / §4.1: slot = table[pos // bs] * bs + pos % bs."""
    return int(table[logical_block(pos, block_size)]) * block_size + block_offset(pos, block_size)


def split_slot(slot: int, block_size: int) -> Tuple[int, int]:
    """MiniPaged-Qwen §11: physical block = slot // bs, offset = slot % bs."""
    return slot // block_size, slot % block_size


def num_logical_blocks(seq_len: int, block_size: int) -> int:
    """MiniPaged-Qwen §4.3: ceil(sequence_length / block_size)."""
    return -(-seq_len // block_size)


def cache_index(physical_block: int, offset: int, kv_head: int):
    """Index of one (token, kv-head) row in a ``[NB, BS, Hkv, D]`` cache."""
    return (physical_block, offset, kv_head)


# -- element interpretation ---------------------------------------------------

def bf16_bits_to_float64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 is the upper half of an IEEE binary32: widen by 16 zero bits."""
    wide = bits.astype(np.uint32) << np.uint32(16)
    return wide.view(np.float32).astype(np.float64)


def to_float64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exact conversion of stored elements to float64."""
    if dtype == "bf16":
        return bf16_bits_to_float64(x)
    return x.astype(np.float64)


# -- cache write: MiniPaged-Qwen §12 -------------------------------------------

def reshape_and_cache(k: np.ndarray, v: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                      slot_mapping: Sequence[int]) -> None:
    """Write token t's K/V rows ``[Hkv, D]`` to ``cache[slot // bs, slot % bs]``.

    ``slot == -1`` marks a padded token: nothing is read or written for it
    (reading of a padding value the pages do not mention).  Any other slot
    outside ``[0, NB * BS)`` is an error.  Plain per-token, per-head loop.
    """
    num_blocks, block_size, num_kv_heads, _ = k_cache.shape
    for t, slot in enumerate(slot_mapping):
        slot = int(slot)
        if slot == -1:
            continue
        if slot < 0 or slot >= num_blocks * block_size:
            raise ValueError(f"slot {slot} outside the pool")
        pb, off = split_slot(slot, block_size)
        for h in range(num_kv_heads):
            k_cache[cache_index(pb, off, h)] = k[t, h]
            v_cache[cache_index(pb, off, h)] = v[t, h]


# -- logical gather: LLM-algo ch.22 Step 4 TODO 4 ------------------------------

def gather(cache: np.ndarray, table: Sequence[int], seq_len: int) -> np.ndarray:
    """Concatenate the table's blocks IN TABLE ORDER (never sorted by physical
    index) and truncate to ``seq_len`` tokens: result ``[seq_len, Hkv, D]``.

    Only the first ceil(seq_len / bs) entries are read, so table padding and
    the unused tail of the last block are never touched (MiniPaged-Qwen §16.6).
    """
    num_blocks, block_size = cache.shape[0], cache.shape[1]
    used = num_logical_blocks(seq_len, block_size)
    if used > len(table):
        raise ValueError("block table shorter than the sequence")
    rows = []
    for lb in range(used):
        pb = int(table[lb])
        if pb < 0 or pb >= num_blocks:
            raise ValueError(f"block {pb} outside the pool")
        rows.append(cache[pb])
    if not rows:
        return cache[:0, 0]
    return np.concatenate(rows, axis=0)[:seq_len]
