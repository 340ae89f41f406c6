"""Capacity ledger, allocation report and tail waste -- oracle only.

* LLM-algo ch.22 Step 4, ``estimate_kv_cache_bytes``: bytes per token count
  K and V (factor 2), layers, kv heads, head dim and element size; a block
  holds ``block_size`` tokens; the pool holds ``num_blocks`` blocks.
  MiniPaged-Qwen §2 gives the same per-token factor (M_KV).
* LLM-algo ch.22 ``allocation_report``: allocated tokens = blocks * bs,
  unused tail = allocated - logical, utilisation = logical / allocated.
* MiniPaged-Qwen §6.2: last-block waste is 0 when L mod bs == 0, else
  bs - (L mod bs).
"""

from __future__ import annotations

from typing import Dict


def kv_cache_bytes(num_blocks: int, block_size: int, num_layers: int, num_kv_heads: int,
                   head_dim: int, dtype_bytes: int) -> Dict[str, int]:
    for v in (num_blocks, block_size, num_layers, num_kv_heads, head_dim, dtype_bytes):
        if v <= 0:
            raise ValueError("every ledger dimension must be positive")
    per_token = 2 * num_layers * num_kv_heads * head_dim * dtype_bytes
    per_block = block_size * per_token
    return {
        "kv_bytes_per_token": per_token,
        "kv_bytes_per_block": per_block,
        "total_cache_bytes": num_blocks * per_block,
    }


def allocation_report(seq_len: int, num_table_blocks: int, block_size: int) -> Dict[str, float]:
    allocated = num_table_blocks * block_size
    return {
        "logical_tokens": seq_len,
        "allocated_tokens": allocated,
        "unused_tail_tokens": allocated - seq_len,
        "utilization": (seq_len / allocated) if allocated else 0.0,
    }


def tail_waste(seq_len: int, block_size: int) -> int:
    r = seq_len % block_size
    return 0 if r == 0 else block_size - r
