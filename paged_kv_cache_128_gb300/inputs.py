"""Seeded synthetic workloads for the paged KV cache path.

This module only draws numbers: shapes, sequence lengths, free-list orders,
the order of host operations that set up a pool, padding positions, and the
q / k / v values.  It holds none of the method's arithmetic (no slots, no
block counts, no attention); both the CUDA path and the CPU oracle consume
what it returns.

Workloads (one decode step each, single layer):

* ``decode_tiny_fp32`` -- fp32, block 4, 16 blocks, 2 sequences cached at
  {6, 11}, Hq 2, Hkv 1, D 8; shuffled pool.
* ``decode_gqa14x2_d64_fp16`` -- fp16, Hq 14, Hkv 2, D 64, block 16, 8192
  blocks, 32 sequences, cached lengths uniform in [1, 2048]; values N(0,1)/2.
* ``decode_gqa28x4_d128_bf16`` -- bf16, Hq 28, Hkv 4, D 128, block 16, 32768
  blocks, 64 sequences, cached lengths uniform in [512, 4096].
* ``decode_long_skewed_bf16`` -- bf16, Hq 32, Hkv 8, D 128, block 16, 40000
  blocks, 8 sequences: two of 32768 and six uniform in [128, 1024], grown
  round-robin in 64-token chunks so their tables interleave.
* ``mixed_batch_bf16`` -- bf16, Hq 32, Hkv 8, D 128, block 32, 65536 blocks;
  256 decode sequences with lognormal(ln 512, 1) lengths capped to
  [1, 8192], a pool fragmented by three rounds of seeded alloc/free churn,
  plus one 4096-token prefill chunk over 8 new sequences (uniform [256, 768]
  rescaled to sum 4096) and 5 % padded (-1) entries in the step's
  slot mapping.

Cached lengths are before the step; the step's decode token is appended
and written first, so attention covers cached + 1 tokens.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional, Tuple

import numpy as np
import torch

BASE_SEED = 20261202

WORKLOADS = ("decode_tiny_fp32", "decode_gqa14x2_d64_fp16", "decode_gqa28x4_d128_bf16",
             "decode_long_skewed_bf16", "mixed_batch_bf16")

TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclass
class Workload:
    name: str
    dtype: str                       # "f32" | "f16" | "bf16"
    block_size: int
    num_blocks: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    scale: float
    value_scale: float
    seed: int
    free_order: Optional[np.ndarray]           # int32 permutation, or None = 0..NB-1
    setup_ops: List[Tuple[str, int, int]]      # ("prefill", id, n) | ("append", id, n) | ("free", id, 0)
    decode_ids: np.ndarray                     # int64 [B], batch order
    cached_lens: np.ndarray                    # int64 [B], before the step
    prefill_lens: np.ndarray = field(default_factory=lambda: np.zeros(0, dtype=np.int64))
    num_pad: int = 0                           # padded (-1) entries in the step's slot mapping
    next_id: int = 0                           # first unused sequence id

    @property
    def num_seqs(self) -> int:
        return int(self.decode_ids.size)

    @property
    def torch_dtype(self) -> torch.dtype:
        return TORCH_DTYPES[self.dtype]

    @property
    def num_step_tokens(self) -> int:
        return int(self.prefill_lens.sum()) + self.num_seqs + self.num_pad


def _decode_setup(ids, lens):
    return [("prefill", int(i), int(n)) for i, n in zip(ids, lens)]


def make_workload(name: str) -> Workload:
    idx = WORKLOADS.index(name)
    seed = BASE_SEED + idx + 1
    rng = np.random.default_rng(seed)
    if name == "decode_tiny_fp32":
        nb = 16
        lens = np.array([6, 11], dtype=np.int64)
        ids = np.arange(2, dtype=np.int64)
        return Workload(name, "f32", 4, nb, 2, 1, 8, 1.0 / np.sqrt(8.0), 1.0, seed,
                        rng.permutation(nb).astype(np.int32), _decode_setup(ids, lens), ids, lens, next_id=2)
    if name == "decode_gqa14x2_d64_fp16":
        nb, B = 8192, 32
        lens = rng.integers(1, 2048, size=B, endpoint=True).astype(np.int64)
        ids = np.arange(B, dtype=np.int64)
        return Workload(name, "f16", 16, nb, 14, 2, 64, 1.0 / 8.0, 0.5, seed,
                        rng.permutation(nb).astype(np.int32), _decode_setup(ids, lens), ids, lens, next_id=B)
    if name == "decode_gqa28x4_d128_bf16":
        nb, B = 32768, 64
        lens = rng.integers(512, 4096, size=B, endpoint=True).astype(np.int64)
        ids = np.arange(B, dtype=np.int64)
        return Workload(name, "bf16", 16, nb, 28, 4, 128, 1.0 / np.sqrt(128.0), 1.0, seed,
                        rng.permutation(nb).astype(np.int32), _decode_setup(ids, lens), ids, lens, next_id=B)
    if name == "decode_long_skewed_bf16":
        nb, B, chunk = 40000, 8, 64
        lens = np.concatenate([[32768, 32768], rng.integers(128, 1024, size=6, endpoint=True)]).astype(np.int64)
        perm = rng.permutation(B)
        lens = lens[perm]
        ids = np.arange(B, dtype=np.int64)
        ops: List[Tuple[str, int, int]] = []
        have = np.zeros(B, dtype=np.int64)
        for i in rng.permutation(B):
            n = int(min(chunk, lens[i]))
            ops.append(("prefill", int(ids[i]), n))
            have[i] = n
        while (have < lens).any():
            for i in rng.permutation(B):
                if have[i] < lens[i]:
                    n = int(min(chunk, lens[i] - have[i]))
                    ops.append(("append", int(ids[i]), n))
                    have[i] += n
        return Workload(name, "bf16", 16, nb, 32, 8, 128, 1.0 / np.sqrt(128.0), 1.0, seed, None, ops, ids, lens,
                        next_id=B)
    if name == "mixed_batch_bf16":
        nb, bs, B = 65536, 32, 256
        ops = []
        next_id = 0
        live: List[Tuple[int, int]] = []
        capacity_tokens = nb * bs
        for _round in range(3):
            used = sum(n for _, n in live)
            while used < 0.6 * capacity_tokens:
                n = int(rng.integers(16, 4096, endpoint=True))
                ops.append(("prefill", next_id, n))
                live.append((next_id, n))
                used += n
                next_id += 1
            order = rng.permutation(len(live))
            gone = set(order[: len(live) // 2].tolist())
            for j in sorted(gone):
                ops.append(("free", live[j][0], 0))
            live = [x for j, x in enumerate(live) if j not in gone]
        lens = np.clip(np.rint(rng.lognormal(np.log(512.0), 1.0, size=B)), 1, 8192).astype(np.int64)
        ids = np.arange(next_id, next_id + B, dtype=np.int64)
        ops += _decode_setup(ids, lens)
        next_id += B
        raw = rng.uniform(256, 768, size=8)
        exact = raw / raw.sum() * 4096
        plens = np.floor(exact).astype(np.int64)
        rem = 4096 - int(plens.sum())
        plens[np.argsort(-(exact - plens), kind="stable")[:rem]] += 1   # largest remainder
        valid = 4096 + B
        num_pad = int(round(0.05 * valid / 0.95))
        return Workload(name, "bf16", bs, nb, 32, 8, 128, 1.0 / np.sqrt(128.0), 1.0, seed, None, ops, ids, lens,
                        prefill_lens=plens, num_pad=num_pad, next_id=next_id)
    raise KeyError(name)


def pad_positions(wl: Workload) -> np.ndarray:
    """Sorted positions of the padded entries in the step's slot mapping."""
    rng = np.random.default_rng(wl.seed + 1000)
    total = wl.num_step_tokens
    return np.sort(rng.choice(total, size=wl.num_pad, replace=False)).astype(np.int64)


@dataclass
class Values:
    q: torch.Tensor               # [B, Hq, D]
    k_step: torch.Tensor          # [N_step, Hkv, D] rows in slot-mapping order
    v_step: torch.Tensor
    k_hist: torch.Tensor          # [sum(cached_lens), Hkv, D] decode sequences' history, batch order
    v_hist: torch.Tensor
    hist_offsets: np.ndarray      # int64 [B + 1]


def make_values(wl: Workload, device: str = "cpu", history: bool = True) -> Values:
    """Seeded q/k/v of the workload's dtype.  On CPU the values are identical
    on every machine for a given torch version; ``device='cuda'`` draws with
    the CUDA generator instead (used where no oracle comparison follows)."""
    g = torch.Generator(device=device)
    g.manual_seed(wl.seed)
    H, D = wl.num_kv_heads, wl.head_dim

    def draw(*shape):
        x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
        return (x * wl.value_scale).to(wl.torch_dtype)

    q = draw(wl.num_seqs, wl.num_heads, D)
    k_step = draw(wl.num_step_tokens, H, D)
    v_step = draw(wl.num_step_tokens, H, D)
    offsets = np.concatenate([[0], np.cumsum(wl.cached_lens)]).astype(np.int64)
    total = int(offsets[-1]) if history else 0
    k_hist = draw(total, H, D)
    v_hist = draw(total, H, D)
    return Values(q, k_step, v_step, k_hist, v_hist, offsets)


def sentinel_bits(dtype: str) -> int:
    """A quiet-NaN pattern used to fill cache slots no sequence owns."""
    return {"f32": 0x7FC00000, "f16": 0x7E00, "bf16": 0x7FC0}[dtype]
