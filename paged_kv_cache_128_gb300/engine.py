"""One layer's paged KV cache on one GPU, driven one decode step at a time.

``PagedDecodeEngine`` owns the host block manager, the device caches and
the pinned/device metadata buffers, and runs the hot path of a serving
step in order:

  a1  host metadata: optional prefill allocation for new sequences (atomic),
      one decode append per running sequence, export of block tables and
      seq_lens, slot mapping with padded (-1) entries; async H2D copy;
  a2  ``reshape_and_cache`` of the step's new K/V (prefill chunk + decode
      tokens) by slot mapping;
  a3-a8  ``paged_decode_attention`` over every running sequence (table
      walk, QK^T, online softmax, PV, split-K and log-sum-exp merge).

The same object builds the pre-step state (a sequence's history is written
through the cache-write kernel with the slots its prefill returned), so the
tests and the benchmark exercise exactly one code path.
"""

from __future__ import annotations

from typing import List, Optional

import numpy as np
import torch

from .block_manager import KVBlockManager
from .inputs import Values, Workload, pad_positions, sentinel_bits
from .kernels import alloc_workspace, decode_plan, paged_decode_attention, reshape_and_cache

_INT_VIEW = {torch.float32: torch.int32, torch.float16: torch.int16, torch.bfloat16: torch.int16}


def _signed(bits: int, width: int) -> int:
    return bits - (1 << width) if bits >= 1 << (width - 1) else bits


class PagedDecodeEngine:
    def __init__(self, wl: Workload, device="cuda", max_steps: int = 64, fill_sentinel: bool = True,
                 blocks_per_split: int = 0):
        self.wl = wl
        self.blocks_per_split = blocks_per_split
        self.device = torch.device(device)
        self.mgr = KVBlockManager(wl.num_blocks, wl.block_size, wl.free_order)
        dt = wl.torch_dtype
        shape = (wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim)
        self.k_cache = torch.empty(shape, dtype=dt, device=self.device)
        self.v_cache = torch.empty(shape, dtype=dt, device=self.device)
        if fill_sentinel:
            iv = _INT_VIEW[dt]
            width = 32 if iv == torch.int32 else 16
            fill = _signed(sentinel_bits(wl.dtype), width)
            self.k_cache.view(iv).fill_(fill)
            self.v_cache.view(iv).fill_(fill)
        B = wl.num_seqs
        self.max_seq_len = int(wl.cached_lens.max()) + 1 + max_steps
        self.max_blocks = -(-self.max_seq_len // wl.block_size)
        self.plan = decode_plan(B, wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.block_size, self.max_seq_len,
                                dt, blocks_per_split)
        self.workspace = alloc_workspace(self.plan, self.device)
        n_step = wl.num_step_tokens
        pin = dict(pin_memory=True)
        self.h_slots = torch.empty(n_step, dtype=torch.int32, **pin)
        self.h_tables = torch.empty(B, self.max_blocks, dtype=torch.int32, **pin)
        self.h_lens = torch.empty(B, dtype=torch.int32, **pin)
        self.d_slots = torch.empty(n_step, dtype=torch.int32, device=self.device)
        self.d_tables = torch.empty(B, self.max_blocks, dtype=torch.int32, device=self.device)
        self.d_lens = torch.empty(B, dtype=torch.int32, device=self.device)
        self.out = torch.empty(B, wl.num_heads, wl.head_dim, dtype=dt, device=self.device)
        pads = pad_positions(wl)
        is_pad = np.zeros(n_step, dtype=bool)
        is_pad[pads] = True
        self.valid_pos = np.nonzero(~is_pad)[0]
        self.pad_pos = pads
        self.n_prefill = int(wl.prefill_lens.sum())
        self.prefill_ids: List[int] = []
        self.next_id = wl.next_id
        self.steps_done = 0
        self._h2d_done = torch.cuda.Event()
        self._h2d_pending = False
        self.history_slots: Optional[np.ndarray] = None

    # ---------------------------------------------------------------- setup
    def setup(self, values: Values) -> None:
        """Replay the workload's setup operations on the manager and write
        every decode sequence's history through the cache-write kernel."""
        wl = self.wl
        per_seq = {int(i): [] for i in wl.decode_ids}
        for op, sid, n in wl.setup_ops:
            if op == "prefill":
                slots = self.mgr.allocate_for_prefill(sid, n)
            elif op == "append":
                slots = self.mgr.append_slots(sid, n)
            else:
                self.mgr.free_sequence(sid)
                continue
            if sid in per_seq:
                per_seq[sid].append(slots)
        hist = [np.concatenate(per_seq[int(i)]) if per_seq[int(i)] else np.zeros(0, np.int32)
                for i in wl.decode_ids]
        self.history_slots = np.concatenate(hist).astype(np.int32) if hist else np.zeros(0, np.int32)
        n = self.history_slots.size
        if n:
            d_hist = torch.from_numpy(self.history_slots).to(self.device)
            k = values.k_hist.to(self.device)
            v = values.v_hist.to(self.device)
            chunk = 1 << 20
            for a in range(0, n, chunk):
                b = min(n, a + chunk)
                reshape_and_cache(k[a:b], v[a:b], self.k_cache, self.v_cache, d_hist[a:b])

    # ------------------------------------------------------------------ step
    def host_metadata(self) -> None:
        """a1: allocate the step's prefill sequences, append one decode slot
        per running sequence, export tables/lens into pinned buffers and
        queue the H2D copies."""
        wl = self.wl
        if self._h2d_pending:
            self._h2d_done.synchronize()       # pinned buffers are about to be rewritten
        slots = self.h_slots.numpy()
        step_slots = np.empty(self.n_prefill + wl.num_seqs, dtype=np.int32)
        if self.n_prefill:
            for sid in self.prefill_ids:
                self.mgr.free_sequence(sid)
            self.prefill_ids = []
            pos = 0
            for n in wl.prefill_lens:
                sid = self.next_id
                self.next_id += 1
                self.mgr.allocate_for_prefill(sid, int(n), step_slots[pos:pos + int(n)])
                self.prefill_ids.append(sid)
                pos += int(n)
        self.mgr.decode_step(wl.decode_ids, self.max_blocks, step_slots[self.n_prefill:], self.h_tables.numpy(),
                             self.h_lens.numpy())
        slots[self.valid_pos] = step_slots
        if self.pad_pos.size:
            slots[self.pad_pos] = -1
        self.d_slots.copy_(self.h_slots, non_blocking=True)
        self.d_tables.copy_(self.h_tables, non_blocking=True)
        self.d_lens.copy_(self.h_lens, non_blocking=True)
        self._h2d_done.record()
        self._h2d_pending = True

    def write_step_kv(self, k_step: torch.Tensor, v_step: torch.Tensor) -> None:
        """a2: cache write of the step's new tokens."""
        reshape_and_cache(k_step, v_step, self.k_cache, self.v_cache, self.d_slots)

    def attention(self, q: torch.Tensor) -> torch.Tensor:
        """a3-a8: decode attention for every running sequence."""
        wl = self.wl
        return paged_decode_attention(self.out, q, self.k_cache, self.v_cache, self.d_tables, self.d_lens,
                                      wl.scale, self.max_seq_len, self.blocks_per_split, self.workspace)

    def step(self, q: torch.Tensor, k_step: torch.Tensor, v_step: torch.Tensor) -> torch.Tensor:
        if self.steps_done + 1 > self.max_seq_len - int(self.wl.cached_lens.max()):
            raise RuntimeError("engine sized for fewer steps")
        self.host_metadata()
        self.write_step_kv(k_step, v_step)
        out = self.attention(q)
        self.steps_done += 1
        return out

    @property
    def launches_per_step(self) -> int:
        return 1 + self.plan.launches

    def algorithmic_bytes(self, seq_lens: np.ndarray) -> dict:
        """Bytes the step must move at minimum: K+V of every attended token
        once, q in and out once, the table entries and lengths used; and the
        cache write (read + write of the valid new rows, plus the slots)."""
        wl = self.wl
        s = 2 if wl.dtype != "f32" else 4
        row = wl.num_kv_heads * wl.head_dim * s
        L = seq_lens.astype(np.int64)
        blocks = -(-L // wl.block_size)
        attn = int(L.sum()) * 2 * row + 2 * wl.num_seqs * wl.num_heads * wl.head_dim * s + 4 * (
            wl.num_seqs + int(blocks.sum()))
        n_valid = self.n_prefill + wl.num_seqs
        write = 2 * 2 * n_valid * row + 4 * wl.num_step_tokens
        return {"attention": attn, "cache_write": write, "step": attn + write}
