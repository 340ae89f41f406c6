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

from typing import Optional

import numpy as np
import torch

from ._lib import check
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
        # One int32 buffer holds a step's metadata (slot mapping, block
        # tables, seq_lens) so it crosses to the device in one copy.  Two
        # pinned host copies alternate between steps, so the host can write
        # step i + 1 while step i's copy may still be queued.
        self._meta_split = (n_step, n_step + B * self.max_blocks)
        meta_len = n_step + B * self.max_blocks + B
        self.h_meta = [torch.empty(meta_len, dtype=torch.int32, pin_memory=True) for _ in range(2)]
        self.d_meta = torch.empty(meta_len, dtype=torch.int32, device=self.device)
        self.d_slots, self.d_tables, self.d_lens = self._views(self.d_meta)
        self._cur = 1
        self._meta_free = [None, None]   # event after which h_meta[i] may be rewritten
        self._meta_events = [torch.cuda.Event(), torch.cuda.Event()]
        self.graphs = None
        self.out = torch.empty(B, wl.num_heads, wl.head_dim, dtype=dt, device=self.device)
        pads = pad_positions(wl)
        is_pad = np.zeros(n_step, dtype=bool)
        is_pad[pads] = True
        self.valid_pos = np.nonzero(~is_pad)[0]
        self.pad_pos = pads
        self.n_prefill = int(wl.prefill_lens.sum())
        self.next_id = wl.next_id
        # inputs of kvbm_prepare_step, kept in place so their addresses are fixed
        self._decode_ids = np.ascontiguousarray(wl.decode_ids, dtype=np.int64)
        self._prefill_lens = np.ascontiguousarray(wl.prefill_lens, dtype=np.int64)
        self._prefill_ids = np.zeros(self._prefill_lens.size, dtype=np.int64)
        self._free_ids = np.zeros(self._prefill_lens.size, dtype=np.int64)
        self._pad_pos = np.ascontiguousarray(pads, dtype=np.int64)
        self._prefilled_once = False
        self._meta_addr = []
        for m in self.h_meta:
            sl, tb, ln = self._views(m)
            self._meta_addr.append((sl.data_ptr(), tb.data_ptr(), ln.data_ptr()))
        self.steps_done = 0
        self.history_slots: Optional[np.ndarray] = None

    def _views(self, meta: torch.Tensor):
        a, b = self._meta_split
        B = self.wl.num_seqs
        return meta[:a], meta[a:b].view(B, self.max_blocks), meta[b:]

    # the pinned metadata of the step written last
    @property
    def h_slots(self) -> torch.Tensor:
        return self._views(self.h_meta[self._cur])[0]

    @property
    def h_tables(self) -> torch.Tensor:
        return self._views(self.h_meta[self._cur])[1]

    @property
    def h_lens(self) -> torch.Tensor:
        return self._views(self.h_meta[self._cur])[2]

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
        """a1 on the host: one native call (kvbm_prepare_step) releases the
        previous step's prefill sequences, allocates this step's, appends
        one decode slot per running sequence, and writes slot mapping (with
        -1 padding), block tables and seq_lens into the next pinned
        metadata buffer."""
        self._cur ^= 1
        ev = self._meta_free[self._cur]
        if ev is not None:
            ev.synchronize()       # the copy that last read this buffer has run
        n_pre = self._prefill_ids.size
        n_free = n_pre if self._prefilled_once else 0   # the previous step's prefills end now
        if n_pre:
            self._free_ids[:] = self._prefill_ids
            self._prefill_ids[:] = np.arange(self.next_id, self.next_id + n_pre)
            self.next_id += n_pre
            self._prefilled_once = True
        slots_a, tables_a, lens_a = self._meta_addr[self._cur]
        st = self.mgr.prepare_step_raw(
            self._free_ids.ctypes.data if n_free else None, n_free,
            self._prefill_ids.ctypes.data if n_pre else None, self._prefill_lens.ctypes.data if n_pre else None,
            n_pre, self._decode_ids.ctypes.data, self._decode_ids.size,
            self._pad_pos.ctypes.data if self._pad_pos.size else None, self._pad_pos.size, self.max_blocks,
            slots_a, tables_a, lens_a)
        check(st, "kvbm_prepare_step")

    def upload_metadata(self) -> None:
        """a1 crossing: one async H2D copy of the step's metadata."""
        self.d_meta.copy_(self.h_meta[self._cur], non_blocking=True)

    def _mark_meta_used(self) -> None:
        ev = self._meta_events[self._cur]
        ev.record()
        self._meta_free[self._cur] = ev

    def write_step_kv(self, k_step: torch.Tensor, v_step: torch.Tensor) -> None:
        """a2: cache write of the step's new tokens."""
        reshape_and_cache(k_step, v_step, self.k_cache, self.v_cache, self.d_slots)

    def attention(self, q: torch.Tensor) -> torch.Tensor:
        """a3-a8: decode attention for every running sequence."""
        wl = self.wl
        return paged_decode_attention(self.out, q, self.k_cache, self.v_cache, self.d_tables, self.d_lens,
                                      wl.scale, self.max_seq_len, self.blocks_per_split, self.workspace)

    def _check_room(self) -> None:
        if self.steps_done + 1 > self.max_seq_len - int(self.wl.cached_lens.max()):
            raise RuntimeError("engine sized for fewer steps")

    def step(self, q: torch.Tensor, k_step: torch.Tensor, v_step: torch.Tensor) -> torch.Tensor:
        """One step with direct launches."""
        self._check_room()
        self.host_metadata()
        self.upload_metadata()
        self._mark_meta_used()
        self.write_step_kv(k_step, v_step)
        out = self.attention(q)
        self.steps_done += 1
        return out

    # ---------------------------------------------------------- CUDA graphs
    def capture(self, q: torch.Tensor, k_step: torch.Tensor, v_step: torch.Tensor, host_io=None) -> None:
        """Capture the device part of a step -- metadata copy, cache write,
        attention -- as two CUDA graphs, one per pinned metadata buffer.
        ``host_io`` = (q_h, k_h, v_h, out_h) pinned host tensors adds the
        inputs' H2D copies into q/k_step/v_step and the output's D2H copy.
        Call after at least one ``step`` so every lazy set-up has run."""
        if self.steps_done == 0:
            raise RuntimeError("run one step before capturing")
        torch.cuda.synchronize()
        graphs = []
        side = torch.cuda.Stream()
        for i in range(2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                self.d_meta.copy_(self.h_meta[i], non_blocking=True)
                if host_io is not None:
                    q.copy_(host_io[0], non_blocking=True)
                    k_step.copy_(host_io[1], non_blocking=True)
                    v_step.copy_(host_io[2], non_blocking=True)
                self.write_step_kv(k_step, v_step)
                out = self.attention(q)
                if host_io is not None:
                    host_io[3].copy_(out, non_blocking=True)
            graphs.append(g)
        torch.cuda.synchronize()
        self.graphs = graphs

    def step_graph(self) -> torch.Tensor:
        """One step: host metadata, then one graph launch for the device part."""
        self._check_room()
        self.host_metadata()
        self.graphs[self._cur].replay()
        self._mark_meta_used()
        self.steps_done += 1
        return self.out

    @property
    def launches_per_step(self) -> int:
        """Library kernels per step: the cache write plus the attention call."""
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
