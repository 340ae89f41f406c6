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

import ctypes

from ._lib import KVError, check, kvstep_config_t, lib
from .block_manager import KVBlockManager
from .inputs import Values, Workload, pad_positions, sentinel_bits
from .kernels import (alloc_workspace, decode_plan, dtype_code, paged_decode_attention, paged_decode_attention_fp8,
                      paged_decode_step, paged_decode_step_fp8, reshape_and_cache, reshape_and_cache_fp8)

_INT_VIEW = {torch.float32: torch.int32, torch.float16: torch.int16, torch.bfloat16: torch.int16}


def _signed(bits: int, width: int) -> int:
    return bits - (1 << width) if bits >= 1 << (width - 1) else bits


class PagedDecodeEngine:
    def __init__(self, wl: Workload, device="cuda", max_steps: int = 64, fill_sentinel: bool = True,
                 blocks_per_split: int = 0, fused: bool = True, kv_cache: str = "native"):
        self.wl = wl
        self.blocks_per_split = blocks_per_split
        # kv_cache "fp8": E4M3 codes with one float32 scale per (token, kv
        # head); the step is the quantised cache write, then fp8 attention
        if kv_cache not in ("native", "fp8"):
            raise ValueError("kv_cache is 'native' or 'fp8'")
        self.fp8 = kv_cache == "fp8"
        # fused: the step's cache write and attention in one paged_decode_step
        # call (one launch with the stream-K kernel); else two calls
        self.fused = fused and blocks_per_split == 0
        self.device = torch.device(device)
        self.mgr = KVBlockManager(wl.num_blocks, wl.block_size, wl.free_order)
        dt = wl.torch_dtype
        shape = (wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim)
        self.k_scales = self.v_scales = None
        if self.fp8:
            self.k_cache = torch.full(shape, 0x7F, dtype=torch.uint8, device=self.device)   # 0x7F: the NaN code
            self.v_cache = torch.full(shape, 0x7F, dtype=torch.uint8, device=self.device)
            sshape = (wl.num_blocks, wl.num_kv_heads, wl.block_size)
            self.k_scales = torch.full(sshape, float("nan"), dtype=torch.float32, device=self.device)
            self.v_scales = torch.full(sshape, float("nan"), dtype=torch.float32, device=self.device)
        else:
            self.k_cache = torch.empty(shape, dtype=dt, device=self.device)
            self.v_cache = torch.empty(shape, dtype=dt, device=self.device)
        if fill_sentinel and not self.fp8:
            iv = _INT_VIEW[dt]
            width = 32 if iv == torch.int32 else 16
            fill = _signed(sentinel_bits(wl.dtype), width)
            self.k_cache.view(iv).fill_(fill)
            self.v_cache.view(iv).fill_(fill)
        B = wl.num_seqs
        self._max_cached = int(wl.cached_lens.max())
        self.max_seq_len = self._max_cached + 1 + max_steps
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
        self._runner = None
        self.out = torch.empty(B, wl.num_heads, wl.head_dim, dtype=dt, device=self.device)
        pads = pad_positions(wl)
        is_pad = np.zeros(n_step, dtype=bool)
        is_pad[pads] = True
        self.valid_pos = np.nonzero(~is_pad)[0]
        self.pad_pos = pads
        self.n_prefill = int(wl.prefill_lens.sum())
        # kvbm_prepare_step puts the prefill slots first, then one decode slot
        # per running sequence, in the non-padded positions: sequence b's new
        # token is row valid_pos[n_prefill + b] of the step's K/V
        rows = self.valid_pos[self.n_prefill:self.n_prefill + B].astype(np.int32)
        self.d_new_rows = torch.from_numpy(np.ascontiguousarray(rows)).to(self.device)
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
                if self.fp8:
                    reshape_and_cache_fp8(k[a:b], v[a:b], self.k_cache, self.v_cache, self.k_scales, self.v_scales,
                                          d_hist[a:b])
                else:
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
        n_free, n_pre = self._advance_ids()
        slots_a, tables_a, lens_a = self._meta_addr[self._cur]
        st = self.mgr.prepare_step_raw(
            self._free_ids.ctypes.data if n_free else None, n_free,
            self._prefill_ids.ctypes.data if n_pre else None, self._prefill_lens.ctypes.data if n_pre else None,
            n_pre, self._decode_ids.ctypes.data, self._decode_ids.size,
            self._pad_pos.ctypes.data if self._pad_pos.size else None, self._pad_pos.size, self.max_blocks,
            slots_a, tables_a, lens_a)
        check(st, "kvbm_prepare_step")

    def _advance_ids(self):
        """This step's sequence ids: the previous step's prefill sequences
        are released and a fresh id is drawn for each new prefill sequence.
        Returns (n_free, n_prefill)."""
        n_pre = self._prefill_ids.size
        n_free = n_pre if self._prefilled_once else 0   # the previous step's prefills end now
        if n_pre:
            self._free_ids[:] = self._prefill_ids
            self._prefill_ids[:] = np.arange(self.next_id, self.next_id + n_pre)
            self.next_id += n_pre
            self._prefilled_once = True
        return n_free, n_pre

    def upload_metadata(self) -> None:
        """a1 crossing: one async H2D copy of the step's metadata."""
        self.d_meta.copy_(self.h_meta[self._cur], non_blocking=True)

    def _mark_meta_used(self) -> None:
        ev = self._meta_events[self._cur]
        ev.record()
        self._meta_free[self._cur] = ev

    def write_step_kv(self, k_step: torch.Tensor, v_step: torch.Tensor) -> None:
        """a2: cache write of the step's new tokens."""
        if self.fp8:
            reshape_and_cache_fp8(k_step, v_step, self.k_cache, self.v_cache, self.k_scales, self.v_scales,
                                  self.d_slots)
        else:
            reshape_and_cache(k_step, v_step, self.k_cache, self.v_cache, self.d_slots)

    def attention(self, q: torch.Tensor) -> torch.Tensor:
        """a3-a8: decode attention for every running sequence."""
        wl = self.wl
        if self.fp8:
            return paged_decode_attention_fp8(self.out, q, self.k_cache, self.v_cache, self.k_scales, self.v_scales,
                                              self.d_tables, self.d_lens, wl.scale, self.max_seq_len, self.workspace)
        return paged_decode_attention(self.out, q, self.k_cache, self.v_cache, self.d_tables, self.d_lens,
                                      wl.scale, self.max_seq_len, self.blocks_per_split, self.workspace)

    def fused_step(self, q: torch.Tensor, k_step: torch.Tensor, v_step: torch.Tensor) -> torch.Tensor:
        """a2-a8 in one paged_decode_step(_fp8) call."""
        wl = self.wl
        if self.fp8:
            return paged_decode_step_fp8(self.out, q, k_step, v_step, self.d_slots, self.d_new_rows, self.k_cache,
                                         self.v_cache, self.k_scales, self.v_scales, self.d_tables, self.d_lens,
                                         wl.scale, self.max_seq_len, self.workspace)
        return paged_decode_step(self.out, q, k_step, v_step, self.d_slots, self.d_new_rows, self.k_cache,
                                 self.v_cache, self.d_tables, self.d_lens, wl.scale, self.max_seq_len,
                                 self.workspace)

    def device_step(self, q: torch.Tensor, k_step: torch.Tensor, v_step: torch.Tensor) -> torch.Tensor:
        """The device part of a step after the metadata copy: a2, then a3-a8."""
        if self.fused:
            return self.fused_step(q, k_step, v_step)
        self.write_step_kv(k_step, v_step)
        return self.attention(q)

    def _check_room(self) -> None:
        if self.steps_done + 1 > self.max_seq_len - self._max_cached:
            raise RuntimeError("engine sized for fewer steps")

    def step(self, q: torch.Tensor, k_step: torch.Tensor, v_step: torch.Tensor) -> torch.Tensor:
        """One step with direct launches."""
        self._check_room()
        self.host_metadata()
        self.upload_metadata()
        self._mark_meta_used()
        out = self.device_step(q, k_step, v_step)
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
                out = self.device_step(q, k_step, v_step)
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

    # ------------------------------------------------------- native runner
    def make_runner(self, host_io: int = 0, stream: Optional[torch.cuda.Stream] = None) -> None:
        """Create the native step runner (kvstep_*): afterwards each
        ``runner_step`` is ONE library call doing a1 (kvbm_prepare_step, the
        async metadata copy on a side stream) and a2-a8 (the fused launch).
        ``host_io`` 1 (or True): the step's q/k/v and output are page-locked
        host buffers that the runner copies in and out on its side streams.
        ``host_io`` 2: q/k/v are staged in the runner's own page-locked slots
        (``runner_stage``) and travel with the metadata in one copy; the
        output is a page-locked host buffer."""
        host_io = int(host_io)
        wl = self.wl
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        ws = self.workspace
        cfg = kvstep_config_t(
            num_seqs=wl.num_seqs, num_heads=wl.num_heads, num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim,
            block_size=wl.block_size, num_blocks=wl.num_blocks, max_blocks_per_seq=self.max_blocks,
            max_seq_len=self.max_seq_len, scale=float(wl.scale), dtype=dtype_code(wl.torch_dtype),
            num_step_tokens=wl.num_step_tokens, k_cache=self.k_cache.data_ptr(), v_cache=self.v_cache.data_ptr(),
            workspace=ws.data_ptr() if ws is not None else None,
            workspace_bytes=ws.numel() if ws is not None else 0, stream=s.cuda_stream, host_io=host_io,
            cache_fp8=1 if self.fp8 else 0, k_scales=self.k_scales.data_ptr() if self.fp8 else None,
            v_scales=self.v_scales.data_ptr() if self.fp8 else None)
        self.close_runner()
        h = ctypes.c_void_p()
        check(lib().kvstep_create(self.mgr._h, ctypes.byref(cfg), ctypes.byref(h)), "kvstep_create")
        self._runner = h
        self._runner_stream = s
        self._runner_host_io = host_io
        self._runner_args = (
            self._decode_ids.ctypes.data, self._decode_ids.size,
            self._pad_pos.ctypes.data if self._pad_pos.size else None, self._pad_pos.size)

    def runner_stage(self, slot: int = -1):
        """host_io 2: page-locked CPU tensors (q, k, v) viewing a staging
        slot of the runner -- slot -1 is the next step's (after its previous
        copy has run), 0..3 a given one (filled before any step)."""
        if getattr(self, "_runner_host_io", 0) != 2:
            raise KVError(1, "runner_stage needs a runner made with host_io=2")
        ptrs = [ctypes.c_void_p() for _ in range(3)]
        got = ctypes.c_int32()
        check(lib().kvstep_stage_buffer(self._runner, int(slot), *[ctypes.byref(x) for x in ptrs],
                                        ctypes.byref(got)), "kvstep_stage_buffer")
        wl = self.wl
        es = torch.empty((), dtype=wl.torch_dtype).element_size()
        shapes = [(wl.num_seqs, wl.num_heads, wl.head_dim), (wl.num_step_tokens, wl.num_kv_heads, wl.head_dim),
                  (wl.num_step_tokens, wl.num_kv_heads, wl.head_dim)]
        views = []
        for ptr, shape in zip(ptrs, shapes):
            nbytes = int(np.prod(shape)) * es
            buf = (ctypes.c_uint8 * nbytes).from_address(ptr.value)
            views.append(torch.frombuffer(buf, dtype=torch.uint8).view(wl.torch_dtype).view(shape))
        return tuple(views)

    def runner_step(self, q: Optional[torch.Tensor], k_step: Optional[torch.Tensor], v_step: Optional[torch.Tensor],
                    out: torch.Tensor) -> None:
        """One step through the native runner (a1-a8 in one call); with
        host_io 2, q/k/v are None (staged with ``runner_stage``)."""
        self._check_room()
        n_free, n_pre = self._advance_ids()
        dec, n_dec, pads, n_pad = self._runner_args
        ptr = lambda t: t.data_ptr() if t is not None else None
        check(lib().kvstep_run(self._runner, ptr(q), ptr(k_step), ptr(v_step), out.data_ptr(),
                               self._free_ids.ctypes.data if n_free else None, n_free,
                               self._prefill_ids.ctypes.data if n_pre else None,
                               self._prefill_lens.ctypes.data if n_pre else None, n_pre, dec, n_dec, pads, n_pad),
              "kvstep_run")
        self.steps_done += 1

    def runner_join(self, stream: Optional[torch.cuda.Stream] = None) -> None:
        """Order ``stream`` (default: the current one) after the runner's work."""
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        check(lib().kvstep_join(self._runner, s.cuda_stream), "kvstep_join")

    def runner_last_metadata(self):
        """Host copies of the runner's last step: (slot mapping, block
        tables [B, max_blocks], seq_lens, decode rows) as numpy arrays."""
        wl = self.wl
        ptrs = [ctypes.c_void_p() for _ in range(4)]
        check(lib().kvstep_last_buffers(self._runner, *[ctypes.byref(p) for p in ptrs]), "kvstep_last_buffers")
        sizes = [wl.num_step_tokens, wl.num_seqs * self.max_blocks, wl.num_seqs, wl.num_seqs]
        arrs = [np.ctypeslib.as_array(ctypes.cast(p, ctypes.POINTER(ctypes.c_int32)), shape=(n,)).copy()
                for p, n in zip(ptrs, sizes)]
        arrs[1] = arrs[1].reshape(wl.num_seqs, self.max_blocks)
        return tuple(arrs)

    def close_runner(self) -> None:
        h = getattr(self, "_runner", None)
        if h:
            lib().kvstep_destroy(h)
            self._runner = None

    def __del__(self):
        try:
            self.close_runner()
        except Exception:
            pass

    @property
    def launches_per_step(self) -> int:
        """Library kernels per step: one fused launch with the stream-K
        kernel, else the cache write plus the attention call's launches."""
        if self.fused and self.plan.kernel == 2:
            return 1
        if self.fp8:
            # the library fuses the fp8 write only for at most two step rows per
            # consumer warp (4 per CTA, two CTAs per SM)
            sms = torch.cuda.get_device_properties(self.device).multi_processor_count
            return 1 if self.fused and self.wl.num_step_tokens <= 2 * sms * 2 * 4 else 2
        return 1 + self.plan.launches

    def algorithmic_bytes(self, seq_lens: np.ndarray) -> dict:
        """Bytes the step must move at minimum: K+V of every attended token
        once, q in and out once, the table entries and lengths used; and the
        cache write (read + write of the valid new rows, plus the slots)."""
        wl = self.wl
        s = 2 if wl.dtype != "f32" else 4
        row = wl.num_kv_heads * wl.head_dim * s
        # a cached row: the dtype's bytes, or fp8 codes plus one float32 scale per head
        crow = wl.num_kv_heads * (wl.head_dim + 4) if self.fp8 else row
        L = seq_lens.astype(np.int64)
        blocks = -(-L // wl.block_size)
        attn = int(L.sum()) * 2 * crow + 2 * wl.num_seqs * wl.num_heads * wl.head_dim * s + 4 * (
            wl.num_seqs + int(blocks.sum()))
        n_valid = self.n_prefill + wl.num_seqs
        write = 2 * n_valid * (row + crow) + 4 * wl.num_step_tokens
        return {"attention": attn, "cache_write": write, "step": attn + write}
