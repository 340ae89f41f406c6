"""Python handle over the native KV block manager (kvbm_* in libpagedkv).

Every operation runs in the C++ library; this class only converts
arguments and turns non-OK statuses into ``KVError``.  Semantics are those
of include/pagedkv.h: MiniPaged-Qwen §8-§9 and §15, the mini-vLLM Block
Manager API, and the LLM-algo ch.22 exercise (atomic prefill, decode
rollback, validated release).
"""

from __future__ import annotations

import ctypes
from typing import Dict, Optional, Sequence, Tuple

import numpy as np

from ._lib import KVError, P32, P64, check, kvbm_stats_t, lib


def _i32(a: np.ndarray):
    return a.ctypes.data_as(P32)


def _i64(a: np.ndarray):
    return a.ctypes.data_as(P64)


def _ids(seq_ids) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(seq_ids, dtype=np.int64).reshape(-1))


class KVBlockManager:
    """Fixed pool of ``num_blocks`` blocks of ``block_size`` slots."""

    def __init__(self, num_blocks: int, block_size: int, initial_free_order: Optional[Sequence[int]] = None):
        self._lib = lib()
        h = ctypes.c_void_p()
        order = None
        if initial_free_order is not None:
            order = np.ascontiguousarray(np.asarray(initial_free_order, dtype=np.int32))
            if order.size != num_blocks:
                raise KVError(1, "kvbm_create")
        check(self._lib.kvbm_create(num_blocks, block_size, _i32(order) if order is not None else None,
                                    ctypes.byref(h)), "kvbm_create")
        self._h = h
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)

    def close(self) -> None:
        if getattr(self, "_h", None):
            self._lib.kvbm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- admission ---------------------------------------------------------------
    def can_allocate(self, num_tokens: int) -> bool:
        ok = ctypes.c_int()
        check(self._lib.kvbm_can_allocate(self._h, num_tokens, ctypes.byref(ok)), "kvbm_can_allocate")
        return bool(ok.value)

    def can_append_slots(self, seq_ids) -> bool:
        ids = _ids(seq_ids)
        ok = ctypes.c_int()
        check(self._lib.kvbm_can_append_slots(self._h, _i64(ids), ids.size, ctypes.byref(ok)),
              "kvbm_can_append_slots")
        return bool(ok.value)

    # -- allocation ----------------------------------------------------------------
    def allocate_for_prefill(self, seq_id: int, num_tokens: int, slots_out: Optional[np.ndarray] = None):
        out = slots_out if slots_out is not None else np.empty(max(num_tokens, 0), dtype=np.int32)
        check(self._lib.kvbm_allocate_for_prefill(self._h, seq_id, num_tokens, _i32(out)),
              "kvbm_allocate_for_prefill")
        return out

    def append_slot_for_decode(self, seq_id: int) -> int:
        slot = ctypes.c_int32()
        check(self._lib.kvbm_append_slot_for_decode(self._h, seq_id, ctypes.byref(slot)),
              "kvbm_append_slot_for_decode")
        return slot.value

    def append_slots(self, seq_id: int, num_tokens: int, slots_out: Optional[np.ndarray] = None):
        out = slots_out if slots_out is not None else np.empty(max(num_tokens, 0), dtype=np.int32)
        check(self._lib.kvbm_append_slots(self._h, seq_id, num_tokens, _i32(out)), "kvbm_append_slots")
        return out

    def decode_step(self, seq_ids, max_blocks: int, slots_out: Optional[np.ndarray] = None,
                    tables_out: Optional[np.ndarray] = None, lens_out: Optional[np.ndarray] = None):
        """One decode append per sequence, then export; all or nothing on OOM.
        The optional outputs must be C-contiguous int32 arrays (they may be
        numpy views of pinned host tensors)."""
        ids = _ids(seq_ids)
        n = ids.size
        slots = slots_out if slots_out is not None else np.empty(n, dtype=np.int32)
        tables = tables_out if tables_out is not None else np.empty((n, max_blocks), dtype=np.int32)
        lens = lens_out if lens_out is not None else np.empty(n, dtype=np.int32)
        check(self._lib.kvbm_decode_step(self._h, _i64(ids), n, max_blocks, _i32(slots), _i32(tables),
                                         _i32(lens)), "kvbm_decode_step")
        return slots, tables, lens

    def prepare_step(self, free_ids, prefill_ids, prefill_lens, decode_ids, pad_positions, max_blocks: int,
                     slots_out: Optional[np.ndarray] = None, tables_out: Optional[np.ndarray] = None,
                     lens_out: Optional[np.ndarray] = None):
        """One step's metadata in one native call (kvbm_prepare_step):
        release ``free_ids``, prefill-allocate ``prefill_ids``/``prefill_lens``,
        append one slot to each of ``decode_ids``, and return (slot mapping
        with -1 at ``pad_positions``, decode block tables, decode seq_lens)."""
        fr, pi, pl, di, pp = (_ids(x) for x in (free_ids, prefill_ids, prefill_lens, decode_ids, pad_positions))
        n_slots = int(pl.sum()) + di.size + pp.size
        slots = slots_out if slots_out is not None else np.empty(n_slots, dtype=np.int32)
        tables = tables_out if tables_out is not None else np.empty((di.size, max_blocks), dtype=np.int32)
        lens = lens_out if lens_out is not None else np.empty(di.size, dtype=np.int32)
        check(self._lib.kvbm_prepare_step(self._h, fr.ctypes.data, fr.size, pi.ctypes.data, pl.ctypes.data, pi.size,
                                          di.ctypes.data, di.size, pp.ctypes.data, pp.size, max_blocks,
                                          slots.ctypes.data, tables.ctypes.data, lens.ctypes.data),
              "kvbm_prepare_step")
        return slots, tables, lens

    def prepare_step_raw(self, *args) -> int:
        """kvbm_prepare_step with pre-computed buffer addresses (hot loops)."""
        return self._lib.kvbm_prepare_step(self._h, *args)

    def free_sequence(self, seq_id: int) -> None:
        check(self._lib.kvbm_free_sequence(self._h, seq_id), "kvbm_free_sequence")

    # -- prefix sharing / copy-on-write ----------------------------------------------
    def fork(self, parent_id: int, child_id: int, prefix_len: int) -> None:
        """New sequence ``child_id`` sharing the blocks of ``parent_id``'s
        first ``prefix_len`` tokens (kvbm_fork)."""
        check(self._lib.kvbm_fork(self._h, parent_id, child_id, prefix_len), "kvbm_fork")

    def take_copies(self) -> Tuple[np.ndarray, np.ndarray]:
        """Queued copy-on-write copies (src, dst) since the last call."""
        n = ctypes.c_int64()
        check(self._lib.kvbm_take_copies(self._h, None, None, 0, ctypes.byref(n)), "kvbm_take_copies")
        src = np.empty(n.value, dtype=np.int32)
        dst = np.empty(n.value, dtype=np.int32)
        if n.value:
            check(self._lib.kvbm_take_copies(self._h, _i32(src), _i32(dst), n.value, ctypes.byref(n)),
                  "kvbm_take_copies")
        return src, dst

    def block_refcount(self, block: int) -> int:
        out = ctypes.c_int32()
        check(self._lib.kvbm_block_refcount(self._h, block, ctypes.byref(out)), "kvbm_block_refcount")
        return out.value

    # -- queries -----------------------------------------------------------------------
    def num_free_blocks(self) -> int:
        n = ctypes.c_int64()
        check(self._lib.kvbm_num_free_blocks(self._h, ctypes.byref(n)), "kvbm_num_free_blocks")
        return n.value

    def free_list(self) -> np.ndarray:
        n = ctypes.c_int64()
        check(self._lib.kvbm_get_free_list(self._h, None, 0, ctypes.byref(n)), "kvbm_get_free_list")
        out = np.empty(n.value, dtype=np.int32)
        check(self._lib.kvbm_get_free_list(self._h, _i32(out), out.size, ctypes.byref(n)), "kvbm_get_free_list")
        return out

    def seq_len(self, seq_id: int) -> int:
        n = ctypes.c_int64()
        check(self._lib.kvbm_seq_len(self._h, seq_id, ctypes.byref(n)), "kvbm_seq_len")
        return n.value

    def block_table(self, seq_id: int) -> np.ndarray:
        n = ctypes.c_int64()
        check(self._lib.kvbm_get_block_table(self._h, seq_id, None, 0, ctypes.byref(n)), "kvbm_get_block_table")
        out = np.empty(n.value, dtype=np.int32)
        check(self._lib.kvbm_get_block_table(self._h, seq_id, _i32(out), out.size, ctypes.byref(n)),
              "kvbm_get_block_table")
        return out

    def export(self, seq_ids, max_blocks: int, tables_out: Optional[np.ndarray] = None,
               lens_out: Optional[np.ndarray] = None):
        ids = _ids(seq_ids)
        tables = tables_out if tables_out is not None else np.empty((ids.size, max_blocks), dtype=np.int32)
        lens = lens_out if lens_out is not None else np.empty(ids.size, dtype=np.int32)
        check(self._lib.kvbm_export(self._h, _i64(ids), ids.size, max_blocks, _i32(tables), _i32(lens)),
              "kvbm_export")
        return tables, lens

    def export_update(self, seq_ids, max_blocks: int, tables: np.ndarray, prev_ids: np.ndarray,
                      prev_nblocks: np.ndarray) -> None:
        """kvbm_export_update: refresh ``tables`` ([n, max_blocks] int32, an
        earlier export described by ``prev_ids`` int64 / ``prev_nblocks``
        int32, both [n] and updated in place) to the current export."""
        ids = _ids(seq_ids)
        for a, dt in ((tables, np.int32), (prev_ids, np.int64), (prev_nblocks, np.int32)):
            if a.dtype != dt or not a.flags.c_contiguous:
                raise KVError(1, "export_update buffers: contiguous int32 tables / int64 ids / int32 counts")
        if tables.shape != (ids.size, max_blocks) or prev_ids.size != ids.size or prev_nblocks.size != ids.size:
            raise KVError(1, "export_update buffer shapes")
        check(self._lib.kvbm_export_update(self._h, _i64(ids), ids.size, max_blocks, _i32(tables), _i64(prev_ids),
                                           _i32(prev_nblocks)), "kvbm_export_update")

    def check_invariants(self) -> bool:
        st = self._lib.kvbm_check_invariants(self._h)
        if st not in (0, 6):
            check(st, "kvbm_check_invariants")
        return st == 0

    def stats(self) -> Dict[str, int]:
        s = kvbm_stats_t()
        check(self._lib.kvbm_stats(self._h, ctypes.byref(s)), "kvbm_stats")
        return {name: getattr(s, name) for name, _ in kvbm_stats_t._fields_}

    def released_ranges(self) -> int:
        """Ranges of consecutive released ids the manager remembers (for
        KV_ERR_DOUBLE_FREE on a second release)."""
        n = ctypes.c_int64()
        check(self._lib.kvbm_released_ranges(self._h, ctypes.byref(n)), "kvbm_released_ranges")
        return n.value

    def allocation_report(self, seq_id: int) -> Dict[str, float]:
        lt, at, ut = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        u = ctypes.c_double()
        check(self._lib.kvbm_allocation_report(self._h, seq_id, ctypes.byref(lt), ctypes.byref(at),
                                               ctypes.byref(ut), ctypes.byref(u)), "kvbm_allocation_report")
        return {"logical_tokens": lt.value, "allocated_tokens": at.value, "unused_tail_tokens": ut.value,
                "utilization": u.value}

    def owner_table(self) -> np.ndarray:
        out = np.empty(self.num_blocks, dtype=np.int64)
        check(self._lib.kvbm_owner_table(self._h, _i64(out), out.size), "kvbm_owner_table")
        return out


def kv_cache_ledger(num_blocks: int, block_size: int, num_layers: int, num_kv_heads: int, head_dim: int,
                    dtype_bytes: int) -> Dict[str, int]:
    a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    check(lib().kv_cache_ledger(num_blocks, block_size, num_layers, num_kv_heads, head_dim, dtype_bytes,
                                ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)), "kv_cache_ledger")
    return {"kv_bytes_per_token": a.value, "kv_bytes_per_block": b.value, "total_cache_bytes": c.value}
