"""ctypes view of libpagedkv.so: loads the in-tree library and declares the
C signatures from include/pagedkv.h.  Argument marshalling only."""

from __future__ import annotations

import ctypes
import os

from ctypes import POINTER, c_char_p, c_double, c_float, c_int, c_int32, c_int64, c_size_t, c_void_p

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpagedkv.so")

KV_OK = 0
STATUS_NAMES = {
    0: "OK", 1: "INVALID_ARG", 2: "OOM", 3: "UNKNOWN_SEQ", 4: "DUPLICATE_SEQ", 5: "DOUBLE_FREE",
    6: "INVARIANT", 7: "CUDA", 8: "DEVICE_BOUNDS", 9: "WORKSPACE", 10: "DEVICE_TIMEOUT", 11: "DEVICE_STEP",
}
DTYPE_F32, DTYPE_F16, DTYPE_BF16 = 0, 1, 2


class KVError(RuntimeError):
    """A non-OK status from the library; ``code`` is the status name."""

    def __init__(self, status: int, where: str):
        self.status = status
        self.code = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{where}: {self.code} ({status_string(status)})")


class kvbm_stats_t(ctypes.Structure):
    _fields_ = [("num_blocks", c_int64), ("block_size", c_int64), ("num_free_blocks", c_int64),
                ("num_sequences", c_int64), ("logical_tokens", c_int64), ("allocated_tokens", c_int64),
                ("unused_tail_tokens", c_int64)]


class kvstep_config_t(ctypes.Structure):
    _fields_ = [("num_seqs", c_int32), ("num_heads", c_int32), ("num_kv_heads", c_int32), ("head_dim", c_int32),
                ("block_size", c_int32), ("num_blocks", c_int64), ("max_blocks_per_seq", c_int32),
                ("max_seq_len", c_int64), ("scale", c_float), ("dtype", c_int32), ("num_step_tokens", c_int64),
                ("k_cache", c_void_p), ("v_cache", c_void_p), ("workspace", c_void_p),
                ("workspace_bytes", c_size_t), ("stream", c_void_p), ("host_io", c_int32),
                ("num_layers", c_int32), ("cache_layer_stride", c_int64), ("cache_fp8", c_int32),
                ("k_scales", c_void_p), ("v_scales", c_void_p)]


P32 = POINTER(c_int32)
P64 = POINTER(c_int64)

# name -> (restype, argtypes), in header order
SIGNATURES = {
    "kv_status_string": (c_char_p, [c_int]),
    "kvbm_create": (c_int, [c_int64, c_int32, P32, POINTER(c_void_p)]),
    "kvbm_destroy": (c_int, [c_void_p]),
    "kvbm_can_allocate": (c_int, [c_void_p, c_int64, POINTER(c_int)]),
    "kvbm_allocate_for_prefill": (c_int, [c_void_p, c_int64, c_int64, P32]),
    "kvbm_append_slot_for_decode": (c_int, [c_void_p, c_int64, P32]),
    "kvbm_append_slots": (c_int, [c_void_p, c_int64, c_int64, P32]),
    "kvbm_fork": (c_int, [c_void_p, c_int64, c_int64, c_int64]),
    "kvbm_take_copies": (c_int, [c_void_p, P32, P32, c_int64, P64]),
    "kvbm_block_refcount": (c_int, [c_void_p, c_int32, P32]),
    "kvbm_can_append_slots": (c_int, [c_void_p, P64, c_int64, POINTER(c_int)]),
    "kvbm_decode_step": (c_int, [c_void_p, P64, c_int64, c_int64, P32, P32, P32]),
    "kvbm_prepare_step": (c_int, [c_void_p, c_void_p, c_int64, c_void_p, c_void_p, c_int64, c_void_p, c_int64,
                                  c_void_p, c_int64, c_int64, c_void_p, c_void_p, c_void_p]),
    "kvbm_free_sequence": (c_int, [c_void_p, c_int64]),
    "kvbm_num_free_blocks": (c_int, [c_void_p, P64]),
    "kvbm_get_free_list": (c_int, [c_void_p, P32, c_int64, P64]),
    "kvbm_seq_len": (c_int, [c_void_p, c_int64, P64]),
    "kvbm_get_block_table": (c_int, [c_void_p, c_int64, P32, c_int64, P64]),
    "kvbm_export": (c_int, [c_void_p, P64, c_int64, c_int64, P32, P32]),
    "kvbm_export_update": (c_int, [c_void_p, P64, c_int64, c_int64, P32, P64, P32]),
    "kvbm_check_invariants": (c_int, [c_void_p]),
    "kvbm_stats": (c_int, [c_void_p, POINTER(kvbm_stats_t)]),
    "kvbm_released_ranges": (c_int, [c_void_p, POINTER(c_int64)]),
    "kvbm_allocation_report": (c_int, [c_void_p, c_int64, P64, P64, P64, POINTER(c_double)]),
    "kvbm_owner_table": (c_int, [c_void_p, P64, c_int64]),
    "kv_cache_ledger": (c_int, [c_int64, c_int64, c_int64, c_int64, c_int64, c_int64, P64, P64, P64]),
    "paged_reshape_and_cache": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_int32,
                                        c_int32, c_int32, c_int64, c_int64, c_int64, c_int, c_void_p]),
    "paged_reshape_and_cache_layers": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_int32,
                                               c_int64, c_int64, c_int64, c_int32, c_int32, c_int32, c_int64,
                                               c_int64, c_int64, c_int, c_void_p]),
    "paged_reshape_and_cache_fp8": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                            c_int64, c_int32, c_int32, c_int32, c_int64, c_int64, c_int64, c_int,
                                            c_void_p]),
    "paged_decode_attention_fp8": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                           c_void_p, c_int32, c_int32, c_int32, c_int32, c_int32, c_int64, c_int32,
                                           c_int64, c_float, c_int, c_void_p, c_size_t, c_void_p]),
    "paged_decode_step_fp8": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_int64,
                                      c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int32,
                                      c_int32, c_int32, c_int32, c_int32, c_int64, c_int32, c_int64, c_float, c_int,
                                      c_void_p, c_size_t, c_void_p]),
    "paged_prefill_attention": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                        c_int64, c_int32, c_int32, c_int32, c_int32, c_int32, c_int64, c_int32, c_int32,
                                        c_float, c_int, c_void_p]),
    "paged_copy_blocks": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_int32, c_int64, c_int32,
                                  c_int32, c_int32, c_int64, c_int, c_void_p]),
    "paged_copy_blocks_fp8": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_int32,
                                      c_int64, c_int32, c_int32, c_int32, c_int64, c_void_p]),
    "paged_decode_plan": (c_int, [c_int32, c_int32, c_int32, c_int32, c_int32, c_int64, c_int32, c_int,
                                  P32, P32, P32, POINTER(c_size_t)]),
    "paged_decode_workspace_size": (c_int, [c_int32, c_int32, c_int32, c_int32, c_int32, c_int64, c_int32,
                                            c_int, POINTER(c_size_t)]),
    "paged_decode_attention": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int32,
                                       c_int32, c_int32, c_int32, c_int32, c_int64, c_int32, c_int64, c_float,
                                       c_int32, c_int, c_void_p, c_size_t, c_void_p]),
    "paged_decode_step": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_int64,
                                  c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32,
                                  c_int32, c_int32, c_int64, c_int32, c_int64, c_float, c_int, c_void_p, c_size_t,
                                  c_void_p]),
    "paged_decode_attention_static_scratch": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                                      c_int32, c_int32, c_int32, c_int32, c_int32, c_int64,
                                                      c_int32, c_int64, c_float, c_int32, c_int, c_void_p]),
    "paged_decode_static_scratch_bytes": (c_size_t, []),
    "kv_device_error": (c_int, [c_int, POINTER(c_int)]),
    "kv_last_cuda_error": (c_char_p, []),
    "kvstep_create": (c_int, [c_void_p, POINTER(kvstep_config_t), POINTER(c_void_p)]),
    "kvstep_destroy": (c_int, [c_void_p]),
    "kvstep_run": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_void_p, c_void_p,
                           c_int64, c_void_p, c_int64, c_void_p, c_int64]),
    "kvstep_join": (c_int, [c_void_p, c_void_p]),
    "kvstep_stage_buffer": (c_int, [c_void_p, c_int32, POINTER(c_void_p), POINTER(c_void_p), POINTER(c_void_p),
                                    POINTER(c_int32)]),
    "kvstep_last_buffers": (c_int, [c_void_p, POINTER(c_void_p), POINTER(c_void_p), POINTER(c_void_p),
                                    POINTER(c_void_p)]),
    "kv_debug_set": (c_int, [c_int, c_int64]),
    "kv_version": (c_char_p, []),
}

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library.  Raises ImportError if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it first with "
                "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc, CUDA 13)")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def status_string(status: int) -> str:
    return lib().kv_status_string(status).decode()


def check(status: int, where: str) -> None:
    if status != KV_OK:
        if status == 7:
            where = f"{where} [{lib().kv_last_cuda_error().decode()}]"
        raise KVError(status, where)
