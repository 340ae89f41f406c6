"""GB300-native paged KV cache: host block manager + sm_103a kernels.

Public API (all work runs in libpagedkv.so; see include/pagedkv.h):

* ``KVBlockManager`` -- host metadata plane (prefill / decode allocation,
  release, export of block tables, seq_lens and slot_mapping).
* ``reshape_and_cache`` -- CUDA cache write by slot_mapping.
* ``paged_decode_attention`` -- CUDA single-query GQA attention through
  block tables, with split-K and a log-sum-exp merge.
* ``paged_decode_step`` -- the step's cache write and decode attention in
  one launch (stream-K kernel), else the two in stream order.
"""

from ._lib import KVError, LIB_PATH, lib  # noqa: F401
from .block_manager import KVBlockManager, kv_cache_ledger  # noqa: F401


def __getattr__(name):
    # the kernel wrappers need torch; import them on first use
    if name in ("reshape_and_cache", "reshape_and_cache_layers", "paged_decode_attention", "paged_decode_step", "copy_blocks", "decode_plan",
                "device_error", "alloc_workspace", "DecodePlan", "reshape_and_cache_fp8",
                "paged_decode_attention_fp8", "paged_decode_step_fp8", "paged_prefill_attention"):
        from . import kernels
        return getattr(kernels, name)
    raise AttributeError(name)
