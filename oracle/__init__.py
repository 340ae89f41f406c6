"""CPU oracle for the paged KV cache hot path -- TEST INFRASTRUCTURE ONLY.

This package is a plain, slow, obviously-correct restatement of what the
paged KV cache computes, written in Python/numpy with float64 arithmetic.
It exists to check the CUDA library; it is not part of the product.  Only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it.  The product package never imports it and has
no CPU fallback that could route through it.

The oracle shares no code with the CUDA library (``csrc/``): no kernels,
headers, helpers, tables or constants.  It takes every input as plain
arrays; the seeded input generators live in their own module and hold none
of the method's arithmetic.

Sources (cited by page title and section throughout):

* "MiniPaged-Qwen: Paged KV Cache 与 KV Block Manager" (blog.zsmgc.love),
  abbreviated *MiniPaged-Qwen* -- address mapping (§3, §4.1), append_token
  (§9), cache layout and slot decomposition (§11), cache write (§12), decode
  attention through block tables (§13), GQA head mapping (§14), invariants
  (§15), internal fragmentation (§6.2).
* "从零实现一个 mini vLLM: Block Manager" (yjxyzxyz.cn), abbreviated
  *mini-vLLM Block Manager* -- prefill allocation, decode slot append,
  release, invariants and the lifecycle example.
* "22. vLLM PagedAttention | vLLM 分页注意力" (datawhalechina
  llm-algo-leetcode), abbreviated *LLM-algo ch.22* -- KVCacheManager
  exercise: atomic prefill, decode growth with rollback, release
  validation, logical gather, capacity ledger, allocation report.

Modules:

* ``block_manager`` -- the reference block manager (free-list policy).
* ``prefix_sharing`` -- the same manager with per-block reference counts,
  forked sequences sharing a prefix, and copy-on-write
  ("paged-attention-impl-detail", section Copy-on-Write共享).
* ``paged_cache``   -- address mapping, scatter (cache write), gather.
* ``attention``     -- float64 decode attention, online-softmax form, and
  the split/merge identity used by split-K.
* ``ledger``        -- KV capacity ledger, allocation report, tail waste.

Every function here is pinned by ``tests/test_oracle_*.py`` against values
the pages print, closed forms, invariants, or a library routine.
"""

from . import attention, block_manager, ledger, paged_cache, prefix_sharing  # noqa: F401
