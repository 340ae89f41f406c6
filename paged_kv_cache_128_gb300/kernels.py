"""Torch-facing wrappers of the CUDA entry points in libpagedkv.

Argument marshalling only: shapes, dtypes and device pointers are read off
the tensors and passed to the C ABI; every step of the computation runs in
the library's kernels.  There is no CPU path: CPU tensors are rejected.
"""

from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Optional

import torch

from ._lib import DTYPE_BF16, DTYPE_F16, DTYPE_F32, KVError, check, lib

_DTYPES = {torch.float32: DTYPE_F32, torch.float16: DTYPE_F16, torch.bfloat16: DTYPE_BF16}


def dtype_code(dtype: torch.dtype) -> int:
    if dtype not in _DTYPES:
        raise KVError(1, f"unsupported dtype {dtype}")
    return _DTYPES[dtype]


def _stream_ptr(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _cuda(t: torch.Tensor, name: str) -> torch.Tensor:
    if not t.is_cuda:
        raise KVError(1, f"{name} must be a CUDA tensor")
    return t


def reshape_and_cache(k: torch.Tensor, v: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      slot_mapping: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> None:
    """Write k/v ``[N, Hkv, D]`` (token stride may exceed Hkv*D) into the
    ``[NB, BS, Hkv, D]`` caches at ``slot_mapping[N]`` (int32, -1 = skip)."""
    for t, n in ((k, "k"), (v, "v"), (k_cache, "k_cache"), (v_cache, "v_cache"), (slot_mapping, "slot_mapping")):
        _cuda(t, n)
    nb, bs, hkv, d = k_cache.shape
    n = slot_mapping.numel()
    if slot_mapping.dtype != torch.int32 or not slot_mapping.is_contiguous():
        raise KVError(1, "slot_mapping must be contiguous int32")
    if k.dtype != k_cache.dtype or v.dtype != k_cache.dtype or v_cache.dtype != k_cache.dtype:
        raise KVError(1, "k, v and the caches must share one dtype")
    if not (k_cache.is_contiguous() and v_cache.is_contiguous() and v_cache.shape == k_cache.shape):
        raise KVError(1, "caches must be contiguous [NB, BS, Hkv, D] of one shape")
    for t in (k, v):
        if t.dim() != 3 or t.shape[0] != n or t.shape[1] != hkv or t.shape[2] != d or t.stride(2) != 1 \
                or t.stride(1) != d:
            raise KVError(1, "k and v must be [N, Hkv, D] with dense heads")
    check(lib().paged_reshape_and_cache(k.data_ptr(), v.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                        slot_mapping.data_ptr(), n, hkv, d, bs, nb, k.stride(0), v.stride(0),
                                        dtype_code(k_cache.dtype), _stream_ptr(stream)),
          "paged_reshape_and_cache")


def reshape_and_cache_layers(k: torch.Tensor, v: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                             slot_mapping: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> None:
    """Write k/v ``[L, N, Hkv, D]`` into L layers' caches ``[L, NB, BS, Hkv,
    D]`` at ``slot_mapping[N]`` (int32, -1 = skip) in one launch: one block
    table and slot mapping serve every layer."""
    for t, n in ((k, "k"), (v, "v"), (k_cache, "k_cache"), (v_cache, "v_cache"), (slot_mapping, "slot_mapping")):
        _cuda(t, n)
    if k_cache.dim() != 5 or not (k_cache.is_contiguous() and v_cache.is_contiguous()) \
            or v_cache.shape != k_cache.shape:
        raise KVError(1, "caches must be contiguous [L, NB, BS, Hkv, D] of one shape")
    layers, nb, bs, hkv, d = k_cache.shape
    n = slot_mapping.numel()
    if slot_mapping.dtype != torch.int32 or not slot_mapping.is_contiguous():
        raise KVError(1, "slot_mapping must be contiguous int32")
    if k.dtype != k_cache.dtype or v.dtype != k_cache.dtype or v_cache.dtype != k_cache.dtype:
        raise KVError(1, "k, v and the caches must share one dtype")
    for t in (k, v):
        if t.dim() != 4 or tuple(t.shape) != (layers, n, hkv, d) or t.stride(3) != 1 or t.stride(2) != d:
            raise KVError(1, "k and v must be [L, N, Hkv, D] with dense heads")
    check(lib().paged_reshape_and_cache_layers(k.data_ptr(), v.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                               slot_mapping.data_ptr(), n, layers, k.stride(0), v.stride(0),
                                               k_cache.stride(0), hkv, d, bs, nb, k.stride(1), v.stride(1),
                                               dtype_code(k_cache.dtype), _stream_ptr(stream)),
          "paged_reshape_and_cache_layers")


def reshape_and_cache_fp8(k: torch.Tensor, v: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                          k_scales: torch.Tensor, v_scales: torch.Tensor, slot_mapping: torch.Tensor,
                          stream: Optional[torch.cuda.Stream] = None) -> None:
    """Quantised cache write: k/v ``[N, Hkv, D]`` (fp16/bf16) to E4M3 codes
    ``[NB, BS, Hkv, D]`` (uint8) with one float32 scale per (token, kv head)
    in ``[NB, Hkv, BS]`` scale arrays, at ``slot_mapping[N]`` (-1 = skip)."""
    for t, n in ((k, "k"), (v, "v"), (k_cache, "k_cache"), (v_cache, "v_cache"), (k_scales, "k_scales"),
                 (v_scales, "v_scales"), (slot_mapping, "slot_mapping")):
        _cuda(t, n)
    if k_cache.dtype != torch.uint8 or v_cache.dtype != torch.uint8 or k_scales.dtype != torch.float32 \
            or v_scales.dtype != torch.float32:
        raise KVError(1, "fp8 caches are uint8 codes with float32 scales")
    nb, bs, hkv, d = k_cache.shape
    if v_cache.shape != k_cache.shape or tuple(k_scales.shape) != (nb, hkv, bs) or v_scales.shape != k_scales.shape:
        raise KVError(1, "caches [NB, BS, Hkv, D], scales [NB, Hkv, BS]")
    if not all(t.is_contiguous() for t in (k_cache, v_cache, k_scales, v_scales, slot_mapping)) \
            or slot_mapping.dtype != torch.int32:
        raise KVError(1, "caches, scales and slot_mapping must be contiguous (slot_mapping int32)")
    n = slot_mapping.numel()
    for t in (k, v):
        if t.dim() != 3 or t.shape[0] != n or t.shape[1] != hkv or t.shape[2] != d or t.stride(2) != 1 \
                or t.stride(1) != d:
            raise KVError(1, "k and v must be [N, Hkv, D] with dense heads")
    check(lib().paged_reshape_and_cache_fp8(k.data_ptr(), v.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                            k_scales.data_ptr(), v_scales.data_ptr(), slot_mapping.data_ptr(), n, hkv,
                                            d, bs, nb, k.stride(0), v.stride(0), dtype_code(k.dtype),
                                            _stream_ptr(stream)), "paged_reshape_and_cache_fp8")


def paged_decode_attention_fp8(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                               k_scales: torch.Tensor, v_scales: torch.Tensor, block_tables: torch.Tensor,
                               seq_lens: torch.Tensor, scale: float, max_seq_len: int,
                               workspace: Optional[torch.Tensor] = None,
                               stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Decode attention over fp8 (E4M3) caches with per-token scales; q and
    out fp16/bf16 ``[B, Hq, D]``."""
    for t, n in ((out, "out"), (q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (k_scales, "k_scales"),
                 (v_scales, "v_scales"), (block_tables, "block_tables"), (seq_lens, "seq_lens")):
        _cuda(t, n)
    B, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    if d2 != d or out.shape != q.shape or out.dtype != q.dtype or k_cache.dtype != torch.uint8:
        raise KVError(1, "shape or dtype mismatch")
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32 or block_tables.dim() != 2 \
            or block_tables.shape[0] != B or seq_lens.numel() != B:
        raise KVError(1, "block_tables must be [B, max_blocks] and seq_lens [B], int32")
    if workspace is None:
        workspace = alloc_workspace(decode_plan(B, hq, hkv, d, bs, max_seq_len, q.dtype), q.device)
    ws_ptr, ws_bytes = (workspace.data_ptr(), workspace.numel()) if workspace is not None else (None, 0)
    check(lib().paged_decode_attention_fp8(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                           k_scales.data_ptr(), v_scales.data_ptr(), block_tables.data_ptr(),
                                           seq_lens.data_ptr(), B, hq, hkv, d, bs, nb, block_tables.shape[1],
                                           max_seq_len, float(scale), dtype_code(q.dtype), ws_ptr, ws_bytes,
                                           _stream_ptr(stream)), "paged_decode_attention_fp8")
    return out


def paged_decode_step_fp8(out: torch.Tensor, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                          slot_mapping: torch.Tensor, new_token_row: torch.Tensor, k_cache: torch.Tensor,
                          v_cache: torch.Tensor, k_scales: torch.Tensor, v_scales: torch.Tensor,
                          block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float, max_seq_len: int,
                          workspace: Optional[torch.Tensor] = None,
                          stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """The step's quantised cache write and decode attention over fp8
    caches in one call (one launch when the rows are 8-byte aligned)."""
    for t, n in ((out, "out"), (q, "q"), (k, "k"), (v, "v"), (slot_mapping, "slot_mapping"),
                 (new_token_row, "new_token_row"), (k_cache, "k_cache"), (v_cache, "v_cache"),
                 (k_scales, "k_scales"), (v_scales, "v_scales"), (block_tables, "block_tables"),
                 (seq_lens, "seq_lens")):
        _cuda(t, n)
    B, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    n = slot_mapping.numel()
    if d2 != d or out.shape != q.shape or out.dtype != q.dtype or k_cache.dtype != torch.uint8 \
            or k.dtype != q.dtype or v.dtype != q.dtype:
        raise KVError(1, "shape or dtype mismatch")
    for t, nm in ((block_tables, "block_tables"), (seq_lens, "seq_lens"), (slot_mapping, "slot_mapping"),
                  (new_token_row, "new_token_row")):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise KVError(1, f"{nm} must be contiguous int32")
    for t in (k, v):
        if t.dim() != 3 or t.shape[0] != n or t.shape[1] != hkv or t.shape[2] != d or t.stride(2) != 1 \
                or t.stride(1) != d:
            raise KVError(1, "k and v must be [N, Hkv, D] with dense heads")
    if workspace is None:
        workspace = alloc_workspace(decode_plan(B, hq, hkv, d, bs, max_seq_len, q.dtype), q.device)
    ws_ptr, ws_bytes = (workspace.data_ptr(), workspace.numel()) if workspace is not None else (None, 0)
    check(lib().paged_decode_step_fp8(out.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                      slot_mapping.data_ptr(), n, k.stride(0), v.stride(0), new_token_row.data_ptr(),
                                      k_cache.data_ptr(), v_cache.data_ptr(), k_scales.data_ptr(), v_scales.data_ptr(),
                                      block_tables.data_ptr(), seq_lens.data_ptr(), B, hq, hkv, d, bs, nb,
                                      block_tables.shape[1], max_seq_len, float(scale), dtype_code(q.dtype), ws_ptr,
                                      ws_bytes, _stream_ptr(stream)), "paged_decode_step_fp8")
    return out


def paged_prefill_attention(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            block_tables: torch.Tensor, seq_lens: torch.Tensor, query_start_loc: torch.Tensor,
                            scale: float, max_query_len: int,
                            stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Chunked prefill: q/out ``[T, Hq, D]``, sequence b's chunk is rows
    ``query_start_loc[b]:query_start_loc[b+1]``, its last positions; each
    chunk token attends causally to its sequence's keys through the table."""
    for t, n in ((out, "out"), (q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"), (block_tables, "block_tables"),
                 (seq_lens, "seq_lens"), (query_start_loc, "query_start_loc")):
        _cuda(t, n)
    if not (q.is_contiguous() and out.is_contiguous() and k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise KVError(1, "q, out and caches must be contiguous")
    nb, bs, hkv, d = k_cache.shape
    T, hq, d2 = q.shape
    B = seq_lens.numel()
    if d2 != d or out.shape != q.shape or out.dtype != q.dtype or k_cache.dtype != q.dtype \
            or v_cache.shape != k_cache.shape or v_cache.dtype != q.dtype:
        raise KVError(1, "shape or dtype mismatch")
    for t, nm in ((block_tables, "block_tables"), (seq_lens, "seq_lens"), (query_start_loc, "query_start_loc")):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise KVError(1, f"{nm} must be contiguous int32")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or query_start_loc.numel() != B + 1:
        raise KVError(1, "block_tables [B, max_blocks], seq_lens [B], query_start_loc [B + 1]")
    check(lib().paged_prefill_attention(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                        block_tables.data_ptr(), seq_lens.data_ptr(), query_start_loc.data_ptr(), T,
                                        B, hq, hkv, d, bs, nb, block_tables.shape[1], max_query_len, float(scale),
                                        dtype_code(q.dtype), _stream_ptr(stream)), "paged_prefill_attention")
    return out


def copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, src: torch.Tensor, dst: torch.Tensor,
                stream: Optional[torch.cuda.Stream] = None) -> None:
    """Copy-on-write copies: block ``dst[i]`` of every layer's K and V cache
    becomes a copy of block ``src[i]`` (int32 device tensors).  Caches are
    ``[NB, BS, Hkv, D]`` or ``[layers, NB, BS, Hkv, D]``, contiguous."""
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache"), (src, "src"), (dst, "dst")):
        _cuda(t, n)
    if not (k_cache.is_contiguous() and v_cache.is_contiguous() and k_cache.shape == v_cache.shape
            and k_cache.dtype == v_cache.dtype):
        raise KVError(1, "caches must be contiguous, of one shape and dtype")
    if src.dtype != torch.int32 or dst.dtype != torch.int32 or src.numel() != dst.numel() \
            or not src.is_contiguous() or not dst.is_contiguous():
        raise KVError(1, "src and dst must be contiguous int32 of one length")
    if k_cache.dim() == 4:
        layers, (nb, bs, hkv, d) = 1, k_cache.shape
        stride = 0
    elif k_cache.dim() == 5:
        layers, nb, bs, hkv, d = k_cache.shape
        stride = k_cache.stride(0)
    else:
        raise KVError(1, "caches must be 4-D or 5-D")
    check(lib().paged_copy_blocks(k_cache.data_ptr(), v_cache.data_ptr(), src.data_ptr(), dst.data_ptr(),
                                  src.numel(), layers, stride, hkv, d, bs, nb, dtype_code(k_cache.dtype),
                                  _stream_ptr(stream)), "paged_copy_blocks")


def copy_blocks_fp8(k_cache: torch.Tensor, v_cache: torch.Tensor, k_scales: torch.Tensor, v_scales: torch.Tensor,
                    src: torch.Tensor, dst: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> None:
    """Copy-on-write copies for fp8 caches: block ``dst[i]`` takes block
    ``src[i]``'s K and V codes (uint8 ``[NB, BS, Hkv, D]``, or with a leading
    layer axis) and scales (float32 ``[NB, Hkv, BS]``, likewise)."""
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache"), (k_scales, "k_scales"), (v_scales, "v_scales"),
                 (src, "src"), (dst, "dst")):
        _cuda(t, n)
    if k_cache.dtype != torch.uint8 or v_cache.shape != k_cache.shape or k_scales.dtype != torch.float32 \
            or v_scales.shape != k_scales.shape or not all(t.is_contiguous() for t in (k_cache, v_cache, k_scales,
                                                                                       v_scales)):
        raise KVError(1, "fp8 caches: contiguous uint8 codes and float32 scales")
    if src.dtype != torch.int32 or dst.dtype != torch.int32 or src.numel() != dst.numel():
        raise KVError(1, "src and dst must be contiguous int32 of one length")
    if k_cache.dim() == 4:
        layers, (nb, bs, hkv, d) = 1, k_cache.shape
        stride = 0
    elif k_cache.dim() == 5:
        layers, nb, bs, hkv, d = k_cache.shape
        stride = k_cache.stride(0)
    else:
        raise KVError(1, "caches must be 4-D or 5-D")
    check(lib().paged_copy_blocks_fp8(k_cache.data_ptr(), v_cache.data_ptr(), k_scales.data_ptr(),
                                      v_scales.data_ptr(), src.data_ptr(), dst.data_ptr(), src.numel(), layers,
                                      stride, hkv, d, bs, nb, _stream_ptr(stream)), "paged_copy_blocks_fp8")


@dataclass
class DecodePlan:
    kernel: int            # 0 = SIMT, 1 = split TMA + tensor cores, 2 = stream-K TMA + tensor cores
    blocks_per_split: int
    num_splits: int
    workspace_bytes: int

    @property
    def launches(self) -> int:
        """Kernels one attention call launches: the split kernels add a merge
        kernel when a sequence spans several splits; stream-K merges inside."""
        return 2 if (self.kernel != 2 and self.num_splits > 1) else 1


def decode_plan(num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                max_seq_len: int, dtype: torch.dtype, blocks_per_split: int = 0) -> DecodePlan:
    k, b, s = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    w = ctypes.c_size_t()
    check(lib().paged_decode_plan(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_seq_len,
                                  blocks_per_split, dtype_code(dtype), ctypes.byref(k), ctypes.byref(b),
                                  ctypes.byref(s), ctypes.byref(w)), "paged_decode_plan")
    return DecodePlan(k.value, b.value, s.value, w.value)


def alloc_workspace(plan: DecodePlan, device) -> Optional[torch.Tensor]:
    if plan.workspace_bytes == 0:
        return None
    return torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device=device)


def paged_decode_attention(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float, max_seq_len: int,
                           blocks_per_split: int = 0, workspace: Optional[torch.Tensor] = None,
                           stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """out[b, qh] = softmax(scale * q[b, qh] K^T) V over seq_lens[b] tokens
    read through block_tables[b]; kvh = qh // (Hq // Hkv).  ``workspace``
    must hold ``decode_plan(...).workspace_bytes`` bytes when that is > 0
    (allocated here if omitted)."""
    for t, n in ((out, "out"), (q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"),
                 (block_tables, "block_tables"), (seq_lens, "seq_lens")):
        _cuda(t, n)
    if not (q.is_contiguous() and out.is_contiguous() and k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise KVError(1, "q, out and caches must be contiguous")
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32 or not block_tables.is_contiguous() \
            or not seq_lens.is_contiguous():
        raise KVError(1, "block_tables and seq_lens must be contiguous int32")
    B, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    if d2 != d or out.shape != q.shape or v_cache.shape != k_cache.shape or out.dtype != q.dtype \
            or k_cache.dtype != q.dtype or v_cache.dtype != q.dtype:
        raise KVError(1, "shape or dtype mismatch")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or seq_lens.numel() != B:
        raise KVError(1, "block_tables must be [B, max_blocks] and seq_lens [B]")
    code = dtype_code(q.dtype)
    ws_ptr, ws_bytes = None, 0
    if workspace is None:
        plan = decode_plan(B, hq, hkv, d, bs, max_seq_len, q.dtype, blocks_per_split)
        workspace = alloc_workspace(plan, q.device)
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    check(lib().paged_decode_attention(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                       block_tables.data_ptr(), seq_lens.data_ptr(), B, hq, hkv, d, bs, nb,
                                       block_tables.shape[1], max_seq_len, float(scale), blocks_per_split, code,
                                       ws_ptr, ws_bytes, _stream_ptr(stream)), "paged_decode_attention")
    return out


def paged_decode_step(out: torch.Tensor, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                      slot_mapping: torch.Tensor, new_token_row: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                      max_seq_len: int, workspace: Optional[torch.Tensor] = None,
                      stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """The step's cache write (``reshape_and_cache(k, v, ..., slot_mapping)``)
    and decode attention in one call: one launch when the stream-K kernel
    applies.  ``new_token_row[b]`` (int32) is the row of k/v holding
    sequence b's newest token, position ``seq_lens[b] - 1``, or -1."""
    for t, n in ((out, "out"), (q, "q"), (k, "k"), (v, "v"), (slot_mapping, "slot_mapping"),
                 (new_token_row, "new_token_row"), (k_cache, "k_cache"), (v_cache, "v_cache"),
                 (block_tables, "block_tables"), (seq_lens, "seq_lens")):
        _cuda(t, n)
    if not (q.is_contiguous() and out.is_contiguous() and k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise KVError(1, "q, out and caches must be contiguous")
    for t, n in ((block_tables, "block_tables"), (seq_lens, "seq_lens"), (slot_mapping, "slot_mapping"),
                 (new_token_row, "new_token_row")):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise KVError(1, f"{n} must be contiguous int32")
    B, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    n = slot_mapping.numel()
    if d2 != d or out.shape != q.shape or v_cache.shape != k_cache.shape or out.dtype != q.dtype \
            or k_cache.dtype != q.dtype or v_cache.dtype != q.dtype or k.dtype != q.dtype or v.dtype != q.dtype:
        raise KVError(1, "shape or dtype mismatch")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or seq_lens.numel() != B \
            or new_token_row.numel() != B:
        raise KVError(1, "block_tables must be [B, max_blocks], seq_lens and new_token_row [B]")
    for t in (k, v):
        if t.dim() != 3 or t.shape[0] != n or t.shape[1] != hkv or t.shape[2] != d or t.stride(2) != 1 \
                or t.stride(1) != d:
            raise KVError(1, "k and v must be [N, Hkv, D] with dense heads")
    ws_ptr, ws_bytes = None, 0
    if workspace is None:
        plan = decode_plan(B, hq, hkv, d, bs, max_seq_len, q.dtype)
        workspace = alloc_workspace(plan, q.device)
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    check(lib().paged_decode_step(out.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), slot_mapping.data_ptr(),
                                  n, k.stride(0), v.stride(0), new_token_row.data_ptr(), k_cache.data_ptr(),
                                  v_cache.data_ptr(), block_tables.data_ptr(), seq_lens.data_ptr(), B, hq, hkv, d, bs,
                                  nb, block_tables.shape[1], max_seq_len, float(scale), dtype_code(q.dtype), ws_ptr,
                                  ws_bytes, _stream_ptr(stream)), "paged_decode_step")
    return out


def device_error(reset: bool = True) -> int:
    """Status recorded by device-side bounds checks / bounded waits (0 = none).
    Synchronises the current device."""
    st = ctypes.c_int()
    check(lib().kv_device_error(1 if reset else 0, ctypes.byref(st)), "kv_device_error")
    return st.value


def paged_decode_attention_static_scratch(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                                          v_cache: torch.Tensor, block_tables: torch.Tensor,
                                          seq_lens: torch.Tensor, scale: float, max_seq_len: int,
                                          blocks_per_split: int = 0,
                                          stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """``paged_decode_attention`` for callers that must not allocate device
    memory: the library's fixed scratch array stands in for the workspace
    (see include/pagedkv.h).  Nothing is allocated here either.  Raises
    KVError(WORKSPACE) when these sizes need more scratch than the array."""
    for t, n in ((out, "out"), (q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache"),
                 (block_tables, "block_tables"), (seq_lens, "seq_lens")):
        _cuda(t, n)
    if not (q.is_contiguous() and out.is_contiguous() and k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise KVError(1, "q, out and caches must be contiguous")
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32 or not block_tables.is_contiguous() \
            or not seq_lens.is_contiguous():
        raise KVError(1, "block_tables and seq_lens must be contiguous int32")
    B, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    if d2 != d or out.shape != q.shape or v_cache.shape != k_cache.shape or out.dtype != q.dtype \
            or k_cache.dtype != q.dtype or v_cache.dtype != q.dtype:
        raise KVError(1, "shape or dtype mismatch")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or seq_lens.numel() != B:
        raise KVError(1, "block_tables must be [B, max_blocks] and seq_lens [B]")
    check(lib().paged_decode_attention_static_scratch(
        out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
        seq_lens.data_ptr(), B, hq, hkv, d, bs, nb, block_tables.shape[1], max_seq_len, float(scale),
        blocks_per_split, dtype_code(q.dtype), _stream_ptr(stream)), "paged_decode_attention_static_scratch")
    return out


# Stream-K test controls (kv_debug_set keys), process-wide.
DEBUG_WAIT_LIMIT_NS = 1
DEBUG_SKIP_TILE = 2
DEBUG_DEFAULTS = {DEBUG_WAIT_LIMIT_NS: 0, DEBUG_SKIP_TILE: -1}


def debug_set(key: int, value: int) -> None:
    """Set one stream-K test control (see kv_debug_set)."""
    check(lib().kv_debug_set(int(key), int(value)), "kv_debug_set")


def debug_reset() -> None:
    """Every stream-K control back to its default."""
    for key, value in DEBUG_DEFAULTS.items():
        debug_set(key, value)


def static_scratch_bytes() -> int:
    """Size of the fixed scratch array behind the no-allocation decode call."""
    return int(lib().paged_decode_static_scratch_bytes())
