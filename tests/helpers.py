"""Shared test helpers: storage conversion between torch tensors and the
oracle's numpy arrays, tolerances, and a small paged-case builder."""

import numpy as np
import torch

from oracle.block_manager import BlockManager as OracleManager
from oracle.paged_cache import reshape_and_cache as oracle_scatter
from oracle.paged_cache import to_float64

# max-abs tolerances against the float64 oracle: fp16 and bf16 are the
# stated bars; fp32 has none stated, 1e-5 covers fp32 accumulation over
# the tested lengths with a wide margin.
TOL = {"f32": 1e-5, "f16": 2e-3, "bf16": 8e-3}
TORCH = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
# significand bits (with the implicit one) of the 16-bit output types
_SIG_BITS = {"f16": 11, "bf16": 8}
_MIN_EXP = {"f16": -14, "bf16": -126}  # smallest normal exponent: below it the ulp stays fixed


def rounding_allowance(ref: np.ndarray, dtype: str) -> np.ndarray:
    """Half an ulp of each exact value in the output dtype: what rounding the
    exact result to that dtype may cost by itself (0 for f32).  For bf16
    outputs above 2 this alone reaches the stated 8e-3 bar, so checks whose
    outputs are that large compare the excess over it with the bar."""
    if dtype not in _SIG_BITS:
        return np.zeros_like(ref)
    e = np.floor(np.log2(np.maximum(np.abs(ref), np.finfo(np.float64).tiny)))
    return np.exp2(np.maximum(e, _MIN_EXP[dtype]) - _SIG_BITS[dtype])
SENTINEL = {"f32": 0x7FC00000, "f16": 0x7E00, "bf16": 0x7FC0}


def to_storage(t: torch.Tensor, dtype: str) -> np.ndarray:
    """CPU copy of a tensor in the oracle's storage form (bf16 as uint16 bits)."""
    t = t.detach().cpu().contiguous()
    if dtype == "bf16":
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


def to_f64(t: torch.Tensor, dtype: str) -> np.ndarray:
    return to_float64(to_storage(t, dtype), dtype)


def sentinel_tensor(shape, dtype: str, device) -> torch.Tensor:
    dt = TORCH[dtype]
    iv = torch.int32 if dtype == "f32" else torch.int16
    width = 32 if dtype == "f32" else 16
    bits = SENTINEL[dtype]
    if bits >= 1 << (width - 1):
        bits -= 1 << width
    t = torch.empty(shape, dtype=dt, device=device)
    t.view(iv).fill_(bits)
    return t


def sentinel_storage(shape, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.full(shape, SENTINEL["f32"], dtype=np.uint32).view(np.float32)
    if dtype == "f16":
        return np.full(shape, SENTINEL["f16"], dtype=np.uint16).view(np.float16)
    return np.full(shape, SENTINEL["bf16"], dtype=np.uint16)


def oracle_paged_pool(lens, nb, bs, hkv, d, dtype, free_order, k_hist, v_hist):
    """Oracle-side pool: prefill each sequence with its length and scatter
    its history (storage arrays) by the oracle manager's slots."""
    ora = OracleManager(nb, bs, free_order)
    kc = sentinel_storage((nb, bs, hkv, d), dtype)
    vc = sentinel_storage((nb, bs, hkv, d), dtype)
    off = 0
    slots_all = []
    for sid, L in enumerate(lens):
        if L == 0:
            slots_all.append([])
            continue
        slots = ora.allocate_for_prefill(sid, L)
        oracle_scatter(k_hist[off:off + L], v_hist[off:off + L], kc, vc, slots)
        slots_all.append(slots)
        off += L
    return ora, kc, vc, slots_all
