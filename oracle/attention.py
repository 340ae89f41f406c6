"""Float64 single-query (decode) attention through block tables -- oracle only.

What it computes (MiniPaged-Qwen §1.1 and §13): for every sequence b and
query head qh, with kv head kvh = floor(qh / (Hq / Hkv)) (MiniPaged-Qwen §14),

    o[b, qh] = sum_j softmax_j(scale * q[b, qh] . K_j) V_j,   j < seq_len[b],

where K_j, V_j are the sequence's logical tokens: its blocks walked in
block-table order and truncated to seq_len (LLM-algo ch.22 Step 4, TODO 4).
"The attention math is unchanged; only the address fetch changes"
(MiniPaged-Qwen §13), so the plain definition is the oracle.

Readings: ``scale`` is an explicit argument (the pages use 1/sqrt(D));
``seq_len == 0`` yields a zero output (the pages do not define it); the
decode token's own K/V is written before attention runs, so ``seq_len``
already counts it (mini-vLLM Block Manager, lifecycle example: the input
token's K/V is written during its own forward).

Also here: the online-softmax form the MiniPaged-Qwen CPU reference keeps
(§17.3), and the split/merge identity behind split-K decoding (partial
(acc, m, l) over disjoint token ranges, merged by their log-sum-exp).  Both
are restatements checked for equality with the two-pass form.
"""

from __future__ import annotations

from typing import List, Sequence, Tuple

import numpy as np

from .paged_cache import gather, to_float64


def kv_head_of(qh: int, num_heads: int, num_kv_heads: int) -> int:
    """MiniPaged-Qwen §14: group = Hq / Hkv, kvh = floor(qh / group)."""
    if num_heads % num_kv_heads != 0:
        raise ValueError("num_heads must be a multiple of num_kv_heads")
    return qh // (num_heads // num_kv_heads)


def attention_one(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """Two-pass softmax attention of one query row over ``K, V [L, D]``."""
    L = K.shape[0]
    if L == 0:
        return np.zeros(V.shape[1], dtype=np.float64)
    s = scale * (K @ q)            # scores [L]
    m = np.max(s)                  # pass 1: max, for a safe exponent
    p = np.exp(s - m)              # pass 2: weights
    return (p @ V) / np.sum(p)


def decode_attention_contiguous(q: np.ndarray, K: np.ndarray, V: np.ndarray,
                                scale: float) -> np.ndarray:
    """``q [Hq, D]``, ``K, V [L, Hkv, D]`` (float64) -> ``o [Hq, D]``."""
    num_heads = q.shape[0]
    num_kv_heads = K.shape[1]
    out = np.zeros((num_heads, V.shape[2]), dtype=np.float64)
    for qh in range(num_heads):
        kvh = kv_head_of(qh, num_heads, num_kv_heads)
        out[qh] = attention_one(q[qh], K[:, kvh, :], V[:, kvh, :], scale)
    return out


def paged_decode_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                           block_tables: Sequence[Sequence[int]], seq_lens: Sequence[int],
                           scale: float, dtype: str) -> np.ndarray:
    """``q [B, Hq, D]`` and caches ``[NB, BS, Hkv, D]`` in storage form.

    Per sequence: gather in table order, truncate, widen to float64, then the
    contiguous definition.  Returns float64 ``[B, Hq, D]``."""
    B, num_heads, D = q.shape
    out = np.zeros((B, num_heads, D), dtype=np.float64)
    qf = to_float64(q, dtype)
    for b in range(B):
        L = int(seq_lens[b])
        K = to_float64(gather(k_cache, block_tables[b], L), dtype)
        V = to_float64(gather(v_cache, block_tables[b], L), dtype)
        out[b] = decode_attention_contiguous(qf[b], K, V, scale)
    return out


# -- online softmax (MiniPaged-Qwen §17.3 CPU reference) ------------------------

def attention_one_online(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """One token at a time: running max m, running sum l, rescaled acc."""
    D = V.shape[1]
    m, l, acc = -np.inf, 0.0, np.zeros(D, dtype=np.float64)
    for j in range(K.shape[0]):
        s = scale * float(K[j] @ q)
        m_new = max(m, s)
        alpha = np.exp(m - m_new) if m != -np.inf else 0.0
        p = np.exp(s - m_new)
        l = l * alpha + p
        acc = acc * alpha + p * V[j]
        m = m_new
    return acc / l if l > 0 else acc


# -- split-K identity -------------------------------------------------------------

def partial_state(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float
                  ) -> Tuple[np.ndarray, float, float]:
    """Unnormalised (acc, m, l) of one token range: acc = sum_j e^{s_j - m} V_j,
    l = sum_j e^{s_j - m}, m = max_j s_j.  An empty range is (0, -inf, 0)."""
    if K.shape[0] == 0:
        return np.zeros(V.shape[1], dtype=np.float64), -np.inf, 0.0
    s = scale * (K @ q)
    m = float(np.max(s))
    p = np.exp(s - m)
    return p @ V, m, float(np.sum(p))


def merge_states(states: List[Tuple[np.ndarray, float, float]]) -> np.ndarray:
    """Log-sum-exp merge: M = max_s m_s, out = sum_s e^{m_s-M} acc_s /
    sum_s e^{m_s-M} l_s.  Ranges with no tokens carry m = -inf and drop out."""
    live = [st for st in states if st[1] != -np.inf]
    if not live:
        return np.zeros_like(states[0][0])
    M = max(st[1] for st in live)
    num = sum(np.exp(st[1] - M) * st[0] for st in live)
    den = sum(np.exp(st[1] - M) * st[2] for st in live)
    return num / den


def chunked_prefill_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """Attention of a sequence's new chunk over its history and the chunk.

    ``q [n, Hq, D]`` are the chunk's queries, the last n of the sequence's
    L tokens; ``K, V [L, Hkv, D]`` its logical keys and values (history,
    then the chunk), float64.  Chunk token t sits at position p = L - n + t
    and attends to keys 0..p (causal within the chunk, all history before
    it): "从零实现一个 mini vLLM: Block Manager" (a chunked prefill allocates
    the chunk's slots, writes their K/V, then attends through the block
    table) and MiniPaged-Qwen §13 (attention over positions read through the
    table).  Each row is the decode attention of that token over its prefix,
    so a chunk of one token is exactly decode.  -> ``o [n, Hq, D]``.
    """
    n = q.shape[0]
    L = K.shape[0]
    if n > L:
        raise ValueError("chunk longer than the sequence")
    out = np.empty(q.shape, dtype=np.float64)
    for t in range(n):
        p = L - n + t
        out[t] = decode_attention_contiguous(q[t], K[:p + 1], V[:p + 1], scale)
    return out
