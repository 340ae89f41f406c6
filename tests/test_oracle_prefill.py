"""Pins for the chunked-prefill oracle (oracle.attention.chunked_prefill_attention).

Independent of its own code: torch's scaled_dot_product_attention in
float64 with an explicit causal-with-offset mask (chunk token t may see keys
0..L-n+t) and the GQA heads repeated; a chunk of one token is decode; the
first token of a sequence with no history returns its own V row exactly;
and changing keys or values after a token's position leaves its output
unchanged (causality), while changing one before it does not; with q = 0
every row is the plain mean of V over its prefix (closed form).
"""

import numpy as np
import pytest
import torch

from oracle.attention import chunked_prefill_attention, decode_attention_contiguous


def _sdpa(q, K, V, scale):
    n, hq, d = q.shape
    L, hkv, _ = K.shape
    g = hq // hkv
    qt = torch.from_numpy(q).permute(1, 0, 2)                       # [Hq, n, D]
    kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(g, 0)
    vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(g, 0)
    pos = torch.arange(L - n, L)[:, None]
    mask = torch.arange(L)[None, :] <= pos                          # [n, L]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    return o.permute(1, 0, 2).numpy()


@pytest.mark.parametrize("n,L,hq,hkv", [(1, 1, 2, 1), (4, 4, 4, 2), (5, 12, 8, 2), (16, 40, 7, 7), (9, 9, 28, 4)])
def test_matches_sdpa_with_offset_causal_mask(n, L, hq, hkv):
    rng = np.random.default_rng(n * 100 + L)
    d = 16
    q = rng.standard_normal((n, hq, d))
    K = rng.standard_normal((L, hkv, d))
    V = rng.standard_normal((L, hkv, d))
    scale = 1.0 / np.sqrt(d)
    assert np.allclose(chunked_prefill_attention(q, K, V, scale), _sdpa(q, K, V, scale), atol=1e-12, rtol=0)


def test_one_token_chunk_is_decode_and_first_token_is_its_value():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((6, 4, 8))
    K = rng.standard_normal((6, 2, 8))
    V = rng.standard_normal((6, 2, 8))
    out = chunked_prefill_attention(q, K, V, 0.4)
    assert np.array_equal(out[0, 0], V[0, 0]) and np.array_equal(out[0, 3], V[0, 1])
    last = chunked_prefill_attention(q[-1:], K, V, 0.4)
    assert np.array_equal(last[0], decode_attention_contiguous(q[-1], K, V, 0.4))


def test_causality():
    rng = np.random.default_rng(4)
    n, L = 5, 11
    q = rng.standard_normal((n, 4, 8))
    K = rng.standard_normal((L, 2, 8))
    V = rng.standard_normal((L, 2, 8))
    base = chunked_prefill_attention(q, K, V, 0.35)
    t = 2
    p = L - n + t
    K2, V2 = K.copy(), V.copy()
    K2[p + 1:] += 3.0
    V2[p + 1:] -= 2.0
    assert np.array_equal(chunked_prefill_attention(q, K2, V2, 0.35)[t], base[t])
    K3 = K.copy()
    K3[p - 1] += 1.0
    assert not np.allclose(chunked_prefill_attention(q, K3, V, 0.35)[t], base[t])
    with pytest.raises(ValueError):
        chunked_prefill_attention(rng.standard_normal((12, 4, 8)), K, V, 0.35)


@pytest.mark.parametrize("ctx", [0, 9])
def test_zero_query_gives_prefix_means(ctx):
    """q = 0 makes every score equal, so chunk token t (position ctx + t)
    returns the plain mean of V over keys 0 .. ctx + t, for every query head
    of its kv head: a closed form that pins the causal bound and the history
    offset without any attention routine."""
    rng = np.random.default_rng(40 + ctx)
    n, hq, hkv, d = 6, 4, 2, 8
    L = ctx + n
    K = rng.standard_normal((L, hkv, d))
    V = rng.standard_normal((L, hkv, d))
    got = chunked_prefill_attention(np.zeros((n, hq, d)), K, V, 0.3)
    for t in range(n):
        p = ctx + t
        for h in range(hq):
            want = V[:p + 1, h // (hq // hkv)].mean(axis=0)
            np.testing.assert_allclose(got[t, h], want, rtol=0, atol=1e-13)
