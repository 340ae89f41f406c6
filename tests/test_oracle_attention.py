"""Pins for the float64 oracle attention.

Each pin comes from outside the oracle's own formula: closed forms (one
token, equal keys, zero query, two tokens = logistic weights), a library
routine (torch's scaled_dot_product_attention in float64, scipy's softmax),
the MiniPaged-Qwen §14 head mapping printed on the page, and brute-force
equalities (online form, split merge).  The last tests plant mistakes in the
oracle and check a pin catches each one.
"""

import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle.attention as att
from oracle.block_manager import BlockManager
from oracle.paged_cache import reshape_and_cache
from tests.conftest import load_golden

G_MAP = load_golden("address_mapping.json")


def _rng(seed):
    return np.random.default_rng(seed)


def _paged_setup(seed, lens, hq, hkv, d, bs, nb=None, dtype=np.float64):
    """Logical K/V per sequence, written into a NaN-filled pool through the
    oracle manager's prefill slots (shuffled free order)."""
    rng = _rng(seed)
    nb = nb or sum(-(-L // bs) for L in lens) + 5
    m = BlockManager(nb, bs, rng.permutation(nb).tolist())
    kc = np.full((nb, bs, hkv, d), np.nan, dtype=dtype)
    vc = np.full((nb, bs, hkv, d), np.nan, dtype=dtype)
    q = rng.standard_normal((len(lens), hq, d)).astype(dtype)
    Ks, Vs = [], []
    for sid, L in enumerate(lens):
        K = rng.standard_normal((L, hkv, d)).astype(dtype)
        V = rng.standard_normal((L, hkv, d)).astype(dtype)
        if L:
            reshape_and_cache(K, V, kc, vc, m.allocate_for_prefill(sid, L))
        Ks.append(K)
        Vs.append(V)
    tables, seq_lens = m.export([s for s, L in enumerate(lens) if L], max(-(-L // bs) for L in lens) + 2)
    # sequences of length 0 have no blocks: give them an all-padding row
    full_tables, it = [], iter(tables)
    for L in lens:
        full_tables.append(next(it) if L else [-1] * len(tables[0]))
    return q, kc, vc, full_tables, list(lens), Ks, Vs


def _sdpa(q, K, V, scale):
    """torch SDPA in float64 on contiguous tensors, kv heads repeated per group."""
    hq, hkv = q.shape[0], K.shape[1]
    g = hq // hkv
    qt = torch.from_numpy(np.ascontiguousarray(q))[:, None, :]              # [Hq, 1, D]
    kt = torch.from_numpy(np.ascontiguousarray(K)).permute(1, 0, 2)          # [Hkv, L, D]
    vt = torch.from_numpy(np.ascontiguousarray(V)).permute(1, 0, 2)
    kt = kt.repeat_interleave(g, dim=0)
    vt = vt.repeat_interleave(g, dim=0)
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)[:, 0, :].numpy()


def test_gqa_mapping_pin():
    g = G_MAP["gqa_mapping"]
    got = [att.kv_head_of(qh, g["num_heads"], g["num_kv_heads"]) for qh in g["query_heads"]]
    assert got == g["kv_heads"]
    with pytest.raises(ValueError):
        att.kv_head_of(0, 6, 4)


@pytest.mark.parametrize("hq,hkv", [(2, 1), (4, 4), (14, 2), (8, 2), (7, 7)])
def test_matches_library_sdpa_through_pages(hq, hkv):
    """Paged oracle attention on shuffled, NaN-padded pools equals torch's
    SDPA on the logically ordered contiguous tensors."""
    lens = [1, 5, 16, 17, 33]
    d, bs = 16, 4
    scale = 1.0 / math.sqrt(d)
    q, kc, vc, tables, seq_lens, Ks, Vs = _paged_setup(hq * 10 + hkv, lens, hq, hkv, d, bs)
    out = att.paged_decode_attention(q, kc, vc, tables, seq_lens, scale, "f64")
    assert np.all(np.isfinite(out))
    for b in range(len(lens)):
        ref = _sdpa(q[b], Ks[b], Vs[b], scale)
        np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-12)


def test_one_token_returns_v0():
    rng = _rng(2)
    q = rng.standard_normal((4, 8))
    K = rng.standard_normal((1, 2, 8))
    V = rng.standard_normal((1, 2, 8))
    out = att.decode_attention_contiguous(q, K, V, 0.3)
    for qh in range(4):
        assert np.array_equal(out[qh], V[0, qh // 2])


def test_equal_keys_or_zero_query_give_mean_of_v():
    rng = _rng(3)
    L, d = 9, 6
    V = rng.standard_normal((L, 1, d))
    K = np.repeat(rng.standard_normal((1, 1, d)), L, axis=0)
    q = rng.standard_normal((1, d))
    np.testing.assert_allclose(att.decode_attention_contiguous(q, K, V, 0.7)[0], V[:, 0].mean(0),
                               rtol=1e-13, atol=1e-13)
    K = rng.standard_normal((L, 1, d))
    np.testing.assert_allclose(att.decode_attention_contiguous(np.zeros((1, d)), K, V, 0.7)[0],
                               V[:, 0].mean(0), rtol=1e-13, atol=1e-13)


def test_two_tokens_logistic_weights():
    """L = 2: weights are sigma(s0 - s1) and sigma(s1 - s0)."""
    rng = _rng(4)
    d = 5
    q = rng.standard_normal(d)
    K = rng.standard_normal((2, d))
    V = rng.standard_normal((2, d))
    scale = 0.45
    s0, s1 = scale * float(q @ K[0]), scale * float(q @ K[1])
    w0 = 1.0 / (1.0 + math.exp(-(s0 - s1)))
    want = w0 * V[0] + (1.0 - w0) * V[1]
    np.testing.assert_allclose(att.attention_one(q, K, V, scale), want, rtol=1e-13, atol=1e-14)


def test_one_hot_values_expose_weights():
    """V = identity rows: the output is the softmax weight vector (scipy)."""
    rng = _rng(5)
    L = 7
    q = rng.standard_normal(L)
    K = rng.standard_normal((L, L))
    out = att.attention_one(q, K, np.eye(L), 0.8)
    np.testing.assert_allclose(out, scipy.special.softmax(0.8 * K @ q), rtol=1e-13, atol=1e-15)


def test_large_scores_do_not_overflow():
    """Scores near 1e3 apart: the winning token's value, no inf/nan."""
    d = 4
    q = np.array([1.0, 0, 0, 0])
    K = np.array([[900.0, 0, 0, 0], [1000.0, 0, 0, 0], [-1000.0, 0, 0, 0]])
    V = np.array([[1.0, 2, 3, 4], [5.0, 6, 7, 8], [9.0, 9, 9, 9]])
    out = att.attention_one(q, K, V, 1.0)
    np.testing.assert_allclose(out, V[1], rtol=0, atol=1e-40)
    assert np.array_equal(att.attention_one_online(q, K, V, 1.0), out)


def test_empty_sequence_gives_zeros():
    q = np.ones((2, 3))
    K = np.zeros((0, 1, 3))
    assert np.array_equal(att.decode_attention_contiguous(q, K, K, 1.0), np.zeros((2, 3)))


@pytest.mark.parametrize("seed", range(5))
def test_online_equals_two_pass(seed):
    rng = _rng(10 + seed)
    L, d = int(rng.integers(1, 60)), 12
    q, K, V = rng.standard_normal(d), 3 * rng.standard_normal((L, d)), rng.standard_normal((L, d))
    np.testing.assert_allclose(att.attention_one_online(q, K, V, 0.5), att.attention_one(q, K, V, 0.5),
                               rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed", range(5))
def test_split_merge_equals_full(seed):
    """Any partition of the tokens into ranges (empty ones included) merged by
    log-sum-exp gives the unsplit result."""
    rng = _rng(20 + seed)
    L, d = int(rng.integers(1, 90)), 8
    q, K, V = rng.standard_normal(d), 2 * rng.standard_normal((L, d)), rng.standard_normal((L, d))
    cuts = sorted(rng.integers(0, L + 1, size=int(rng.integers(0, 6))).tolist())
    edges = [0] + cuts + [L, L]
    states = [att.partial_state(q, K[a:b], V[a:b], 0.6) for a, b in zip(edges[:-1], edges[1:])]
    np.testing.assert_allclose(att.merge_states(states), att.attention_one(q, K, V, 0.6),
                               rtol=1e-12, atol=1e-12)


# -- planted mistakes: each must be caught by a pin above ------------------------

def test_planted_wrong_head_mapping_is_caught(monkeypatch):
    monkeypatch.setattr(att, "kv_head_of", lambda qh, hq, hkv: qh % hkv)
    with pytest.raises(AssertionError):
        test_gqa_mapping_pin()
    with pytest.raises(AssertionError):
        test_matches_library_sdpa_through_pages(8, 2)


def test_planted_dropped_scale_is_caught(monkeypatch):
    orig = att.attention_one
    monkeypatch.setattr(att, "attention_one", lambda q, K, V, scale: orig(q, K, V, 1.0))
    with pytest.raises(AssertionError):
        test_matches_library_sdpa_through_pages(4, 4)


def test_planted_sorted_gather_is_caught(monkeypatch):
    import oracle.paged_cache as pc
    orig = pc.gather
    monkeypatch.setattr(att, "gather", lambda cache, table, L: orig(
        cache, sorted(table[: -(-L // cache.shape[1])]) + list(table[-(-L // cache.shape[1]):]), L))
    with pytest.raises(AssertionError):
        test_matches_library_sdpa_through_pages(2, 1)


def test_planted_untruncated_tail_is_caught(monkeypatch):
    import oracle.paged_cache as pc
    orig = pc.gather

    def whole_blocks(cache, table, L):
        bs = cache.shape[1]
        return orig(cache, table, -(-L // bs) * bs)

    monkeypatch.setattr(att, "gather", whole_blocks)
    with pytest.raises(AssertionError):
        test_matches_library_sdpa_through_pages(2, 1)
