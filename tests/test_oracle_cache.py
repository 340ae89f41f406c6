"""Pins for the oracle cache write (scatter) and logical gather."""

import numpy as np
import pytest

from oracle.block_manager import BlockManager
from oracle.paged_cache import bf16_bits_to_float64, gather, reshape_and_cache, split_slot
from tests.conftest import load_golden

G_CH22 = load_golden("llm_algo_ch22.json")
G_MAP = load_golden("address_mapping.json")


def _cache(nb, bs, h, d, fill=np.nan):
    return np.full((nb, bs, h, d), fill, dtype=np.float32)


def test_gather_fill_case():
    """LLM-algo ch.22 Case 1: three blocks filled 1, 2, 3; length 9."""
    g = G_CH22["gather_fill"]
    m = BlockManager(10, 4)
    m.allocate_for_prefill(1, 6)
    for _ in range(3):
        m.append_slot_for_decode(1)
    cache = _cache(10, 4, 1, g["head_dim"])
    for b, val in zip(m.block_table(1), g["fill"]):
        cache[b] = val
    out = gather(cache, m.block_table(1), m.seq_len(1))[:, 0, :]
    assert list(out.shape) == g["shape"]
    assert [float(r[0]) for r in out] == g["rows"]
    assert np.all(out == out[:, :1])


def test_gather_non_contiguous_table_order():
    """LLM-algo ch.22 Case 1b: table [3, 1] is read in table order."""
    g = G_CH22["gather_non_contiguous"]
    cache = _cache(g["num_blocks"], g["block_size"], 1, g["head_dim"])
    for b, val in g["fill"].items():
        cache[int(b)] = val
    out = gather(cache, g["table"], g["seq_len"])[:, 0, :]
    assert [float(r[0]) for r in out] == g["rows"]


def test_gather_boundary_truncation():
    """LLM-algo ch.22 Case 2: prompt 4 + one decode -> (5, 8), tail truncated."""
    g = G_CH22["boundary"]
    m = BlockManager(g["num_blocks"], g["block_size"])
    m.allocate_for_prefill(2, g["prompt_len"])
    assert len(m.block_table(2)) == g["blocks_after_prefill"]
    m.append_slot_for_decode(2)
    assert len(m.block_table(2)) == g["blocks_after_decode"]
    cache = _cache(g["num_blocks"], g["block_size"], 1, g["head_dim"])
    cache[m.block_table(2)[0]] = 7.0
    cache[m.block_table(2)[1]] = 8.0
    out = gather(cache, m.block_table(2), m.seq_len(2))[:, 0, :]
    assert list(out.shape) == g["shape"]
    assert [float(r[0]) for r in out] == g["rows"]


def test_gather_never_reads_padding():
    cache = _cache(4, 2, 1, 2, fill=5.0)
    out = gather(cache, [2, -1, -1], 2)         # padding entries past the used blocks
    assert out.shape == (2, 1, 2)
    assert gather(cache, [], 0).shape == (0, 1, 2)
    with pytest.raises(ValueError):
        gather(cache, [2, -1], 3)               # needs 2 blocks: the second is padding


def test_scatter_decomposition_pins():
    """MiniPaged-Qwen §11/§12: slot 10 -> block 2 offset 2; slot 36 -> block 9
    offset 0 (block size 4).  Every other row keeps its sentinel."""
    bs, h, d = 4, 3, 5
    k_cache = _cache(12, bs, h, d)
    v_cache = _cache(12, bs, h, d)
    rng = np.random.default_rng(0)
    k = rng.standard_normal((3, h, d)).astype(np.float32)
    v = rng.standard_normal((3, h, d)).astype(np.float32)
    cases = G_MAP["slot_decomposition"]["cases"]
    slots = [cases[0]["slot"], -1, cases[1]["slot"]]
    reshape_and_cache(k, v, k_cache, v_cache, slots)
    written = {(c["physical_block"], c["block_offset"]): t for c, t in zip(cases, (0, 2))}
    for pb in range(12):
        for off in range(bs):
            if (pb, off) in written:
                t = written[(pb, off)]
                assert np.array_equal(k_cache[pb, off], k[t])
                assert np.array_equal(v_cache[pb, off], v[t])
            else:
                assert np.all(np.isnan(k_cache[pb, off])) and np.all(np.isnan(v_cache[pb, off]))
    with pytest.raises(ValueError):
        reshape_and_cache(k[:1], v[:1], k_cache, v_cache, [12 * bs])
    with pytest.raises(ValueError):
        reshape_and_cache(k[:1], v[:1], k_cache, v_cache, [-2])


def test_scatter_then_gather_is_identity():
    """Writing a sequence's prompt by its prefill slots and gathering it back
    returns the prompt, for shuffled pools and every block size."""
    rng = np.random.default_rng(1)
    for bs in (1, 2, 4, 16):
        nb = 64
        order = rng.permutation(nb).tolist()
        m = BlockManager(nb, bs, order)
        kc = np.full((nb, bs, 2, 3), 0xFFFF, dtype=np.uint16)
        vc = kc.copy()
        for sid, n in enumerate((1, bs, 3 * bs + 1)):
            x = rng.integers(0, 0x7F00, size=(n, 2, 3), dtype=np.uint16)
            y = rng.integers(0, 0x7F00, size=(n, 2, 3), dtype=np.uint16)
            slots = m.allocate_for_prefill(sid, n)
            reshape_and_cache(x, y, kc, vc, slots)
            assert np.array_equal(gather(kc, m.block_table(sid), n), x)
            assert np.array_equal(gather(vc, m.block_table(sid), n), y)
            for t, s in enumerate(slots):
                pb, off = split_slot(s, bs)
                assert m.block_table(sid).index(pb) == t // bs and off == t % bs


def test_bf16_widening():
    """bfloat16 is the top 16 bits of binary32: 0x3F80 -> 1.0, 0xC000 -> -2.0,
    0x3F81 -> 1 + 2^-7, 0x7F80 -> +inf, 0x0001 -> smallest subnormal 2^-133."""
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x7F80, 0x0001, 0x8000], dtype=np.uint16)
    want = np.array([1.0, -2.0, 1.0 + 2.0 ** -7, np.inf, 2.0 ** -133, -0.0])
    got = bf16_bits_to_float64(bits)
    assert np.array_equal(got, want)
    assert np.signbit(got[-1])
