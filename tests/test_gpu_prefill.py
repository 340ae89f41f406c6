"""GPU parity of chunked-prefill attention (paged_prefill_attention).

Each sequence holds ctx tokens of history and a chunk of n new tokens (its
last n positions; all L = ctx + n tokens are written through the cache
write first).  Every chunk row must match the float64 oracle
(oracle.attention.chunked_prefill_attention) on the sequence's logical K/V,
within the dtype's tolerance: chunks with and without history, chunks
crossing query tiles and 128-key tiles, one-token chunks (decode), GQA
ratios 1 to 8 (the tensor-core kernel packs 1, 2, 4 or 8 heads of a group
into one 128-row tile), head_dim 64 and 128, block sizes 16 to 128 (tcgen05
kernel) and 4 and 8 (mma.sync kernel), and the mixed-batch workload's
4096-token prefill chunk (sampled rows).  Unused cache slots hold a NaN
sentinel, so a tail slot that reached the output would show.
"""

import math

import numpy as np
import pytest
import torch

import paged_kv_cache_128_gb300 as pk
from oracle.attention import chunked_prefill_attention
from paged_kv_cache_128_gb300.inputs import make_values, make_workload
from tests.helpers import TOL, TORCH, rounding_allowance, sentinel_tensor, to_f64

pytestmark = pytest.mark.gpu


def _run(dtype, hq, hkv, d, bs, seqs, seed, value_scale=0.5, sample_rows=None, max_query_len=None):
    """seqs: list of (history length, chunk length); every sequence has at
    least one token.  max_query_len defaults to the longest chunk."""
    rng = np.random.default_rng(seed)
    g = torch.Generator().manual_seed(seed)
    dt = TORCH[dtype]
    lens = [c + n for c, n in seqs]
    nb = sum(-(-L // bs) for L in lens) + 3
    mgr = pk.KVBlockManager(nb, bs, rng.permutation(nb).tolist())
    dev = torch.device("cuda")
    kc = sentinel_tensor((nb, bs, hkv, d), dtype, dev)
    vc = sentinel_tensor((nb, bs, hkv, d), dtype, dev)
    Ks, Vs = [], []
    for sid, L in enumerate(lens):
        slots = torch.from_numpy(mgr.allocate_for_prefill(sid, L)).to(dev)
        k = (torch.randn(L, hkv, d, generator=g) * value_scale).to(dt)
        v = (torch.randn(L, hkv, d, generator=g) * value_scale).to(dt)
        pk.reshape_and_cache(k.to(dev), v.to(dev), kc, vc, slots)
        Ks.append(k)
        Vs.append(v)
    maxb = max(-(-L // bs) for L in lens) + 1
    tables, seq_lens = mgr.export(list(range(len(seqs))), maxb)
    qsl = np.concatenate([[0], np.cumsum([n for _, n in seqs])]).astype(np.int32)
    T = int(qsl[-1])
    q = (torch.randn(T, hq, d, generator=g) * value_scale).to(dt)
    out = sentinel_tensor((T, hq, d), dtype, dev)
    scale = 1.0 / math.sqrt(d)
    pk.device_error()
    pk.paged_prefill_attention(out, q.to(dev), kc, vc, torch.from_numpy(tables).to(dev),
                               torch.from_numpy(seq_lens).to(dev), torch.from_numpy(qsl).to(dev), scale,
                               max_query_len if max_query_len is not None else max(n for _, n in seqs))
    assert pk.device_error() == 0
    got = to_f64(out, dtype)
    assert np.all(np.isfinite(got))
    q64 = to_f64(q, dtype)
    worst = 0.0
    for b, (c, n) in enumerate(seqs):
        K, V = to_f64(Ks[b], dtype), to_f64(Vs[b], dtype)
        rows = range(n) if sample_rows is None else sorted(set(rng.integers(0, n, sample_rows).tolist()))
        for t in rows:
            p = c + t
            ref = chunked_prefill_attention(q64[qsl[b] + t:qsl[b] + t + 1], K[:p + 1], V[:p + 1], scale)[0]
            # the stated bar applies beyond the output's own rounding (half an
            # ulp of the exact value), which the rows of short spans drawn at
            # N(0, 1) reach by themselves
            worst = max(worst, float(np.max(np.abs(got[qsl[b] + t] - ref) - rounding_allowance(ref, dtype))))
    return worst


CASES = [
    ("bf16", 8, 2, 128, 16, [(0, 1), (0, 5), (0, 64), (0, 65), (0, 200), (13, 7), (100, 1), (300, 130), (31, 33)]),
    ("f16", 14, 2, 64, 16, [(0, 63), (5, 64), (40, 129), (0, 1)]),
    ("bf16", 32, 8, 128, 32, [(0, 256), (17, 95), (64, 64)]),
    ("f16", 4, 4, 128, 32, [(7, 40), (0, 3), (500, 70)]),
    ("bf16", 16, 2, 128, 64, [(0, 300), (257, 129), (1000, 17)]),
    ("f16", 4, 2, 64, 128, [(5, 250), (128, 128), (0, 1)]),
    ("bf16", 8, 2, 128, 8, [(0, 70), (20, 45), (0, 1)]),
    ("f16", 6, 3, 64, 4, [(3, 33), (0, 9)]),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-g{c[1] // c[2]}-d{c[3]}-bs{c[4]}")
def test_prefill_matches_oracle(case):
    dtype, hq, hkv, d, bs, seqs = case
    worst = _run(dtype, hq, hkv, d, bs, seqs, seed=len(seqs) + d)
    assert worst <= TOL[dtype], f"max abs err {worst:.3e}"


def test_prefill_mixed_batch_chunk():
    """The mixed-batch workload's prefill chunk: 8 new sequences, 4096
    tokens in all, Hq 32, Hkv 8, D 128, bs 32 (sampled rows of each)."""
    wl = make_workload("mixed_batch_bf16")
    seqs = [(0, int(n)) for n in wl.prefill_lens]
    assert sum(n for _, n in seqs) == 4096
    worst = _run("bf16", wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.block_size, seqs, seed=5, value_scale=1.0,
                 sample_rows=12)
    assert worst <= TOL["bf16"], f"max abs err {worst:.3e}"


def test_prefill_mixed_batch_chunk_with_history():
    """The benchmark's prefill case: the mixed-batch chunk (8 sequences, 4096
    tokens) with 2048 tokens of history before each chunk; every row of
    every sequence against the oracle."""
    wl = make_workload("mixed_batch_bf16")
    seqs = [(2048, int(n)) for n in wl.prefill_lens]
    worst = _run("bf16", wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.block_size, seqs, seed=6, value_scale=1.0)
    assert worst <= TOL["bf16"], f"max abs err {worst:.3e}"


@pytest.mark.parametrize("bs", [16, 8], ids=["tcgen05", "mma_sync"])
def test_prefill_chunk_longer_than_max_query_len_is_reported(bs):
    """A grid sized by a max_query_len below the longest chunk cannot reach
    that chunk's last rows: the launch records KV_ERR_DEVICE_BOUNDS."""
    dev = torch.device("cuda")
    nb, hkv, d, hq = 64, 2, 64, 4
    g = torch.Generator().manual_seed(3)
    kc = (torch.randn(nb, bs, hkv, d, generator=g) * 0.5).half().to(dev)
    vc = (torch.randn(nb, bs, hkv, d, generator=g) * 0.5).half().to(dev)
    maxb = 300 // bs + 1
    tables = torch.arange(maxb, dtype=torch.int32, device=dev).view(1, -1)
    lens = torch.tensor([300], dtype=torch.int32, device=dev)
    qsl = torch.tensor([0, 300], dtype=torch.int32, device=dev)   # one chunk of 300 rows
    q = (torch.randn(300, hq, d, generator=g) * 0.5).half().to(dev)
    out = torch.zeros(300, hq, d, dtype=torch.float16, device=dev)
    pk.device_error()
    pk.paged_prefill_attention(out, q, kc, vc, tables, lens, qsl, 0.125, 20)   # grid for 20 rows or so
    assert pk.device_error() == 8
    pk.paged_prefill_attention(out, q, kc, vc, tables, lens, qsl, 0.125, 300)  # the true bound: no error
    assert pk.device_error() == 0


def test_prefill_chunk_longer_than_sequence_is_reported():
    dev = torch.device("cuda")
    nb, bs, hkv, d, hq = 8, 16, 2, 64, 4
    kc = torch.zeros(nb, bs, hkv, d, dtype=torch.float16, device=dev)
    vc = torch.zeros_like(kc)
    tables = torch.tensor([[0, 1, 2, -1]], dtype=torch.int32, device=dev)
    lens = torch.tensor([10], dtype=torch.int32, device=dev)
    qsl = torch.tensor([0, 12], dtype=torch.int32, device=dev)    # 12 chunk tokens, sequence of 10
    q = torch.randn(12, hq, d, device=dev).half()
    out = torch.full((12, hq, d), 7.0, dtype=torch.float16, device=dev)
    pk.device_error()
    pk.paged_prefill_attention(out, q, kc, vc, tables, lens, qsl, 0.125, 12)
    assert pk.device_error() == 8
    assert torch.all(out == 7.0)                                   # nothing written


def test_prefill_chunk_past_the_query_rows_is_reported():
    dev = torch.device("cuda")
    nb, bs, hkv, d, hq = 8, 16, 2, 64, 4
    kc = torch.zeros(nb, bs, hkv, d, dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    tables = torch.tensor([[0, 1, 2, -1]], dtype=torch.int32, device=dev)
    lens = torch.tensor([40], dtype=torch.int32, device=dev)
    qsl = torch.tensor([0, 20], dtype=torch.int32, device=dev)    # 20 chunk rows, q holds 12
    q = torch.randn(12, hq, d, device=dev).bfloat16()
    out = torch.full((12, hq, d), 7.0, dtype=torch.bfloat16, device=dev)
    pk.device_error()
    pk.paged_prefill_attention(out, q, kc, vc, tables, lens, qsl, 0.125, 20)
    assert pk.device_error() == 8
    assert torch.all(out == 7.0)


@pytest.mark.parametrize("bs", [16, 8], ids=["tcgen05", "mma_sync"])
def test_prefill_empty_chunks_between_others(bs):
    """Sequences whose chunk is empty (n = 0) sit between others: they own
    no rows of q/out, and every other chunk still matches the oracle."""
    seqs = [(5, 0), (30, 17), (3, 0), (100, 1), (0, 40), (7, 0)]
    worst = _run("bf16", 8, 2, 128, bs, seqs, seed=21)
    assert worst <= TOL["bf16"], f"max abs err {worst:.3e}"


@pytest.mark.parametrize("bs", [32, 4], ids=["tcgen05", "mma_sync"])
def test_prefill_grid_larger_than_the_chunks(bs):
    """max_query_len is only an upper bound: a grid sized for 4x the longest
    chunk gives the same rows."""
    seqs = [(12, 70), (0, 129)]
    worst = _run("f16", 4, 2, 64, bs, seqs, seed=22, max_query_len=4 * 129)
    assert worst <= TOL["f16"], f"max abs err {worst:.3e}"


def test_prefill_without_query_rows_launches_nothing():
    dev = torch.device("cuda")
    kc = torch.zeros(4, 16, 2, 64, dtype=torch.float16, device=dev)
    vc = torch.zeros_like(kc)
    tables = torch.tensor([[0, 1]], dtype=torch.int32, device=dev)
    lens = torch.tensor([20], dtype=torch.int32, device=dev)
    qsl = torch.tensor([0, 0], dtype=torch.int32, device=dev)
    q = torch.empty(0, 4, 64, dtype=torch.float16, device=dev)
    out = torch.empty_like(q)
    pk.device_error()
    pk.paged_prefill_attention(out, q, kc, vc, tables, lens, qsl, 0.125, 0)
    torch.cuda.synchronize()
    assert pk.device_error() == 0


def test_prefill_attention_over_a_runner_step():
    """One mixed-batch serving step through the native step runner allocates
    the step's 8 new sequences and writes their chunk K/V.  Chunked-prefill
    attention over the runner's own block tables then matches the oracle,
    whose K/V are the step's original rows, found through the step's slot
    mapping on the host (sampled chunk rows of every sequence)."""
    from paged_kv_cache_128_gb300.engine import PagedDecodeEngine

    wl = make_workload("mixed_batch_bf16")
    dev = torch.device("cuda")
    vals = make_values(wl, device="cuda")
    eng = PagedDecodeEngine(wl, dev, max_steps=2)
    eng.setup(vals)
    eng.make_runner()
    out = torch.empty_like(vals.q)
    eng.runner_step(vals.q, vals.k_step, vals.v_step, out)
    eng.runner_join()
    torch.cuda.synchronize()
    slots, _, _, _ = eng.runner_last_metadata()
    ids = eng._prefill_ids.copy()
    lens = np.asarray(eng._prefill_lens, dtype=np.int64)
    bs = wl.block_size
    tables, seq_lens = eng.mgr.export(ids.tolist(), int(max(-(-lens // bs))))
    assert np.array_equal(seq_lens, lens)
    row_of_slot = {int(s): r for r, s in enumerate(slots) if s >= 0}
    qsl = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    g = torch.Generator().manual_seed(31)
    q = torch.randn(int(qsl[-1]), wl.num_heads, wl.head_dim, generator=g).to(wl.torch_dtype)
    got = torch.full(q.shape, float("nan"), dtype=wl.torch_dtype, device=dev)
    scale = float(wl.scale)
    pk.device_error()
    pk.paged_prefill_attention(got, q.to(dev), eng.k_cache, eng.v_cache, torch.from_numpy(tables).to(dev),
                               torch.from_numpy(seq_lens).to(dev), torch.from_numpy(qsl).to(dev), scale,
                               int(lens.max()))
    torch.cuda.synchronize()
    assert pk.device_error() == 0
    got64, q64 = to_f64(got, "bf16"), to_f64(q, "bf16")
    k_rows, v_rows = to_f64(vals.k_step, "bf16"), to_f64(vals.v_step, "bf16")
    rng = np.random.default_rng(32)
    worst = 0.0
    for b in range(ids.size):
        n = int(lens[b])
        rows = [row_of_slot[int(tables[b, i // bs]) * bs + i % bs] for i in range(n)]
        K, V = k_rows[rows], v_rows[rows]
        for t in sorted(set(rng.integers(0, n, 10).tolist()) | {0, n - 1}):
            ref = chunked_prefill_attention(q64[qsl[b] + t:qsl[b] + t + 1], K[:t + 1], V[:t + 1], scale)[0]
            worst = max(worst, float(np.max(np.abs(got64[qsl[b] + t] - ref))))
    assert worst <= TOL["bf16"], f"max abs err {worst:.3e}"
    eng.close_runner()
