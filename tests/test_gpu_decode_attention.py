"""GPU parity of paged decode attention against the float64 oracle.

Each case builds one pool twice: on the product side (native manager ->
slots -> CUDA cache write) and on the oracle side (oracle manager -> slots
-> oracle scatter).  Tables must match bit-exactly; outputs must be within
the dtype's max-abs tolerance of the oracle.  Unused slots hold NaN, so a
read past a sequence's end or of table padding shows up as NaN.
"""

import math

import numpy as np
import pytest
import torch

import paged_kv_cache_128_gb300 as pk
from oracle.attention import paged_decode_attention as oracle_attention
from tests.helpers import TOL, TORCH, oracle_paged_pool, sentinel_tensor, to_f64, to_storage

pytestmark = pytest.mark.gpu


def run_case(dtype, hq, hkv, d, bs, lens, seed, bps=0, nb=None, scale=None, value_scale=1.0, max_seq_len=None,
             repeat=1, workspace=None, expect_error=0):
    rng = np.random.default_rng(seed)
    B = len(lens)
    nb = nb or sum(-(-L // bs) for L in lens) + 3
    order = rng.permutation(nb).tolist()
    g = torch.Generator().manual_seed(seed)
    dt = TORCH[dtype]
    total = int(sum(lens))
    q = (torch.randn(B, hq, d, generator=g) * value_scale).to(dt)
    k_hist = (torch.randn(total, hkv, d, generator=g) * value_scale).to(dt)
    v_hist = (torch.randn(total, hkv, d, generator=g) * value_scale).to(dt)
    scale = scale if scale is not None else 1.0 / math.sqrt(d)
    dev = torch.device("cuda")

    # product side
    mgr = pk.KVBlockManager(nb, bs, order)
    slots = [mgr.allocate_for_prefill(sid, L) for sid, L in enumerate(lens) if L > 0]
    slots = np.concatenate(slots) if slots else np.zeros(0, np.int32)
    kc = sentinel_tensor((nb, bs, hkv, d), dtype, dev)
    vc = sentinel_tensor((nb, bs, hkv, d), dtype, dev)
    if total:
        pk.reshape_and_cache(k_hist.to(dev), v_hist.to(dev), kc, vc, torch.from_numpy(slots).to(dev))
    max_blocks = max(-(-L // bs) for L in lens) + 2
    tables = np.full((B, max_blocks), -1, dtype=np.int32)
    seq_lens = np.zeros(B, dtype=np.int32)
    live = [sid for sid, L in enumerate(lens) if L > 0]
    if live:
        t, l = mgr.export(live, max_blocks)
        tables[live] = t
        seq_lens[live] = l
    out = torch.empty(B, hq, d, dtype=dt, device=dev)
    pk.paged_decode_attention(out, q.to(dev), kc, vc, torch.from_numpy(tables).to(dev),
                              torch.from_numpy(seq_lens).to(dev), scale, max_seq_len or max(max(lens), 1), bps,
                              workspace=workspace)
    assert pk.device_error() == expect_error
    if expect_error:
        return None, None
    if repeat > 1:
        # the partition fixes the combine order: every call is bit-identical
        d_q, d_t, d_l = q.to(dev), torch.from_numpy(tables).to(dev), torch.from_numpy(seq_lens).to(dev)
        again = torch.empty_like(out)
        for _ in range(repeat - 1):
            again.fill_(0)
            pk.paged_decode_attention(again, d_q, kc, vc, d_t, d_l, scale, max_seq_len or max(max(lens), 1), bps,
                                      workspace=workspace)
            assert torch.equal(again, out)
        assert pk.device_error() == 0

    # oracle side
    ora, kco, vco, _ = oracle_paged_pool(lens, nb, bs, hkv, d, dtype, order, to_storage(k_hist, dtype),
                                         to_storage(v_hist, dtype))
    t_o = np.full((B, max_blocks), -1, dtype=np.int32)
    if live:
        t_o[live] = np.asarray(ora.export(live, max_blocks)[0], dtype=np.int32)
    assert np.array_equal(tables, t_o)
    ref = oracle_attention(to_storage(q, dtype), kco, vco, t_o.tolist(), list(lens), scale, dtype)
    got = to_f64(out, dtype)
    assert np.all(np.isfinite(got))
    err = np.max(np.abs(got - ref))
    assert err <= TOL[dtype], f"max abs err {err:.3e} > {TOL[dtype]:.1e}"
    return got, ref


LENS_A = [1, 15, 16, 17, 100, 257, 600]
LENS_B = [33, 1, 64, 0, 129, 31, 512, 2]


@pytest.mark.parametrize("dtype,hq,hkv,d,bs", [
    ("f16", 14, 2, 64, 16),      # G = 7, the small GQA workload's heads
    ("bf16", 28, 4, 128, 16),    # G = 7, the mid-size workload's heads
    ("bf16", 32, 8, 128, 16),    # G = 4
    ("bf16", 32, 8, 128, 32),    # G = 4, block 32 (mixed batch)
    ("f16", 8, 8, 128, 16),      # G = 1 (MHA)
    ("bf16", 16, 2, 64, 32),     # G = 8
    ("f16", 32, 2, 128, 16),     # G = 16 (two n-tiles)
    ("bf16", 24, 2, 64, 16),     # G = 12
    ("bf16", 4, 2, 256, 16),     # D = 256
    ("f16", 6, 2, 256, 32),      # D = 256, block 32
])
def test_tensor_core_path(dtype, hq, hkv, d, bs):
    plan = pk.decode_plan(len(LENS_A), hq, hkv, d, bs, max(LENS_A), TORCH[dtype])
    assert plan.kernel == 2                                   # stream-K by default
    run_case(dtype, hq, hkv, d, bs, LENS_A, seed=hq * 1000 + d + bs)
    assert pk.decode_plan(len(LENS_A), hq, hkv, d, bs, max(LENS_A), TORCH[dtype], 5).kernel == 1
    run_case(dtype, hq, hkv, d, bs, LENS_A, seed=hq * 1000 + d + bs, bps=5)   # split kernel


def test_wide_group_d256_takes_split_kernel():
    """head_dim 256 with 12 query heads per kv head: the stream-K kernel's
    stage ring and merge area would exceed shared memory, so the plan takes
    the split tensor-core kernel, which must still match the oracle."""
    plan = pk.decode_plan(len(LENS_A), 24, 2, 256, 16, max(LENS_A), TORCH["bf16"])
    assert plan.kernel == 1
    run_case("bf16", 24, 2, 256, 16, LENS_A, seed=2562)


@pytest.mark.parametrize("dtype,hq,hkv,d,bs", [
    ("f32", 2, 1, 8, 4),         # the tiny fp32 workload's shape
    ("f32", 6, 2, 32, 16),
    ("f32", 8, 1, 100, 7),       # odd block size, head dim not a multiple of 32
    ("f16", 6, 3, 96, 16),       # head dim the tensor-core kernel does not take
    ("bf16", 8, 4, 128, 8),      # block size the tensor-core kernel does not take
    ("bf16", 48, 2, 64, 16),     # G = 24: several head groups per kv head
])
def test_simt_path(dtype, hq, hkv, d, bs):
    plan = pk.decode_plan(len(LENS_B), hq, hkv, d, bs, max(LENS_B), TORCH[dtype])
    assert plan.kernel == 0
    run_case(dtype, hq, hkv, d, bs, LENS_B, seed=hq * 100 + d + bs)


@pytest.mark.parametrize("dtype,hq,hkv,d,bs", [("bf16", 28, 4, 128, 16), ("f16", 14, 2, 64, 16),
                                              ("bf16", 32, 8, 128, 32), ("f32", 4, 2, 16, 4)])
def test_split_invariance(dtype, hq, hkv, d, bs):
    """Any split size gives the oracle's answer (within tolerance)."""
    lens = [700, 1, 300, 48, 1025]
    outs = []
    for bps in (0, 1, 2, 3, 7, 1000):
        got, ref = run_case(dtype, hq, hkv, d, bs, lens, seed=7, bps=bps)
        outs.append(got)
    for o in outs[1:]:
        assert np.max(np.abs(o - outs[0])) <= 2 * TOL[dtype]


@pytest.mark.parametrize("dtype,hq,hkv,d,bs,lens", [
    ("bf16", 16, 2, 64, 32, LENS_A),                    # fewer cost positions than CTAs: pieces from global
    ("bf16", 28, 4, 128, 16, [700, 1, 300, 48, 1025] * 4),  # pieces copied into freed stages
    ("f16", 8, 1, 128, 16, [20000]),                     # one unit over every CTA: more than 32 pieces
])
def test_stream_k_repeated_calls_identical(dtype, hq, hkv, d, bs, lens):
    """Forty calls on the same inputs: each must equal the first bit for bit
    (and the first the oracle).  An owner that read a later piece before it
    was published would make some call differ."""
    run_case(dtype, hq, hkv, d, bs, lens, seed=4242 + d, repeat=40)


def test_stream_k_more_ctas_than_tiles():
    """A generous max_seq_len makes the stream-K grid larger than the tile
    count, so some CTAs get empty ranges between the parts of one unit."""
    run_case("bf16", 8, 2, 128, 16, [40, 3, 70], seed=21, max_seq_len=20000)
    run_case("f16", 14, 2, 64, 16, [1, 2, 33], seed=22, max_seq_len=50000)


def test_zero_length_rows_are_zero():
    got, _ = run_case("bf16", 8, 2, 128, 16, [0, 5, 0, 40], seed=3)
    assert np.all(got[0] == 0) and np.all(got[2] == 0)
    got, _ = run_case("f32", 4, 2, 8, 4, [0, 3], seed=4)
    assert np.all(got[0] == 0)


def test_long_sequence_auto_split():
    lens = [6000, 17, 3000]
    run_case("bf16", 32, 8, 128, 16, lens, seed=11)
    plan = pk.decode_plan(3, 4, 2, 32, 16, 6000, torch.float32)
    assert plan.kernel == 0 and plan.num_splits > 1
    run_case("f32", 4, 2, 32, 16, lens, seed=12)


def test_closed_form_single_token_and_equal_keys():
    """L = 1 returns V0 exactly (after one rounding); constant keys give the
    mean of V -- closed forms, on the tensor-core path."""
    dev = torch.device("cuda")
    nb, bs, hkv, d, hq = 8, 16, 2, 64, 8
    kc = sentinel_tensor((nb, bs, hkv, d), "bf16", dev)
    vc = sentinel_tensor((nb, bs, hkv, d), "bf16", dev)
    v = torch.randn(20, hkv, d, device=dev).to(torch.bfloat16)
    krow = torch.randn(1, hkv, d, device=dev).to(torch.bfloat16).expand(20, hkv, d).contiguous()
    slots = torch.arange(3 * bs, 3 * bs + 20, dtype=torch.int32, device=dev)
    pk.reshape_and_cache(krow, v, kc, vc, slots)
    tables = torch.tensor([[3, 4], [3, 4]], dtype=torch.int32, device=dev)
    lens = torch.tensor([1, 20], dtype=torch.int32, device=dev)
    q = torch.randn(2, hq, d, device=dev).to(torch.bfloat16)
    out = torch.empty_like(q)
    pk.paged_decode_attention(out, q, kc, vc, tables, lens, 0.125, 20)
    G = hq // hkv
    for qh in range(hq):
        assert torch.equal(out[0, qh], v[0, qh // G])
        mean = v[:, qh // G].double().mean(0)
        assert torch.max(torch.abs(out[1, qh].double() - mean)) <= 8e-3


def test_table_entry_outside_pool_is_reported():
    dev = torch.device("cuda")
    kc = torch.zeros(4, 16, 1, 64, dtype=torch.float16, device=dev)
    q = torch.zeros(1, 2, 64, dtype=torch.float16, device=dev)
    out = torch.empty_like(q)
    pk.device_error()
    pk.paged_decode_attention(out, q, kc, kc, torch.tensor([[2, 9]], dtype=torch.int32, device=dev),
                              torch.tensor([20], dtype=torch.int32, device=dev), 0.1, 20)
    assert pk.device_error() == 8
    pk.paged_decode_attention(out, q, kc, kc, torch.tensor([[2, 1]], dtype=torch.int32, device=dev),
                              torch.tensor([40], dtype=torch.int32, device=dev), 0.1, 40)
    assert pk.device_error() == 8      # seq_len beyond the table row


def test_workspace_too_small_is_rejected():
    dev = torch.device("cuda")
    kc = torch.zeros(512, 16, 1, 64, dtype=torch.float16, device=dev)
    q = torch.zeros(1, 2, 64, dtype=torch.float16, device=dev)
    out = torch.empty_like(q)
    tables = torch.arange(512, dtype=torch.int32, device=dev)[None]
    lens = torch.tensor([8000], dtype=torch.int32, device=dev)
    plan = pk.decode_plan(1, 2, 1, 64, 16, 8000, torch.float16)
    assert plan.workspace_bytes > 0
    ws = torch.empty(plan.workspace_bytes - 256, dtype=torch.uint8, device=dev)
    with pytest.raises(pk.KVError) as e:
        pk.paged_decode_attention(out, q, kc, kc, tables, lens, 0.1, 8000, workspace=ws)
    assert e.value.code == "WORKSPACE"
