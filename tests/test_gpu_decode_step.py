"""GPU parity of paged_decode_step, the step's cache write and decode
attention in one call.

For every case the same step runs twice on identical pools: once through
``paged_decode_step`` and once as ``reshape_and_cache`` followed by
``paged_decode_attention``.  Outputs and both whole caches must be
bit-identical (the fused launch does the same copy and the same
arithmetic), and the output must be within tolerance of the float64 oracle
evaluated on each sequence's logical K/V, which includes the token written
in the step.
"""

import math

import numpy as np
import pytest
import torch

import paged_kv_cache_128_gb300 as pk
from oracle.attention import paged_decode_attention as oracle_attention
from oracle.block_manager import BlockManager as OracleManager
from oracle.paged_cache import reshape_and_cache as oracle_scatter
from paged_kv_cache_128_gb300.engine import PagedDecodeEngine
from paged_kv_cache_128_gb300.inputs import WORKLOADS, make_values, make_workload
from tests.helpers import TOL, TORCH, sentinel_storage, sentinel_tensor, to_f64, to_storage

pytestmark = pytest.mark.gpu


def build_step(dtype, hq, hkv, d, bs, cached, has_new, n_prefill, n_pad, seed, value_scale=1.0):
    """A pool holding each sequence's history and one step's new rows.

    Sequence b holds cached[b] tokens before the step and cached[b] + 1
    after it.  When has_new[b], its newest token is written by the step
    (row new_row[b]); otherwise that token is already in the cache and
    new_row[b] = -1.  The step also writes n_prefill rows of a sequence
    outside the batch and holds n_pad padded (-1) rows; rows are shuffled.
    K and V values are N(0, 1) * value_scale.
    """
    rng = np.random.default_rng(seed)
    g = torch.Generator().manual_seed(seed)
    B = len(cached)
    lens = [c + 1 for c in cached]
    nb = sum(-(-L // bs) for L in lens) + -(-max(n_prefill, 1) // bs) + 4
    order = rng.permutation(nb).tolist()
    mgr = pk.KVBlockManager(nb, bs, order)
    ora = OracleManager(nb, bs, order)
    slots = []
    for sid, L in enumerate(lens):
        s = mgr.allocate_for_prefill(sid, L)
        assert list(s) == ora.allocate_for_prefill(sid, L)
        slots.append(np.asarray(s, dtype=np.int64))
    pre_slots = np.zeros(0, dtype=np.int64)
    if n_prefill:
        pre_slots = np.asarray(mgr.allocate_for_prefill(B, n_prefill), dtype=np.int64)
        assert list(pre_slots) == ora.allocate_for_prefill(B, n_prefill)
    dt = TORCH[dtype]
    q = torch.randn(B, hq, d, generator=g).to(dt)
    k_all = [(torch.randn(L, hkv, d, generator=g) * value_scale).to(dt) for L in lens]
    v_all = [(torch.randn(L, hkv, d, generator=g) * value_scale).to(dt) for L in lens]
    k_pre = (torch.randn(n_prefill, hkv, d, generator=g) * value_scale).to(dt)
    v_pre = (torch.randn(n_prefill, hkv, d, generator=g) * value_scale).to(dt)

    # history: everything but the step's new tokens
    hist_slots, hist_k, hist_v = [], [], []
    for b in range(B):
        keep = cached[b] + (0 if has_new[b] else 1)
        hist_slots.append(slots[b][:keep])
        hist_k.append(k_all[b][:keep])
        hist_v.append(v_all[b][:keep])
    # the step: prefill rows, new decode rows, pads, in shuffled order
    items = [("pre", i) for i in range(n_prefill)] + [("dec", b) for b in range(B) if has_new[b]]
    items += [("pad", i) for i in range(n_pad)]
    perm = rng.permutation(len(items))
    items = [items[i] for i in perm]
    n = len(items)
    step_k = torch.randn(n, hkv, d, generator=g).to(dt)   # pads carry random rows that must land nowhere
    step_v = torch.randn(n, hkv, d, generator=g).to(dt)
    step_slots = np.full(n, -1, dtype=np.int64)
    new_row = np.full(B, -1, dtype=np.int32)
    for r, (kind, i) in enumerate(items):
        if kind == "pre":
            step_k[r], step_v[r], step_slots[r] = k_pre[i], v_pre[i], pre_slots[i]
        elif kind == "dec":
            step_k[r], step_v[r], step_slots[r] = k_all[i][cached[i]], v_all[i][cached[i]], slots[i][cached[i]]
            new_row[i] = r
    max_blocks = max(-(-L // bs) for L in lens) + 1
    tables, seq_lens = mgr.export(list(range(B)), max_blocks)
    t_o, l_o = ora.export(list(range(B)), max_blocks)
    assert np.array_equal(np.asarray(tables), np.asarray(t_o, dtype=np.int32))
    return dict(nb=nb, q=q, lens=lens, tables=np.asarray(tables, dtype=np.int32),
                seq_lens=np.asarray(seq_lens, dtype=np.int32), hist_slots=np.concatenate(hist_slots),
                hist_k=torch.cat(hist_k), hist_v=torch.cat(hist_v), step_k=step_k, step_v=step_v,
                step_slots=step_slots, new_row=new_row, k_all=k_all, v_all=v_all, k_pre=k_pre, v_pre=v_pre,
                pre_slots=pre_slots, slots=slots)


def run_both(c, dtype, bs, hkv, d, scale, bad_row=None):
    dev = torch.device("cuda")
    kc = sentinel_tensor((c["nb"], bs, hkv, d), dtype, dev)
    vc = sentinel_tensor((c["nb"], bs, hkv, d), dtype, dev)
    if c["hist_slots"].size:
        pk.reshape_and_cache(c["hist_k"].to(dev), c["hist_v"].to(dev), kc, vc,
                             torch.from_numpy(c["hist_slots"].astype(np.int32)).to(dev))
    kc2, vc2 = kc.clone(), vc.clone()
    q = c["q"].to(dev)
    sk, sv = c["step_k"].to(dev), c["step_v"].to(dev)
    slots = torch.from_numpy(c["step_slots"].astype(np.int32)).to(dev)
    rows = c["new_row"].copy()
    if bad_row is not None:
        rows[bad_row[0]] = bad_row[1]
    rows = torch.from_numpy(rows).to(dev)
    tables = torch.from_numpy(c["tables"]).to(dev)
    lens = torch.from_numpy(c["seq_lens"]).to(dev)
    max_len = int(c["seq_lens"].max())
    out = torch.empty_like(q)
    pk.paged_decode_step(out, q, sk, sv, slots, rows, kc, vc, tables, lens, scale, max_len)
    status = pk.device_error()
    out2 = torch.empty_like(q)
    pk.reshape_and_cache(sk, sv, kc2, vc2, slots)
    pk.paged_decode_attention(out2, q, kc2, vc2, tables, lens, scale, max_len)
    assert pk.device_error() == 0
    return status, out, out2, (kc, vc), (kc2, vc2)


def oracle_out(c, dtype, bs, hkv, d, scale):
    kco = sentinel_storage((c["nb"], bs, hkv, d), dtype)
    vco = sentinel_storage((c["nb"], bs, hkv, d), dtype)
    for b, L in enumerate(c["lens"]):
        oracle_scatter(to_storage(c["k_all"][b], dtype), to_storage(c["v_all"][b], dtype), kco, vco,
                       c["slots"][b].tolist())
    if c["pre_slots"].size:
        oracle_scatter(to_storage(c["k_pre"], dtype), to_storage(c["v_pre"], dtype), kco, vco,
                       c["pre_slots"].tolist())
    return oracle_attention(to_storage(c["q"], dtype), kco, vco, c["tables"].tolist(), c["lens"], scale, dtype), \
        kco, vco


def bits(t):
    return t.view(torch.int32 if t.dtype == torch.float32 else torch.int16)


CASES = [
    # dtype, hq, hkv, d, bs, cached lengths (before the step)
    ("f16", 14, 2, 64, 16, [0, 15, 16, 31, 32, 33, 47, 100, 511, 1000]),
    ("bf16", 28, 4, 128, 16, [0, 1, 16, 31, 63, 64, 200, 777, 2047]),
    ("bf16", 32, 8, 128, 32, [0, 31, 32, 95, 96, 300, 1023, 4100]),
    ("f16", 16, 2, 128, 32, [5, 64, 65, 129, 900]),
    ("bf16", 16, 1, 256, 16, [7, 17, 250]),
    ("f32", 4, 2, 64, 16, [0, 3, 16, 40]),            # SIMT kernel: the two-launch form
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-g{c[1] // c[2]}-d{c[3]}-bs{c[4]}")
@pytest.mark.parametrize("mode", ["all_new", "some_new"])
def test_step_equals_write_then_attention(case, mode):
    dtype, hq, hkv, d, bs, cached = case
    seed = 7 + len(cached) + (0 if mode == "all_new" else 100)
    rng = np.random.default_rng(seed)
    has_new = [True] * len(cached) if mode == "all_new" else list(rng.random(len(cached)) < 0.5)
    c = build_step(dtype, hq, hkv, d, bs, cached, has_new, n_prefill=37, n_pad=5, seed=seed)
    scale = 1.0 / math.sqrt(d)
    status, out, out2, caches, caches2 = run_both(c, dtype, bs, hkv, d, scale)
    assert status == 0
    assert torch.equal(bits(out), bits(out2))
    for a, b in zip(caches, caches2):
        assert torch.equal(bits(a), bits(b))
    ref, kco, vco = oracle_out(c, dtype, bs, hkv, d, scale)
    got = to_f64(out, dtype)
    assert np.all(np.isfinite(got))
    err = np.max(np.abs(got - ref))
    assert err <= TOL[dtype], f"max abs err {err:.3e}"
    # the cache after the step holds exactly the oracle's scatter, bit for bit
    for t, o in zip(caches, (kco, vco)):
        assert np.array_equal(to_storage(t, dtype).view(np.uint8), o.view(np.uint8))


def test_inconsistent_new_row_is_reported():
    """A new-token row whose slot is not the sequence's newest position, and
    a row past the step, are recorded as DEVICE_STEP (reads stay in bounds)."""
    dtype, hq, hkv, d, bs, cached = CASES[0]
    c = build_step(dtype, hq, hkv, d, bs, cached, [True] * len(cached), n_prefill=8, n_pad=2, seed=3)
    scale = 1.0 / math.sqrt(d)
    other = int(c["new_row"][1])
    status, *_ = run_both(c, dtype, bs, hkv, d, scale, bad_row=(4, other))
    assert status == 11  # KV_ERR_DEVICE_STEP
    status, *_ = run_both(c, dtype, bs, hkv, d, scale, bad_row=(4, len(c["step_slots"]) + 3))
    assert status == 11


@pytest.mark.parametrize("name", WORKLOADS)
def test_engine_fused_equals_unfused(name):
    """The engine's fused step and its two-call step give bit-identical
    outputs and caches over several steps of every workload."""
    wl = make_workload(name)
    dev = torch.device("cuda")
    vals = make_values(wl, device="cuda")
    fused = PagedDecodeEngine(wl, dev, max_steps=4)
    plain = PagedDecodeEngine(wl, dev, max_steps=4, fused=False)
    fused.setup(vals)
    plain.setup(vals)
    for _ in range(3):
        a = fused.step(vals.q, vals.k_step, vals.v_step).clone()
        b = plain.step(vals.q, vals.k_step, vals.v_step).clone()
        assert torch.equal(bits(a), bits(b))
    assert torch.equal(bits(fused.k_cache), bits(plain.k_cache))
    assert torch.equal(bits(fused.v_cache), bits(plain.v_cache))
    assert pk.device_error() == 0
