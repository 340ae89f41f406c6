"""Full-size workloads, run through the same engine and launch
configuration the benchmark times, checked against the oracle:

* host metadata (slot mapping with padding, block tables, seq_lens) is
  bit-exact against the oracle manager replaying the same operations;
* every written cache row equals its input row bit for bit, and the number
  of rows that differ from the NaN sentinel equals the number written
  (a property that holds at any size);
* every sequence's attention output is within tolerance of the float64
  oracle evaluated on that sequence's logical K/V.
"""

import numpy as np
import pytest
import torch

import paged_kv_cache_128_gb300 as pk
from oracle.attention import decode_attention_contiguous
from oracle.block_manager import BlockManager as OracleManager
from paged_kv_cache_128_gb300.engine import PagedDecodeEngine
from paged_kv_cache_128_gb300.inputs import WORKLOADS, make_values, make_workload, pad_positions
from tests.helpers import SENTINEL, TOL, to_f64

pytestmark = pytest.mark.gpu


def _oracle_step(wl):
    """Replay setup + one step on the oracle manager; return (history slots in
    batch order, step slot mapping, tables, lens)."""
    ora = OracleManager(wl.num_blocks, wl.block_size, None if wl.free_order is None else wl.free_order.tolist())
    hist = {int(i): [] for i in wl.decode_ids}
    for op, sid, n in wl.setup_ops:
        if op == "prefill":
            s = ora.allocate_for_prefill(sid, n)
        elif op == "append":
            s = ora.append_slots(sid, n)
        else:
            ora.free_sequence(sid)
            continue
        if sid in hist:
            hist[sid] += s
    hist_slots = np.array([x for i in wl.decode_ids for x in hist[int(i)]], dtype=np.int64)
    step = []
    nid = wl.next_id
    for n in wl.prefill_lens:
        step += ora.allocate_for_prefill(nid, int(n))
        nid += 1
    step += ora.decode_step(wl.decode_ids.tolist())
    total = wl.num_step_tokens
    pads = set(pad_positions(wl).tolist())
    mapping = np.empty(total, dtype=np.int64)
    it = iter(step)
    for pos in range(total):
        mapping[pos] = -1 if pos in pads else next(it)
    return ora, hist_slots, mapping


def _rows_equal(cache, slots, rows):
    """Bitwise equality of cache rows at `slots` with `rows` (on the GPU)."""
    hkv, d = cache.shape[2], cache.shape[3]
    flat = cache.view(-1, hkv, d)
    iv = torch.int32 if cache.dtype == torch.float32 else torch.int16
    idx = torch.from_numpy(np.asarray(slots, dtype=np.int64)).to(cache.device)
    return torch.equal(flat.index_select(0, idx).view(iv), rows.to(cache.device).view(iv))


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "two_calls"])
@pytest.mark.parametrize("name", WORKLOADS)
def test_workload_step_matches_oracle(name, fused):
    wl = make_workload(name)
    vals = make_values(wl)
    dev = torch.device("cuda")
    eng = PagedDecodeEngine(wl, dev, max_steps=4, fused=fused)
    eng.setup(vals)
    pk.device_error()
    out = eng.step(vals.q.to(dev), vals.k_step.to(dev), vals.v_step.to(dev))
    torch.cuda.synchronize()
    assert pk.device_error() == 0

    # host metadata: bit-exact
    ora, hist_slots, mapping = _oracle_step(wl)
    assert np.array_equal(eng.history_slots.astype(np.int64), hist_slots)
    assert np.array_equal(eng.h_slots.numpy().astype(np.int64), mapping)
    tables, lens = ora.export(wl.decode_ids.tolist(), eng.max_blocks)
    assert np.array_equal(eng.h_tables.numpy(), np.asarray(tables, dtype=np.int32))
    assert np.array_equal(eng.h_lens.numpy(), np.asarray(lens, dtype=np.int32))
    assert eng.mgr.check_invariants() and ora.invariants_ok()

    # cache writes: bit-exact rows, and nothing else touched
    assert _rows_equal(eng.k_cache, hist_slots, vals.k_hist)
    assert _rows_equal(eng.v_cache, hist_slots, vals.v_hist)
    valid = np.nonzero(mapping >= 0)[0]
    assert _rows_equal(eng.k_cache, mapping[valid], vals.k_step[valid])
    assert _rows_equal(eng.v_cache, mapping[valid], vals.v_step[valid])
    iv = torch.int32 if wl.dtype == "f32" else torch.int16
    s = SENTINEL[wl.dtype]
    s = s - (1 << 16) if (iv == torch.int16 and s >= 1 << 15) else s
    for cache in (eng.k_cache, eng.v_cache):
        touched = (cache.view(iv).view(-1, wl.head_dim) != s).any(dim=1).sum().item()
        assert touched == (hist_slots.size + valid.size) * wl.num_kv_heads

    # attention: every sequence against the float64 oracle on logical K/V
    n_pre = int(wl.prefill_lens.sum())
    got = to_f64(out, wl.dtype)
    q64 = to_f64(vals.q, wl.dtype)
    off = vals.hist_offsets
    worst = 0.0
    for b in range(wl.num_seqs):
        row = valid[n_pre + b]        # this sequence's decode token in the step
        K = np.concatenate([to_f64(vals.k_hist[off[b]:off[b + 1]], wl.dtype),
                            to_f64(vals.k_step[row:row + 1], wl.dtype)])
        V = np.concatenate([to_f64(vals.v_hist[off[b]:off[b + 1]], wl.dtype),
                            to_f64(vals.v_step[row:row + 1], wl.dtype)])
        assert K.shape[0] == lens[b]
        ref = decode_attention_contiguous(q64[b], K, V, wl.scale)
        worst = max(worst, float(np.max(np.abs(got[b] - ref))))
    assert worst <= TOL[wl.dtype], f"{name}: max abs err {worst:.3e}"


@pytest.mark.parametrize("name", ["decode_gqa14x2_d64_fp16", "mixed_batch_bf16"])
def test_graph_steps_match_direct_steps(name):
    """The benchmark replays each step's device part as a CUDA graph; its
    outputs, cache writes and metadata equal those of direct launches."""
    wl = make_workload(name)
    dev = torch.device("cuda")
    vals = make_values(wl, device="cuda")
    direct = PagedDecodeEngine(wl, dev, max_steps=6)
    graphed = PagedDecodeEngine(wl, dev, max_steps=6)
    direct.setup(vals)
    graphed.setup(vals)
    a = direct.step(vals.q, vals.k_step, vals.v_step).clone()
    b = graphed.step(vals.q, vals.k_step, vals.v_step).clone()
    assert torch.equal(a, b)
    graphed.capture(vals.q, vals.k_step, vals.v_step)
    for _ in range(4):
        a = direct.step(vals.q, vals.k_step, vals.v_step).clone()
        b = graphed.step_graph().clone()
        torch.cuda.synchronize()
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        assert torch.equal(direct.h_tables, graphed.h_tables) and torch.equal(direct.h_lens, graphed.h_lens)
    assert torch.equal(direct.k_cache.view(torch.int16), graphed.k_cache.view(torch.int16))
    assert pk.device_error() == 0
