"""The path the benchmark times -- the native step runner driven for many
steps -- checked step by step against the oracle.

Each step is one ``kvstep_run`` call: the manager's metadata for the step
(the previous step's prefill sequences released, this step's allocated
atomically, one decode append per running sequence, padded slots), tables
updated in place in the runner's rotating buffers, one copy to the device,
and the fused cache-write + attention launch.  Beside it the oracle replays
the same operations on its own manager and keeps every decode sequence's
logical K/V itself (its history, then the row each step appends), so
nothing on the oracle side comes from the device.  Per step:

* slot mapping (with the -1 pads), block tables and seq_lens are bit-exact
  ("MiniPaged-Qwen: Paged KV Cache 与 KV Block Manager" §9 append across
  block boundaries, §16.2 exported tables; "从零实现一个 mini vLLM: Block
  Manager", ModelRunner inputs);
* every valid row of the step (prefill chunk and decode tokens) sits in the
  cache at the oracle's slot, bit for bit (§11-§12 cache write);
* every decode sequence's output is within the stated tolerance of the
  float64 attention over its logical K/V (§13 decode through the table,
  §14 GQA).

Each step draws new q/k/v, and the lengths grow across block boundaries.
``host_io`` 0 is the benchmark's device-resident leg; 2 its end-to-end leg
(q/k/v staged in the runner's page-locked slots, the output copied back to
a page-locked host buffer).
"""

import numpy as np
import pytest
import torch

import paged_kv_cache_128_gb300 as pk
from oracle.attention import decode_attention_contiguous
from oracle.block_manager import BlockManager as OracleManager
from paged_kv_cache_128_gb300.engine import PagedDecodeEngine
from paged_kv_cache_128_gb300.inputs import make_values, make_workload, pad_positions
from tests.helpers import TOL, to_f64

pytestmark = pytest.mark.gpu

STEPS = 9


class OracleReplay:
    """The workload's host operations on the oracle manager, plus each decode
    sequence's logical K/V in float64 (history, then one row per step)."""

    def __init__(self, wl, vals, steps):
        self.wl = wl
        fo = None if wl.free_order is None else wl.free_order.tolist()
        self.mgr = OracleManager(wl.num_blocks, wl.block_size, fo)
        for op, sid, n in wl.setup_ops:
            if op == "prefill":
                self.mgr.allocate_for_prefill(sid, n)
            elif op == "append":
                self.mgr.append_slots(sid, n)
            else:
                self.mgr.free_sequence(sid)
        self.lens = [int(x) for x in wl.cached_lens]
        kh = to_f64(vals.k_hist, wl.dtype)
        vh = to_f64(vals.v_hist, wl.dtype)
        off = vals.hist_offsets
        shape = (wl.num_kv_heads, wl.head_dim)
        self.K, self.V = [], []
        for b, L in enumerate(self.lens):
            k = np.empty((L + steps,) + shape)
            v = np.empty((L + steps,) + shape)
            k[:L] = kh[off[b]:off[b + 1]]
            v[:L] = vh[off[b]:off[b + 1]]
            self.K.append(k)
            self.V.append(v)
        del kh, vh
        self.pads = set(pad_positions(wl).tolist())
        self.next_id = wl.next_id
        self.live_prefills = []

    def step(self):
        """One step's operations: release the previous step's prefill
        sequences, prefill this step's new ones, one decode append each.
        Returns the step's slot mapping (pads -1)."""
        wl = self.wl
        for sid in self.live_prefills:
            self.mgr.free_sequence(sid)
        new = list(range(self.next_id, self.next_id + wl.prefill_lens.size))
        self.next_id += len(new)
        slots = []
        for sid, n in zip(new, wl.prefill_lens):
            slots += self.mgr.allocate_for_prefill(sid, int(n))
        self.live_prefills = new
        slots += self.mgr.decode_step(wl.decode_ids.tolist())
        it = iter(slots)
        return np.array([-1 if pos in self.pads else next(it) for pos in range(wl.num_step_tokens)], dtype=np.int64)

    def append_rows(self, k_rows, v_rows):
        """Each decode sequence's new position gets its step row (float64)."""
        for b in range(len(self.lens)):
            self.K[b][self.lens[b]] = k_rows[b]
            self.V[b][self.lens[b]] = v_rows[b]
            self.lens[b] += 1

    def attention(self, q64):
        return [decode_attention_contiguous(q64[b], self.K[b][:L], self.V[b][:L], self.wl.scale)
                for b, L in enumerate(self.lens)]


def _rows_at(cache, slots):
    hkv, d = cache.shape[2], cache.shape[3]
    idx = torch.from_numpy(np.asarray(slots, dtype=np.int64)).to(cache.device)
    return cache.view(-1, hkv, d).index_select(0, idx)


def _bits(t):
    return t.view(torch.int32 if t.dtype == torch.float32 else torch.int16)


@pytest.mark.parametrize("host_io", [0, 2], ids=["device_io", "staged_io"])
@pytest.mark.parametrize("name", ["decode_gqa14x2_d64_fp16", "mixed_batch_bf16"])
def test_runner_steps_match_oracle(name, host_io):
    wl = make_workload(name)
    dev = torch.device("cuda")
    vals = make_values(wl)                                   # CPU draw: the oracle sees the same numbers
    eng = PagedDecodeEngine(wl, dev, max_steps=STEPS + 2)    # unused slots hold NaN
    eng.setup(vals)
    ora = OracleReplay(wl, vals, STEPS)
    eng.make_runner(host_io=host_io)
    out_h = torch.empty(vals.q.shape, dtype=vals.q.dtype, pin_memory=True)
    out_d = torch.empty_like(vals.q, device=dev)
    g = torch.Generator().manual_seed(wl.seed + 77)
    crossings = 0
    pk.device_error()
    for step in range(STEPS):
        def draw(*shape):
            return (torch.randn(*shape, generator=g) * wl.value_scale).to(wl.torch_dtype)
        q = draw(wl.num_seqs, wl.num_heads, wl.head_dim)
        k = draw(wl.num_step_tokens, wl.num_kv_heads, wl.head_dim)
        v = draw(wl.num_step_tokens, wl.num_kv_heads, wl.head_dim)
        if host_io == 2:
            for dst, src in zip(eng.runner_stage(-1), (q, k, v)):
                dst.copy_(src)
            eng.runner_step(None, None, None, out_h)
        else:
            kd, vd = k.to(dev), v.to(dev)
            eng.runner_step(q.to(dev), kd, vd, out_d)
        eng.runner_join()
        torch.cuda.synchronize()
        assert pk.device_error() == 0, f"step {step}"

        # metadata, bit-exact
        mapping = ora.step()
        slots, tables, lens, rows = eng.runner_last_metadata()
        assert np.array_equal(slots.astype(np.int64), mapping), f"step {step}: slot mapping"
        o_tables, o_lens = ora.mgr.export(wl.decode_ids.tolist(), eng.max_blocks)
        assert np.array_equal(tables, np.asarray(o_tables, dtype=np.int32)), f"step {step}: block tables"
        assert np.array_equal(lens, np.asarray(o_lens, dtype=np.int32)), f"step {step}: seq_lens"
        crossings += int(sum(1 for L in o_lens if (L - 1) % wl.block_size == 0))

        # cache write: every valid row of the step at the oracle's slot, bit for bit
        valid = np.nonzero(mapping >= 0)[0]
        assert torch.equal(_bits(_rows_at(eng.k_cache, mapping[valid]).cpu()), _bits(k[valid]))
        assert torch.equal(_bits(_rows_at(eng.v_cache, mapping[valid]).cpu()), _bits(v[valid]))

        # attention: every decode sequence against the float64 oracle
        n_pre = int(wl.prefill_lens.sum())
        dec_rows = valid[n_pre:n_pre + wl.num_seqs]      # decode tokens follow the prefill chunk
        assert np.array_equal(rows, dec_rows.astype(np.int32))
        ora.append_rows(to_f64(k[dec_rows], wl.dtype), to_f64(v[dec_rows], wl.dtype))
        got = to_f64(out_h if host_io == 2 else out_d, wl.dtype)
        ref = ora.attention(to_f64(q, wl.dtype))
        worst = max(float(np.max(np.abs(got[b] - ref[b]))) for b in range(wl.num_seqs))
        assert worst <= TOL[wl.dtype], f"{name} step {step}: max abs err {worst:.3e}"
    assert crossings > 0          # some decode append opened a new block during the steps
    assert eng.mgr.check_invariants() and ora.mgr.invariants_ok()
    eng.close_runner()
