"""GPU parity of the native step runner (kvstep_*).

The runner does a whole serving step in one library call: the manager's
metadata into a page-locked buffer, an async copy on a side stream, and the
fused cache-write + attention launch after an event wait.  Driven for
several steps, it must reproduce the Python-driven step bit for bit:
outputs, caches, host metadata and each decode sequence's row in the step.
With host I/O it also copies q/k/v in and the output out itself.
"""

import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_128_gb300 as pk
from paged_kv_cache_128_gb300._lib import KVError, check, kvstep_config_t, lib
from paged_kv_cache_128_gb300.engine import PagedDecodeEngine
from paged_kv_cache_128_gb300.inputs import make_values, make_workload

pytestmark = pytest.mark.gpu

NAMES = ["decode_tiny_fp32", "decode_gqa14x2_d64_fp16", "decode_long_skewed_bf16", "mixed_batch_bf16"]


def bits(t):
    return t.view(torch.int32 if t.dtype == torch.float32 else torch.int16)


@pytest.mark.parametrize("name", NAMES)
@pytest.mark.parametrize("host_io", [0, 1, 2], ids=["device_io", "host_io", "staged_io"])
def test_runner_matches_python_step(name, host_io):
    wl = make_workload(name)
    dev = torch.device("cuda")
    vals = make_values(wl, device="cuda")
    ref = PagedDecodeEngine(wl, dev, max_steps=12)
    run = PagedDecodeEngine(wl, dev, max_steps=12)
    ref.setup(vals)
    run.setup(vals)
    run.make_runner(host_io=host_io)
    if host_io == 1:
        q, k, v = (t.cpu().pin_memory() for t in (vals.q, vals.k_step, vals.v_step))
        out = torch.empty(vals.q.shape, dtype=vals.q.dtype, pin_memory=True)
    elif host_io == 2:
        q = k = v = None
        out = torch.empty(vals.q.shape, dtype=vals.q.dtype, pin_memory=True)
    else:
        q, k, v, out = vals.q, vals.k_step, vals.v_step, torch.empty_like(vals.q)
    for _ in range(9):  # every metadata buffer is reused (its tables updated, not rewritten)
        a = ref.step(vals.q, vals.k_step, vals.v_step).clone()
        if host_io == 2:  # this step's slot, written after its previous copy has run
            for dst, src in zip(run.runner_stage(-1), (vals.q, vals.k_step, vals.v_step)):
                dst.copy_(src.cpu())
        run.runner_step(q, k, v, out)
        run.runner_join()
        torch.cuda.synchronize()
        assert torch.equal(bits(a), bits(out.to(dev)))
        slots, tables, lens, rows = run.runner_last_metadata()
        assert np.array_equal(slots, ref.h_slots.numpy())
        assert np.array_equal(tables, ref.h_tables.numpy())
        assert np.array_equal(lens, ref.h_lens.numpy())
        assert np.array_equal(rows, ref.d_new_rows.cpu().numpy())
    assert torch.equal(bits(ref.k_cache), bits(run.k_cache))
    assert torch.equal(bits(ref.v_cache), bits(run.v_cache))
    assert pk.device_error() == 0
    run.close_runner()


def test_runner_rejects_bad_steps():
    wl = make_workload("decode_gqa14x2_d64_fp16")
    dev = torch.device("cuda")
    vals = make_values(wl, device="cuda")
    eng = PagedDecodeEngine(wl, dev, max_steps=4)
    eng.setup(vals)
    eng.make_runner()
    out = torch.empty_like(vals.q)
    ids = eng._decode_ids
    # n_decode must be the configured batch
    st = lib().kvstep_run(eng._runner, vals.q.data_ptr(), vals.k_step.data_ptr(), vals.v_step.data_ptr(),
                          out.data_ptr(), None, 0, None, None, 0, ids.ctypes.data, ids.size - 1, None, 0)
    assert st == 1
    # an unknown sequence: the manager's error, nothing launched
    bad = ids.copy()
    bad[3] = 10 ** 9
    st = lib().kvstep_run(eng._runner, vals.q.data_ptr(), vals.k_step.data_ptr(), vals.v_step.data_ptr(),
                          out.data_ptr(), None, 0, None, None, 0, bad.ctypes.data, bad.size, None, 0)
    assert st == 3
    # then a good step still runs and matches a direct one
    eng.runner_step(vals.q, vals.k_step, vals.v_step, out)
    eng.runner_join()
    torch.cuda.synchronize()
    assert pk.device_error() == 0
    h = ctypes.c_void_p()
    with pytest.raises(KVError):   # an empty configuration is rejected before anything is allocated
        check(lib().kvstep_create(eng.mgr._h, ctypes.byref(kvstep_config_t(num_seqs=0)), ctypes.byref(h)),
              "kvstep_create")
    eng.close_runner()


@pytest.mark.parametrize("name", ["decode_gqa28x4_d128_bf16", "mixed_batch_bf16"])
def test_runner_fp8_cache_matches_python_step(name):
    """With fp8 caches the runner's step (quantised write, then fp8
    attention) equals the Python-driven step bit for bit: outputs, codes and
    scales."""
    wl = make_workload(name)
    dev = torch.device("cuda")
    vals = make_values(wl, device="cuda")
    ref = PagedDecodeEngine(wl, dev, max_steps=4, kv_cache="fp8")
    run = PagedDecodeEngine(wl, dev, max_steps=4, kv_cache="fp8")
    ref.setup(vals)
    run.setup(vals)
    run.make_runner()
    out = torch.empty_like(vals.q)
    for _ in range(3):
        a = ref.step(vals.q, vals.k_step, vals.v_step).clone()
        run.runner_step(vals.q, vals.k_step, vals.v_step, out)
        run.runner_join()
        torch.cuda.synchronize()
        assert torch.equal(bits(a), bits(out))
    assert torch.equal(ref.k_cache, run.k_cache) and torch.equal(ref.v_cache, run.v_cache)
    assert torch.equal(ref.k_scales.view(torch.int32), run.k_scales.view(torch.int32))
    assert torch.equal(ref.v_scales.view(torch.int32), run.v_scales.view(torch.int32))
    assert pk.device_error() == 0
    run.close_runner()
