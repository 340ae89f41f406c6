"""GPU parity of multi-layer pools: one block table and one slot mapping
serve several layers' caches ([layers, NB, BS, Hkv, D]).

* ``reshape_and_cache_layers`` writes every layer in one launch; each
  layer's cache must equal the oracle's scatter of that layer's rows, bit
  for bit, with padded rows landing nowhere.
* The native step runner with several layers builds and copies the step's
  metadata once and launches one fused step per layer: every layer's output
  must equal a single-layer ``paged_decode_step`` on a twin pool bit for
  bit, and the float64 oracle within tolerance.
"""

import ctypes
import math

import numpy as np
import pytest
import torch

import paged_kv_cache_128_gb300 as pk
from oracle.attention import decode_attention_contiguous
from oracle.paged_cache import reshape_and_cache as oracle_scatter
from paged_kv_cache_128_gb300._lib import check, kvstep_config_t, lib
from paged_kv_cache_128_gb300.kernels import alloc_workspace, decode_plan, dtype_code
from tests.helpers import TOL, TORCH, sentinel_storage, sentinel_tensor, to_f64, to_storage

pytestmark = pytest.mark.gpu


def bits(t):
    return t.view(torch.int32 if t.dtype == torch.float32 else torch.int16)


@pytest.mark.parametrize("dtype,layers,hkv,d,bs", [("bf16", 3, 4, 128, 16), ("f16", 5, 2, 64, 32),
                                                   ("f32", 2, 1, 8, 4)])
def test_cache_write_all_layers(dtype, layers, hkv, d, bs):
    rng = np.random.default_rng(layers)
    g = torch.Generator().manual_seed(layers)
    nb, n = 40, 57
    slots = rng.permutation(nb * bs)[:n].astype(np.int32)
    slots[rng.choice(n, 6, replace=False)] = -1                   # padded rows
    dt = TORCH[dtype]
    k = torch.randn(layers, n, hkv, d, generator=g).to(dt)
    v = torch.randn(layers, n, hkv, d, generator=g).to(dt)
    dev = torch.device("cuda")
    kc = sentinel_tensor((layers, nb, bs, hkv, d), dtype, dev)
    vc = sentinel_tensor((layers, nb, bs, hkv, d), dtype, dev)
    pk.device_error()
    pk.reshape_and_cache_layers(k.to(dev), v.to(dev), kc, vc, torch.from_numpy(slots).to(dev))
    assert pk.device_error() == 0
    for layer in range(layers):
        ko = sentinel_storage((nb, bs, hkv, d), dtype)
        vo = sentinel_storage((nb, bs, hkv, d), dtype)
        oracle_scatter(to_storage(k[layer], dtype), to_storage(v[layer], dtype), ko, vo, slots.tolist())
        assert np.array_equal(to_storage(kc[layer], dtype).view(np.uint8), ko.view(np.uint8))
        assert np.array_equal(to_storage(vc[layer], dtype).view(np.uint8), vo.view(np.uint8))


def _pool(layers, nb, bs, hkv, d, dtype, lens, seed, value_scale=1.0):
    rng = np.random.default_rng(seed)
    g = torch.Generator().manual_seed(seed)
    dt = TORCH[dtype]
    dev = torch.device("cuda")
    mgr = pk.KVBlockManager(nb, bs, rng.permutation(nb).tolist())
    kc = sentinel_tensor((layers, nb, bs, hkv, d), dtype, dev)
    vc = sentinel_tensor((layers, nb, bs, hkv, d), dtype, dev)
    hist_k, hist_v = [], []
    for sid, L in enumerate(lens):
        slots = torch.from_numpy(mgr.allocate_for_prefill(sid, L)).to(dev)
        kk = (torch.randn(layers, L, hkv, d, generator=g) * value_scale).to(dt)
        vv = (torch.randn(layers, L, hkv, d, generator=g) * value_scale).to(dt)
        pk.reshape_and_cache_layers(kk.to(dev), vv.to(dev), kc, vc, slots)
        hist_k.append(kk)
        hist_v.append(vv)
    return mgr, kc, vc, hist_k, hist_v


def test_runner_layers_share_metadata():
    dtype, layers, hq, hkv, d, bs, nb = "bf16", 4, 16, 4, 128, 16, 600
    dt = TORCH[dtype]
    dev = torch.device("cuda")
    # Values N(0, 1) / 2 as in the small-model workload: with a handful of
    # N(0, 1) tokens, outputs above 2 make half a bf16 ulp alone 4e-3 and the
    # stated 8e-3 bar unattainable for any rounding to bf16.
    lens = [15, 16, 33, 100, 333, 512, 47]
    B = len(lens)
    ids = np.arange(B, dtype=np.int64)
    mgr_r, kc_r, vc_r, hk, hv = _pool(layers, nb, bs, hkv, d, dtype, lens, seed=3, value_scale=0.5)
    mgr_p, kc_p, vc_p, _, _ = _pool(layers, nb, bs, hkv, d, dtype, lens, seed=3, value_scale=0.5)
    max_len, max_blocks = 600, 600 // bs + 1
    scale = 1.0 / math.sqrt(d)
    ws = alloc_workspace(decode_plan(B, hq, hkv, d, bs, max_len, dt), dev)
    cfg = kvstep_config_t(num_seqs=B, num_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs, num_blocks=nb,
                          max_blocks_per_seq=max_blocks, max_seq_len=max_len, scale=scale, dtype=dtype_code(dt),
                          num_step_tokens=B, k_cache=kc_r.data_ptr(), v_cache=vc_r.data_ptr(),
                          workspace=ws.data_ptr(), workspace_bytes=ws.numel(),
                          stream=torch.cuda.current_stream().cuda_stream, host_io=0, num_layers=layers,
                          cache_layer_stride=kc_r.stride(0))
    h = ctypes.c_void_p()
    check(lib().kvstep_create(mgr_r._h, ctypes.byref(cfg), ctypes.byref(h)), "kvstep_create")
    g = torch.Generator().manual_seed(77)
    rows = torch.arange(B, dtype=torch.int32, device=dev)
    logical_k = [x.clone() for x in hk]
    logical_v = [x.clone() for x in hv]
    try:
        for step in range(3):
            q = (torch.randn(layers, B, hq, d, generator=g) * 0.5).to(dt)
            kn = (torch.randn(layers, B, hkv, d, generator=g) * 0.5).to(dt)
            vn = (torch.randn(layers, B, hkv, d, generator=g) * 0.5).to(dt)
            qd, knd, vnd = q.to(dev), kn.to(dev), vn.to(dev)
            out_r = torch.empty(layers, B, hq, d, dtype=dt, device=dev)
            check(lib().kvstep_run(h, qd.data_ptr(), knd.data_ptr(), vnd.data_ptr(), out_r.data_ptr(), None, 0,
                                   None, None, 0, ids.ctypes.data, B, None, 0), "kvstep_run")
            check(lib().kvstep_join(h, torch.cuda.current_stream().cuda_stream), "kvstep_join")
            # twin: the same step, one single-layer fused call per layer
            slots, tables, lens_now = mgr_p.decode_step(ids, max_blocks)
            d_slots, d_tables, d_lens = (torch.from_numpy(a).to(dev) for a in (slots, tables, lens_now))
            out_p = torch.empty_like(out_r)
            for layer in range(layers):
                pk.paged_decode_step(out_p[layer], qd[layer], knd[layer], vnd[layer], d_slots, rows, kc_p[layer],
                                     vc_p[layer], d_tables, d_lens, scale, max_len)
            torch.cuda.synchronize()
            assert pk.device_error() == 0
            assert torch.equal(bits(out_r), bits(out_p))
            worst = 0.0
            for b in range(B):
                logical_k[b] = torch.cat([logical_k[b], kn[:, b:b + 1]], dim=1)
                logical_v[b] = torch.cat([logical_v[b], vn[:, b:b + 1]], dim=1)
                for layer in range(layers):
                    ref = decode_attention_contiguous(to_f64(q[layer, b], dtype), to_f64(logical_k[b][layer], dtype),
                                                      to_f64(logical_v[b][layer], dtype), scale)
                    worst = max(worst, float(np.max(np.abs(to_f64(out_r[layer, b], dtype) - ref))))
            assert worst <= TOL[dtype], f"step {step}: max abs err {worst:.3e}"
        assert torch.equal(bits(kc_r), bits(kc_p)) and torch.equal(bits(vc_r), bits(vc_p))
    finally:
        lib().kvstep_destroy(h)
