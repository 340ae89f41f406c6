"""GPU parity of prefix sharing with copy-on-write.

* ``copy_blocks`` copies whole blocks of every layer bit for bit, and
  skips (and reports) pairs outside the pool.
* Decode over forked sequences: children share their parent's prefix blocks
  (kvbm_fork); each step appends one token to every sequence, applies the
  queued copy-on-write copies on the device, then runs the fused cache write
  + attention.  Every sequence's cache, read back through its table, must
  equal its own logical K/V bit for bit (parent prefix, then its own
  tokens), and attention must match the float64 oracle on those tensors.
"""

import math

import numpy as np
import pytest
import torch

import paged_kv_cache_128_gb300 as pk
from paged_kv_cache_128_gb300 import kernels as pk_kernels
from oracle.attention import decode_attention_contiguous
from tests.helpers import TOL, TORCH, sentinel_tensor, to_f64

pytestmark = pytest.mark.gpu


def bits(t):
    return t.view(torch.int32 if t.dtype == torch.float32 else torch.int16)


@pytest.mark.parametrize("layers", [1, 3])
def test_copy_blocks_bit_exact(layers):
    g = torch.Generator().manual_seed(11 + layers)
    nb, bs, hkv, d = 64, 16, 2, 128
    shape = (nb, bs, hkv, d) if layers == 1 else (layers, nb, bs, hkv, d)
    k = torch.randn(shape, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(shape, generator=g).to(torch.bfloat16).cuda()
    src = torch.tensor([3, 7, 20, 41, 5], dtype=torch.int32)
    dst = torch.tensor([50, 2, 63, 0, 33], dtype=torch.int32)
    k_want, v_want = k.clone(), v.clone()
    kw = k_want.view(-1, nb, bs, hkv, d)
    vw = v_want.view(-1, nb, bs, hkv, d)
    for s, t in zip(src.tolist(), dst.tolist()):
        kw[:, t] = kw[:, s]
        vw[:, t] = vw[:, s]
    pk.device_error()
    pk.copy_blocks(k, v, src.cuda(), dst.cuda())
    assert pk.device_error() == 0
    assert torch.equal(bits(k), bits(k_want)) and torch.equal(bits(v), bits(v_want))
    # a pair outside the pool is skipped and reported; the others still copy
    k2, v2 = k.clone(), v.clone()
    pk.copy_blocks(k2, v2, torch.tensor([1, nb + 5], dtype=torch.int32).cuda(),
                   torch.tensor([4, 6], dtype=torch.int32).cuda())
    assert pk.device_error() == 8
    kw2 = k.view(-1, nb, bs, hkv, d).clone()
    kw2[:, 4] = kw2[:, 1]
    assert torch.equal(bits(k2.view(-1, nb, bs, hkv, d)), bits(kw2))


@pytest.mark.parametrize("dtype,hq,hkv,d,bs", [("bf16", 8, 2, 128, 16), ("f16", 14, 2, 64, 32)])
def test_decode_over_forked_sequences(dtype, hq, hkv, d, bs):
    rng = np.random.default_rng(5)
    g = torch.Generator().manual_seed(5)
    dt = TORCH[dtype]
    nb = 400
    order = rng.permutation(nb).tolist()
    mgr = pk.KVBlockManager(nb, bs, order)
    dev = torch.device("cuda")
    kc = sentinel_tensor((nb, bs, hkv, d), dtype, dev)
    vc = sentinel_tensor((nb, bs, hkv, d), dtype, dev)
    logical_k, logical_v = {}, {}
    sid = 0
    for _ in range(5):                                        # parents
        L = int(rng.integers(20, 300))
        slots = mgr.allocate_for_prefill(sid, L)
        kk = torch.randn(L, hkv, d, generator=g).to(dt)
        vv = torch.randn(L, hkv, d, generator=g).to(dt)
        pk.reshape_and_cache(kk.to(dev), vv.to(dev), kc, vc, torch.from_numpy(slots).to(dev))
        logical_k[sid], logical_v[sid] = kk, vv
        parent = sid
        sid += 1
        for _ in range(2):                                    # children sharing a prefix of it
            plen = int(rng.integers(1, L + 1))
            mgr.fork(parent, sid, plen)
            logical_k[sid], logical_v[sid] = kk[:plen].clone(), vv[:plen].clone()
            sid += 1
    assert mgr.check_invariants()
    assert not mgr.take_copies()[0].size                      # forks copy nothing
    ids = list(range(sid))
    B = len(ids)
    max_blocks = 300 // bs + 8
    scale = 1.0 / math.sqrt(d)
    q = torch.randn(B, hq, d, generator=g).to(dt)
    rows = torch.arange(B, dtype=torch.int32, device=dev)
    copies_seen = 0
    for step in range(4):
        slots, tables, lens = mgr.decode_step(ids, max_blocks)
        src, dst = mgr.take_copies()
        copies_seen += src.size
        if src.size:                                          # copies before this step's writes
            pk.copy_blocks(kc, vc, torch.from_numpy(src).to(dev), torch.from_numpy(dst).to(dev))
        kn = torch.randn(B, hkv, d, generator=g).to(dt)
        vn = torch.randn(B, hkv, d, generator=g).to(dt)
        for i, s in enumerate(ids):
            logical_k[s] = torch.cat([logical_k[s], kn[i:i + 1]])
            logical_v[s] = torch.cat([logical_v[s], vn[i:i + 1]])
        out = torch.empty(B, hq, d, dtype=dt, device=dev)
        pk.paged_decode_step(out, q.to(dev), kn.to(dev), vn.to(dev), torch.from_numpy(slots).to(dev), rows, kc, vc,
                             torch.from_numpy(tables).to(dev), torch.from_numpy(lens).to(dev), scale,
                             int(lens.max()))
        assert pk.device_error() == 0
        assert mgr.check_invariants()
        got = to_f64(out, dtype)
        q64 = to_f64(q, dtype)
        worst = 0.0
        for i, s in enumerate(ids):
            assert lens[i] == logical_k[s].shape[0]
            ref = decode_attention_contiguous(q64[i], to_f64(logical_k[s], dtype), to_f64(logical_v[s], dtype),
                                              scale)
            worst = max(worst, float(np.max(np.abs(got[i] - ref))))
        assert worst <= TOL[dtype], f"step {step}: max abs err {worst:.3e}"
    assert copies_seen > 0                                    # the case exercised copy-on-write
    # every sequence reads back exactly its own tokens through its table
    flat_k, flat_v = kc.view(-1, hkv, d), vc.view(-1, hkv, d)
    for s in ids:
        table = mgr.block_table(s)
        L = mgr.seq_len(s)
        pos = np.arange(L)
        slot = torch.from_numpy(table[pos // bs].astype(np.int64) * bs + pos % bs).to(dev)
        assert torch.equal(bits(flat_k.index_select(0, slot)), bits(logical_k[s].to(dev)))
        assert torch.equal(bits(flat_v.index_select(0, slot)), bits(logical_v[s].to(dev)))


def test_step_runner_applies_copies():
    """The native step runner takes the copies its decode appends queue and
    copies the blocks before its fused launch: over forked sequences its
    outputs and caches equal those of the same steps driven from Python."""
    import ctypes

    from paged_kv_cache_128_gb300._lib import check, kvstep_config_t, lib
    from paged_kv_cache_128_gb300.kernels import alloc_workspace, decode_plan, dtype_code

    dtype, hq, hkv, d, bs, nb = "bf16", 8, 2, 128, 16, 300
    dt = TORCH[dtype]
    dev = torch.device("cuda")
    sides = []
    for _ in range(2):
        rng = np.random.default_rng(9)
        g = torch.Generator().manual_seed(9)
        mgr = pk.KVBlockManager(nb, bs, rng.permutation(nb).tolist())
        kc = sentinel_tensor((nb, bs, hkv, d), dtype, dev)
        vc = sentinel_tensor((nb, bs, hkv, d), dtype, dev)
        sid = 0
        for _ in range(4):
            L = int(rng.integers(10, 200))
            slots = mgr.allocate_for_prefill(sid, L)
            pk.reshape_and_cache(torch.randn(L, hkv, d, generator=g).to(dt).to(dev),
                                 torch.randn(L, hkv, d, generator=g).to(dt).to(dev), kc, vc,
                                 torch.from_numpy(slots).to(dev))
            parent = sid
            sid += 1
            for _ in range(2):
                mgr.fork(parent, sid, int(rng.integers(1, L + 1)))
                sid += 1
        sides.append((mgr, kc, vc))
    B = sid
    ids = np.arange(B, dtype=np.int64)
    max_blocks, max_len = 200 // bs + 8, 200 + 16
    scale = 1.0 / math.sqrt(d)
    g = torch.Generator().manual_seed(1)
    q = torch.randn(B, hq, d, generator=g).to(dt).to(dev)
    plan = decode_plan(B, hq, hkv, d, bs, max_len, dt)
    ws = alloc_workspace(plan, dev)
    mgr_r, kc_r, vc_r = sides[1]
    cfg = kvstep_config_t(num_seqs=B, num_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs, num_blocks=nb,
                          max_blocks_per_seq=max_blocks, max_seq_len=max_len, scale=scale, dtype=dtype_code(dt),
                          num_step_tokens=B, k_cache=kc_r.data_ptr(), v_cache=vc_r.data_ptr(),
                          workspace=ws.data_ptr() if ws is not None else None,
                          workspace_bytes=ws.numel() if ws is not None else 0,
                          stream=torch.cuda.current_stream().cuda_stream, host_io=0)
    h = ctypes.c_void_p()
    check(lib().kvstep_create(mgr_r._h, ctypes.byref(cfg), ctypes.byref(h)), "kvstep_create")
    mgr_p, kc_p, vc_p = sides[0]
    rows = torch.arange(B, dtype=torch.int32, device=dev)
    copies = 0
    try:
        for _ in range(5):
            kn = torch.randn(B, hkv, d, generator=g).to(dt).to(dev)
            vn = torch.randn(B, hkv, d, generator=g).to(dt).to(dev)
            # Python-driven step
            slots, tables, lens = mgr_p.decode_step(ids, max_blocks)
            src, dst = mgr_p.take_copies()
            copies += src.size
            if src.size:
                pk.copy_blocks(kc_p, vc_p, torch.from_numpy(src).to(dev), torch.from_numpy(dst).to(dev))
            out_p = torch.empty(B, hq, d, dtype=dt, device=dev)
            pk.paged_decode_step(out_p, q, kn, vn, torch.from_numpy(slots).to(dev), rows, kc_p, vc_p,
                                 torch.from_numpy(tables).to(dev), torch.from_numpy(lens).to(dev), scale, max_len)
            # runner step
            out_r = torch.empty_like(out_p)
            check(lib().kvstep_run(h, q.data_ptr(), kn.data_ptr(), vn.data_ptr(), out_r.data_ptr(), None, 0, None,
                                   None, 0, ids.ctypes.data, B, None, 0), "kvstep_run")
            check(lib().kvstep_join(h, torch.cuda.current_stream().cuda_stream), "kvstep_join")
            torch.cuda.synchronize()
            assert torch.equal(bits(out_p), bits(out_r))
        assert copies > 0
        assert torch.equal(bits(kc_p), bits(kc_r)) and torch.equal(bits(vc_p), bits(vc_r))
        assert pk.device_error() == 0
    finally:
        lib().kvstep_destroy(h)


def test_copy_blocks_fp8_bit_exact():
    """fp8 caches: each copied block's codes and scales equal the source's,
    and every other block is untouched."""
    dev = torch.device("cuda")
    nb, bs, hkv, d = 40, 16, 2, 128
    g = torch.Generator(device=dev).manual_seed(3)
    kc = torch.randint(0, 256, (nb, bs, hkv, d), generator=g, device=dev, dtype=torch.int32).to(torch.uint8)
    vc = torch.randint(0, 256, (nb, bs, hkv, d), generator=g, device=dev, dtype=torch.int32).to(torch.uint8)
    ks = torch.rand(nb, hkv, bs, generator=g, device=dev)
    vs = torch.rand(nb, hkv, bs, generator=g, device=dev)
    src = torch.tensor([3, 7, 0, 39], dtype=torch.int32, device=dev)
    dst = torch.tensor([10, 20, 21, 5], dtype=torch.int32, device=dev)
    want = [t.clone() for t in (kc, vc, ks, vs)]
    for t in want:
        t[dst.long()] = t[src.long()]
    pk_kernels.copy_blocks_fp8(kc, vc, ks, vs, src, dst)
    torch.cuda.synchronize()
    assert pk.device_error() == 0
    for got, w in zip((kc, vc, ks.view(torch.int32), vs.view(torch.int32)),
                      (want[0], want[1], want[2].view(torch.int32), want[3].view(torch.int32))):
        assert torch.equal(got, w)


def test_fp8_step_runner_applies_copies():
    """The step runner with fp8 caches over forked sequences: the copies its
    appends queue are applied (codes and scales) before its launch, and its
    outputs, codes and scales equal the same steps driven from Python."""
    import ctypes

    from paged_kv_cache_128_gb300._lib import check, kvstep_config_t, lib
    from paged_kv_cache_128_gb300.kernels import alloc_workspace, decode_plan, dtype_code

    hq, hkv, d, bs, nb = 8, 2, 128, 16, 300
    dt = torch.bfloat16
    dev = torch.device("cuda")
    sides = []
    for _ in range(2):
        rng = np.random.default_rng(19)
        g = torch.Generator().manual_seed(19)
        mgr = pk.KVBlockManager(nb, bs, rng.permutation(nb).tolist())
        kc = torch.full((nb, bs, hkv, d), 0x7F, dtype=torch.uint8, device=dev)
        vc = torch.full_like(kc, 0x7F)
        ks = torch.full((nb, hkv, bs), float("nan"), device=dev)
        vs = torch.full_like(ks, float("nan"))
        sid = 0
        for _ in range(4):
            L = int(rng.integers(10, 200))
            slots = mgr.allocate_for_prefill(sid, L)
            pk.reshape_and_cache_fp8(torch.randn(L, hkv, d, generator=g).to(dt).to(dev),
                                     torch.randn(L, hkv, d, generator=g).to(dt).to(dev), kc, vc, ks, vs,
                                     torch.from_numpy(slots).to(dev))
            parent = sid
            sid += 1
            for _ in range(2):
                mgr.fork(parent, sid, int(rng.integers(1, L + 1)))
                sid += 1
        sides.append((mgr, kc, vc, ks, vs))
    B = sid
    ids = np.arange(B, dtype=np.int64)
    max_blocks, max_len = 200 // bs + 8, 200 + 16
    scale = 1.0 / math.sqrt(d)
    g = torch.Generator().manual_seed(2)
    q = torch.randn(B, hq, d, generator=g).to(dt).to(dev)
    plan = decode_plan(B, hq, hkv, d, bs, max_len, dt)
    ws = alloc_workspace(plan, dev)
    mgr_r, kc_r, vc_r, ks_r, vs_r = sides[1]
    cfg = kvstep_config_t(num_seqs=B, num_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs, num_blocks=nb,
                          max_blocks_per_seq=max_blocks, max_seq_len=max_len, scale=scale, dtype=dtype_code(dt),
                          num_step_tokens=B, k_cache=kc_r.data_ptr(), v_cache=vc_r.data_ptr(),
                          workspace=ws.data_ptr(), workspace_bytes=ws.numel(),
                          stream=torch.cuda.current_stream().cuda_stream, host_io=0, cache_fp8=1,
                          k_scales=ks_r.data_ptr(), v_scales=vs_r.data_ptr())
    h = ctypes.c_void_p()
    check(lib().kvstep_create(mgr_r._h, ctypes.byref(cfg), ctypes.byref(h)), "kvstep_create")
    mgr_p, kc_p, vc_p, ks_p, vs_p = sides[0]
    rows = torch.arange(B, dtype=torch.int32, device=dev)
    copies = 0
    try:
        for _ in range(5):
            kn = torch.randn(B, hkv, d, generator=g).to(dt).to(dev)
            vn = torch.randn(B, hkv, d, generator=g).to(dt).to(dev)
            slots, tables, lens = mgr_p.decode_step(ids, max_blocks)
            src, dst = mgr_p.take_copies()
            copies += src.size
            if src.size:
                pk_kernels.copy_blocks_fp8(kc_p, vc_p, ks_p, vs_p, torch.from_numpy(src).to(dev),
                                           torch.from_numpy(dst).to(dev))
            out_p = torch.empty(B, hq, d, dtype=dt, device=dev)
            pk.paged_decode_step_fp8(out_p, q, kn, vn, torch.from_numpy(slots).to(dev), rows, kc_p, vc_p, ks_p, vs_p,
                                     torch.from_numpy(tables).to(dev), torch.from_numpy(lens).to(dev), scale, max_len)
            out_r = torch.empty_like(out_p)
            check(lib().kvstep_run(h, q.data_ptr(), kn.data_ptr(), vn.data_ptr(), out_r.data_ptr(), None, 0, None,
                                   None, 0, ids.ctypes.data, B, None, 0), "kvstep_run")
            check(lib().kvstep_join(h, torch.cuda.current_stream().cuda_stream), "kvstep_join")
            torch.cuda.synchronize()
            assert torch.equal(bits(out_p), bits(out_r))
        assert copies > 0
        assert torch.equal(kc_p, kc_r) and torch.equal(vc_p, vc_r)
        assert torch.equal(ks_p.view(torch.int32), ks_r.view(torch.int32))
        assert torch.equal(vs_p.view(torch.int32), vs_r.view(torch.int32))
        assert pk.device_error() == 0
    finally:
        lib().kvstep_destroy(h)
