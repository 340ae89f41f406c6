"""GPU parity of the cache-write kernel: bit-exact against the oracle
scatter over the whole pool (sentinel-filled, so any stray byte shows)."""

import numpy as np
import pytest
import torch

import paged_kv_cache_128_gb300 as pk
from oracle.paged_cache import reshape_and_cache as oracle_scatter
from tests.helpers import TORCH, sentinel_storage, sentinel_tensor, to_storage

pytestmark = pytest.mark.gpu


def _case(dtype, n, nb, bs, hkv, d, n_pad, seed):
    g = torch.Generator().manual_seed(seed)
    rng = np.random.default_rng(seed)
    k = torch.randn(n, hkv, d, generator=g).to(TORCH[dtype])
    v = torch.randn(n, hkv, d, generator=g).to(TORCH[dtype])
    slots = rng.choice(nb * bs, size=n, replace=False).astype(np.int32)
    if n_pad:
        slots[rng.choice(n, size=n_pad, replace=False)] = -1
    return k, v, slots


@pytest.mark.parametrize("dtype,n,nb,bs,hkv,d,n_pad,extra", [
    ("f32", 2, 16, 4, 1, 8, 0, 0),          # the tiny fp32 workload's shape
    ("f32", 37, 32, 4, 3, 20, 5, 0),        # 240-byte rows: 16-byte vectors
    ("f16", 300, 64, 16, 2, 64, 15, 0),
    ("bf16", 513, 128, 16, 4, 128, 26, 0),
    ("bf16", 700, 64, 32, 8, 128, 35, 0),
    ("f16", 90, 32, 16, 8, 256, 9, 0),      # 4 KB rows: two rounds of a lane's vectors
    ("f32", 45, 16, 16, 4, 160, 4, 0),      # 2560-byte rows: a partial second round
    ("f16", 50, 16, 8, 3, 12, 3, 0),        # 72-byte rows: 8-byte vectors
    ("bf16", 40, 16, 8, 1, 6, 2, 0),        # 12-byte rows: 4-byte vectors
    ("bf16", 33, 16, 4, 1, 3, 1, 0),        # 6-byte rows: 2-byte elements
    ("bf16", 200, 64, 16, 4, 128, 10, 128 * 4 * 2),   # k/v rows inside a packed qkv buffer
])
def test_scatter_bit_exact(dtype, n, nb, bs, hkv, d, n_pad, extra):
    k, v, slots = _case(dtype, n, nb, bs, hkv, d, n_pad, seed=n + nb + d)
    dev = torch.device("cuda")
    kc = sentinel_tensor((nb, bs, hkv, d), dtype, dev)
    vc = sentinel_tensor((nb, bs, hkv, d), dtype, dev)
    if extra:
        base_k = torch.empty(n, hkv * d + extra, dtype=TORCH[dtype], device=dev)
        base_v = torch.empty_like(base_k)
        base_k[:, : hkv * d] = k.reshape(n, hkv * d).to(dev)
        base_v[:, : hkv * d] = v.reshape(n, hkv * d).to(dev)
        kd = base_k.as_strided((n, hkv, d), (hkv * d + extra, d, 1))
        vd = base_v.as_strided((n, hkv, d), (hkv * d + extra, d, 1))
    else:
        kd, vd = k.to(dev), v.to(dev)
    pk.reshape_and_cache(kd, vd, kc, vc, torch.from_numpy(slots).to(dev))
    assert pk.device_error() == 0
    ko = sentinel_storage((nb, bs, hkv, d), dtype)
    vo = sentinel_storage((nb, bs, hkv, d), dtype)
    oracle_scatter(to_storage(k, dtype), to_storage(v, dtype), ko, vo, slots.tolist())
    assert np.array_equal(to_storage(kc, dtype).view(np.uint8), ko.view(np.uint8))
    assert np.array_equal(to_storage(vc, dtype).view(np.uint8), vo.view(np.uint8))


def test_empty_and_all_padded():
    dev = torch.device("cuda")
    kc = sentinel_tensor((8, 16, 2, 64), "bf16", dev)
    vc = sentinel_tensor((8, 16, 2, 64), "bf16", dev)
    before = kc.clone()
    z = torch.empty(0, 2, 64, dtype=torch.bfloat16, device=dev)
    pk.reshape_and_cache(z, z, kc, vc, torch.empty(0, dtype=torch.int32, device=dev))
    k = torch.randn(5, 2, 64, device=dev).to(torch.bfloat16)
    pk.reshape_and_cache(k, k, kc, vc, torch.full((5,), -1, dtype=torch.int32, device=dev))
    assert torch.equal(kc.view(torch.int16), before.view(torch.int16))
    assert pk.device_error() == 0


def test_last_slot_and_out_of_pool_slot():
    """The last slot of the pool is writable; a slot past it is skipped by
    the kernel's bounds check and reported, and nothing else changes."""
    dev = torch.device("cuda")
    nb, bs = 8, 16
    kc = sentinel_tensor((nb, bs, 2, 64), "f16", dev)
    vc = sentinel_tensor((nb, bs, 2, 64), "f16", dev)
    k = torch.randn(3, 2, 64, device=dev).to(torch.float16)
    slots = torch.tensor([nb * bs - 1, nb * bs, -7], dtype=torch.int32, device=dev)
    pk.device_error()      # clear
    pk.reshape_and_cache(k, k, kc, vc, slots)
    assert pk.device_error() == 8      # KV_ERR_DEVICE_BOUNDS
    assert torch.equal(kc[nb - 1, bs - 1], k[0])
    assert int((kc.view(torch.int16) != 0x7E00).sum()) == 2 * 64
    assert pk.device_error() == 0      # reset by the previous read


def test_rejects_bad_arguments():
    dev = torch.device("cuda")
    kc = torch.zeros(4, 4, 1, 8, device=dev)
    k = torch.zeros(2, 1, 8, device=dev)
    with pytest.raises(pk.KVError):
        pk.reshape_and_cache(k, k, kc, kc, torch.zeros(2, dtype=torch.int64, device=dev))
    with pytest.raises(pk.KVError):
        pk.reshape_and_cache(k.half(), k.half(), kc, kc, torch.zeros(2, dtype=torch.int32, device=dev))
