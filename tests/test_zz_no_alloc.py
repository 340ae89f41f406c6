"""The no-allocation decode entry point, for callers that may not allocate
device memory (their GPU memory belongs to another allocator, or allocation
is not allowed where they run): it must give the workspace call's answer
using only the library's fixed scratch array.

Collected last on purpose (file name), so a run that stops at the first
failure has run every other test before this one.  It is self-contained and
passes alone in a fresh process or after the rest of the suite."""

import math

import numpy as np
import pytest
import torch

import paged_kv_cache_128_gb300 as pk
from oracle.attention import decode_attention_contiguous
from paged_kv_cache_128_gb300 import kernels
from tests.helpers import to_f64

pytestmark = pytest.mark.gpu

TOL = {torch.float16: 2e-3, torch.bfloat16: 8e-3}
NAME = {torch.float16: "f16", torch.bfloat16: "bf16"}


def _case(dtype, hq, hkv, d, bs, lens, seed):
    dev = torch.device("cuda")
    g = torch.Generator().manual_seed(seed)
    rng = np.random.default_rng(seed)
    nb = sum(-(-L // bs) for L in lens) + 4
    mgr = pk.KVBlockManager(nb, bs, rng.permutation(nb).tolist())
    slots = np.concatenate([mgr.allocate_for_prefill(i, L) for i, L in enumerate(lens)])
    total = int(sum(lens))
    kc = torch.zeros(nb, bs, hkv, d, dtype=dtype, device=dev)
    vc = torch.zeros_like(kc)
    k = torch.randn(total, hkv, d, generator=g).to(dtype).to(dev)
    v = torch.randn(total, hkv, d, generator=g).to(dtype).to(dev)
    pk.reshape_and_cache(k, v, kc, vc, torch.from_numpy(slots).to(dev))
    max_blocks = max(-(-L // bs) for L in lens) + 1
    tables, seq_lens = mgr.export(list(range(len(lens))), max_blocks)
    q1 = torch.randn(len(lens), hq, d, generator=g).to(dtype).to(dev)
    q2 = torch.randn(len(lens), hq, d, generator=g).to(dtype).to(dev)
    return (kc, vc, torch.from_numpy(tables).to(dev), torch.from_numpy(seq_lens).to(dev), q1, q2, k, v)


def _oracle(q, k, v, lens, scale, dtype):
    """float64 attention of each sequence over its own rows (sequence i
    holds rows sum(lens[:i]) .. sum(lens[:i+1]) - 1, written in that order)."""
    name = NAME[dtype]
    q64, k64, v64 = to_f64(q, name), to_f64(k, name), to_f64(v, name)
    off = np.concatenate([[0], np.cumsum(lens)])
    return np.stack([decode_attention_contiguous(q64[i], k64[off[i]:off[i + 1]], v64[off[i]:off[i + 1]], scale)
                     for i in range(len(lens))])


@pytest.mark.parametrize("dtype,hq,hkv,d,bs,lens", [
    (torch.bfloat16, 28, 4, 128, 16, [1, 700, 2049, 33, 4096, 512]),   # stream-K, cut sequences
    (torch.float16, 14, 2, 64, 16, [5, 2048, 17, 999]),
])
def test_static_scratch_matches_workspace_call_twice(dtype, hq, hkv, d, bs, lens):
    kc, vc, tables, seq_lens, q1, q2, k, v = _case(dtype, hq, hkv, d, bs, lens, seed=len(lens) + hq)
    scale = 1.0 / math.sqrt(d)
    max_len = max(lens)
    assert pk.decode_plan(len(lens), hq, hkv, d, bs, max_len, dtype).kernel == 2   # the stream-K kernel, which has scratch
    for q in (q1, q2):                      # two calls in a row share the scratch array
        ref = torch.empty_like(q)
        pk.paged_decode_attention(ref, q, kc, vc, tables, seq_lens, scale, max_len)
        got = torch.empty_like(q)
        kernels.paged_decode_attention_static_scratch(got, q, kc, vc, tables, seq_lens, scale, max_len)
        torch.cuda.synchronize()
        assert pk.device_error() == 0
        # same kernel, same plan, same partition: the same bits, whatever the
        # scratch array held from the call before
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
        want = _oracle(q, k, v, lens, scale, dtype)
        err = float(np.max(np.abs(to_f64(got, NAME[dtype]) - want)))
        assert err <= TOL[dtype], err


def test_static_scratch_rejects_sizes_beyond_its_maximum():
    """8 query heads per kv head at head dim 256: the stream-K kernel's
    partial rows need more than the array holds."""
    dev = torch.device("cuda")
    d, hq, hkv, bs = 256, 16, 2, 16
    plan = pk.decode_plan(2, hq, hkv, d, bs, 4096, torch.bfloat16)
    assert plan.kernel == 2
    assert plan.workspace_bytes > kernels.static_scratch_bytes()
    kc = torch.zeros(8, bs, hkv, d, dtype=torch.bfloat16, device=dev)
    q = torch.zeros(2, hq, d, dtype=torch.bfloat16, device=dev)
    out = torch.full_like(q, 7.0)
    tables = torch.zeros(2, 4, dtype=torch.int32, device=dev)
    lens = torch.ones(2, dtype=torch.int32, device=dev)
    with pytest.raises(pk.KVError) as e:
        kernels.paged_decode_attention_static_scratch(out, q, kc, kc, tables, lens, 0.1, 4096)
    assert e.value.code == "WORKSPACE"
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())          # nothing was launched
