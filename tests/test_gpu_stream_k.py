"""The stream-K decode kernel's workspace flags and bounded waits.

The kernel gives each CTA an equal share of the batch's tiles; a sequence
cut by those ranges is finished by the CTA holding its first tiles, which
waits (bounded) for the later pieces' ready flags.  These tests check,
against the float64 oracle ("MiniPaged-Qwen: Paged KV Cache 与 KV Block
Manager" §13-§14: decode attention through the block table with the GQA
head map):

* a workspace holding arbitrary bytes needs no clearing (the flags carry a
  tag unique to each call), and repeated calls give the same bits;
* sequences cut into dozens of pieces (32k tokens, 8 kv heads);
* failure detection without a fault: with a short wait limit and one tile
  that is never loaded, the launch ends, the device error word reads
  KV_ERR_DEVICE_TIMEOUT, and the next calls on the same context are
  correct.
"""

import pytest
import torch

import paged_kv_cache_128_gb300 as pk
from paged_kv_cache_128_gb300 import kernels
from tests.test_gpu_decode_attention import run_case

pytestmark = pytest.mark.gpu

KV_ERR_DEVICE_TIMEOUT = 10
LENS_MIX = [700, 1, 300, 48, 1025, 4096, 17, 2500] * 3


@pytest.fixture(autouse=True)
def default_controls():
    kernels.debug_reset()
    yield
    kernels.debug_reset()


@pytest.mark.parametrize("fill", ["ones", "random"])
def test_workspace_needs_no_clearing(fill):
    lens = LENS_MIX
    plan = pk.decode_plan(len(lens), 32, 8, 128, 32, max(lens), torch.bfloat16)
    assert plan.kernel == 2
    dev = torch.device("cuda")
    if fill == "ones":
        ws = torch.full((plan.workspace_bytes,), 0xFF, dtype=torch.uint8, device=dev)
    else:
        g = torch.Generator(device=dev).manual_seed(5)
        ws = torch.randint(0, 256, (plan.workspace_bytes,), generator=g, device=dev, dtype=torch.int32).to(torch.uint8)
    run_case("bf16", 32, 8, 128, 32, lens, seed=73, workspace=ws, repeat=3)


def test_long_sequences_cut_into_many_pieces():
    """Two 32k-token sequences over 8 kv heads among short ones (the long
    skewed batch's shape): each long (sequence, kv head) spans many CTAs'
    ranges."""
    run_case("bf16", 32, 8, 128, 16, [32768, 100, 32768, 50, 1000], seed=74, repeat=3)


def test_bounded_wait_runs_out_and_the_gpu_stays_usable():
    """CTA 0 never loads the third tile of its range: the consumer's wait for
    it runs out after 2 ms (and the waits behind it, each bounded), the
    launch ends and records KV_ERR_DEVICE_TIMEOUT; then the same call with
    the controls back at their defaults matches the oracle, and so do later
    calls: the context stays usable."""
    lens = [4096] * 8 + [1000] * 8       # CTA 0's first range holds far more than three tiles
    kernels.debug_set(kernels.DEBUG_WAIT_LIMIT_NS, 2_000_000)
    kernels.debug_set(kernels.DEBUG_SKIP_TILE, 2)
    pk.device_error()
    run_case("bf16", 28, 4, 128, 16, lens, seed=75, expect_error=KV_ERR_DEVICE_TIMEOUT)
    kernels.debug_reset()
    run_case("bf16", 28, 4, 128, 16, lens, seed=75)           # the context is healthy: correct, no error
    run_case("f16", 14, 2, 64, 16, LENS_MIX, seed=76, repeat=3)
