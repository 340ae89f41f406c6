"""Benchmark of the paged KV cache hot path on one GB300 (or N replicas).

A step is one serving decode step of one layer for the whole batch:
host metadata (decode appends, prefill allocation, table export, slot
mapping, H2D), the cache write of the step's new K/V, and paged decode
attention with split-K and the log-sum-exp merge.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl native|reference]

Prints one JSON line on rank 0.  ``value`` is algorithmic HBM bytes of the
step (K/V of every attended token read once, q/out, table entries and
lengths, plus the cache write) per second of device time, summed over
ranks; each rank runs its own replica of the workload (weak scaling, no
data-path collective).  Steps are issued back to back through the native
step runner (one library call per step: host metadata, async H2D copy on a
side stream, one fused cache-write + attention launch), so the host builds
step i + 1's metadata and its copy runs while the GPU runs step i; steps
rotate over enough replica pools that no step finds its K/V in L2.  The
roofline object times the step's device launch alone, L2 flushed before
each.

The default workload is the mixed continuous-batching step (256 decode
sequences, a 4096-token prefill chunk, 5 % padded slots; bf16, Hq 32,
Hkv 8, D 128, block 32), the largest of the five.  ``roofline_by_workload``
times the fused-step launch of the three single-layer decode batches held
to 70 % of HBM peak in the same run.  ``cpu_baseline`` is the float64
oracle on one host thread; ``cpu_baseline_all_cores`` runs it on every host
core at once.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attn HBM GB/s (% of ~8 TB/s peak) and decode tokens/s at 1 GB300"
DEFAULT_WORKLOAD = "mixed_batch_bf16"
# workloads whose fused-step launch is also timed (L2 flushed) in every
# default run: the three single-layer decode batches held to 70 % of HBM peak
TARGET_WORKLOADS = ("decode_gqa14x2_d64_fp16", "decode_gqa28x4_d128_bf16", "decode_long_skewed_bf16")
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="native", choices=("native", "reference"))
    ap.add_argument("--kv-cache", default="native", choices=("native", "fp8"),
                    help="cache element type: the workload's dtype, or fp8 E4M3 codes with per-token scales "
                         "(head_dim 128 workloads)")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--no-target-rooflines", action="store_true",
                    help="skip the per-workload launch timings of the 70 %% target workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="--impl reference: seconds of oracle time for the whole run (steps + warm-up)")
    ap.add_argument("--prefill", action="store_true",
                    help="time chunked-prefill attention instead of the decode step: the mixed-batch workload's "
                         "4096-token prefill chunk, one JSON line per --prefill-context")
    ap.add_argument("--prefill-context", default="0,2048",
                    help="--prefill: comma-separated history lengths (tokens already cached per sequence)")
    ap.add_argument("--layers", type=int, default=0,
                    help="time a multi-layer decode step instead: the workload's decode batch over this many "
                         "layers' caches under one block table, through the native runner (metadata once per step, "
                         "one fused launch per layer); decode-only workloads")
    ap.add_argument("--cache-write", action="store_true",
                    help="time the cache write alone instead (paged_reshape_and_cache, or the quantised "
                         "paged_reshape_and_cache_fp8 with --kv-cache fp8) on the workload's first step: its new "
                         "K/V rows scattered to their slots, L2 flushed before each call")
    ap.add_argument("--profile-calls", type=int, default=0,
                    help="only set the workload up and run this many attention calls (L2 flushed before each); "
                         "the small case used under ncu")
    return ap.parse_args()


# ----------------------------------------------------------------- helpers

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _code_only(text):
    """C++/CUDA source without comments and blank lines: a comment edit
    leaves the compiled kernel, and so this hash, unchanged."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":  # string or character literal, escapes skipped
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(line.rstrip() for line in "".join(out).splitlines() if line.strip())


def kernel_source_hash():
    """Hash of the decode kernels' source (comments and blank lines left out)."""
    h = hashlib.sha256()
    for rel in ("paged_kv_cache_128_gb300/csrc/paged_decode.cu", "paged_kv_cache_128_gb300/csrc/common.cuh"):
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per fused step call from a committed ncu summary, if it
    was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "decode_step_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    entry = rec.get(workload)
    if not entry or entry.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    return entry.get("dram_bytes_per_call")


class ClockSampler:
    """nvidia-smi sampling (200 ms) of SM clock and throttle reasons."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------- oracle timing

ORACLE_SNIPPET = r"""
import json, sys, time
sys.path.insert(0, {root!r})
import numpy as np
from oracle.block_manager import BlockManager
from oracle.paged_cache import reshape_and_cache
from oracle.attention import paged_decode_attention
from paged_kv_cache_128_gb300.inputs import make_workload, make_values, pad_positions
import torch

wl = make_workload({name!r})
vals = make_values(wl, history=False)
def st(t):
    t = t.contiguous()
    return t.view(torch.int16).numpy().view(np.uint16) if wl.dtype == "bf16" else t.numpy()
budget = {budget}
# sample: S decode sequences from batch position F on (a bounded slice of the same step)
F = {first} % wl.num_seqs
S = min(wl.num_seqs - F, {max_seqs})
def setup():
    mgr = BlockManager(wl.num_blocks, wl.block_size, None if wl.free_order is None else wl.free_order.tolist())
    shape = (wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim)
    kc = np.zeros(shape, dtype=st(vals.k_step[:1]).dtype)
    vc = np.zeros_like(kc)
    ids = set(int(i) for i in wl.decode_ids[F:F + S])
    # history of the sampled sequences only, seeded per sample
    g = torch.Generator().manual_seed(wl.seed + 7919 * (F + 1))
    def draw(n):
        x = torch.randn(n, wl.num_kv_heads, wl.head_dim, generator=g) * wl.value_scale
        return st(x.to(wl.torch_dtype))
    for op, sid, n in wl.setup_ops:
        if op == "prefill":
            s = mgr.allocate_for_prefill(sid, n)
        elif op == "append":
            s = mgr.append_slots(sid, n)
        else:
            mgr.free_sequence(sid); continue
        if sid in ids:
            reshape_and_cache(draw(n), draw(n), kc, vc, s)
    return mgr, kc, vc
mgr, kc, vc = setup()
sample_ids = wl.decode_ids[F:F + S].tolist()
q = st(vals.q[F:F + S])
k_new = st(vals.k_step[F:F + S]); v_new = st(vals.v_step[F:F + S])
if {sync}:   # several copies run at once: start timing together
    print("READY", flush=True)
    sys.stdin.readline()
elapsed, steps, bytes_total = 0.0, 0, 0
es = 4 if wl.dtype == "f32" else 2
row = wl.num_kv_heads * wl.head_dim * es
while elapsed < budget and steps < 10000:
    if not mgr.can_append_slots(sample_ids):   # pool exhausted by growth: rebuild, untimed
        mgr, kc, vc = setup()
    t0 = time.perf_counter()
    slots = mgr.decode_step(sample_ids)
    mb = max(len(mgr.block_table(s)) for s in sample_ids)
    tables, lens = mgr.export(sample_ids, mb)
    reshape_and_cache(k_new, v_new, kc, vc, slots)
    paged_decode_attention(q, kc, vc, tables, lens, wl.scale, wl.dtype)
    elapsed += time.perf_counter() - t0
    steps += 1
    L = np.asarray(lens, dtype=np.int64)
    bytes_total += int(L.sum()) * 2 * row + 2 * S * wl.num_heads * wl.head_dim * es \
        + 4 * (S + int((-(-L // wl.block_size)).sum())) + 2 * 2 * S * row + 4 * S
print(json.dumps({{"seconds": elapsed, "steps": steps, "seqs": S, "bytes": bytes_total,
                  "tokens": steps * S}}))
"""


def _oracle_env():
    env = dict(os.environ)
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[var] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    return env


def run_oracle_sample(name, budget, max_seqs, first=0):
    code = ORACLE_SNIPPET.format(root=ROOT, name=name, budget=budget, max_seqs=max_seqs, first=first, sync=False)
    proc = subprocess.run([sys.executable, "-c", code], env=_oracle_env(), stdout=subprocess.PIPE,
                          stderr=subprocess.PIPE, text=True, timeout=budget * 20 + 300)
    if proc.returncode != 0:
        raise RuntimeError("oracle sample failed:\n" + proc.stderr[-2000:])
    return json.loads(proc.stdout.strip().splitlines()[-1])


def run_oracle_parallel(name, budget, max_seqs, procs):
    """``procs`` single-threaded oracle processes at once, process i on the
    8 sequences from batch position 8 i (sequences are independent); they
    set up, then start their timed loops together.  Returns the summed
    bytes and tokens, and the longest timed loop."""
    code = [ORACLE_SNIPPET.format(root=ROOT, name=name, budget=budget, max_seqs=max_seqs, first=i * max_seqs,
                                  sync=True) for i in range(procs)]
    ps = [subprocess.Popen([sys.executable, "-c", c], env=_oracle_env(), stdin=subprocess.PIPE,
                           stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True) for c in code]
    try:
        for p in ps:
            line = p.stdout.readline()
            if not line.startswith("READY"):
                raise RuntimeError("oracle process failed during set-up:\n" + p.stderr.read()[-2000:])
        for p in ps:
            p.stdin.write("go\n")
            p.stdin.flush()
        outs = [p.communicate(timeout=budget * 20 + 300) for p in ps]
    finally:
        for p in ps:
            if p.poll() is None:
                p.kill()
    res = []
    for p, (out, err) in zip(ps, outs):
        if p.returncode != 0:
            raise RuntimeError("oracle process failed:\n" + err[-2000:])
        res.append(json.loads(out.strip().splitlines()[-1]))
    return {"seconds": max(r["seconds"] for r in res), "bytes": sum(r["bytes"] for r in res),
            "tokens": sum(r["tokens"] for r in res), "seqs": sum(r["seqs"] for r in res),
            "steps": min(r["steps"] for r in res)}


def cpu_baseline(name, budget):
    r = run_oracle_sample(name, budget, max_seqs=8)
    gbs = r["bytes"] / r["seconds"] / 1e9
    return {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": (f"float64 numpy oracle, one host thread: {r['steps']} decode steps of the first "
                       f"{r['seqs']} sequences of {name} (manager append + export, cache write, attention), "
                       f"{r['seconds']:.1f} s"),
            "decode_tokens_per_s": r["tokens"] / r["seconds"]}


def cpu_baseline_all_cores(name, budget):
    """The same oracle loop on every host core: one single-threaded process
    per core, each over its own 8 sequences of the batch."""
    from paged_kv_cache_128_gb300.inputs import make_workload
    cores = os.cpu_count() or 1
    procs = max(1, min(cores, make_workload(name).num_seqs // 8))
    r = run_oracle_parallel(name, budget, 8, procs)
    gbs = r["bytes"] / r["seconds"] / 1e9
    return {"value": gbs, "unit": "GB/s", "cores": procs, "kind": "oracle",
            "sample": (f"float64 numpy oracle, {procs} single-threaded processes at once on {cores} host cores, "
                       f"each over its own 8 sequences of {name} ({r['seqs']} in all; manager append + export, "
                       f"cache write, attention), at least {r['steps']} decode steps each, {r['seconds']:.1f} s"),
            "decode_tokens_per_s": r["tokens"] / r["seconds"]}


# ------------------------------------------------------------- native arm

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int, device="cpu") -> float:
    """The largest x over the ranks of the process group (x itself for one
    rank): the timed region of a multi-replica run is the slowest rank's."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def flushed_launch_time(eng, q, k_step, v_step, calls, l2, dev):
    """Mean device time of the step's device launch alone, and its
    algorithmic bytes.  Launches are queued behind a GPU-side delay, so the
    events bracket device time only.  Before each call L2 is flushed (write
    2x L2, then read 2x L2 of other data) and the step's metadata is copied
    host to device again, as every step does before its kernels: K/V come
    from HBM, the block tables and lengths from where the step's copy left
    them.  The event clock ticks in steps of about 2 us, so the mean over
    the calls is taken (a median would snap to a tick)."""
    import torch
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    flush_read = torch.ones(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)
    meta_h = eng.d_meta.cpu().pin_memory()
    ms = []
    for _ in range(calls):
        flush.zero_()
        flush_read.sum()
        eng.d_meta.copy_(meta_h, non_blocking=True)
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(200000)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        eng.device_step(q, k_step, v_step)
        b.record()
        b.synchronize()
        ms.append(a.elapsed_time(b))
    call_s = statistics.fmean(ms[2:] if len(ms) > 4 else ms) / 1e3
    # the step's device kernels after the metadata copy (one fused launch of
    # the cache write + attention with the stream-K kernel), over the lengths
    # in the metadata it was given
    return call_s, eng.algorithmic_bytes(eng._views(meta_h)[2].numpy())["step"]


def target_rooflines(args, dev, l2, peak, peak_kind):
    """The fused-step launch of each 70 %-target workload, timed as the
    headline roofline is (one pool each, L2 flushed before every call)."""
    import torch
    from paged_kv_cache_128_gb300.engine import PagedDecodeEngine
    from paged_kv_cache_128_gb300.inputs import make_values, make_workload
    out = {}
    calls = max(args.steps, 30)
    for name in TARGET_WORKLOADS:
        if name == args.workload:
            continue
        wl = make_workload(name)
        if args.kv_cache == "fp8" and wl.head_dim != 128:
            continue  # fp8 caches are built for head_dim 128 only
        eng = PagedDecodeEngine(wl, dev, max_steps=2, fill_sentinel=False, kv_cache=args.kv_cache)
        vals = make_values(wl, device="cuda")
        eng.setup(vals)
        eng.step(vals.q, vals.k_step, vals.v_step)
        torch.cuda.synchronize()
        call_s, nbytes = flushed_launch_time(eng, vals.q, vals.k_step, vals.v_step, calls, l2, dev)
        achieved = nbytes / call_s / 1e9
        out[name] = {"bound": "hbm", "achieved": achieved, "peak": peak,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback", "unit": "GB/s", "frac": achieved / peak,
                     "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                     "traffic": recorded_traffic(name if args.kv_cache == "native" else f"{name}:fp8"),
                     "algorithmic_bytes_per_call": nbytes, "mean_call_us": call_s * 1e6, "calls": calls,
                     "plan": {0: "simt_split", 1: "tma_mma_split", 2: "tma_mma_stream_k"}[eng.plan.kernel]}
        del eng, vals
        torch.cuda.empty_cache()
    return out


def run_native(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import paged_kv_cache_128_gb300 as pk
    from paged_kv_cache_128_gb300.engine import PagedDecodeEngine
    from paged_kv_cache_128_gb300.inputs import make_values, make_workload

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = make_workload(args.workload)
    pk.lib()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size

    def barrier():
        if world > 1:
            dist.barrier()

    # Replicas: consecutive steps use different pools until more than 3x L2
    # has streamed, so no step finds its K/V in L2 and no flush is needed.
    probe = PagedDecodeEngine(wl, dev, max_steps=1, fill_sentinel=False, kv_cache=args.kv_cache)
    attn_bytes0 = probe.algorithmic_bytes(wl.cached_lens + 1)["attention"]
    pool_bytes = 2 * probe.k_cache.numel() * probe.k_cache.element_size()
    del probe
    torch.cuda.empty_cache()
    replicas = int(min(16, max(1, -(-3 * l2 // attn_bytes0)), max(1, (48 << 30) // pool_bytes)))
    per_replica = -(-(2 * (args.steps + args.warmup)) // replicas) + 8
    engines = []
    vals = None
    for r in range(replicas):
        eng = PagedDecodeEngine(wl, dev, max_steps=per_replica, fill_sentinel=False, kv_cache=args.kv_cache)
        vals = make_values(wl, device="cuda") if vals is None else vals
        eng.setup(vals)
        engines.append(eng)
    q, k_step, v_step = vals.q, vals.k_step, vals.v_step
    for eng in engines:            # one direct step each (lazy set-up), then the native step runner,
        eng.step(q, k_step, v_step)    # primed with one step so no runner's first step is timed
        eng.make_runner()
        eng.runner_step(q, k_step, v_step, eng.out)
        eng.runner_join()
    torch.cuda.synchronize()

    def run_step(i):
        eng = engines[i % replicas]
        eng.runner_step(q, k_step, v_step, eng.out)
        return eng

    def join_all():
        for eng in engines:
            eng.runner_join()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    for i in range(args.warmup):
        run_step(i)
    torch.cuda.synchronize()
    # ---------------- device-resident throughput (pipelined steps) ----------------
    marks = []
    barrier()
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.perf_counter()
    t_start.record()
    for i in range(args.steps):
        eng = run_step(args.warmup + i)
        marks.append((eng, eng.steps_done))
    join_all()
    t_end.record()
    torch.cuda.synchronize()
    barrier()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    t_steps = t_start.elapsed_time(t_end) / 1e3
    step_bytes, tokens = 0, 0
    for eng, done in marks:                  # lengths after that step's append
        lens = eng.wl.cached_lens + done
        step_bytes += eng.algorithmic_bytes(lens)["step"]
        tokens += eng.wl.num_seqs
    t_steps_max = max_over_ranks(t_steps, world, dev)
    value_gbs = step_bytes * world / t_steps_max / 1e9
    tokens_per_s = tokens * world / t_steps_max
    status = pk.device_error()

    # ---------------- the step's device launch alone (the roofline kernel) ----------------
    # Launches are queued behind a GPU-side delay, so the events bracket
    # device time only.  Before each call L2 is flushed (write 2x L2, then
    # read 2x L2 of other data) and the step's metadata is copied host to
    # device again, as every step does before its kernels: K/V come from
    # HBM, the block tables and lengths from where the step's copy left them.
    # The event clock ticks in steps of about 2 us, so the mean over many
    # calls is taken (the median would snap to a tick).
    eng0 = engines[0]
    attn_call_s, attn_bytes = flushed_launch_time(eng0, q, k_step, v_step, max(args.steps, 10), l2, dev)

    # ---------------- end to end through host buffers ----------------
    # The step's q/k/v sit in the runners' page-locked staging slots (host_io
    # 2: written once per slot here, as a caller writes the inputs it has),
    # and every step copies its slot -- metadata, q, k and v -- host to
    # device in one copy and the output back to a page-locked host buffer,
    # on the runners' side streams, inside the timed region.
    q_h = q.cpu()
    k_h = k_step.cpu()
    v_h = v_step.cpu()
    outs_h = [torch.empty(q.shape, dtype=q.dtype, pin_memory=True) for _ in engines]
    for r, eng in enumerate(engines):
        eng.make_runner(host_io=2)
        for slot in range(4):
            for dst, src in zip(eng.runner_stage(slot), (q_h, k_h, v_h)):
                dst.copy_(src)
        eng.runner_step(None, None, None, outs_h[r])   # primed: no runner's first step is timed
        eng.runner_join()

    def run_e2e(i):
        eng = engines[i % replicas]
        eng.runner_step(None, None, None, outs_h[i % replicas])
        return eng

    for i in range(args.warmup):
        run_e2e(i)
    join_all()
    torch.cuda.synchronize()
    barrier()
    e_marks = []
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.steps):
        eng = run_e2e(i)
        e_marks.append((eng, eng.steps_done))
    join_all()
    e1.record()
    torch.cuda.synchronize()
    t_e2e = max_over_ranks(e0.elapsed_time(e1) / 1e3, world, dev)
    e2e_bytes = sum(eng.algorithmic_bytes(eng.wl.cached_lens + done)["step"] for eng, done in e_marks)
    e2e_gbs = e2e_bytes * world / t_e2e / 1e9
    # per step: q, k, v and the metadata buffer (slot mapping, tables, lengths, decode rows) in; out back
    h2d = (q.numel() + k_step.numel() + v_step.numel()) * q.element_size() + 4 * (engines[0].d_meta.numel() +
                                                                                    wl.num_seqs)
    d2h = outs_h[0].numel() * outs_h[0].element_size()
    status = status or pk.device_error()

    peak, peak_kind = measured_peak()
    achieved = attn_bytes / attn_call_s / 1e9
    traffic = recorded_traffic(args.workload if args.kv_cache == "native" else f"{args.workload}:fp8")
    plan = engines[0].plan
    result = {
        "metric": METRIC,
        "value": value_gbs,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": t_steps_max / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": wl.dtype,
        "data": "synthetic (seeded; no dataset on the source pages)",
        "config": {
            "workload": wl.name,
            "kv_cache": "fp8 E4M3 codes + float32 scale per (token, kv head)" if args.kv_cache == "fp8" else wl.dtype,
            "num_seqs": wl.num_seqs, "num_heads": wl.num_heads, "num_kv_heads": wl.num_kv_heads,
            "head_dim": wl.head_dim, "block_size": wl.block_size, "num_blocks": wl.num_blocks,
            "mean_seq_len": float(np.mean(wl.cached_lens)) + 1,
            "prefill_tokens_per_step": int(wl.prefill_lens.sum()), "padded_slots_per_step": wl.num_pad,
            "l2": (f"inputs larger than L2: steps rotate over {replicas} replica pools so more than 3x L2 "
                   "streams between two uses of one pool; the roofline loop flushes L2 before each call"),
            "pipelining": "host metadata of a step overlaps device work of the previous steps",
            "step_driver": ("native step runner (kvstep_run): one library call per step does the host "
                            "metadata, the async H2D copy on a side stream and the fused launch"),
            "parallelism": f"replicas x{world}",
            "plan": {"kernel": {0: "simt_split", 1: "tma_mma_split", 2: "tma_mma_stream_k"}[plan.kernel],
                     "blocks_per_split": plan.blocks_per_split, "num_splits": plan.num_splits},
        },
        "decode_tokens_per_s": tokens_per_s,
        "hbm_frac_of_nominal_8tbs": value_gbs / world / NOMINAL_HBM_GBS,
        "roofline": {
            "bound": "hbm",
            "kernel": ("paged_decode_step call: one cooperative stream-K launch doing the cache write and "
                       "decode attention" if eng0.fused and plan.kernel == 2 else
                       "paged_reshape_and_cache_fp8 + paged_decode_attention_fp8 calls" if eng0.fp8 else
                       "paged_reshape_and_cache + paged_decode_attention calls"),
            "achieved": achieved,
            "peak": peak,
            "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback",
            "unit": "GB/s",
            "frac": achieved / peak,
            "traffic": traffic,
            "algorithmic_bytes_per_call": attn_bytes,
            "mean_call_us": attn_call_s * 1e6,
            "call_setup": ("L2 flushed, then the step's metadata copied host to device (as each step does); "
                           "K/V read from HBM"),
        },
        "e2e": {"value": e2e_gbs, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": t_e2e / args.steps * 1e3},
        "gpu_launches": args.steps * engines[0].launches_per_step,
        "clocks": clk,
        "device_error": status,
        "wall_s_timed_region": wall,
    }
    # ---------------- the fused-step launch of the 70 % target workloads ----------------
    if not args.no_target_rooflines:
        for e in engines:
            e.close_runner()
        engines.clear()
        marks.clear()
        e_marks.clear()
        eng = eng0 = None
        torch.cuda.empty_cache()
        result["roofline_by_workload"] = target_rooflines(args, dev, l2, peak, peak_kind)
        status = status or pk.device_error()
        result["device_error"] = status
    if rank == 0 and not args.no_cpu_baseline:
        try:
            result["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_budget)
        except Exception as exc:  # reported, not fatal
            result["cpu_baseline"] = {"value": None, "error": str(exc)[-300:]}
        try:
            result["cpu_baseline_all_cores"] = cpu_baseline_all_cores(args.workload, args.cpu_budget)
        except Exception as exc:  # reported, not fatal
            result["cpu_baseline_all_cores"] = {"value": None, "error": str(exc)[-300:]}
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result))


# ---------------------------------------------------------- reference arm

def run_reference(args):
    """The oracle as it stands, on one host thread, over the workload's first
    8 sequences: one bounded run of about --ref-seconds x K / (K + W)
    seconds of timed decode steps (its set-up is the untimed warm-up).
    Under torchrun only rank 0 runs and prints; the others exit at once."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from paged_kv_cache_128_gb300.inputs import make_workload
    wl = make_workload(args.workload)
    total = max(1, args.steps + args.warmup)
    budget = max(0.05, args.ref_seconds * max(1, args.steps) / total)
    r = run_oracle_sample(args.workload, budget, max_seqs=min(8, wl.num_seqs))
    secs = r["seconds"]
    gbs = r["bytes"] / secs / 1e9
    out = {
        "impl": "reference",
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": secs / max(1, r["steps"]) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic (seeded)", "config": {"workload": wl.name},
        "decode_tokens_per_s": r["tokens"] / secs,
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": (f"float64 numpy oracle on one host thread: {r['steps']} decode steps of the "
                                    f"first {r['seqs']} sequences (manager append + export, cache write, "
                                    f"attention), {secs:.1f} s timed")},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out))


def run_profile_calls(args):
    """One engine, one step, then ``--profile-calls`` device steps (the fused
    cache write + attention launch) with L2 flushed before each: a short,
    fixed launch sequence for ncu captures."""
    import torch

    import paged_kv_cache_128_gb300 as pk
    from paged_kv_cache_128_gb300.engine import PagedDecodeEngine
    from paged_kv_cache_128_gb300.inputs import make_values, make_workload

    dev = torch.device("cuda")
    wl = make_workload(args.workload)
    eng = PagedDecodeEngine(wl, dev, max_steps=4, fill_sentinel=False, kv_cache=args.kv_cache)
    vals = make_values(wl, device="cuda")
    eng.setup(vals)
    eng.step(vals.q, vals.k_step, vals.v_step)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    for _ in range(args.profile_calls):
        flush.zero_()
        eng.device_step(vals.q, vals.k_step, vals.v_step)
    torch.cuda.synchronize()
    status = pk.device_error()
    ab = eng.algorithmic_bytes(wl.cached_lens + 1)
    print(json.dumps({"workload": wl.name, "calls": args.profile_calls, "plan": eng.plan.__dict__,
                      "fused": eng.fused, "attention_bytes": ab["attention"], "step_bytes": ab["step"],
                      "device_error": status}))
    if status:
        sys.exit(1)


# ----------------------------------------------------------- cache write

def run_cache_write(args):
    """The standalone cache write of the workload's first step (the call the
    two-call step and the history set-up make), L2 flushed before each call,
    CUDA events on the launching stream around the launch only (queued
    behind a GPU-side delay).  Algorithmic bytes: each valid new row read
    once and written once (fp8: its codes and per-head scales), plus the
    slot of every row.  With --profile-calls only that many calls run (the
    small fixed launch sequence for ncu)."""
    import torch

    import paged_kv_cache_128_gb300 as pk
    from paged_kv_cache_128_gb300.engine import PagedDecodeEngine
    from paged_kv_cache_128_gb300.inputs import make_values, make_workload

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak, peak_kind = measured_peak()
    wl = make_workload(args.workload)
    eng = PagedDecodeEngine(wl, dev, max_steps=2, fill_sentinel=False, kv_cache=args.kv_cache)
    vals = make_values(wl, device="cuda")
    eng.setup(vals)
    eng.step(vals.q, vals.k_step, vals.v_step)  # the step's slot mapping now sits on the device
    torch.cuda.synchronize()
    nbytes = eng.algorithmic_bytes(eng._views(eng.d_meta.cpu())[2].numpy())["cache_write"]
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    flush_read = torch.ones(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)
    if args.profile_calls:
        for _ in range(args.profile_calls):
            flush.zero_()
            eng.write_step_kv(vals.k_step, vals.v_step)
        torch.cuda.synchronize()
        status = pk.device_error()
        print(json.dumps({"workload": wl.name, "cache_write_calls": args.profile_calls, "kv_cache": args.kv_cache,
                          "bytes_per_call": nbytes, "device_error": status}))
        if status:
            sys.exit(1)
        return
    for _ in range(max(args.warmup, 3)):
        eng.write_step_kv(vals.k_step, vals.v_step)
    torch.cuda.synchronize()
    calls = max(min(args.steps, 200), 30)
    clocks = ClockSampler(0)
    clocks.start()
    ms = []
    for _ in range(calls):
        flush.zero_()
        flush_read.sum()
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(200000)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        eng.write_step_kv(vals.k_step, vals.v_step)
        b.record()
        b.synchronize()
        ms.append(a.elapsed_time(b))
    clk = clocks.stop()
    status = pk.device_error()
    call_s = statistics.fmean(ms[2:]) / 1e3
    gbs = nbytes / call_s / 1e9
    kernel = "cache_write_fp8_kernel" if args.kv_cache == "fp8" else "reshape_and_cache_kernel"
    print(json.dumps({"metric": "standalone cache write HBM GB/s", "value": gbs, "unit": "GB/s",
                      "higher_is_better": True, "mean_call_us": call_s * 1e6, "calls": calls,
                      "bytes_per_call": nbytes, "rows": int(eng.n_prefill + wl.num_seqs),
                      "roofline": {"bound": "hbm", "kernel": kernel, "achieved": gbs, "peak": peak,
                                   "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)", "unit": "GB/s",
                                   "frac": gbs / peak},
                      "config": {"workload": wl.name, "kv_cache": args.kv_cache, "l2": "flushed before each call"},
                      "clocks": clk, "device_error": status}))
    if status:
        sys.exit(1)


# ------------------------------------------------------ chunked prefill

def prefill_setup(ctx, dev, seed=5):
    """The mixed-batch workload's prefill chunk (8 new sequences, 4096 tokens
    split U[256, 768]-like by the workload generator; bf16, Hq 32, Hkv 8,
    D 128, bs 32), each sequence with ``ctx`` tokens of history before its
    chunk.  K/V of every position go through the cache write into pool
    blocks taken in a seeded shuffled order; values N(0, 1)."""
    import numpy as np
    import torch
    import paged_kv_cache_128_gb300 as pk
    from paged_kv_cache_128_gb300.inputs import make_workload
    wl = make_workload("mixed_batch_bf16")
    chunks = [int(n) for n in wl.prefill_lens]
    lens = [ctx + n for n in chunks]
    bs, hkv, d, hq = wl.block_size, wl.num_kv_heads, wl.head_dim, wl.num_heads
    nb = sum(-(-L // bs) for L in lens) + 8
    rng = np.random.default_rng(seed)
    mgr = pk.KVBlockManager(nb, bs, rng.permutation(nb).tolist())
    g = torch.Generator(device=dev).manual_seed(seed)
    kc = torch.empty(nb, bs, hkv, d, dtype=torch.bfloat16, device=dev)
    vc = torch.empty_like(kc)
    for sid, L in enumerate(lens):
        slots = torch.from_numpy(mgr.allocate_for_prefill(sid, L)).to(dev)
        k = torch.randn(L, hkv, d, generator=g, device=dev).to(torch.bfloat16)
        v = torch.randn(L, hkv, d, generator=g, device=dev).to(torch.bfloat16)
        pk.reshape_and_cache(k, v, kc, vc, slots)
    tables, seq_lens = mgr.export(list(range(len(lens))), max(-(-L // bs) for L in lens))
    qsl = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    T = int(qsl[-1])
    q = torch.randn(T, hq, d, generator=g, device=dev).to(torch.bfloat16)
    out = torch.empty_like(q)
    args = (out, q, kc, vc, torch.from_numpy(tables).to(dev), torch.from_numpy(seq_lens).to(dev),
            torch.from_numpy(qsl).to(dev), 1.0 / d ** 0.5, max(chunks))
    # causal work: chunk token t of a sequence attends ctx + t + 1 keys; 4 D
    # flops per (query head, key): 2 D for q.k and 2 D for p v
    keys = sum(ctx + t + 1 for n in chunks for t in range(n))
    return {"args": args, "flops": keys * hq * d * 4, "tokens": T, "seqs": len(chunks), "hq": hq, "hkv": hkv,
            "d": d, "bs": bs, "kv_bytes": 2 * sum(lens) * hkv * d * 2, "lens": lens, "chunks": chunks,
            "tables": tables, "qsl": qsl}


def prefill_cpu_baseline(w, budget_s=6.0):
    """The float64 oracle (one host thread) on a bounded sample of the same
    call: the first sequence's K/V gathered through its block table, then
    chunk rows from its last one backwards until about ``budget_s`` pass;
    causal TFLOP/s of the rows done."""
    import numpy as np
    import torch
    from oracle.attention import chunked_prefill_attention
    from oracle.paged_cache import gather, to_float64

    out, q, kc, vc = w["args"][:4]
    scale, bs = w["args"][7], w["bs"]
    L, n = int(w["lens"][0]), int(w["chunks"][0])

    def f64(t):
        return to_float64(t.contiguous().view(torch.int16).numpy().view(np.uint16), "bf16")

    nblk = -(-L // bs)
    table = [int(x) for x in w["tables"][0, :nblk]]
    idx = torch.tensor(table, dtype=torch.long, device=kc.device)
    K = gather(f64(kc.index_select(0, idx).cpu()), list(range(nblk)), L)
    V = gather(f64(vc.index_select(0, idx).cpu()), list(range(nblk)), L)
    q64 = f64(q[: n].cpu())
    t0 = time.perf_counter()
    flops, rows = 0, 0
    for t in range(n - 1, -1, -1):
        p_pos = L - n + t
        chunked_prefill_attention(q64[t:t + 1], K[:p_pos + 1], V[:p_pos + 1], scale)
        flops += (p_pos + 1) * w["hq"] * w["d"] * 4
        rows += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "sample": f"float64 numpy oracle, one host thread: the last {rows} chunk rows of the first sequence "
                      f"(history + chunk {L} tokens, all {w['hq']} query heads), {dt:.1f} s"}


def run_prefill(args):
    """Chunked-prefill attention (one launch per call) on the mixed-batch
    prefill chunk, L2 flushed before each timed call, events on the launching
    stream around the launch only (queued behind a GPU-side delay)."""
    import torch
    import paged_kv_cache_128_gb300 as pk
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, peak_kind = float(json.load(f)["bf16_tflops"]), "measured (cuBLAS bf16 burst)"
    except Exception:
        peak, peak_kind = 1900.0, "fallback"
    for ctx in [int(c) for c in args.prefill_context.split(",")]:
        w = prefill_setup(ctx, dev)
        pk.device_error()
        if args.profile_calls:
            for _ in range(args.profile_calls):
                flush.zero_()
                pk.paged_prefill_attention(*w["args"])
            torch.cuda.synchronize()
            print(json.dumps({"profile_calls": args.profile_calls, "history_tokens": ctx,
                              "device_error": pk.device_error()}))
            continue
        for _ in range(max(args.warmup, 3)):
            pk.paged_prefill_attention(*w["args"])
        torch.cuda.synchronize()
        clocks = ClockSampler(0)
        clocks.start()
        ms = []
        stream = torch.cuda.current_stream()
        for _ in range(args.steps):
            flush.zero_()
            if hasattr(torch.cuda, "_sleep"):
                torch.cuda._sleep(100000)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            pk.paged_prefill_attention(*w["args"], stream=stream)
            b.record(stream)
            b.synchronize()
            ms.append(a.elapsed_time(b))
        clk = clocks.stop()
        t = statistics.fmean(ms) / 1e3
        tflops = w["flops"] / t / 1e12
        # end to end: q copied in from page-locked host memory and the output
        # copied back, every call, inside the timed region
        out_d, q_d = w["args"][0], w["args"][1]
        q_h = q_d.cpu().pin_memory()
        out_h = torch.empty(out_d.shape, dtype=out_d.dtype, pin_memory=True)
        e2e_steps = max(10, args.steps // 4)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(e2e_steps):
            q_d.copy_(q_h, non_blocking=True)
            pk.paged_prefill_attention(*w["args"], stream=stream)
            out_h.copy_(out_d, non_blocking=True)
        b.record(stream)
        b.synchronize()
        t_e2e = a.elapsed_time(b) / 1e3 / e2e_steps
        status = pk.device_error()
        cpu = None if args.no_cpu_baseline else prefill_cpu_baseline(w)
        print(json.dumps({
            "metric": "chunked-prefill paged attention TFLOP/s (causal flops) at 1 GB300",
            "value": round(tflops, 2), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": round(t * 1e3, 5), "higher_is_better": True,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "mixed_batch_bf16 prefill chunk", "sequences": w["seqs"],
                       "chunk_tokens": w["tokens"], "history_tokens": ctx, "num_heads": w["hq"],
                       "num_kv_heads": w["hkv"], "head_dim": w["d"], "block_size": w["bs"],
                       "kv_bytes": w["kv_bytes"], "l2": "flushed before each call"},
            "roofline": {"bound": "tensor", "achieved": round(tflops, 2), "peak": peak, "unit": "TFLOP/s",
                         "frac": round(tflops / peak, 4), "peak_kind": peak_kind, "flops_per_call": w["flops"],
                         "traffic": None},
            "e2e": {"value": round(w["flops"] / t_e2e / 1e12, 2), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": q_d.numel() * q_d.element_size(),
                    "d2h_bytes_per_step": out_d.numel() * out_d.element_size(),
                    "ms_per_step": round(t_e2e * 1e3, 5), "l2": "not flushed between calls"},
            "cpu_baseline": cpu,
            "gpu_launches": args.steps, "clocks": clk, "device_error": status}))
        if status:
            sys.exit(1)


# ------------------------------------------------------ multi-layer steps

def run_layers(args):
    """A decode step over ``--layers`` layers' caches sharing one block
    table ("MiniPaged-Qwen" §16.3): the native runner builds and copies the
    step's metadata once and launches one fused cache-write + attention
    kernel per layer.  Steps rotate over replica pools until more than 3x L2
    streams between two uses of one; one layer alone is timed the same way
    for comparison.  K/V values are random normal (not checked here: the
    multi-layer GPU tests check them against the oracle)."""
    import ctypes
    import numpy as np
    import torch
    import paged_kv_cache_128_gb300 as pk
    from paged_kv_cache_128_gb300._lib import check, kvstep_config_t, lib
    from paged_kv_cache_128_gb300.inputs import make_workload
    from paged_kv_cache_128_gb300.kernels import alloc_workspace, decode_plan, dtype_code

    wl = make_workload(args.workload)
    if wl.prefill_lens.size or wl.num_pad:
        raise SystemExit("--layers takes a decode-only workload")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    dt = wl.torch_dtype
    B, hq, hkv, d, bs, nb = wl.num_seqs, wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.block_size, wl.num_blocks
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    es = torch.empty((), dtype=dt).element_size()
    row = hkv * d * es
    ids = np.ascontiguousarray(wl.decode_ids, dtype=np.int64)
    steps, warm = max(args.steps, 1), max(args.warmup, 3)
    results = {}
    for layers in (1, args.layers):
        per_layer = int(wl.cached_lens.sum()) * 2 * row
        replicas = int(max(1, min(16, -(-3 * l2 // (per_layer * layers)))))
        max_len = int(wl.cached_lens.max()) + 1 + (steps + warm) // replicas + 4
        maxb = -(-max_len // bs)
        runners = []
        for _ in range(replicas):
            mgr = pk.KVBlockManager(nb, bs, wl.free_order)
            for sid, n in zip(wl.decode_ids.tolist(), wl.cached_lens.tolist()):
                mgr.allocate_for_prefill(int(sid), int(n))
            kc = torch.empty(layers, nb, bs, hkv, d, dtype=dt, device=dev).normal_()
            vc = torch.empty_like(kc).normal_()
            ws = alloc_workspace(decode_plan(B, hq, hkv, d, bs, max_len, dt), dev)
            cfg = kvstep_config_t(num_seqs=B, num_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
                                  num_blocks=nb, max_blocks_per_seq=maxb, max_seq_len=max_len, scale=float(wl.scale),
                                  dtype=dtype_code(dt), num_step_tokens=B, k_cache=kc.data_ptr(),
                                  v_cache=vc.data_ptr(), workspace=ws.data_ptr() if ws is not None else None,
                                  workspace_bytes=ws.numel() if ws is not None else 0,
                                  stream=torch.cuda.current_stream().cuda_stream, host_io=0, num_layers=layers,
                                  cache_layer_stride=kc.stride(0))
            h = ctypes.c_void_p()
            check(lib().kvstep_create(mgr._h, ctypes.byref(cfg), ctypes.byref(h)), "kvstep_create")
            q = torch.randn(layers, B, hq, d, device=dev, dtype=dt)
            k = torch.randn(layers, B, hkv, d, device=dev, dtype=dt)
            v = torch.randn(layers, B, hkv, d, device=dev, dtype=dt)
            runners.append([h, q, k, v, torch.empty_like(q), mgr, kc, vc, ws, 0])

        def step(i):
            r = runners[i % replicas]
            check(lib().kvstep_run(r[0], r[1].data_ptr(), r[2].data_ptr(), r[3].data_ptr(), r[4].data_ptr(), None,
                                   0, None, None, 0, ids.ctypes.data, B, None, 0), "kvstep_run")
            r[9] += 1
            return r[9]

        for i in range(max(warm, replicas)):
            step(i)
        for r in runners:
            check(lib().kvstep_join(r[0], torch.cuda.current_stream().cuda_stream), "kvstep_join")
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        nbytes = 0
        wall0 = time.perf_counter()
        a.record()
        for i in range(steps):
            done = step(i)
            lens = wl.cached_lens + done   # after this step's append
            nbytes += layers * (int(lens.sum()) * 2 * row + 2 * B * hq * d * es + 4 * (B + int((-(-lens // bs)).sum()))
                                + 2 * 2 * B * row + 4 * B)
        host_s = (time.perf_counter() - wall0) / steps
        for r in runners:
            check(lib().kvstep_join(r[0], torch.cuda.current_stream().cuda_stream), "kvstep_join")
        b.record()
        torch.cuda.synchronize()
        t = a.elapsed_time(b) / 1e3
        results[layers] = {"step_us": t / steps * 1e6, "per_layer_us": t / steps / layers * 1e6,
                           "gbs": nbytes / t / 1e9, "host_us_per_step": host_s * 1e6,
                           "decode_tokens_per_s": B * steps / t, "replicas": replicas}
        for r in runners:
            lib().kvstep_destroy(r[0])
        del runners
        torch.cuda.empty_cache()
    status = pk.device_error()
    print(json.dumps({"metric": "multi-layer decode step GB/s (algorithmic bytes of every layer) at 1 GB300",
                      "value": results[args.layers]["gbs"], "unit": "GB/s", "n_gpus": 1, "steps": steps,
                      "warmup": warm, "ms_per_step": results[args.layers]["step_us"] / 1e3, "higher_is_better": True,
                      "dtype": wl.dtype, "data": "synthetic (random normal K/V)",
                      "config": {"workload": wl.name, "layers": args.layers,
                                 "l2": "inputs larger than L2: steps rotate over replica pools"},
                      "layers": {str(k): v for k, v in results.items()}, "device_error": status}))
    if status:
        sys.exit(1)


def main():
    args = parse_args()
    if args.layers:
        run_layers(args)
        return
    if args.prefill:
        run_prefill(args)
        return
    if args.cache_write:
        run_cache_write(args)
        return
    if args.profile_calls:
        run_profile_calls(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
