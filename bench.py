"""Benchmark: TurboQuant paged-KV decode step on GB300.

One step = the whole hot path for one decode iteration of a batch:
  tq_store of the step's new token per sequence (rotate, quantise, pack,
  write through slot_mapping) + tq_decode (rotate q, split-K attention over
  the packed cache, LSE reduce).

Workload (default): batch 32 x context 4096, n_q 32, n_kv 8, d 128, block 16,
preset 4bit_nc, bf16 inputs with one x8 outlier channel per head, block table
a random permutation. ``value`` = logical packed-KV bytes read per step /
step time (GB/s). Extra keys report decode tok/s, store Mtok/s (8192-token
prefill chunk) and the split kernel's roofline.

L2 hygiene: three copies of the cache (3 x 143 MB, each larger than L2) are
rotated between steps, so no step finds its cache in L2.

The K timed steps are launched eagerly through the binding. The same K steps
replayed from CUDA graphs (one captured step per cache copy, as a serving loop
replays its decode step) are timed too and reported as ``graph_ms_per_step``
(null, with ``config.graph`` saying why, if capture fails).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tq|reference]
  python bench.py --op dequant [--steps K] [--warmup W]   (full dequantisation alone)

``--impl reference`` times the CPU oracle (test infrastructure) on a bounded
sample of the same workload; N > 1 runs weak-scaling replicas (each rank its
own batch; there is no data exchange in this path).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode KV-read GB/s & % of HBM peak; decode tok/s; store Mtok/s (d=128 4bit_nc)"
WORKLOAD = "gqa"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, burst copy)"
    except Exception:
        return 6800.0, "fallback (6.8 TB/s)"


def _profile_traffic(kernel_file: str, summary: str):
    """Per-launch DRAM bytes from a committed ncu summary, if it matches the
    current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", summary)
    try:
        text = open(path).read()
        src = open(os.path.join(ROOT, "turboquant_paged_kv_gb300", "csrc", kernel_file), "rb").read()
    except OSError:
        return None
    h = hashlib.sha256(src).hexdigest()[:16]
    m_hash = re.search(r"source_sha256_16:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    if not m_hash or not m_bytes or m_hash.group(1) != h:
        return None
    return int(m_bytes.group(1))


class ClockSampler:
    """nvidia-smi sampling during the timed region (clocks + throttle reasons)."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: str):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.25)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_workload(rank: int):
    """Rank ``rank``'s replica of the workload: same shapes, its own seed
    (weak scaling: every rank decodes a whole batch of its own)."""
    import workloads
    return workloads.get(WORKLOAD, seed=rank)


def max_over_ranks(values, device, world: int):
    """Element-wise max of per-rank timings (ms) over all ranks."""
    import torch
    vals = torch.tensor(list(values), dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(vals, op=dist.ReduceOp.MAX)
    return vals.tolist()


def whole_job_gbs(world: int, bytes_per_rank: int, ms: float) -> float:
    """Whole-job throughput: bytes all ranks read in one step / the slowest rank's step."""
    return world * bytes_per_rank / (ms * 1e-3) / 1e9


def all_ranks_ok(ok: bool, device, world: int) -> bool:
    """True only if ``ok`` holds on every rank (one max-reduce; every rank
    calls it, so no rank can wait for a peer that took another branch)."""
    return max_over_ranks([0.0 if ok else 1.0], device, world)[0] == 0.0


def merge_timings(values, optional, device, world: int):
    """Max over ranks of ``values`` (ms) and of ``optional`` (ms or None), in
    one collective; the optional timing is None unless every rank has one."""
    got = max_over_ranks(list(values) + [optional or 0.0, 1.0 if optional is None else 0.0], device, world)
    return got[:len(values)], (None if got[-1] else got[-2])


_ORACLE_STEP_SCRIPT = """
import os, sys, time, json
sys.path.insert(0, {root!r})
sys.path.insert(0, os.path.join({root!r}, "tests"))
import numpy as np, workloads
from parity import OracleCache
from oracle import store as ost
w = workloads.get({workload!r}, batch=1, seed={seed})
inp = workloads.make_inputs(w)
oc = OracleCache(w, inp).fill()
q = inp.q.double().numpy()
k, v = oc.kv[0]
last = inp.fill_slots.numpy()[-1:]
times = []
for _ in range({steps}):
    t0 = time.perf_counter()
    ost.store(k[-1:].double().numpy(), v[-1:].double().numpy(), last, oc.cache, oc.lay, oc.preset, oc.cent, oc.mid)
    oc.decode(q)
    times.append(time.perf_counter() - t0)
print(json.dumps({{"times": times, "bytes": int(inp.seq_lens.sum()) * w.n_kv * oc.lay.slot_bytes}}))
"""

_SINGLE_THREAD_ENV = dict(OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")


def _oracle_child(workload: str, steps: int, seed: int) -> subprocess.Popen:
    code = _ORACLE_STEP_SCRIPT.format(root=ROOT, workload=workload, seed=seed, steps=steps)
    return subprocess.Popen([sys.executable, "-c", code], env=dict(os.environ, **_SINGLE_THREAD_ENV),
                            stdout=subprocess.PIPE, text=True)


def _oracle_result(proc: subprocess.Popen):
    out, _ = proc.communicate()
    if proc.returncode != 0:
        raise RuntimeError(f"oracle child exited {proc.returncode}")
    r = json.loads(out.strip().splitlines()[-1])
    return r["times"], r["bytes"]


def _oracle_steps(workload: str, steps: int):
    """Time the oracle in a single-threaded child process (spawned, no CUDA):
    one sequence of the workload is oracle-stored once, then each step is the
    oracle store of one new token plus the oracle decode of all query heads
    of that sequence. Returns (list of step seconds, bytes read per step)."""
    return _oracle_result(_oracle_child(workload, steps, 0))


def _oracle_steps_all_cores(workload: str, steps: int, procs: int):
    """The same oracle step in ``procs`` single-threaded child processes at
    once, each on a sequence of its own (seeds 0 .. procs-1). Returns the
    aggregate bytes per second over the children's timed steps (the first two
    steps of each are warm-up)."""
    children = [_oracle_child(workload, steps, seed) for seed in range(procs)]
    results = [_oracle_result(c) for c in children]
    return sum(nbytes / statistics.mean(times[2:]) for times, nbytes in results)


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    import workloads
    w = workloads.get(WORKLOAD)
    times, nbytes = _oracle_steps(WORKLOAD, args.warmup + args.steps)
    step_s = statistics.mean(times[args.warmup:])
    gbs = nbytes / step_s / 1e9
    sample = (f"1 of {w.batch} sequences ({w.fixed_len} tokens, {w.n_kv} KV heads): oracle store of one new "
              f"token + oracle decode of {w.n_q} query heads, per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD}: {w.note}, d {w.d}, block {w.block_size}, {w.preset}"},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_tq(args):
    import numpy as np
    import torch

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    from turboquant_paged_kv_gb300 import build as tqbuild
    if rank == 0:
        tqbuild.build()
    if world > 1:
        torch.distributed.barrier()
    import turboquant_paged_kv_gb300 as tq
    import workloads

    w = rank_workload(rank)
    inp = workloads.make_inputs(w, device=dev)
    # seq_lens and the block table are written long before each decode (the
    # kernel right before it is tq_store), so the split kernel may plan before
    # waiting for that kernel
    cfg = tq.make_config(w.preset, w.n_q, w.n_kv, block_size=w.block_size, partition_tokens=args.partition,
                         flags=tq.TQ_FLAG_INDICES_READY)
    cb = tq.tq_build_codebook(w.d, 4)
    lay = tq.tq_layout_for(cfg)
    n_copies = 3
    caches = [torch.empty(inp.num_blocks * lay.block_bytes, dtype=torch.uint8, device=dev)]
    # fill the cache: every cached position of every sequence
    for b in range(w.batch):
        k, v = inp.kv_for_sequence(b, dev)
        s0 = dict(inp.fill_order)[b]
        tq.tq_store(cfg, cb, k, v, inp.fill_slots[s0: s0 + k.shape[0]], caches[0])
    for _ in range(n_copies - 1):
        caches.append(caches[0].clone())
    torch.cuda.synchronize()

    B, L = w.batch, w.fixed_len
    seq_lens = inp.seq_lens
    table = inp.block_table
    max_len = int(seq_lens.max().item())
    last_slots = table[torch.arange(B, device=dev), (seq_lens - 1) // w.block_size].to(torch.int64) * w.block_size \
        + ((seq_lens - 1) % w.block_size).to(torch.int64)
    g = torch.Generator(device=dev)
    g.manual_seed(1234 + rank)
    new_k = torch.randn(B, w.n_kv, w.d, generator=g, device=dev).to(torch.bfloat16)
    new_v = torch.randn(B, w.n_kv, w.d, generator=g, device=dev).to(torch.bfloat16)
    q = inp.q
    out = torch.empty(B, w.n_q, w.d, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(tq.tq_decode_workspace_size(cfg, B, max_len), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    kv_bytes = int(seq_lens.sum().item()) * w.n_kv * lay.slot_bytes

    def step(i):
        cache = caches[i % n_copies]
        tq.tq_store(cfg, cb, new_k, new_v, last_slots, cache)
        tq.tq_decode(cfg, cb, q, cache, table, seq_lens, max_len, out, ws)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    props = torch.cuda.get_device_properties(dev)
    gpu_id = ("GPU-" + str(props.uuid)) if getattr(props, "uuid", None) else str(dev.index or 0)
    with ClockSampler(gpu_id) as clk:
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        ev0.record(stream)
        for i in range(args.steps):
            step(i)
        ev1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        eager_ms = ev0.elapsed_time(ev1) / args.steps

        # ---- the same K steps replayed from CUDA graphs (one per cache copy),
        # as a serving loop runs its decode step
        graph_ms, graph_note, graphs = None, "captured", []
        try:
            for c in range(n_copies):
                gr = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gr):
                    step(c)
                graphs.append(gr)
        except RuntimeError as exc:   # capture refused: only the eager steps count
            graphs, graph_note = [], "capture failed: %s" % str(exc).splitlines()[0][:120]
        # every rank times the graphs only if every rank captured them
        if all_ranks_ok(bool(graphs), dev, world):
            for i in range(args.warmup):
                graphs[i % n_copies].replay()
            torch.cuda.synchronize()
            if world > 1:
                torch.distributed.barrier()
            ev0.record(stream)
            for i in range(args.steps):
                graphs[i % n_copies].replay()
            ev1.record(stream)
            torch.cuda.synchronize()
            if world > 1:
                torch.distributed.barrier()
            graph_ms = ev0.elapsed_time(ev1) / args.steps
        elif graphs:
            graph_note = "capture failed on another rank"
        step_ms = eager_ms

        # ---- split kernel alone (the dominant kernel), same stream, rotated caches
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = max(args.steps, 20)
        e0.record(stream)
        for i in range(reps):
            tq.tq_decode_partials(cfg, cb, q, caches[i % n_copies], table, seq_lens, max_len, ws)
        e1.record(stream)
        torch.cuda.synchronize()
        split_ms = e0.elapsed_time(e1) / reps

    # ---- store throughput on an 8192-token prefill chunk (random distinct slots)
    n_store = 8192
    st_k = torch.randn(n_store, w.n_kv, w.d, generator=g, device=dev).to(torch.bfloat16)
    st_v = torch.randn(n_store, w.n_kv, w.d, generator=g, device=dev).to(torch.bfloat16)
    st_slots = torch.randperm(inp.num_blocks * w.block_size, generator=g, device=dev)[:n_store].to(torch.int64)
    scratch = caches[1]
    for _ in range(3):
        tq.tq_store(cfg, cb, st_k, st_v, st_slots, scratch)
    e0.record(stream)
    st_reps = 50
    for _ in range(st_reps):
        tq.tq_store(cfg, cb, st_k, st_v, st_slots, scratch)
    e1.record(stream)
    torch.cuda.synchronize()
    store_ms = e0.elapsed_time(e1) / st_reps

    # ---- end to end through the public API with host buffers
    # the step's inputs packed into one pinned host buffer and one device
    # buffer (each part 256-byte aligned): one host->device copy per step
    parts = [q, new_k, new_v, last_slots, seq_lens, table]
    offs, total = [], 0
    for t in parts:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    pack_h = torch.empty(total, dtype=torch.uint8).pin_memory()
    pack_d = torch.empty(total, dtype=torch.uint8, device=dev)

    def view(buf, t, off):
        return buf[off: off + t.numel() * t.element_size()].view(t.dtype).view(t.shape)

    for t, off in zip(parts, offs):
        view(pack_h, t, off).copy_(t.cpu())
    q_d, nk_d, nv_d, sl_d, lens_d, tab_d = (view(pack_d, t, off) for t, off in zip(parts, offs))
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = total
    d2h = out_h.numel() * out_h.element_size()

    def e2e_step(i):
        pack_d.copy_(pack_h, non_blocking=True)
        cache = caches[i % n_copies]
        tq.tq_store(cfg, cb, nk_d, nv_d, sl_d, cache)
        tq.tq_decode(cfg, cb, q_d, cache, tab_d, lens_d, max_len, out, ws)
        out_h.copy_(out, non_blocking=True)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(args.steps):
        e2e_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps

    # ---- max over ranks
    (step_ms, split_ms, store_ms, e2e_ms), graph_ms = merge_timings([step_ms, split_ms, store_ms, e2e_ms], graph_ms,
                                                                    dev, world)
    clocks = clk.summary()

    if rank == 0:
        peak, peak_src = _peaks()
        gbs = whole_job_gbs(world, kv_bytes, step_ms)
        split_gbs = kv_bytes / (split_ms * 1e-3) / 1e9
        line = {
            "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16 mma / f32 accumulate over 4-bit codes", "data": "synthetic",
            "config": {"workload": f"{WORKLOAD}: {w.note}, d {w.d}, block {w.block_size}, {w.preset}, bf16 in/out",
                       "partition_tokens": args.partition, "split": "stream-K: equal tile ranges per warp" if args.partition == 0 else "fixed partitions",
                       "l2": "3 rotated cache copies of %.0f MB each (> L2)" % (caches[0].numel() / 1e6),
                       "kv_bytes_per_step": kv_bytes, "graph": graph_note},
            "graph_ms_per_step": graph_ms,
            "decode_tok_s": world * B / (step_ms * 1e-3),
            "hbm_frac_step": gbs / world / peak,
            "store_mtok_s": n_store / (store_ms * 1e-3) / 1e6,
            "store_gbs": n_store * (w.n_kv * (2 * w.d * 2 + lay.slot_bytes) + 8) / (store_ms * 1e-3) / 1e9,
            "roofline": {"kernel": "split_kernel (tq_decode_partials)", "bound": "hbm", "achieved": split_gbs,
                         "peak": peak, "unit": "GB/s", "frac": split_gbs / peak,
                         "traffic": _profile_traffic("tq_decode.cu", "decode_split_gqa.md"),
                         "peak_source": peak_src, "ms_per_launch": split_ms,
                         "algorithmic_bytes_per_launch": kv_bytes},
            "e2e": {"value": whole_job_gbs(world, kv_bytes, e2e_ms), "unit": "GB/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": 3 * args.steps,
            "clocks": clocks,
        }
        if not args.no_cpu_baseline:
            times, nbytes = _oracle_steps(WORKLOAD, 8)
            step_s = statistics.mean(times[2:])
            line["cpu_baseline"] = {
                "value": nbytes / step_s / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
                "sample": f"1 of {B} sequences ({L} tokens, {w.n_kv} KV heads, {w.n_q} query heads): "
                          "oracle store of one new token + oracle decode, mean of 6 steps after 2 warm-up",
            }
            # the same oracle on every host core at once (one sequence per core)
            procs = max(1, min(len(os.sched_getaffinity(0)), B))
            try:
                line["cpu_baseline"]["all_cores"] = {
                    "value": _oracle_steps_all_cores(WORKLOAD, 8, procs) / 1e9, "unit": "GB/s", "cores": procs,
                    "sample": f"{procs} sequences at once, one single-threaded process each, same steps",
                }
            except Exception as exc:   # a reported extra: never lose the line over it
                line["cpu_baseline"]["all_cores"] = {"unavailable": str(exc)[:120]}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_dequant(args):
    """``--op dequant``: tq_dequant of the whole gqa cache (32 x 4096 positions,
    8 KV heads) to bf16 keys and values in the original basis, one launch per
    step, timed alone with CUDA events. Each launch reads 141 MB of packed
    slots and writes 537 MB, far more than L2, so consecutive launches find
    nothing in L2.
    Prints one JSON line of its own (not the decode step's)."""
    import torch

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    from turboquant_paged_kv_gb300 import build as tqbuild
    tqbuild.build()
    import turboquant_paged_kv_gb300 as tq
    import workloads

    w = workloads.get(WORKLOAD)
    inp = workloads.make_inputs(w, device=dev)
    cfg = tq.make_config(w.preset, w.n_q, w.n_kv, block_size=w.block_size)
    cb = tq.tq_build_codebook(w.d, 4)
    lay = tq.tq_layout_for(cfg)
    cache = torch.empty(inp.num_blocks * lay.block_bytes, dtype=torch.uint8, device=dev)
    for b in range(w.batch):
        k, v = inp.kv_for_sequence(b, dev)
        s0 = dict(inp.fill_order)[b]
        tq.tq_store(cfg, cb, k, v, inp.fill_slots[s0: s0 + k.shape[0]], cache)
    max_len = inp.max_seq_len
    shape = (w.batch, max_len, w.n_kv, w.d)
    k_out = torch.empty(shape, dtype=torch.bfloat16, device=dev)
    v_out = torch.empty(shape, dtype=torch.bfloat16, device=dev)
    positions = int(inp.seq_lens.sum().item()) * w.n_kv
    nbytes = positions * (lay.slot_bytes + 2 * w.d * 2)    # packed slot in, bf16 key + value out
    stream = torch.cuda.current_stream()

    def step():
        tq.tq_dequant(cfg, cb, cache, inp.block_table, inp.seq_lens, max_len, k_out, v_out)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    props = torch.cuda.get_device_properties(dev)
    gpu_id = ("GPU-" + str(props.uuid)) if getattr(props, "uuid", None) else "0"
    with ClockSampler(gpu_id) as clk:
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    peak, peak_src = _peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    print(json.dumps({
        "op": "dequant", "metric": "full dequant GB/s (packed slots read + bf16 K/V written)",
        "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "dtype": "f32 arithmetic, bf16 out", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD}: {w.note}, d {w.d}, block {w.block_size}, {w.preset}, bf16 out",
                   "l2": "each launch moves %.0f MB (> L2)" % (nbytes / 1e6), "bytes_per_launch": nbytes},
        "roofline": {"kernel": "dequant_kernel (tq_dequant)", "bound": "hbm", "achieved": gbs, "peak": peak,
                     "unit": "GB/s", "frac": gbs / peak, "peak_source": peak_src, "ms_per_launch": ms,
                     "algorithmic_bytes_per_launch": nbytes},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
    }), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="tq", choices=["tq", "reference"])
    ap.add_argument("--partition", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--op", default="decode", choices=["decode", "dequant"],
                    help="decode: the decode step (default); dequant: tq_dequant of the gqa cache alone")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.op == "dequant":
        return run_dequant(args)
    return run_reference(args) if args.impl == "reference" else run_tq(args)


if __name__ == "__main__":
    sys.exit(main())
