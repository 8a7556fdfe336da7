"""Benchmark: TurboQuant paged-KV decode step on GB300.

One step = the whole hot path for one decode iteration of a batch:
  tq_store of the step's new token per sequence (rotate, quantise, pack,
  write through slot_mapping) + tq_decode (rotate q, split-K attention over
  the packed cache, LSE reduce).

Workloads (``--workload``; the default is the one the headline metric is
quoted on):

  gqa   batch 32 x context 4096, n_q 32, n_kv 8, 4bit_nc, bf16 inputs with one
        x8 outlier channel per head, block table a random permutation
  k3v4  batch 64, contexts uniform in [512, 16384], n_q 32, n_kv 8, k3v4_nc
  k8v4  batch 128 x 8192, n_q 32, n_kv 8, k8v4 (e4m3 keys); its store line
        is the workload's own 8192-token prefill chunk
  long  batch 4 x 131072, n_q 64, n_kv 8, 4bit_nc, Student-t outlier channels
  3bit  the gqa shape with the 3bit_nc preset (3-bit keys and 3-bit values)
  all   every workload above, one JSON line each

``value`` = logical packed-KV bytes read per step / step time (GB/s). Each
line also carries decode tok/s, the split kernel's roofline (the dominant
kernel), the store kernel's roofline on an 8192-token prefill chunk, an
end-to-end number through the public API with host buffers, and the CPU
oracle timed on a bounded sample of the same workload.

L2 hygiene: three copies of the cache (each larger than the 129 MB L2) are
rotated between steps, so no step finds its cache in L2.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tq|reference]
                  [--workload gqa|k3v4|k8v4|long|all] [--partition P]
  python bench.py --op dequant [--steps K] [--warmup W]   (full dequantisation alone)
  python bench.py --op store [--workload W]               (the prefill-chunk store alone)
  python bench.py --op prod                               (TurboQuant_prod keys: scores + store)
  python bench.py --op continue                           (128-query continuation chunks vs per-query decode)

``--impl reference`` times the CPU oracle (test infrastructure) on a bounded
sample of the same workload. N > 1 runs weak-scaling replicas, one process
per GPU (each rank its own batch; there is no data exchange in this path):
under torchrun the ranks come from the environment; without it bench.py
starts the N ranks itself. ``--dry-run`` runs the multi-rank host logic on
the CPU (gloo) without touching a GPU.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import socket
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode KV-read GB/s & % of HBM peak; decode tok/s; store Mtok/s (d=128 4bit_nc)"
WORKLOADS = ("gqa", "k3v4", "k8v4", "long", "3bit")
DEFAULT_WORKLOAD = "gqa"
# tokens of one sequence the CPU oracle handles per step in the baseline legs
ORACLE_SAMPLE_TOKENS = 8192
STORE_TOKENS = 8192


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, burst copy)"
    except Exception:
        return 6800.0, "fallback (6.8 TB/s)"


def _tensor_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst cuBLAS bf16 GEMM)"
    except Exception:
        return 1900.0, "fallback (1.9 PFLOP/s bf16 burst)"


def _profile_field(kernel_file: str, summary: str, field: str):
    """A number from a committed ncu summary under profiles/, if the summary's
    recorded source hash matches the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", summary)
    try:
        text = open(path).read()
        src = open(os.path.join(ROOT, "turboquant_paged_kv_gb300", "csrc", kernel_file), "rb").read()
    except OSError:
        return None
    h = hashlib.sha256(src).hexdigest()[:16]
    m_hash = re.search(r"source_sha256_16:\s*([0-9a-f]+)", text)
    m_val = re.search(re.escape(field) + r":\s*([0-9.]+)", text)
    if not m_hash or not m_val or m_hash.group(1) != h:
        return None
    v = float(m_val.group(1))
    return int(v) if v.is_integer() else v


def key_bits(preset: str):
    """Codebook bits of a preset's keys (None for e4m3 keys)."""
    return {"4bit_nc": 4, "k3v4_nc": 3, "3bit_nc": 3}.get(preset)


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


# ---------------------------------------------------------------- ranks

def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_workload(rank: int, name: str = DEFAULT_WORKLOAD):
    """Rank ``rank``'s replica of the workload: same shapes, its own seed
    (weak scaling: every rank decodes a whole batch of its own)."""
    import workloads
    return workloads.get(name, seed=rank)


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


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_entry(rank: int, world: int, port: int, argv):
    """One self-launched rank: the environment torchrun would give it, then
    the ordinary entry point."""
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    rc = main(argv)
    if rc:
        raise SystemExit(rc)


def launch_ranks(n: int, argv, dry_run: bool) -> int:
    """Start ``n`` ranks of this script (spawned processes, one per GPU) when
    no launcher set the rank environment. Refuses, with a non-zero exit,
    to run more ranks than there are visible GPUs."""
    if not dry_run:
        import torch
        have = torch.cuda.device_count() if torch.cuda.is_available() else 0
        if have < n:
            print(json.dumps({"error": f"--gpus {n} needs {n} visible GPUs, found {have}"}), flush=True)
            return 2
    import torch.multiprocessing as mp
    mp.start_processes(_rank_entry, args=(n, _free_port(), argv), nprocs=n, join=True, start_method="spawn")
    return 0


def run_dry(args) -> int:
    """The multi-rank host logic with no GPU: process group over gloo, each
    rank's replica workload, the max-over-ranks of (stand-in) step timings
    and the whole-job value, printed by rank 0."""
    import torch
    import torch.distributed as dist
    world, rank, _ = _dist()
    if world > 1:
        dist.init_process_group("gloo")
    try:
        import workloads
        w = rank_workload(rank, args.workload if args.workload != "all" else DEFAULT_WORKLOAD)
        inp = workloads.make_inputs(workloads.get(w.name + "_small", seed=w.seed)
                                    if w.name + "_small" in workloads.WORKLOADS else w)
        kv_bytes = int(w.batch) * (w.fixed_len or 1) * w.n_kv
        mine = 1.0 + rank                      # stand-in step time (ms)
        (step_ms,) = max_over_ranks([mine], torch.device("cpu"), world)
        seeds = max_over_ranks([float(w.seed)], torch.device("cpu"), world)
        if rank == 0:
            print(json.dumps({"dry_run": True, "n_gpus": world, "workload": w.name, "max_step_ms": step_ms,
                              "max_seed": seeds[0], "q_checksum_rank0": float(inp.q.float().sum()),
                              "value": whole_job_gbs(world, kv_bytes, step_ms)}), flush=True)
    finally:
        if world > 1:
            dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------- CPU oracle

_ORACLE_STEP_SCRIPT = """
import os, sys, time, json
sys.path.insert(0, {root!r})
sys.path.insert(0, os.path.join({root!r}, "tests"))
import numpy as np, workloads
from parity import OracleCache
from oracle import store as ost
base = workloads.get({workload!r})
over = dict(batch=1, seed={seed}, store_tokens=0, store_extra_blocks=0)
if base.fixed_len:
    over["fixed_len"] = min(base.fixed_len, {cap})
else:
    over["len_range"] = (min(base.len_range[0], {cap}), min(base.len_range[1], {cap}))
w = workloads.get({workload!r}, **over)
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
print(json.dumps({{"times": times, "bytes": int(inp.seq_lens.sum()) * w.n_kv * oc.lay.slot_bytes,
                  "tokens": int(inp.seq_lens.sum())}}))
"""

_SINGLE_THREAD_ENV = dict(OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")


def _oracle_child(workload: str, steps: int, seed: int) -> subprocess.Popen:
    code = _ORACLE_STEP_SCRIPT.format(root=ROOT, workload=workload, seed=seed, steps=steps,
                                      cap=ORACLE_SAMPLE_TOKENS)
    return subprocess.Popen([sys.executable, "-c", code], env=dict(os.environ, **_SINGLE_THREAD_ENV),
                            stdout=subprocess.PIPE, text=True)


def _oracle_result(proc: subprocess.Popen):
    out, _ = proc.communicate()
    if proc.returncode != 0:
        raise RuntimeError(f"oracle child exited {proc.returncode}")
    r = json.loads(out.strip().splitlines()[-1])
    return r["times"], r["bytes"], r["tokens"]


def _oracle_steps(workload: str, steps: int):
    """Time the oracle in a single-threaded child process (spawned, no CUDA):
    one sequence of the workload (at most ORACLE_SAMPLE_TOKENS positions) is
    oracle-stored once, then each step is the oracle store of one new token
    plus the oracle decode of all query heads of that sequence. Returns (list
    of step seconds, bytes read per step, tokens of the sequence)."""
    return _oracle_result(_oracle_child(workload, steps, 0))


def _oracle_steps_all_cores(workload: str, steps: int, procs: int):
    """The same oracle step in ``procs`` single-threaded child processes at
    once, each on a sequence of its own (seeds 0 .. procs-1). Returns the
    aggregate bytes per second over the children's timed steps (the first two
    steps of each are warm-up)."""
    children = [_oracle_child(workload, steps, seed) for seed in range(procs)]
    results = [_oracle_result(c) for c in children]
    return sum(nbytes / statistics.mean(times[2:]) for times, nbytes, _ in results)


def _sample_text(w, tokens: int) -> str:
    return (f"1 of {w.batch} sequences, {tokens} positions ({w.n_kv} KV heads, {w.n_q} query heads; "
            f"sequences longer than {ORACLE_SAMPLE_TOKENS} positions are cut there): oracle store of one "
            "new token + oracle decode")


def _workload_text(w, extra: str = "") -> str:
    return f"{w.name}: {w.note}, d {w.d}, block {w.block_size}, {w.preset}{extra}"


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    import workloads
    for name in (WORKLOADS if args.workload == "all" else (args.workload,)):
        w = workloads.get(name)
        times, nbytes, tokens = _oracle_steps(name, args.warmup + args.steps)
        step_s = statistics.mean(times[args.warmup:])
        gbs = nbytes / step_s / 1e9
        line = {
            "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": _workload_text(w)},
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": _sample_text(w, tokens) + ", per step"},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm

class DecodeCase:
    """One workload's inputs, filled caches and step buffers on the device."""

    def __init__(self, tq, name: str, rank: int, dev, partition: int, n_copies: int = 3):
        import torch
        import workloads
        self.tq = tq
        self.w = w = rank_workload(rank, name)
        self.inp = inp = workloads.make_inputs(w, device=dev)
        # seq_lens and the block table are written long before each decode (the
        # kernel right before it is tq_store), so the split kernel may plan before
        # waiting for that kernel
        self.cfg = tq.make_config(w.preset, w.n_q, w.n_kv, block_size=w.block_size, partition_tokens=partition,
                                  flags=tq.TQ_FLAG_INDICES_READY)
        bits = key_bits(w.preset)
        self.cb = tq.tq_build_codebook(w.d, bits) if bits else None
        self.lay = lay = tq.tq_layout_for(self.cfg)
        caches = [torch.empty(inp.num_blocks * lay.block_bytes, dtype=torch.uint8, device=dev)]
        for b in range(w.batch):   # every cached position of every sequence
            k, v = inp.kv_for_sequence(b, dev)
            s0 = dict(inp.fill_order)[b]
            tq.tq_store(self.cfg, self.cb, k, v, inp.fill_slots[s0: s0 + k.shape[0]], caches[0])
            del k, v
        for _ in range(n_copies - 1):
            caches.append(caches[0].clone())
        self.caches = caches
        torch.cuda.synchronize()
        B = w.batch
        self.seq_lens = inp.seq_lens
        self.table = inp.block_table
        self.max_len = int(inp.seq_lens.max().item())
        last = (inp.seq_lens - 1).to(torch.int64)
        self.last_slots = (self.table[torch.arange(B, device=dev), last // w.block_size].to(torch.int64)
                           * w.block_size + last % w.block_size)
        self.gen = torch.Generator(device=dev)
        self.gen.manual_seed(1234 + rank)
        self.new_k = torch.randn(B, w.n_kv, w.d, generator=self.gen, device=dev).to(torch.bfloat16)
        self.new_v = torch.randn(B, w.n_kv, w.d, generator=self.gen, device=dev).to(torch.bfloat16)
        self.q = inp.q
        self.out = torch.empty(B, w.n_q, w.d, dtype=torch.bfloat16, device=dev)
        self.ws = torch.empty(tq.tq_decode_workspace_size(self.cfg, B, self.max_len), dtype=torch.uint8,
                              device=dev)
        self.kv_bytes = int(inp.seq_lens.sum().item()) * w.n_kv * lay.slot_bytes

    def step(self, i):
        """One decode step: tq_store of every sequence's new token, then
        tq_decode over all positions (three launches)."""
        tq = self.tq
        cache = self.caches[i % len(self.caches)]
        tq.tq_store(self.cfg, self.cb, self.new_k, self.new_v, self.last_slots, cache)
        tq.tq_decode(self.cfg, self.cb, self.q, cache, self.table, self.seq_lens, self.max_len, self.out, self.ws)

    def step_fused(self, i):
        """The same step in one call, tq_decode_append (the split kernel stores
        the new tokens; two launches)."""
        cache = self.caches[i % len(self.caches)]
        self.tq.tq_decode_append(self.cfg, self.cb, self.q, self.new_k, self.new_v, cache, self.table,
                                 self.seq_lens, self.max_len, self.out, self.ws)

    def split_only(self, i):
        self.tq.tq_decode_partials(self.cfg, self.cb, self.q, self.caches[i % len(self.caches)], self.table,
                                   self.seq_lens, self.max_len, self.ws)

    def store_chunk(self, dev):
        """The store leg's inputs: the workload's own prefill chunk when it has
        one (k8v4), else 8192 bf16 tokens through random distinct slots."""
        import torch
        w = self.w
        if w.store_tokens:
            k, v, slots = self.inp.store_chunk(dev)
            return k, v, slots
        k = torch.randn(STORE_TOKENS, w.n_kv, w.d, generator=self.gen, device=dev).to(torch.bfloat16)
        v = torch.randn(STORE_TOKENS, w.n_kv, w.d, generator=self.gen, device=dev).to(torch.bfloat16)
        slots = torch.randperm(self.inp.num_blocks * w.block_size, generator=self.gen, device=dev)[:STORE_TOKENS]
        return k, v, slots.to(torch.int64)


def _events(n=2):
    import torch
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def time_device(fn, reps: int, stream) -> float:
    """Mean ms per call of ``fn(i)``, CUDA events on the launching stream."""
    import torch
    e0, e1 = _events()
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(reps):
        fn(i)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def run_workload(tq, name: str, args, dev, world: int, rank: int):
    import torch

    c = DecodeCase(tq, name, rank, dev, args.partition)
    w = c.w
    stream = torch.cuda.current_stream()
    # the first timed loop after start-up runs ~2.5 us/step slow on gqa whatever
    # it times, so the one-call step (reported beside) is timed first and the
    # headline step after W warm-up steps of its own
    for i in range(args.warmup):
        c.step_fused(i)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()

    props = torch.cuda.get_device_properties(dev)
    gpu_id = ("GPU-" + str(props.uuid)) if getattr(props, "uuid", None) else str(dev.index or 0)
    with ClockSampler(gpu_id) as clk:
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        fused_ms = time_device(c.step_fused, args.steps, stream)
        for i in range(args.warmup):
            c.step(i)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        step_ms = time_device(c.step, args.steps, stream)
        if world > 1:
            torch.distributed.barrier()

        # ---- the same K steps replayed from CUDA graphs (one per cache copy),
        # as a serving loop runs its decode step
        graph_ms, graph_note, graphs = None, "captured", []
        try:
            for j in range(len(c.caches)):
                gr = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gr):
                    c.step(j)
                graphs.append(gr)
        except RuntimeError as exc:   # capture refused: only the eager steps count
            graphs, graph_note = [], "capture failed: %s" % str(exc).splitlines()[0][:120]
        if all_ranks_ok(bool(graphs), dev, world):
            for i in range(args.warmup):
                graphs[i % len(graphs)].replay()
            graph_ms = time_device(lambda i: graphs[i % len(graphs)].replay(), args.steps, stream)
        elif graphs:
            graph_note = "capture failed on another rank"
        del graphs

        # ---- split kernel alone (the dominant kernel), same stream, rotated caches
        for i in range(3):
            c.split_only(i)
        split_ms = time_device(c.split_only, max(args.steps, 100), stream)

    # ---- store throughput on a prefill chunk
    st_k, st_v, st_slots = c.store_chunk(dev)
    scratch = c.caches[1]
    n_store = st_k.shape[0]

    def store_once(_i):
        tq.tq_store(c.cfg, c.cb, st_k, st_v, st_slots, scratch)

    for i in range(3):
        store_once(i)
    store_ms = time_device(store_once, 200, stream)

    # ---- end to end through the public API with host buffers. Every step
    # copies its inputs (packed in one pinned buffer, 256-byte aligned parts)
    # host -> device, runs store + decode and copies the output back, and the
    # host waits for that output before the next step, as a serving loop that
    # samples the next token does. Timed on the host clock.
    parts = [c.q, c.new_k, c.new_v, c.seq_lens, c.table, c.last_slots]
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
    q_d, nk_d, nv_d, lens_d, tab_d, sl_d = (view(pack_d, t, off) for t, off in zip(parts, offs))
    out_h = torch.empty(c.out.shape, dtype=c.out.dtype).pin_memory()
    h2d_fused = offs[-1]   # the slots go last: the fused call does not take them
    h2d = total
    d2h = out_h.numel() * out_h.element_size()

    def e2e_fused(i):   # the same step in one call
        pack_d[:h2d_fused].copy_(pack_h[:h2d_fused], non_blocking=True)
        cache = c.caches[i % len(c.caches)]
        tq.tq_decode_append(c.cfg, c.cb, q_d, nk_d, nv_d, cache, tab_d, lens_d, c.max_len, c.out, c.ws)
        out_h.copy_(c.out, non_blocking=True)
        stream.synchronize()   # the host reads this step's output

    def e2e_two_call(i):
        pack_d.copy_(pack_h, non_blocking=True)
        cache = c.caches[i % len(c.caches)]
        tq.tq_store(c.cfg, c.cb, nk_d, nv_d, sl_d, cache)
        tq.tq_decode(c.cfg, c.cb, q_d, cache, tab_d, lens_d, c.max_len, c.out, c.ws)
        out_h.copy_(c.out, non_blocking=True)
        stream.synchronize()

    def host_time(fn):
        for i in range(args.warmup):
            fn(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(args.steps):
            fn(i)
        return (time.perf_counter() - t0) * 1e3 / args.steps

    e2e_fused_ms = host_time(e2e_fused)   # reported beside, timed first (see above)
    e2e_ms = host_time(e2e_two_call)

    # ---- max over ranks
    (step_ms, split_ms, store_ms, e2e_ms, fused_ms, e2e_fused_ms), graph_ms = merge_timings(
        [step_ms, split_ms, store_ms, e2e_ms, fused_ms, e2e_fused_ms], graph_ms, dev, world)
    clocks = clk.summary()
    if rank != 0:
        return None
    peak, peak_src = _peaks()
    gbs = whole_job_gbs(world, c.kv_bytes, step_ms)
    split_gbs = c.kv_bytes / (split_ms * 1e-3) / 1e9
    store_bytes = n_store * (w.n_kv * (2 * w.d * 2 + c.lay.slot_bytes) + 8)
    store_gbs = store_bytes / (store_ms * 1e-3) / 1e9
    split_note = ("stream-K: equal slice ranges per CTA" if args.partition == 0
                  else f"fixed partitions of {args.partition} positions")
    line = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16 mma / f32 accumulate over %s codes" % ("e4m3 key" if w.preset == "k8v4" else
                                                             "%d-bit key" % key_bits(w.preset)),
        "value_bits": c.lay.value_bits,
        "data": "synthetic",
        "config": {"workload": _workload_text(w, ", bf16 in/out"),
                   "partition_tokens": args.partition, "split": split_note,
                   "l2": "%d rotated cache copies of %.0f MB each (> L2)" % (len(c.caches), c.caches[0].numel() / 1e6),
                   "kv_bytes_per_step": c.kv_bytes, "graph": graph_note},
        "graph_ms_per_step": graph_ms,
        "step_timing": ("eager launches through the binding: tq_store of the step's new tokens then tq_decode, "
                        "timed after fused_ms_per_step (the same step as one tq_decode_append call) and W warm-up "
                        "steps of its own; graph_ms_per_step: the same steps replayed from CUDA graphs"),
        "fused_ms_per_step": fused_ms,
        "decode_tok_s": world * w.batch / (step_ms * 1e-3),
        "hbm_frac_step": gbs / world / peak,
        "store_mtok_s": n_store / (store_ms * 1e-3) / 1e6,
        "roofline": {"kernel": "split_kernel (tq_decode_partials)", "bound": "hbm", "achieved": split_gbs,
                     "peak": peak, "unit": "GB/s", "frac": split_gbs / peak,
                     "traffic": _profile_field("tq_decode.cu", f"decode_split_{name}.md", "dram_bytes_per_launch"),
                     "peak_source": peak_src, "ms_per_launch": split_ms,
                     "algorithmic_bytes_per_launch": c.kv_bytes},
        "store_roofline": {"kernel": "store_kernel (tq_store), %d-token prefill chunk" % n_store, "bound": "hbm",
                           "achieved": store_gbs, "peak": peak, "unit": "GB/s", "frac": store_gbs / peak,
                           "issue_frac": _profile_field("tq_store.cu", f"store_{name}.md", "issue_active_frac"),
                           "traffic": _profile_field("tq_store.cu", f"store_{name}.md", "dram_bytes_per_launch"),
                           "peak_source": peak_src, "ms_per_launch": store_ms,
                           "algorithmic_bytes_per_launch": store_bytes, "mtok_s": n_store / (store_ms * 1e-3) / 1e6},
        "e2e": {"value": whole_job_gbs(world, c.kv_bytes, e2e_ms), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "call": "tq_store then tq_decode",
                "timing": "host clock; each step ends when the host has the step's output",
                "fused": {"value": whole_job_gbs(world, c.kv_bytes, e2e_fused_ms), "ms_per_step": e2e_fused_ms,
                          "h2d_bytes_per_step": h2d_fused, "call": "tq_decode_append (timed first)"}},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        times, nbytes, tokens = _oracle_steps(name, 8)
        step_s = statistics.mean(times[2:])
        line["cpu_baseline"] = {
            "value": nbytes / step_s / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": _sample_text(w, tokens) + ", mean of 6 steps after 2 warm-up",
        }
        procs = max(1, min(len(os.sched_getaffinity(0)), w.batch))
        try:
            line["cpu_baseline"]["all_cores"] = {
                "value": _oracle_steps_all_cores(name, 8, procs) / 1e9, "unit": "GB/s", "cores": procs,
                "sample": f"{procs} sequences at once, one single-threaded process each, same steps",
            }
        except Exception as exc:   # a reported extra: never lose the line over it
            line["cpu_baseline"]["all_cores"] = {"unavailable": str(exc)[:120]}
    return line


def run_tq(args):
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

    for name in (WORKLOADS if args.workload == "all" else (args.workload,)):
        line = run_workload(tq, name, args, dev, world, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        torch.cuda.empty_cache()
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

    w = workloads.get(DEFAULT_WORKLOAD)
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

    def step(_i=0):
        tq.tq_dequant(cfg, cb, cache, inp.block_table, inp.seq_lens, max_len, k_out, v_out)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    props = torch.cuda.get_device_properties(dev)
    gpu_id = ("GPU-" + str(props.uuid)) if getattr(props, "uuid", None) else "0"
    with ClockSampler(gpu_id) as clk:
        ms = time_device(step, max(args.steps, 50), stream)
    peak, peak_src = _peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    print(json.dumps({
        "op": "dequant", "metric": "full dequant GB/s (packed slots read + bf16 K/V written)",
        "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": max(args.steps, 50), "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "dtype": "f32 arithmetic, bf16 out", "data": "synthetic",
        "config": {"workload": _workload_text(w, ", bf16 out"),
                   "l2": "each launch moves %.0f MB (> L2)" % (nbytes / 1e6), "bytes_per_launch": nbytes},
        "roofline": {"kernel": "dequant_mma_kernel (tq_dequant)", "bound": "hbm", "achieved": gbs, "peak": peak,
                     "unit": "GB/s", "frac": gbs / peak, "peak_source": peak_src, "ms_per_launch": ms,
                     "traffic": _profile_field("tq_dequant.cu", "dequant_gqa.md", "dram_bytes_per_launch"),
                     "algorithmic_bytes_per_launch": nbytes},
        "gpu_launches": max(args.steps, 50),
        "clocks": clk.summary(),
    }), flush=True)
    return 0


def run_store(args):
    """``--op store``: tq_store of the workload's prefill chunk (8192 bf16
    tokens through random distinct slots; k8v4: its own chunk) into an empty
    cache, one launch per step, timed alone with CUDA events. Prints one JSON
    line of its own with the store kernel's roofline."""
    import torch

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    from turboquant_paged_kv_gb300 import build as tqbuild
    tqbuild.build()
    import turboquant_paged_kv_gb300 as tq
    import workloads

    name = DEFAULT_WORKLOAD if args.workload == "all" else args.workload
    w = workloads.get(name)
    cfg = tq.make_config(w.preset, w.n_q, w.n_kv, block_size=w.block_size)
    bits = key_bits(w.preset)
    cb = tq.tq_build_codebook(w.d, bits) if bits else None
    lay = tq.tq_layout_for(cfg)
    g = torch.Generator(device=dev)
    g.manual_seed(1234)
    if w.store_tokens:
        k, v, slots = workloads.make_inputs(w, device=dev).store_chunk(dev)
        num_blocks = int(slots.max().item()) // w.block_size + 1
    else:
        num_blocks = 2 * STORE_TOKENS // w.block_size
        k = torch.randn(STORE_TOKENS, w.n_kv, w.d, generator=g, device=dev).to(torch.bfloat16)
        v = torch.randn(STORE_TOKENS, w.n_kv, w.d, generator=g, device=dev).to(torch.bfloat16)
        slots = torch.randperm(num_blocks * w.block_size, generator=g, device=dev)[:STORE_TOKENS].to(torch.int64)
    cache = torch.zeros(num_blocks * lay.block_bytes, dtype=torch.uint8, device=dev)
    n = k.shape[0]
    nbytes = n * (w.n_kv * (2 * w.d * 2 + lay.slot_bytes) + 8)
    stream = torch.cuda.current_stream()

    def step(_i=0):
        tq.tq_store(cfg, cb, k, v, slots, cache)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    props = torch.cuda.get_device_properties(dev)
    gpu_id = ("GPU-" + str(props.uuid)) if getattr(props, "uuid", None) else "0"
    reps = max(args.steps, 200)
    with ClockSampler(gpu_id) as clk:
        ms = time_device(step, reps, stream)
    peak, peak_src = _peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    print(json.dumps({
        "op": "store", "metric": "store Mtok/s and GB/s (bf16 K/V read + packed slots written)",
        "value": n / (ms * 1e-3) / 1e6, "unit": "Mtok/s", "n_gpus": 1, "steps": reps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "dtype": "f32 arithmetic, bf16 in", "data": "synthetic",
        "config": {"workload": _workload_text(w, f", {n}-token prefill chunk, random distinct slots"),
                   "bytes_per_launch": nbytes},
        "roofline": {"kernel": "store_kernel (tq_store)", "bound": "hbm", "achieved": gbs, "peak": peak,
                     "unit": "GB/s", "frac": gbs / peak, "peak_source": peak_src, "ms_per_launch": ms,
                     "issue_frac": _profile_field("tq_store.cu", f"store_{name}.md", "issue_active_frac"),
                     "traffic": _profile_field("tq_store.cu", f"store_{name}.md", "dram_bytes_per_launch"),
                     "algorithmic_bytes_per_launch": nbytes},
        "gpu_launches": reps,
        "clocks": clk.summary(),
    }), flush=True)
    return 0


_PROD_ORACLE_SCRIPT = """
import os, sys, time, json
sys.path.insert(0, {root!r})
import numpy as np, workloads
from oracle import codebook as ocb
from oracle import qjl
w = workloads.get("prod", batch=1, fixed_len={tokens})
inp = workloads.make_inputs(w)
lay = qjl.prod_tile_layout(w.d, w.block_size, w.n_kv, 2)
cent = ocb.codebook(w.d, 2)
S = workloads.projection(w).double().numpy()
cache = np.zeros(inp.num_blocks * lay.block_bytes, dtype=np.uint8)
k = inp.kv_for_sequence(0, "cpu")[0].double().numpy()
qjl.prod_store(k, inp.fill_slots.numpy(), S, cache, lay, cent, ocb.midpoints_fp32(cent))
q = inp.q.double().numpy()
times = []
for _ in range({steps}):
    t0 = time.perf_counter()
    qjl.prod_scores(q, S, cache, lay, cent, inp.block_table.numpy(), inp.seq_lens.numpy(), {tokens})
    times.append(time.perf_counter() - t0)
print(json.dumps({{"times": times}}))
"""
PROD_ORACLE_TOKENS = 4096


def run_prod(args):
    """``--op prod``: the TurboQuant_prod key path (2-bit Lloyd-Max code + 1-bit
    QJL residual signs) on the gqa shape, 32 x 4096 positions, n_q 32, n_kv 8:
    each step is tq_prod_scores of every query head against every cached key
    (a query-prep launch and the scores launch); four copies of the 54.5 MB
    cache are rotated so no step finds its keys in L2. The line also carries
    tq_prod_store of an 8192-token bf16 prefill chunk (its contraction, the
    projection S r, runs on tensor cores with fp16 hi/lo operands) and the
    oracle's prod_scores
    on one whole sequence
    (4096 positions). Prints one JSON line of its own."""
    import torch

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    from turboquant_paged_kv_gb300 import build as tqbuild
    tqbuild.build()
    import turboquant_paged_kv_gb300 as tq
    import workloads

    w = workloads.get("prod")
    inp = workloads.make_inputs(w, device=dev)
    cfg = tq.make_config("prod3", w.n_q, w.n_kv, block_size=w.block_size)
    cb = tq.tq_build_codebook(w.d, 2)
    lay = tq.tq_prod_layout_for(cfg)
    S = workloads.projection(w, dev)
    caches = [torch.empty(inp.num_blocks * lay.block_bytes, dtype=torch.uint8, device=dev) for _ in range(4)]
    for b in range(w.batch):
        k = inp.kv_for_sequence(b, dev)[0]
        s0 = dict(inp.fill_order)[b]
        tq.tq_prod_store(cfg, cb, S, k, inp.fill_slots[s0: s0 + k.shape[0]], caches[0])
    for c in caches[1:]:
        c.copy_(caches[0])
    L = inp.max_seq_len
    positions = int(inp.seq_lens.sum().item())
    scores = torch.empty(w.batch, w.n_q, L, dtype=torch.float32, device=dev)
    ws = torch.empty(tq.tq_prod_scores_workspace_size(cfg, w.batch), dtype=torch.uint8, device=dev)
    nbytes = positions * w.n_kv * lay.slot_bytes + scores.numel() * 4 + inp.q.numel() * 2
    stream = torch.cuda.current_stream()

    def step(i=0):
        tq.tq_prod_scores(cfg, cb, S, inp.q, caches[i % 4], inp.block_table, inp.seq_lens, L, scores, ws)

    # store leg: an 8192-token prefill chunk through random distinct slots
    g = torch.Generator(device=dev)
    g.manual_seed(1234)
    nblk = 2 * STORE_TOKENS // w.block_size
    kst = torch.randn(STORE_TOKENS, w.n_kv, w.d, generator=g, device=dev).to(torch.bfloat16)
    sst = torch.randperm(nblk * w.block_size, generator=g, device=dev)[:STORE_TOKENS].to(torch.int64)
    cst = torch.zeros(nblk * lay.block_bytes, dtype=torch.uint8, device=dev)

    def store(_i=0):
        tq.tq_prod_store(cfg, cb, S, kst, sst, cst)

    for _ in range(args.warmup):
        step()
        store()
    torch.cuda.synchronize()
    props = torch.cuda.get_device_properties(dev)
    gpu_id = ("GPU-" + str(props.uuid)) if getattr(props, "uuid", None) else "0"
    reps = max(args.steps, 100)
    with ClockSampler(gpu_id) as clk:
        ms = time_device(step, reps, stream)
        ms_store = time_device(store, 20, stream)
    peak, peak_src = _peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    store_tflops = STORE_TOKENS * w.n_kv * 2 * w.d * w.d / (ms_store * 1e-3) / 1e12
    tpeak, tpeak_src = _tensor_peak()
    line = {
        "op": "prod", "metric": "TurboQuant_prod scores GB/s (packed prod keys read + fp32 scores written); keys/s",
        "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": reps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "dtype": "f32 arithmetic, f16 query operands on tensor cores, bf16 in",
        "data": "synthetic",
        "config": {"workload": _workload_text(w), "l2": "4 cache copies of %.1f MB rotated" %
                   (positions * w.n_kv * lay.slot_bytes / 1e6), "bytes_per_launch": nbytes},
        "keys_per_s": positions * w.n_kv / (ms * 1e-3),
        "roofline": {"kernel": "prod_query_kernel + prod_scores_kernel (one tq_prod_scores call)", "bound": "hbm",
                     "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak, "peak_source": peak_src,
                     "ms_per_launch": ms, "algorithmic_bytes_per_launch": nbytes,
                     "traffic": _profile_field("tq_prod.cu", "prod_scores_prod.md", "dram_bytes_per_launch")},
        "store": {"kernel": "prod_store_kernel (tq_prod_store)", "tokens": STORE_TOKENS,
                  "mtok_s": STORE_TOKENS / (ms_store * 1e-3) / 1e6, "ms_per_launch": ms_store,
                  "roofline": {"bound": "tensor", "achieved": store_tflops, "peak": tpeak,
                               "unit": "TFLOP/s", "frac": store_tflops / tpeak,
                               "peak_source": tpeak_src + " (the projection runs on f16 operands, bf16's rate)",
                               "flops_per_launch": STORE_TOKENS * w.n_kv * 2 * w.d * w.d,
                               "traffic": _profile_field("tq_prod_store.cu", "prod_store_prod.md",
                                                         "dram_bytes_per_launch")}},
        "gpu_launches": 2 * reps + 20,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        code = _PROD_ORACLE_SCRIPT.format(root=ROOT, tokens=PROD_ORACLE_TOKENS, steps=30)
        out = subprocess.run([sys.executable, "-c", code], env=dict(os.environ, **_SINGLE_THREAD_ENV),
                             capture_output=True, text=True, check=True).stdout
        t = statistics.mean(json.loads(out.strip().splitlines()[-1])["times"][1:])
        obytes = PROD_ORACLE_TOKENS * w.n_kv * lay.slot_bytes + w.n_q * PROD_ORACLE_TOKENS * 4
        line["cpu_baseline"] = {"value": obytes / t / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                "keys_per_s": PROD_ORACLE_TOKENS * w.n_kv / t,
                                "sample": f"1 sequence x {PROD_ORACLE_TOKENS} positions, 8 KV heads x 4 query "
                                          "heads each: oracle prod_scores"}
    print(json.dumps(line), flush=True)
    return 0


CONT_CHUNK = 128


def run_continue(args):
    """``--op continue``: continuation chunks. 32 sequences, each a 4096-token
    cached history plus a 128-token chunk already stored (4224 positions, gqa
    heads: n_q 32, n_kv 8, 4bit_nc; 145 MB of packed slots, above L2), served
    by tq_continue (each KV tile read once per 64 / G = 16 queries) and, for
    comparison, by the per-query path: tq_decode with 4096 requests of lengths
    4097 .. 4224. Prints one JSON line of its own."""
    import torch

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    from turboquant_paged_kv_gb300 import build as tqbuild
    tqbuild.build()
    import turboquant_paged_kv_gb300 as tq
    import workloads

    base = workloads.get(DEFAULT_WORKLOAD)
    w = workloads.get(DEFAULT_WORKLOAD, fixed_len=base.fixed_len + CONT_CHUNK)
    inp = workloads.make_inputs(w, device=dev)
    cfg = tq.make_config(w.preset, w.n_q, w.n_kv, block_size=w.block_size)
    cb = tq.tq_build_codebook(w.d, 4)
    lay = tq.tq_layout_for(cfg)
    cache = torch.empty(inp.num_blocks * lay.block_bytes, dtype=torch.uint8, device=dev)
    for b in range(w.batch):
        k, v = inp.kv_for_sequence(b, dev)
        s0 = dict(inp.fill_order)[b]
        tq.tq_store(cfg, cb, k, v, inp.fill_slots[s0: s0 + k.shape[0]], cache)
    L = inp.max_seq_len
    total = w.batch * CONT_CHUNK
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    q = torch.randn(total, w.n_q, w.d, generator=g, device=dev).to(torch.bfloat16)
    qs = (torch.arange(w.batch + 1, dtype=torch.int32, device=dev) * CONT_CHUNK)
    out = torch.empty(total, w.n_q, w.d, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(tq.tq_continue_workspace_size(cfg, total, L), dtype=torch.uint8, device=dev)
    # per-query path: one decode request per chunk query
    lens_pq = (torch.arange(CONT_CHUNK, dtype=torch.int32, device=dev) + (L - CONT_CHUNK + 1)).repeat(w.batch)
    table_pq = inp.block_table.repeat_interleave(CONT_CHUNK, dim=0).contiguous()
    out_pq = torch.empty_like(out)
    ws_pq = torch.empty(tq.tq_decode_workspace_size(cfg, total, L), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def cont(_i=0):
        tq.tq_continue(cfg, cb, q, qs, CONT_CHUNK, cache, inp.block_table, inp.seq_lens, L, out, ws)

    def per_query(_i=0):
        tq.tq_decode(cfg, cb, q, cache, table_pq, lens_pq, L, out_pq, ws_pq)

    for _ in range(args.warmup):
        cont()
        per_query()
    torch.cuda.synchronize()
    err = (out.float() - out_pq.float()).abs().max().item()
    props = torch.cuda.get_device_properties(dev)
    gpu_id = ("GPU-" + str(props.uuid)) if getattr(props, "uuid", None) else "0"
    reps = max(args.steps, 50)
    with ClockSampler(gpu_id) as clk:
        ms = time_device(cont, reps, stream)
        ms_pq = time_device(per_query, max(reps // 10, 5), stream)
    peak, peak_src = _peaks()
    slot_bytes = w.n_kv * lay.slot_bytes
    unique = w.batch * L * slot_bytes                              # every cached slot once
    G = w.n_q // w.n_kv
    passes = -(-CONT_CHUNK * G // 64)                              # query groups of 64 / G queries
    cont_reads = sum(w.batch * min(L, L - CONT_CHUNK + min(CONT_CHUNK, 64 // G * (i + 1))) * slot_bytes
                     for i in range(passes))
    pq_reads = w.batch * sum(L - CONT_CHUNK + 1 + i for i in range(CONT_CHUNK)) * slot_bytes
    gbs = unique / (ms * 1e-3) / 1e9
    # algorithmic tensor work: every (query, query head) against every position it sees,
    # d multiply-adds for the score and d for the output (2 flops each)
    seen = w.batch * sum(L - CONT_CHUNK + 1 + i for i in range(CONT_CHUNK))
    flops = seen * w.n_q * w.d * 4
    tflops = flops / (ms * 1e-3) / 1e12
    tpeak, tpeak_src = _tensor_peak()
    print(json.dumps({
        "op": "continue", "metric": "continuation chunk queries/s (128-query chunks over 4096-token histories)",
        "value": total / (ms * 1e-3), "unit": "queries/s", "n_gpus": 1, "steps": reps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "dtype": "f32 softmax/accumulate, f16 tensor-core operands, bf16 in/out",
        "data": "synthetic",
        "config": {"workload": _workload_text(w, f", last {CONT_CHUNK} positions of each sequence are the chunk"),
                   "l2": "the packed cache is %.0f MB (> L2)" % (unique / 1e6)},
        "per_query_path": {"ms_per_step": ms_pq, "queries_per_s": total / (ms_pq * 1e-3),
                           "kernel": "tq_decode, one request per chunk query", "speedup_of_continue": ms_pq / ms,
                           "max_abs_diff_vs_continue": err},
        "kv_bytes_read": {"continue": cont_reads, "per_query": pq_reads, "unique": unique,
                          "ratio": pq_reads / cont_reads},
        "roofline": {"kernel": "cont_kernel + cont_reduce_kernel (one tq_continue call)", "bound": "tensor",
                     "achieved": tflops, "peak": tpeak, "unit": "TFLOP/s", "frac": tflops / tpeak,
                     "peak_source": tpeak_src, "ms_per_launch": ms, "algorithmic_flops_per_launch": flops,
                     "note": "flops = (query, query head) x visible position x d x 4 (QK and PV multiply-adds); "
                             "mma.sync f16 operands with fp16 hi/lo query and probability parts, so the tensor "
                             "pipe does twice the algorithmic work",
                     "traffic": _profile_field("tq_continue.cu", "continue_gqa.md", "dram_bytes_per_launch"),
                     "hbm": {"achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                             "bytes": unique, "note": "every packed slot once; the kernel reads the history "
                                                      f"{passes} times (once per query group), the repeats from L2"}},
        "gpu_launches": 2 * reps + 2 * max(reps // 10, 5),
        "clocks": clk.summary(),
    }), flush=True)
    return 0


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="tq", choices=["tq", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=WORKLOADS + ("all",))
    ap.add_argument("--partition", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--dry-run", action="store_true",
                    help="run the multi-rank host logic on the CPU (gloo) without a GPU")
    ap.add_argument("--op", default="decode", choices=["decode", "dequant", "store", "prod", "continue"],
                    help="decode: the decode step (default); dequant: tq_dequant of the gqa cache alone; "
                         "store: tq_store of the workload's prefill chunk alone; prod: the TurboQuant_prod "
                         "key path (scores + store); continue: 128-query continuation chunks")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    return args


def main(argv=None):
    argv = sys.argv[1:] if argv is None else list(argv)
    args = parse_args(argv)
    world, _, _ = _dist()
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        return launch_ranks(args.gpus, argv, args.dry_run)
    if "WORLD_SIZE" in os.environ and args.gpus != world:
        print(json.dumps({"error": f"--gpus {args.gpus} but the launcher started {world} ranks"}), flush=True)
        return 2
    if args.dry_run:
        return run_dry(args)
    if args.op == "dequant":
        return run_dequant(args)
    if args.op == "store":
        return run_store(args)
    if args.op == "prod":
        return run_prod(args)
    if args.op == "continue":
        return run_continue(args)
    return run_reference(args) if args.impl == "reference" else run_tq(args)


if __name__ == "__main__":
    sys.exit(main())
