"""Benchmark: paged KV-cache write + paged decode attention on one GB300.

One step = the batch's new tokens (one per sequence, the last token of its
context) written into the paged cache, then decode attention over the whole
paged context, on the Llama-3-8B-shaped decode workload (B=64, H=32,
KVH=8, D=128, block 16, context lengths uniform in [512, 4096], shuffled
physical blocks, garbage table tails, bf16), synthetic and seeded.  By
default a step is one pkv_write_decode_attention launch (`--mode
two-launch`: pkv_write, then pkv_decode_attention).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--workload NAME] [--mode fused|two-launch] [--no-graph]

Prints one JSON line.  `value` is the step's algorithmic bytes (K/V rows
used, q, out, table prefix, lengths, plus the write's rows and slots) per
second of device time over the K timed steps, all ranks together.  The K
timed steps are captured once as a CUDA graph and replayed, so the host's
launch rate stays out of the timed region (`--no-graph`: every step
launched from the host).  The `roofline` block is for the attention kernel
(with the write, when fused): its algorithmic bytes over its time per step
(graph: the replay's CUDA-event span over K; `--no-graph`: the mean of the
per-launch CUDA events on its stream), against the measured HBM copy
bandwidth.  `--impl reference` times
the oracle (plain fp64 C on the host cores) on bounded samples of the same
workload instead.  Under torchrun (N > 1) every rank runs its own
independent batch (weak scaling, no collective on the data path); time is
the max over ranks.  `--workload` picks another of the five workloads (the
per-step one cycles through its 32 steps).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from concurrent.futures import ThreadPoolExecutor

import torch
import torch.distributed as dist

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_67_gb300 import workloads as wl  # noqa: E402

METRIC = "paged decode attn achieved HBM GB/s (% of peak) + write_kv GB/s, 1×GB300"
WORKLOAD = "llama8b_bf16"
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------ helpers

WORKLOAD_TEXT = {
    "llama8b_bf16": ("B=64 H=32 KVH=8 D=128 block_size=16, context_lens U[512,4096], shuffled "
                     "blocks from a 1.25x pool, garbage table tails, q/k/v~N(0,1) bf16"),
    "long_bf16": ("B=8 H=32 KVH=8 D=128 block_size=16, context_lens U[16384,32768], shuffled "
                  "blocks, garbage table tails, bf16"),
    "mqa_bf16": ("B=128 H=16 KVH=1 D=256 block_size=32, context_lens log-uniform [1,8192], "
                 "shuffled blocks, garbage table tails, bf16"),
    "step_bf16": ("256 sequences (200 live, 56 padded: slot -1, length 0) H=64 KVH=8 D=128 "
                  "block_size=16, context_lens U[1,2048], 32 decode steps cycled, bf16"),
    "tiny_fp32": "B=4 H=4 KVH=2 D=64 block_size=16, context_lens U[1,100], fp32",
}


def config_block(workload=WORKLOAD, mode="fused", dec_bytes=None, wr_bytes=None, world=1,
                 graph=False):
    step = ("pkv_write_decode_attention (new token of every sequence written, then attention "
            "over the context that counts it, one launch)" if mode == "fused" else
            "pkv_write of the new tokens, then pkv_decode_attention")
    c = {"workload": f"{workload}: {WORKLOAD_TEXT[workload]}; step = {step}",
         "parallelism": f"{world} independent replica batch(es), no collective"}
    if graph:
        c["launch"] = "the timed steps replayed from one CUDA graph"
    if dec_bytes is not None:
        c["l2"] = f"inputs larger than L2 ({dec_bytes / 1e6:.0f} MB of K/V per step, no flush)"
        c["decode_bytes_per_step"] = dec_bytes
        c["write_bytes_per_step"] = wr_bytes
    return c


TRAFFIC_RECORDS = os.path.join("profiles", "decode_traffic.txt")


def decode_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    captures (one record per kernel and workload, `kernel | workload |
    sources_sha256 | bytes_per_launch`), or None when there is none for them
    or the kernel's sources have changed since it was taken."""
    path = os.path.join(ROOT, TRAFFIC_RECORDS)
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    for line in lines:
        if not line.strip() or line.lstrip().startswith("#"):
            continue
        parts = [x.strip() for x in line.split("|")]
        if len(parts) != 4 or parts[0] != kernel or parts[1] != workload:
            continue
        try:
            if parts[2] != sources_sha256(kernel):
                return None
            return int(parts[3])
        except (ValueError, OSError):
            return None
    return None


def code_only(text):
    """C/C++/CUDA source without its comments and with whitespace runs
    collapsed: what the compiler sees, so that a comment edit does not read
    as a kernel change."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


KERNEL_SOURCES = {
    "pkv_decode_tc_kernel": ("pkv_decode_tc.cu", "pkv_device.cuh"),
    "pkv_decode_wide_kernel": ("pkv_decode_wide.cu", "pkv_device.cuh", "pkv_tcgen05.cuh"),
    "pkv_decode_simt_kernel": ("pkv_decode_simt.cu", "pkv_device.cuh"),
    "pkv_decode_xpacked_kernel": ("pkv_decode_xpacked.cu", "pkv_device.cuh"),
}


def sources_sha256(kernel="pkv_decode_tc_kernel"):
    """Digest of what a decode kernel's launches are built from: its own
    file, the shared device headers it uses and the plan (partition
    choice) in the API file, comments left out."""
    import hashlib
    import re
    csrc = os.path.join(ROOT, "paged_kv_cache_67_gb300", "csrc")
    family = kernel.split("<")[0]
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[family]:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(code_only(fh.read()).encode())
    with open(os.path.join(csrc, "pkv_api.cu"), encoding="utf-8") as fh:
        api = fh.read()
    m = re.search(r"\nbool make_plan\(.*?\n}\n", api, re.S)
    h.update(code_only(m.group(0) if m else api).encode())
    return h.hexdigest()


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock and throttle samples, each stamped with the host's
    monotonic clock, from before the first warm-up to the end of the run.
    A timed region reports the samples inside it plus the nearest one on
    each side of it, so a region shorter than the sampling period (20 steps
    of ~0.1 ms) still has two.  Read-only queries: no GPU setting changes."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu = gpu_index
        self.period_ms = period_ms
        self.proc = None
        self.thread = None
        self.samples = []     # (monotonic seconds, csv line)
        self.lock = threading.Lock()

    def start(self, wait_s: float = 5.0):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
            return self
        t_end = time.monotonic() + wait_s
        while time.monotonic() < t_end and not self.samples and self.proc.poll() is None:
            time.sleep(0.01)
        return self

    def _read(self):
        for line in self.proc.stdout:
            with self.lock:
                self.samples.append((time.monotonic(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=5)
            self.proc = None

    def __enter__(self):
        return self.start()

    def __exit__(self, *exc):
        self.stop()

    def window(self, t0: float, t1: float, wait_s: float = 2.0):
        """Summary of the samples taken between t0 and t1 (monotonic), with
        the last one before t0 and the first one after t1 (waited for)."""
        if self.proc is not None:
            t_end = time.monotonic() + wait_s
            while time.monotonic() < t_end and self.proc.poll() is None:
                with self.lock:
                    if self.samples and self.samples[-1][0] > t1:
                        break
                time.sleep(0.005)
        with self.lock:
            samples = list(self.samples)
        inside = [ln for ts, ln in samples if t0 <= ts <= t1]
        before = [ln for ts, ln in samples if ts < t0][-1:]
        after = [ln for ts, ln in samples if ts > t1][:1]
        out = self.summarize(before + inside + after)
        out["inside_region"] = len(inside)
        return out

    @staticmethod
    def summarize(lines):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def aggregate(elapsed_s: float, units: float, world: int, device=None):
    """Whole-job throughput of weakly scaled ranks: every rank's units over
    the slowest rank's time (max over ranks)."""
    if world <= 1:
        return units / elapsed_s, elapsed_s, units
    t = torch.tensor([elapsed_s, units], dtype=torch.float64, device=device)
    tmax = t[:1].clone()
    dist.all_reduce(tmax, op=dist.ReduceOp.MAX)
    tsum = t[1:].clone()
    dist.all_reduce(tsum, op=dist.ReduceOp.SUM)
    return float(tsum.item()) / float(tmax.item()), float(tmax.item()), float(tsum.item())


def barrier(world):
    if world > 1:
        dist.barrier()


# ------------------------------------------------------------ CPU (oracle)

def oracle_units(inp):
    """(sequence, KV head) units: the oracle's bounded-sample granularity."""
    cfg = inp.cfg
    return [(b, kvh) for b in range(cfg.B) for kvh in range(cfg.KVH) if int(inp.context_lens[b]) > 0]


def unit_bytes(inp, b, elem):
    cfg = inp.cfg
    n = int(inp.context_lens[b])
    return 2 * n * cfg.D * elem + 2 * cfg.G * cfg.D * elem + (-(-n // cfg.bs)) * 4 + 4


def run_oracle_units(oracle, cpu, units, threads):
    """Decode the given (sequence, KV head) units with the oracle, one unit
    per task, on `threads` host threads (ctypes releases the GIL)."""
    cfg = cpu["cfg"]
    out = cpu["out"]

    def one(u):
        b, kvh = u
        oracle.decode(cpu["q"], cpu["k"], cpu["v"], cpu["tables"], cpu["lens"], cpu["scale"],
                      seqs=(b, b + 1), heads=(kvh * cfg.G, (kvh + 1) * cfg.G), out=out)

    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(one, units))


def cpu_copy(inp):
    return {"cfg": inp.cfg, "q": inp.q.cpu(), "k": inp.k_cache.cpu(), "v": inp.v_cache.cpu(),
            "tables": inp.block_tables.cpu(), "lens": inp.context_lens.cpu(), "scale": inp.scale,
            "out": torch.zeros(inp.q.shape, dtype=inp.q.dtype)}


def cpu_baseline(inp, elem, seconds=10.0):
    """The oracle on the host cores over the workload's units, repeated
    until `seconds` have passed (at least one unit)."""
    import oracle
    oracle.build()
    cpu = cpu_copy(inp)
    threads = max(1, min(os.cpu_count() or 1, 64))
    units = oracle_units(inp)
    g = torch.Generator().manual_seed(0)
    order = [units[i] for i in torch.randperm(len(units), generator=g).tolist()]
    done_bytes, done_units, t0 = 0, 0, time.perf_counter()
    i = 0
    while True:
        chunk = [order[(i + j) % len(order)] for j in range(threads)]
        run_oracle_units(oracle, cpu, chunk, threads)
        i += threads
        done_units += len(chunk)
        done_bytes += sum(unit_bytes(inp, b, elem) for b, _ in chunk)
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    # the same units on one thread, a shorter sample
    one_bytes, one_units, t1 = 0, 0, time.perf_counter()
    while True:
        b_u = order[(i + one_units) % len(order)]
        run_oracle_units(oracle, cpu, [b_u], 1)
        one_units += 1
        one_bytes += unit_bytes(inp, b_u[0], elem)
        if time.perf_counter() - t1 >= seconds / 3:
            break
    dt1 = time.perf_counter() - t1
    return {"value": done_bytes / dt / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": (f"{done_units} (sequence, KV head) units of the {inp.cfg.name} workload "
                       f"({done_units / len(units):.2f} decode passes over its {len(units)} units), "
                       f"fp64 C oracle, {dt:.1f} s on {threads} threads"),
            "single_thread": {"value": one_bytes / dt1 / 1e9, "unit": "GB/s",
                              "sample": f"{one_units} units on one thread, {dt1:.1f} s"}}


def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle
    oracle.build()
    cfg = wl.CONFIGS[args.workload]
    elem = torch.empty((), dtype=cfg.dtype).element_size()
    inp = wl.make_decode_inputs(cfg, seed=1234, device="cpu")
    cpu = cpu_copy(inp)
    threads = max(1, min(os.cpu_count() or 1, 64))
    units = oracle_units(inp)
    g = torch.Generator().manual_seed(1)
    order = [units[i] for i in torch.randperm(len(units), generator=g).tolist()]
    # each step: one unit per thread (a bounded sample of the batch)
    pos = 0

    def step():
        nonlocal pos
        chunk = [order[(pos + j) % len(order)] for j in range(threads)]
        pos += threads
        run_oracle_units(oracle, cpu, chunk, threads)
        return sum(unit_bytes(inp, b, elem) for b, _ in chunk)

    for _ in range(args.warmup):
        step()
    total, t0 = 0, time.perf_counter()
    for _ in range(args.steps):
        total += step()
    dt = time.perf_counter() - t0
    value = total / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / max(args.steps, 1) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_block(args.workload, args.mode),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle",
                         "sample": f"{threads} (sequence, KV head) units per step, rotating"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# -------------------------------------------------------------- GPU (lib)

DECODE_CONFIG_ORDER = ("long_bf16", "mqa_bf16", "step_bf16", "tiny_fp32")
KERNEL_CHOICES = {"auto": -1, "cuda-core": 0, "tc": 1, "wide": 2}


def make_step_inputs(cfg, inp, rank, dev, elem):
    """Device inputs of each distinct step (one for a single-step workload:
    the new token is the last of every context; the per-step workload's 32
    appends otherwise) with their algorithmic bytes."""
    steps = []
    if cfg.steps > 1:
        st = wl.make_steps(inp, seed=4321 + rank, device=dev)
        lens_c, slots_c = st.lens.cpu(), st.slots.cpu()
        for s in range(cfg.steps):
            steps.append(dict(q=st.q[s], k=st.k[s], v=st.v[s], slots=st.slots[s],
                              tables=st.tables[s], lens=st.lens[s],
                              dec=wl.decode_bytes(lens_c[s], cfg.B, cfg.H, cfg.KVH, cfg.D, cfg.bs, elem),
                              wr=wl.write_bytes(slots_c[s], cfg.KVH, cfg.D, elem)))
    else:
        positions = [int(n) - 1 if int(n) > 0 else None for n in inp.context_lens]
        wb = wl.make_write_batch(inp, positions, seed=4321 + rank, device=dev)
        steps.append(dict(q=inp.q, k=wb.k, v=wb.v, slots=wb.slot_mapping,
                          tables=inp.block_tables.to(dev), lens=inp.context_lens.to(dev),
                          dec=wl.decode_bytes(inp.context_lens, cfg.B, cfg.H, cfg.KVH, cfg.D,
                                              cfg.bs, elem),
                          wr=wl.write_bytes(wb.slot_mapping.cpu(), cfg.KVH, cfg.D, elem)))
    return steps


def max_context(cfg):
    """The host-side bound on the context lengths the bench passes as
    max_context_len: the longest first-step context, plus the appended
    tokens of a multi-step workload."""
    return cfg.len_hi + (cfg.steps if cfg.steps > 1 else 0)


def kernel_name(cfg, mode, kernel=-1):
    import paged_kv_cache_67_gb300 as pkv
    P, _, kern = pkv.pkv_decode_plan(cfg.B, cfg.H, cfg.KVH, cfg.D, cfg.bs, cfg.table_width,
                                     max_context(cfg), dtype=cfg.dtype)
    if kernel >= 0:
        kern = kernel
    t = {torch.bfloat16: "bf16", torch.float16: "fp16", torch.float32: "fp32"}[cfg.dtype]
    if kern == 2:  # the fused step on this kernel is pkv_write followed by it
        return f"pkv_decode_wide_kernel<{cfg.D}, {t}>"
    base = f"pkv_decode_tc_kernel<{cfg.D}, {t}" if kern == 1 else f"pkv_decode_simt_kernel<{t}"
    return base + (", append>" if mode == "fused" else ">")


def l2_bytes(dev):
    try:
        return int(torch.cuda.get_device_properties(dev).L2_cache_size)
    except Exception:
        return 126 * 2**20


class DecodeRun:
    """One decode workload on the GPU, as the bench times it: `copies`
    independent input sets (each with its cache pool, tables, queries and
    the step inputs) cycled step by step, one output buffer, one workspace.
    A step is pkv_write_decode_attention (mode "fused") or pkv_write then
    pkv_decode_attention (mode "two-launch", where `kernel` >= 0 names the
    decode kernel); layout "xpacked" runs the packed-layout pair."""

    def __init__(self, pkv, name, dev, rank, mode="fused", kernel=-1, copies=1,
                 layout="token-major"):
        self.pkv, self.name, self.dev = pkv, name, dev
        self.cfg = cfg = wl.CONFIGS[name]
        self.elem = torch.empty((), dtype=cfg.dtype).element_size()
        self.mode, self.kernel, self.layout = mode, kernel, layout
        self.fused = mode == "fused" and layout == "token-major"
        self.sets = []
        for c in range(copies):
            seed = 1234 + rank + 7919 * c
            inp = wl.make_decode_inputs(cfg, seed=seed, device=dev)
            steps = make_step_inputs(cfg, inp, rank + 7919 * c, dev, self.elem)
            kx = vx = None
            if layout == "xpacked":
                nb = inp.k_cache.shape[0]
                kx = inp.k_cache.view(nb, cfg.bs, cfg.KVH, cfg.D // 8, 8).permute(0, 2, 3, 1, 4).contiguous()
                vx = inp.v_cache.permute(0, 2, 3, 1).contiguous()
            self.sets.append(dict(inp=inp, steps=steps, kx=kx, vx=vx))
        self.order = [(c, s) for s in range(len(self.sets[0]["steps"])) for c in range(copies)]
        self.inp = self.sets[0]["inp"]
        self.out = torch.empty_like(self.inp.q)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.max_ctx = max_context(cfg)
        self.ws = pkv.DecodeWorkspace(cfg.B, cfg.H, cfg.KVH, cfg.D, cfg.bs, cfg.table_width,
                                      self.max_ctx, 0, device=dev)
        self.kname = (kernel_name(cfg, mode, kernel) if layout == "token-major" else
                      f"pkv_decode_xpacked_kernel<{cfg.D}, bf16>")
        # launches per step: the fused entry is one
        self.launches_per_step = 1 if self.fused else 2

    def entry(self, i):
        c, s = self.order[i % len(self.order)]
        return self.sets[c], self.sets[c]["steps"][s]

    def step_bytes(self, i):
        _, st = self.entry(i)
        return st["dec"] + st["wr"]

    def kernel_bytes(self, i):
        """Algorithmic bytes of the timed decode launch (the write's too when
        the step is fused)."""
        _, st = self.entry(i)
        return st["dec"] + (st["wr"] if self.fused else 0)

    def write(self, i, stream):
        set_, st = self.entry(i)
        inp = set_["inp"]
        if set_["kx"] is not None:
            self.pkv.pkv_write_xpacked(set_["kx"], set_["vx"], st["k"], st["v"], st["slots"],
                                       err_flags=self.err, stream=stream)
        else:
            self.pkv.pkv_write(inp.k_cache, inp.v_cache, st["k"], st["v"], st["slots"],
                               err_flags=self.err, stream=stream)

    def decode(self, i, stream):
        pkv = self.pkv
        set_, st = self.entry(i)
        inp = set_["inp"]
        kw = dict(max_context_len=self.max_ctx, workspace=self.ws, err_flags=self.err, stream=stream)
        if set_["kx"] is not None:
            pkv.pkv_decode_attention_xpacked(self.out, st["q"], set_["kx"], set_["vx"], st["tables"],
                                             st["lens"], inp.scale, **kw)
        elif self.fused:
            pkv.pkv_write_decode_attention(self.out, st["q"], st["k"], st["v"], st["slots"],
                                           inp.k_cache, inp.v_cache, st["tables"], st["lens"],
                                           inp.scale, **kw)
        elif self.kernel >= 0:
            pkv.pkv_decode_attention_with_kernel(self.out, st["q"], inp.k_cache, inp.v_cache,
                                                 st["tables"], st["lens"], inp.scale, self.kernel, **kw)
        else:
            pkv.pkv_decode_attention(self.out, st["q"], inp.k_cache, inp.v_cache, st["tables"],
                                     st["lens"], inp.scale, **kw)

    def step(self, i, stream, ev=None):
        if not self.fused:
            self.write(i, stream)
        if ev is not None:
            ev[0].record(stream)
        self.decode(i, stream)
        if ev is not None:
            ev[1].record(stream)

    def check_flags(self, when):
        if int(self.err.item()) != 0:
            raise RuntimeError(f"{self.name}: device error flags {int(self.err.item()):#x} {when}")

    def warmup(self, n, stream):
        for i in range(max(n, len(self.order))):
            self.step(i, stream)
        torch.cuda.synchronize()
        self.check_flags("during warm-up")

    def time_graph(self, steps, stream, world, sampler):
        """The timed steps captured once as a CUDA graph and replayed between
        CUDA events on the launching stream: (elapsed s, clocks)."""
        cap = torch.cuda.Stream(self.dev)
        cap.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(graph, stream=cap):
                for i in range(steps):
                    self.step(i, cap)
        torch.cuda.synchronize()
        t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        h0 = time.monotonic()
        torch.cuda.nvtx.range_push("timed")
        t_start.record(stream)
        graph.replay()
        t_end.record(stream)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
        h1 = time.monotonic()
        barrier(world)
        self.check_flags("in the timed region")
        del graph
        return t_start.elapsed_time(t_end) * 1e-3, sampler.window(h0, h1)

    def time_launches(self, steps, stream, world, sampler, flush=None):
        """Every timed step launched from the host, the decode launch between
        its own CUDA events on its stream; with `flush` (a buffer larger than
        L2) the buffer is rewritten before every step, outside the events.
        Returns (elapsed s, mean decode ms, median decode ms, clocks)."""
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        h0 = time.monotonic()
        torch.cuda.nvtx.range_push("timed")
        t_start.record(stream)
        for i in range(steps):
            if flush is not None:
                flush.add_(1)
            self.step(i, stream, evs[i])
        t_end.record(stream)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
        h1 = time.monotonic()
        barrier(world)
        self.check_flags("in the timed region")
        ms = [a.elapsed_time(b) for a, b in evs]
        return (t_start.elapsed_time(t_end) * 1e-3, statistics.mean(ms), statistics.median(ms),
                sampler.window(h0, h1))


def flop_per_byte(cfg):
    """Decode arithmetic per byte of K/V read: per key and value row of D
    elements, 2 * D flops of scores and 2 * D of weighted sum for each of
    the G = H / KVH query heads, over 2 * D * element bytes."""
    el = torch.empty((), dtype=cfg.dtype).element_size()
    return round(2 * (cfg.H // cfg.KVH) / el, 2)


def config_entry(run, args, stream, world, sampler, peak, flush):
    """One workload of the `configs` block: its decode kernel timed at the
    run's K and W, against the HBM peak.  Without `flush` the timed steps
    are replayed from one CUDA graph (the run's input sets, cycled, are
    larger than L2); with it every step is launched from the host after the
    L2 is flushed."""
    run.warmup(args.warmup, stream)
    cycle_bytes = sum(run.step_bytes(i) for i in range(len(run.order)))
    if not flush:
        elapsed, clocks = run.time_graph(args.steps, stream, world, sampler)
        kern_ms = elapsed * 1e3 / args.steps
        timing = (f"{args.steps} steps replayed from one CUDA graph; "
                  + (f"{len(run.sets)} independent input sets cycled, " if len(run.sets) > 1 else "")
                  + f"inputs larger than L2 ({cycle_bytes / len(run.order) / 1e6:.0f} MB per step"
                  + (f", {cycle_bytes / 1e6:.0f} MB per cycle" if len(run.sets) > 1 else "")
                  + "), no flush")
    else:
        buf = torch.zeros(2 * l2_bytes(run.dev) // 4 + 1, dtype=torch.float32, device=run.dev)
        elapsed, _, kern_ms, clocks = run.time_launches(args.steps, stream, world, sampler, buf)
        timing = (f"{args.steps} host-launched steps, a {buf.numel() * 4 / 1e6:.0f} MB buffer "
                  f"rewritten before each (L2 flush), CUDA events around each decode launch "
                  f"(median)")
        del buf
    kb = statistics.mean(run.kernel_bytes(i) for i in range(args.steps))
    achieved = kb / (kern_ms * 1e-3) / 1e9
    gather = None if flush else measure_gather(run.pkv, run, stream)
    traffic = decode_traffic(run.kname, run.name)
    if traffic is not None and len(run.sets) > 1:
        # the record is of the first input set: scaled to the cycle's mean bytes
        traffic = round(traffic * kb / run.kernel_bytes(0))
    return {
        "workload": f"{run.name}: {WORKLOAD_TEXT[run.name]}",
        "step": "pkv_write_decode_attention" if run.fused else "pkv_write + pkv_decode_attention",
        "kernel": run.kname, "kernel_us": round(kern_ms * 1e3, 2),
        "bytes_per_launch": round(kb), "achieved": round(achieved, 1), "unit": "GB/s",
        "peak": peak, "frac": round(achieved / peak, 4), "bound": "hbm",
        "traffic": traffic, "flop_per_byte": flop_per_byte(run.cfg),
        "ms_per_step": round(elapsed * 1e3 / args.steps, 4), "timing": timing,
        "gpu_launches": args.steps * run.launches_per_step, "clocks": clocks,
        **({"gather_read_gbs": gather["gbs"],
            "frac_of_gather_read": round(achieved / gather["gbs"], 4),
            "gather_what": gather["what"] + ("; the first input set" if len(run.sets) > 1 else "")}
           if gather else {}),
    }


def measure_copy(pkv, dev, stream):
    """In-run copy bandwidth of 1 GiB buffers: the library's own copy kernel
    (pkv_hbm_copy), and torch's copy_ for context; read + write bytes."""
    src = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    dst = torch.empty_like(src)
    res = {}
    for name, fn in (("pkv_hbm_copy", lambda: pkv.pkv_hbm_copy(dst, src, stream=stream)),
                     ("torch_copy", lambda: dst.copy_(src))):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(10)]
        for a, b in evs:
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        ms = min(a.elapsed_time(b) for a, b in evs)
        res[name] = round(2 * src.numel() / (ms * 1e-3) / 1e9, 1)
    del src, dst
    return res


def measure_fma(pkv, dev, stream):
    """In-run fp32 multiply-add rate of the CUDA cores (pkv_fp32_fma_peak:
    eight blocks of 256 threads per SM, eight chains per thread), plain fmaf
    and paired fma.rn.f32x2; TFLOP/s, best of 5 launches of ~1 ms."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    out = torch.empty(8 * sms, dtype=torch.float32, device=dev)
    iters = 16384
    flops = out.numel() * pkv.FMA_THREADS * pkv.FMA_CHAINS * iters * 2
    res = {}
    for name, paired in (("fmaf", False), ("fma_f32x2", True)):
        for _ in range(3):
            pkv.pkv_fp32_fma_peak(out, iters, 1.0, 1.0, paired=paired, stream=stream)
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(5)]
        for a, b in evs:
            a.record(stream)
            pkv.pkv_fp32_fma_peak(out, iters, 1.0, 1.0, paired=paired, stream=stream)
            b.record(stream)
        torch.cuda.synchronize()
        ms = min(a.elapsed_time(b) for a, b in evs)
        res[name] = round(flops / (ms * 1e-3) / 1e12, 1)
    if not torch.equal(out.cpu(), torch.full_like(out.cpu(), float(pkv.FMA_CHAINS * iters))):
        raise RuntimeError("pkv_fp32_fma_peak: chains did not reach their exact value")
    return {"fmaf_tflops": res["fmaf"], "fma_f32x2_tflops": res["fma_f32x2"],
            "tflops": max(res.values()),
            "what": f"pkv_fp32_fma_peak: {out.numel()} blocks x {pkv.FMA_THREADS} threads x "
                    f"{pkv.FMA_CHAINS} chains x {iters} multiply-adds, best of 5"}


def gather_orders(pkv, dev, stream):
    """The gather yardstick over the 8B-shaped batch's blocks in three
    orders -- table order (the pages' random placement), sorted by physical
    block, and one contiguous run of the pool -- K and V one launch each;
    GB/s, best of 10.  Prints one JSON line."""
    cfg = wl.CONFIGS["llama8b_bf16"]
    inp = wl.make_decode_inputs(cfg, seed=1234, device=dev)
    lens = [int(x) for x in inp.context_lens]
    blocks = [blk for b, n in enumerate(lens) for blk in inp.owned[b][:-(-n // cfg.bs)]]
    bb = cfg.bs * cfg.KVH * cfg.D * torch.empty((), dtype=cfg.dtype).element_size()
    sink = torch.zeros(1, dtype=torch.int64, device=dev)
    res = {"workload": "llama8b_bf16 (seed 1234)", "blocks": len(blocks),
           "pool_blocks": int(inp.k_cache.shape[0]), "unit": "GB/s"}
    for name, order in (("table_order", blocks), ("sorted", sorted(blocks)),
                        ("contiguous", list(range(len(blocks))))):
        idx = torch.tensor(order, dtype=torch.int32, device=dev)

        def both():
            for cache in (inp.k_cache, inp.v_cache):
                pkv.pkv_hbm_gather_read(cache, idx, bb, bb, sink, stream=stream, check_bounds=False)

        for _ in range(3):
            both()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(10)]
        for a, b in evs:
            a.record(stream)
            both()
            b.record(stream)
        torch.cuda.synchronize()
        ms = min(a.elapsed_time(b) for a, b in evs)
        res[name] = round(2 * len(order) * bb / (ms * 1e-3) / 1e9, 1)
    print(json.dumps(res), flush=True)


def measure_gather(pkv, run, stream):
    """In-run read bandwidth of the batch's own access pattern without the
    arithmetic: every cache block the first input set's sequences use (K
    then V), whole, in table order, read in one launch (as the decode reads
    them) by pkv_hbm_gather_read_pair; best of 10."""
    inp, cfg = run.inp, run.cfg
    lens = [int(x) for x in inp.context_lens]
    blocks = [blk for b, n in enumerate(lens) for blk in inp.owned[b][:-(-n // cfg.bs)]]
    idx = torch.tensor(blocks, dtype=torch.int32, device=run.dev)
    block_bytes = cfg.bs * cfg.KVH * cfg.D * run.elem
    sink = torch.zeros(1, dtype=torch.int64, device=run.dev)
    pkv.pkv_hbm_gather_read_pair(inp.k_cache, inp.v_cache, idx, block_bytes, block_bytes, sink,
                                 stream=stream)

    def both():
        pkv.pkv_hbm_gather_read_pair(inp.k_cache, inp.v_cache, idx, block_bytes, block_bytes, sink,
                                     stream=stream, check_bounds=False)

    for _ in range(3):
        both()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(10)]
    for a, b in evs:
        a.record(stream)
        both()
        b.record(stream)
    torch.cuda.synchronize()
    ms = min(a.elapsed_time(b) for a, b in evs)
    nbytes = 2 * len(blocks) * block_bytes
    return {"gbs": round(nbytes / (ms * 1e-3) / 1e9, 1), "bytes": nbytes, "blocks": len(blocks),
            "what": (f"every cache block the {cfg.name} batch uses ({len(blocks)} blocks of "
                     f"{block_bytes} B, K then V), whole, in table order, by the library's "
                     f"gather-read kernel in one launch (pkv_hbm_gather_read_pair): the batch's access pattern "
                     f"without the arithmetic; best of 10")}


def run_gpu(args, world, rank, local):
    from paged_kv_cache_67_gb300 import build as libbuild
    import paged_kv_cache_67_gb300 as pkv

    libbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    peak, peak_kind = hbm_peak()
    sampler = ClockSampler(local).start()
    try:
        return _run_gpu(args, world, rank, dev, stream, peak, peak_kind, sampler, pkv)
    finally:
        sampler.stop()


def _run_gpu(args, world, rank, dev, stream, peak, peak_kind, sampler, pkv):
    run = DecodeRun(pkv, args.workload, dev, rank, mode=args.mode,
                    kernel=KERNEL_CHOICES[args.kernel], layout=args.layout)
    cfg, inp = run.cfg, run.inp
    extra = {}
    if not args.only_decode:
        # write_kv on a bulk fill (every context token of the batch): GB/s
        bulk = wl.make_bulk_fill(inp, seed=99 + rank, device=dev)
        bulk_bytes = wl.write_bytes(bulk.slot_mapping, cfg.KVH, cfg.D, run.elem)

        def bulk_write():
            pkv.pkv_write(inp.k_cache, inp.v_cache, bulk.k, bulk.v, bulk.slot_mapping,
                          err_flags=run.err, stream=stream)

        for _ in range(3):
            bulk_write()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(20)]
        for a, b in evs:
            a.record(stream)
            bulk_write()
            b.record(stream)
        torch.cuda.synchronize()
        bulk_ms = statistics.median(a.elapsed_time(b) for a, b in evs)
        bulk_gbs = bulk_bytes / (bulk_ms * 1e-3) / 1e9
        extra["write_kv"] = {"value": round(bulk_gbs, 1), "unit": "GB/s",
                             "frac": round(bulk_gbs / peak, 4), "tokens": int(bulk.slot_mapping.numel()),
                             "bytes": bulk_bytes, "us": round(bulk_ms * 1e3, 2),
                             "what": "bulk fill: every context token of the workload, random order"}
        del bulk  # the pool now holds the bulk-fill values; the decode reads those
        copy = measure_copy(pkv, dev, stream)
        if args.layout == "token-major":
            extra["gather_read_in_run"] = measure_gather(pkv, run, stream)
        extra["hbm_copy_gbs_in_run"] = copy["pkv_hbm_copy"]
        extra["hbm_copy_in_run"] = {"pkv_hbm_copy_gbs": copy["pkv_hbm_copy"],
                                    "torch_copy_gbs": copy["torch_copy"],
                                    "what": "1 GiB buffers, read + write bytes, best of 10, "
                                            "pkv_hbm_copy is the library's own copy kernel"}
        extra["fma_fp32_in_run"] = measure_fma(pkv, dev, stream)

    run.warmup(args.warmup, stream)
    if args.graph:
        elapsed, clocks = run.time_graph(args.steps, stream, world, sampler)
        dec_ms = elapsed * 1e3 / args.steps  # back-to-back graph nodes: the per-step time
    else:
        elapsed, dec_ms, _, clocks = run.time_launches(args.steps, stream, world, sampler)
    step_bytes = [run.step_bytes(i) for i in range(args.steps)]
    value, tmax, _ = aggregate(elapsed, sum(step_bytes) / 1e9, world, dev)
    kern_bytes = statistics.mean(run.kernel_bytes(i) for i in range(args.steps))
    dec_bytes = statistics.mean(st["dec"] for st in run.sets[0]["steps"])
    wr_bytes = statistics.mean(st["wr"] for st in run.sets[0]["steps"])

    e2e = None
    if not args.only_decode:
        e2e = run_e2e(args, world, dev, pkv, run, stream, sum(step_bytes))

    achieved = kern_bytes / (dec_ms * 1e-3) / 1e9
    configs = None
    if args.configs == "all" and not args.only_decode and args.layout == "token-major":
        configs = run_configs(args, world, rank, dev, stream, peak, sampler, pkv, exclude=args.workload)
    if rank != 0:
        return None
    cpu = None
    if world == 1 and not args.only_decode and not args.no_cpu_baseline:
        cpu = cpu_baseline(inp, run.elem)
    dt = {torch.bfloat16: "bf16", torch.float16: "fp16", torch.float32: "fp32"}[cfg.dtype]
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tmax / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dt, "data": "synthetic",
        "config": config_block(args.workload, run.mode, round(dec_bytes), round(wr_bytes), world,
                               args.graph),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": decode_traffic(run.kname, args.workload),
                     "kernel": run.kname, "bytes_per_launch": round(kern_bytes),
                     "peak_source": ("measured (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                                     else "fallback 6.8 TB/s"),
                     "kernel_us": round(dec_ms * 1e3, 2), "flop_per_byte": flop_per_byte(cfg),
                     **({"frac_of_gather_read": round(achieved / extra["gather_read_in_run"]["gbs"], 4)}
                        if "gather_read_in_run" in extra else {})},
        **extra,
        "e2e": e2e,
        "gpu_launches": args.steps * run.launches_per_step,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    if configs is not None:
        line["configs"] = configs
    print(json.dumps(line), flush=True)
    return line


def input_sets(cfg, rank, dev):
    """(input sets, flush) for timing a workload without a warm L2: one set
    when a step's bytes exceed twice L2; else enough independent sets (up to
    four) that one cycle of them does; else one set and an L2 flush before
    every step."""
    elem = torch.empty((), dtype=cfg.dtype).element_size()
    lens = wl.draw_lengths(cfg, 1234 + rank)
    per_set = wl.decode_bytes(lens, cfg.B, cfg.H, cfg.KVH, cfg.D, cfg.bs, elem)
    need = 2 * l2_bytes(dev)
    if per_set > need:
        return 1, False
    copies = -(-need // max(per_set, 1)) + 1
    return (copies, False) if copies <= 4 else (1, True)


def run_configs(args, world, rank, dev, stream, peak, sampler, pkv, exclude):
    """The other workloads at the same K and W: one entry each."""
    out = {}
    for name in DECODE_CONFIG_ORDER:
        if name == exclude:
            continue
        copies, flush = input_sets(wl.CONFIGS[name], rank, dev)
        run = DecodeRun(pkv, name, dev, rank, mode="fused", copies=copies)
        out[name] = config_entry(run, args, stream, world, sampler, peak, flush)
        del run
        torch.cuda.empty_cache()
    for name in sorted(wl.PREFILL_CONFIGS):
        out[name] = prefill_entry(args, world, rank, dev, stream, sampler, pkv, name)
        torch.cuda.empty_cache()
    return out


def prefill_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]), float(pk["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 1900.0, 1700.0, "fallback"


def prefill_timed(args, world, rank, dev, stream, sampler, pkv, name):
    """Causal varlen prefill over the paged cache, each launch between CUDA
    events: (cfg, inputs, flops per launch, elapsed s, mean ms, clocks)."""
    cfg = wl.PREFILL_CONFIGS[name]
    inp = wl.make_prefill_inputs(cfg, seed=1234 + rank, device=dev)
    tables, cu, lens = inp.block_tables.to(dev), inp.cu_seqlens_q.to(dev), inp.context_lens.to(dev)
    out = torch.empty_like(inp.q)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    flops = wl.prefill_flops(inp.context_lens, inp.cu_seqlens_q, cfg.H, cfg.D)

    def step():
        pkv.pkv_prefill_attention(out, inp.q, inp.k_cache, inp.v_cache, tables, cu, lens, inp.scale,
                                  max_q_len=inp.max_q_len, err_flags=err, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    h0 = time.monotonic()
    t_start.record(stream)
    for a, b in evs:
        a.record(stream)
        step()
        b.record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    h1 = time.monotonic()
    barrier(world)
    if int(err.item()) != 0:
        raise RuntimeError(f"{name}: device error flags {int(err.item()):#x}")
    elapsed = t_start.elapsed_time(t_end) * 1e-3
    k_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    return cfg, inp, flops, elapsed, k_ms, sampler.window(h0, h1)


def prefill_text(name, cfg, inp):
    return (f"{name}: B={cfg.B} H={cfg.H} KVH={cfg.KVH} D={cfg.D} block_size={cfg.bs}, "
            f"context_lens U[{cfg.len_lo},{cfg.len_hi}], even sequences prefill the whole prompt, "
            f"odd ones a chunk of U[{cfg.chunk_lo},{cfg.chunk_hi}] queries on a cached prefix; "
            f"{int(inp.cu_seqlens_q[-1])} queries")


def prefill_entry(args, world, rank, dev, stream, sampler, pkv, name):
    cfg, inp, flops, elapsed, k_ms, clocks = prefill_timed(args, world, rank, dev, stream, sampler,
                                                           pkv, name)
    peak, peak_s, src = prefill_peaks()
    achieved = flops / (k_ms * 1e-3) / 1e12
    return {"workload": prefill_text(name, cfg, inp), "step": "pkv_prefill_attention",
            "kernel": f"pkv_prefill_tc_kernel<{cfg.D}, bf16>", "kernel_us": round(k_ms * 1e3, 2),
            "flops_per_launch": flops, "achieved": round(achieved, 1), "unit": "TFLOP/s",
            "peak": peak, "frac": round(achieved / peak, 4),
            "frac_of_sustained": round(achieved / peak_s, 4), "bound": "tensor",
            "peak_source": f"{src} (MEASURED_PEAKS.json bf16_tflops)", "traffic": None,
            "ms_per_step": round(elapsed * 1e3 / args.steps, 4),
            "timing": (f"{args.steps} host-launched launches, CUDA events around each (mean); "
                       "q, out and K/V larger than L2, no flush"),
            "gpu_launches": args.steps, "clocks": clocks}


def run_prefill(args, world, rank, local):
    """Causal varlen prefill attention over the paged cache: TFLOP/s of the
    tensor-core kernel against the measured bf16 matmul peak."""
    from paged_kv_cache_67_gb300 import build as libbuild
    import paged_kv_cache_67_gb300 as pkv

    libbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(local).start()
    try:
        cfg, inp, flops, elapsed, k_ms, clocks = prefill_timed(args, world, rank, dev, stream,
                                                               sampler, pkv, args.workload)
    finally:
        sampler.stop()
    value, tmax, _ = aggregate(elapsed, flops * args.steps / 1e12, world, dev)
    if rank != 0:
        return None
    peak, peak_s, src = prefill_peaks()
    achieved = flops / (k_ms * 1e-3) / 1e12
    line = {
        "metric": "paged causal prefill attn achieved TFLOP/s", "value": round(value, 1),
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tmax / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": prefill_text(args.workload, cfg, inp),
                   "flops_per_step": flops,
                   "l2": "q, out and K/V larger than L2, no flush"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "frac_of_sustained": round(achieved / peak_s, 4), "traffic": None,
                     "kernel": f"pkv_prefill_tc_kernel<{cfg.D}, bf16>",
                     "peak_source": f"{src} (MEASURED_PEAKS.json bf16_tflops)",
                     "kernel_us": round(k_ms * 1e3, 2)},
        "e2e": None, "gpu_launches": args.steps, "clocks": clocks, "cpu_baseline": None,
    }
    print(json.dumps(line), flush=True)
    return line


def run_e2e(args, world, dev, pkv, run, stream, total_bytes):
    """The same steps end to end through the public API: each step's inputs
    copied in from pinned host memory, the output landing in pinned host
    memory and waited for.

    A step's inputs sit in one pinned host buffer (each tensor at a 256-byte
    aligned offset) and go over in one copy (a prepared pkv_copy_async) into a
    device buffer that the kernels read through views, the way a serving loop
    stages a batch; the fused step is a prepared call on those views (its
    checks and argument marshalling done once, as a loop that reuses its
    buffers would) whose output is the pinned host buffer itself: the kernel
    stores the result across to the host, with no copy after the launch."""
    steps = run.sets[0]["steps"]
    inp, out, ws, err, max_ctx = run.inp, run.out, run.ws, run.err, run.max_ctx
    S = len(steps)
    keys = ("q", "k", "v", "slots", "tables", "lens")
    offs, off = {}, 0
    for k in keys:
        offs[k] = off
        off += (steps[0][k].numel() * steps[0][k].element_size() + 255) // 256 * 256
    blob_bytes = off

    def views(buf):
        return {k: buf[offs[k]:offs[k] + steps[0][k].numel() * steps[0][k].element_size()]
                .view(steps[0][k].dtype).view(steps[0][k].shape) for k in keys}

    host = []
    for s in range(S):
        hb = torch.empty(blob_bytes, dtype=torch.uint8).pin_memory()
        for k, t in views(hb).items():
            t.copy_(steps[s][k].cpu())
        host.append(hb)
    dblob = torch.empty(blob_bytes, dtype=torch.uint8, device=dev)
    dbuf = views(dblob)
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = blob_bytes
    d2h = h_out.numel() * h_out.element_size()

    # the fused step through a prepared call: checked and marshalled once,
    # then enqueued every step on the same (refilled) device buffers
    fused_call = None
    if run.fused:
        fused_call = pkv.prepare_write_decode_attention(
            h_out, dbuf["q"], dbuf["k"], dbuf["v"], dbuf["slots"], inp.k_cache, inp.v_cache,
            dbuf["tables"], dbuf["lens"], inp.scale, max_context_len=max_ctx, workspace=ws,
            err_flags=err, stream=stream)

    copy_in = [pkv.prepare_copy_async(dblob, hb, stream=stream) for hb in host]

    def e2e_step(i):
        copy_in[i % S]()
        if fused_call is not None:
            fused_call()
        else:
            pkv.pkv_write(inp.k_cache, inp.v_cache, dbuf["k"], dbuf["v"], dbuf["slots"],
                          err_flags=err, stream=stream)
            pkv.pkv_decode_attention(h_out, dbuf["q"], inp.k_cache, inp.v_cache, dbuf["tables"],
                                     dbuf["lens"], inp.scale, max_context_len=max_ctx,
                                     workspace=ws, err_flags=err, stream=stream)
        stream.synchronize()  # the caller reads the result every step

    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup, S)):
            e2e_step(i)
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(args.steps):
            e2e_step(i)
        torch.cuda.synchronize()
        e2e_elapsed = time.perf_counter() - t0
    barrier(world)
    e2e_value, _, _ = aggregate(e2e_elapsed, total_bytes / 1e9, world, dev)
    return {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="lib", choices=["lib", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only-decode", action="store_true",
                    help="warm-up + timed steps only (no bulk fill, e2e, CPU baseline or other "
                         "workloads): for profiling")
    ap.add_argument("--workload", default=WORKLOAD,
                    choices=sorted(wl.CONFIGS) + sorted(wl.PREFILL_CONFIGS),
                    help="the batch the steps run on (default: the Llama-3-8B-shaped decode)")
    ap.add_argument("--configs", default="all", choices=["all", "none"],
                    help="all (default): also time every other workload at the same steps and "
                         "warm-up, one entry each under `configs`")
    ap.add_argument("--mode", default="fused", choices=["fused", "two-launch"],
                    help="fused: one pkv_write_decode_attention launch per step; two-launch: "
                         "pkv_write then pkv_decode_attention")
    ap.add_argument("--kernel", default="auto", choices=sorted(KERNEL_CHOICES),
                    help="with --mode two-launch: the decode kernel to run instead of the plan's "
                         "(pkv_decode_attention_with_kernel), to compare kernels on one batch")
    ap.add_argument("--graph", dest="graph", action="store_true", default=True,
                    help="replay the timed steps from one CUDA graph (the default)")
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="launch every timed step from the host, each decode launch between "
                         "its own CUDA events")
    ap.add_argument("--gather-orders", action="store_true",
                    help="only the gather yardstick over the 8B-shaped batch's blocks in table "
                         "order, sorted and contiguous (one JSON line)")
    ap.add_argument("--layout", default="token-major", choices=["token-major", "xpacked"],
                    help="xpacked: the layout experiment (caches in vLLM's packed layout, "
                         "write + decode in two launches; with --only-decode)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.layout == "xpacked" and not args.only_decode:
        ap.error("--layout xpacked goes with --only-decode")
    if args.layout == "xpacked":
        args.mode = "two-launch"
    if args.kernel != "auto" and args.mode != "two-launch":
        ap.error("--kernel goes with --mode two-launch")
    world, rank, local = dist_setup()
    try:
        if args.gather_orders:
            if rank == 0:
                from paged_kv_cache_67_gb300 import build as libbuild
                import paged_kv_cache_67_gb300 as pkv
                libbuild.build()
                torch.cuda.set_device(local)
                dev = torch.device("cuda", local)
                gather_orders(pkv, dev, torch.cuda.current_stream(dev))
        elif args.impl == "reference":
            run_reference(args, world, rank)
        elif args.workload in wl.PREFILL_CONFIGS:
            run_prefill(args, world, rank, local)
        else:
            run_gpu(args, world, rank, local)
    finally:
        if world > 1 and dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
