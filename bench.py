"""Benchmark: paged KV-cache write + paged decode attention on one GB300.

One step = pkv_write of the batch's new tokens (one per sequence, the last
token of its context) followed by pkv_decode_attention over the whole paged
context, on the Llama-3-8B-shaped decode workload (B=64, H=32, KVH=8,
D=128, block 16, context lengths uniform in [512, 4096], shuffled physical
blocks, garbage table tails, bf16), synthetic and seeded.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line.  `value` is the step's algorithmic bytes (K/V rows
used, q, out, table prefix, lengths, plus the write's rows and slots) per
second of device time over the K timed steps, all ranks together.  The
`roofline` block is for the decode kernel alone: its algorithmic bytes over
its mean launch time from CUDA events on its stream, against the measured
HBM copy bandwidth.  `--impl reference` times the oracle (plain fp64 C on
the host cores) on bounded samples of the same workload instead.
Under torchrun (N > 1) every rank runs its own independent batch (weak
scaling, no collective on the data path); time is the max over ranks.
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

def config_block(dec_bytes=None, wr_bytes=None, world=1):
    c = {"workload": (f"{WORKLOAD}: B=64 H=32 KVH=8 D=128 block_size=16, context_lens "
                      "U[512,4096], shuffled blocks from a 1.25x pool, garbage table tails, "
                      "q/k/v~N(0,1) bf16; step = pkv_write of 64 new tokens + "
                      "pkv_decode_attention"),
         "parallelism": f"{world} independent replica batch(es), no collective"}
    if dec_bytes is not None:
        c["l2"] = f"inputs larger than L2 ({dec_bytes / 1e6:.0f} MB of K/V per step, no flush)"
        c["decode_bytes_per_step"] = dec_bytes
        c["write_bytes_per_step"] = wr_bytes
    return c


def decode_traffic():
    """DRAM bytes per decode launch from the committed ncu capture, or None
    when the decode kernel's sources have changed since it was taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "decode_traffic.txt")
    try:
        rec = dict(line.split() for line in open(path) if line.strip() and not line.startswith("#"))
        h = hashlib.sha256()
        for f in ("pkv_decode_tc.cu", "pkv_device.cuh", "pkv_api.cu"):
            with open(os.path.join(ROOT, "paged_kv_cache_67_gb300", "csrc", f), "rb") as fh:
                h.update(fh.read())
        return int(rec["bytes_per_launch"]) if h.hexdigest() == rec["sources_sha256"] else None
    except Exception:
        return None


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
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
    return {"value": done_bytes / dt / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": (f"{done_units} (sequence, KV head) units of the {WORKLOAD} workload "
                       f"({done_units / len(units):.2f} decode passes over its {len(units)} units), "
                       f"fp64 C oracle, {dt:.1f} s on {threads} threads")}


def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle
    oracle.build()
    cfg = wl.CONFIGS[WORKLOAD]
    elem = 2
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
        "config": dict(config_block(), sample=f"{threads} (sequence, KV head) units per step"),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle",
                         "sample": f"{threads} (sequence, KV head) units per step, rotating"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# -------------------------------------------------------------- GPU (lib)

def run_gpu(args, world, rank, local):
    from paged_kv_cache_67_gb300 import build as libbuild
    import paged_kv_cache_67_gb300 as pkv

    libbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = wl.CONFIGS[WORKLOAD]
    elem = 2
    inp = wl.make_decode_inputs(cfg, seed=1234 + rank, device=dev)
    positions = [int(n) - 1 for n in inp.context_lens]
    wb = wl.make_write_batch(inp, positions, seed=4321 + rank, device=dev)
    tables = inp.block_tables.to(dev)
    lens = inp.context_lens.to(dev)
    q = inp.q
    out = torch.empty_like(q)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    max_ctx = cfg.len_hi
    ws = pkv.DecodeWorkspace(cfg.B, cfg.H, cfg.KVH, cfg.D, cfg.bs, cfg.table_width, max_ctx, 0,
                             device=dev)
    stream = torch.cuda.current_stream(dev)
    dec_bytes = wl.decode_bytes(inp.context_lens, cfg.B, cfg.H, cfg.KVH, cfg.D, cfg.bs, elem)
    wr_bytes = wl.write_bytes(wb.slot_mapping, cfg.KVH, cfg.D, elem)
    step_bytes = dec_bytes + wr_bytes
    peak, peak_kind = hbm_peak()

    def write():
        pkv.pkv_write(inp.k_cache, inp.v_cache, wb.k, wb.v, wb.slot_mapping, err_flags=err,
                      stream=stream)

    def decode():
        pkv.pkv_decode_attention(out, q, inp.k_cache, inp.v_cache, tables, lens, inp.scale,
                                 max_context_len=max_ctx, workspace=ws, err_flags=err,
                                 stream=stream)

    extra = {}
    if not args.only_decode:
        # write_kv on a bulk fill (every context token, ~147k tokens): GB/s
        bulk = wl.make_bulk_fill(inp, seed=99 + rank, device=dev)
        bulk_bytes = wl.write_bytes(bulk.slot_mapping, cfg.KVH, cfg.D, elem)

        def bulk_write():
            pkv.pkv_write(inp.k_cache, inp.v_cache, bulk.k, bulk.v, bulk.slot_mapping,
                          err_flags=err, stream=stream)

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

        # in-run copy bandwidth of a 1 GiB buffer (context for the measured peak)
        src = torch.empty(1 << 29, dtype=torch.bfloat16, device=dev)
        dst = torch.empty_like(src)
        for _ in range(3):
            dst.copy_(src)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(10):
            dst.copy_(src)
        e1.record(stream)
        torch.cuda.synchronize()
        extra["hbm_copy_gbs_in_run"] = round(10 * 2 * src.numel() * 2 / (e0.elapsed_time(e1) * 1e-3) / 1e9, 1)
        del src, dst

    # warm-up
    for _ in range(args.warmup):
        write()
        decode()
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error flags {int(err.item()):#x} during warm-up")

    # timed region: K steps; each decode launch bracketed by events on its stream
    dec_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("timed")
    with ClockSampler(local) as clocks:
        t_start.record(stream)
        for i in range(args.steps):
            write()
            dec_ev[i][0].record(stream)
            decode()
            dec_ev[i][1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    barrier(world)
    elapsed = t_start.elapsed_time(t_end) * 1e-3
    dec_ms = statistics.mean(a.elapsed_time(b) for a, b in dec_ev)
    launches = 2 * args.steps
    if int(err.item()) != 0:
        raise RuntimeError(f"device error flags {int(err.item()):#x} in the timed region")
    value, tmax, _ = aggregate(elapsed, step_bytes * args.steps / 1e9, world, dev)

    e2e = None
    if not args.only_decode:
        # end to end through the public API: pinned host inputs in, result out
        h_q = q.cpu().pin_memory()
        h_k, h_v = wb.k.cpu().pin_memory(), wb.v.cpu().pin_memory()
        h_slots = wb.slot_mapping.cpu().pin_memory()
        h_tables, h_lens = inp.block_tables.cpu().pin_memory(), inp.context_lens.cpu().pin_memory()
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        d_q, d_k, d_v = torch.empty_like(q), torch.empty_like(wb.k), torch.empty_like(wb.v)
        d_slots, d_tables, d_lens = (torch.empty_like(wb.slot_mapping), torch.empty_like(tables),
                                     torch.empty_like(lens))
        h2d = sum(t.numel() * t.element_size() for t in (h_q, h_k, h_v, h_slots, h_tables, h_lens))
        d2h = h_out.numel() * h_out.element_size()

        def e2e_step():
            d_q.copy_(h_q, non_blocking=True)
            d_k.copy_(h_k, non_blocking=True)
            d_v.copy_(h_v, non_blocking=True)
            d_slots.copy_(h_slots, non_blocking=True)
            d_tables.copy_(h_tables, non_blocking=True)
            d_lens.copy_(h_lens, non_blocking=True)
            pkv.pkv_write(inp.k_cache, inp.v_cache, d_k, d_v, d_slots, err_flags=err, stream=stream)
            pkv.pkv_decode_attention(out, d_q, inp.k_cache, inp.v_cache, d_tables, d_lens, inp.scale,
                                     max_context_len=max_ctx, workspace=ws, err_flags=err,
                                     stream=stream)
            h_out.copy_(out, non_blocking=True)
            stream.synchronize()  # the caller reads the result every step

        for _ in range(max(3, args.warmup)):
            e2e_step()
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            e2e_step()
        torch.cuda.synchronize()
        e2e_elapsed = time.perf_counter() - t0
        barrier(world)
        e2e_value, _, _ = aggregate(e2e_elapsed, step_bytes * args.steps / 1e9, world, dev)
        e2e = {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h}

    achieved = dec_bytes / (dec_ms * 1e-3) / 1e9
    if rank != 0:
        return None
    cpu = None
    if world == 1 and not args.only_decode and not args.no_cpu_baseline:
        cpu = cpu_baseline(inp, elem)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tmax / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_block(dec_bytes, wr_bytes, world),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": decode_traffic(),
                     "kernel": "pkv_decode_tc_kernel<128, bf16>",
                     "peak_source": ("measured (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                                     else "fallback 6.8 TB/s"),
                     "decode_us": round(dec_ms * 1e3, 2)},
        **extra,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks.summary(),
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="lib", choices=["lib", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only-decode", action="store_true",
                    help="warm-up + timed steps only (no bulk fill, e2e or CPU baseline): for profiling")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_gpu(args, world, rank, local)
    finally:
        if world > 1 and dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
