#!/usr/bin/env python
"""Bench of the GB300 DLRMv1 inference forward (samples/s and us/batch).

A step is one dlrm_forward over one batch of the named synthetic workload
(default: batch 2048, bottom 13-512-256-64, 3 tables x 100k x 64, one index
per bag, top 70-512-256-1, fp32). Timing: W untimed warm-up steps, then K
steps, each preceded by an L2 flush (a 256 MB write, larger than the 129 MB
L2) and timed with CUDA events on the launching stream; the K event times are
summed. One JSON line on stdout (rank 0).

Extra objects on the line:
  e2e        the same metric through dlrm_forward_host (pinned host buffers,
             H2D of dense/indices/offsets and D2H of the output in the timed
             region)
  graph      the forward captured once in a CUDA graph and replayed
  stages_us  per-stage device time from the library's event profiling mode
  roofline   the dominant stage against its bound (FP32 FFMA peak from SM
             count x 128 lanes x 2 x 2070 MHz, or measured HBM GB/s)
  configs    the forward on the other workloads (64-sample 3-table, 2048-sample
             32-table, the 11 x 5 batch x tables sweep, and the 65536-sample
             26-table Zipf workload): us/batch, samples/s, plan, whole-forward
             roofline fraction
  gather_b65536_k26_zipf  the standalone multi-table gather on the 13.3 GB
             26-table workload (bags of 20, Zipf(1.05)) plus a uniform-index
             control, algorithmic GB/s against measured HBM GB/s; under
             "general_bags" the same tables through embedding_bag_multi with
             bags of random lengths 0..40 over general offsets, sum / mean / max
  cpu_baseline  the CPU oracle (fp64, all host cores) on a bounded sample

--impl reference times the CPU oracle as the reference arm (there is no
runnable reference implementation; the pages hold no code for this path).
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "DLRM fwd samples/sec & µs/batch at bs=2048; gather HBM GB/s vs roofline"
UNIT = "samples/s"
FLUSH_BYTES = 256 << 20
FP32_LANES_PER_SM = 128
SM_MAX_MHZ_DEFAULT = 2070.0
# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one ncu
# capture of the kernel as built now on the named workload; a kernel change
# invalidates the entry.
NCU_TRAFFIC = {("fused", "b2048_k3"): 3175168}
# DRAM bytes (read + write) of one standalone gather launch on the full 26 x 1M x 128
# tables, bags of 20 (ncu dram__bytes_read.sum + dram__bytes_write.sum, one pass):
# table-major bag order lets repeats of a row within a table's pass hit L2, so the
# DRAM traffic is below the algorithmic bytes even for uniform indices
NCU_GATHER_DRAM = {"zipf": 3.33e9 + 0.858e9, "uniform": 15.07e9 + 0.869e9}


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="b2048_k3")
    ap.add_argument("--math", choices=["fp32", "fp32_ffma", "tf32", "bf16", "tf32x3"],
                    default="fp32",
                    help="arithmetic of the timed model's MLPs (fp32 is the parity mode)")
    ap.add_argument("--config-math", choices=["fp32", "fp32_ffma", "tf32", "bf16", "tf32x3"],
                    default="fp32",
                    help="arithmetic of the other workloads' forwards under `configs` (their "
                         "roofline fraction is against the pipes their plan uses)")
    ap.add_argument("--seed", type=int, default=1234)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads' forward measurements")
    ap.add_argument("--no-gather", action="store_true",
                    help="skip the 13.3 GB standalone-gather measurement")
    ap.add_argument("--profile-steps", type=int, default=200)
    ap.add_argument("--path", choices=["auto", "fused", "layerwise"], default="auto",
                    help="kernel plan of the forward handle (default: the library's choice)")
    ap.add_argument("--only-gather", action="store_true",
                    help="time only the standalone gathers of the 26-table workload "
                         "(uniform bags of 20 and general bags, Zipf and uniform indices)")
    ap.add_argument("--gather-rows", type=int, default=0,
                    help="rows per table for --only-gather (default: the workload's 1M; "
                         "smaller tables keep an ncu capture to a few GB)")
    ap.add_argument("--only-forward", action="store_true",
                    help="time the device forward only (for ncu launch lists)")
    ap.add_argument("--rows", type=int, default=0,
                    help="rows per table of the timed model (default: the workload's; "
                         "smaller tables keep an ncu capture to a few GB)")
    ap.add_argument("--batch", type=int, default=0,
                    help="batch of the timed model (default: the workload's)")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm_gbs=float(p["hbm_gbs"]), bf16_tflops=float(p["bf16_tflops"]),
                    sm_max_mhz=float(p.get("sm_max_mhz", SM_MAX_MHZ_DEFAULT)), source="measured")
    except Exception:
        return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, sm_max_mhz=SM_MAX_MHZ_DEFAULT,
                    source="fallback")


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.windows = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def mark(self, t0: float, t1: float):
        self.windows.append((t0, t1))

    def finish(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        return summarise_clocks(out, self.windows)


THROTTLES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def summarise_clocks(text: str, windows) -> dict:
    """SM clocks and active throttle reasons from `nvidia-smi --query-gpu=
    ClockSampler.FIELDS --format=csv,noheader,nounits` rows, keeping the samples
    inside the timed windows (epoch seconds, +-0.15 s; all samples when none
    fall inside). `verdict` names a run these clocks would reject: a hardware or
    thermal slowdown, or a median SM clock below 90% of max with no reason
    active (a clock lock left by someone); sw_power_cap is kept and noted."""
    rows = []
    for rec in csv.reader(io.StringIO(text)):
        if len(rec) < 10:
            continue
        try:
            ts = time.mktime(time.strptime(rec[0].strip().split(".")[0], "%Y/%m/%d %H:%M:%S"))
            frac = float("0." + rec[0].strip().split(".")[1]) if "." in rec[0] else 0.0
            rows.append(dict(t=ts + frac, sm=float(rec[2]), smax=float(rec[3]),
                             power=float(rec[4]) if rec[4].strip() not in ("", "[N/A]") else None,
                             hw=rec[6].strip(), hwt=rec[7].strip(), swt=rec[8].strip(),
                             swp=rec[9].strip()))
        except Exception:
            continue
    inside = [r for r in rows if any(a - 0.15 <= r["t"] <= b + 0.15 for a, b in windows)]
    used = inside if inside else rows
    if not used:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
    reasons = set()
    for r in used:
        for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                          ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
            if r[key].lower().startswith("active"):
                reasons.add(name)
    med = statistics.median(r["sm"] for r in used)
    smax = max(r["smax"] for r in used)
    bad = [name for name in THROTTLES if name in reasons]
    if bad:
        verdict = "rejected: " + ", ".join(bad)
    elif med < 0.9 * smax and "sw_power_cap" not in reasons:
        verdict = "rejected: SM clock below max with no reason active (a clock lock?)"
    else:
        verdict = "ok"
    return {"sm_mhz": med, "sm_max_mhz": smax, "reasons": sorted(reasons), "verdict": verdict,
            "samples": len(used), "samples_in_timed_region": len(inside)}


# ---------------------------------------------------------------- oracle timing

def time_oracle(inp, batch, budget_s, max_samples=None, threads=None):
    """Oracle samples/s on a bounded sample: whole batches (or a prefix of one)
    repeated until budget_s of CPU time has run, on `threads` host threads (all
    cores by default)."""
    import numpy as np
    import oracle
    lib = oracle.load()
    threads = threads or os.cpu_count() or 1
    probe_ids = np.arange(min(batch, 64))
    t0 = time.perf_counter()
    oracle.forward(inp, sample_ids=probe_ids, threads=threads, lib=lib)
    per_sample = max((time.perf_counter() - t0) / len(probe_ids), 1e-7)
    n = int(min(batch, max(1, budget_s / per_sample / 2)))
    if max_samples:
        n = min(n, max_samples)
    ids = np.arange(n)
    done, t_start = 0, time.perf_counter()
    reps = 0
    while True:
        oracle.forward(inp, sample_ids=ids, threads=threads, lib=lib)
        done += n
        reps += 1
        if time.perf_counter() - t_start >= budget_s:
            break
    dt = time.perf_counter() - t_start
    return dict(value=done / dt, unit=UNIT, cores=threads, kind="oracle",
                sample=f"{n} of {batch} samples x {reps} repetitions ({dt:.1f} s, fp64, "
                       f"{threads} thread{'s' if threads != 1 else ''})")


# ---------------------------------------------------------------- ranks

def max_over_ranks(local_ms: float, dist=None, device=None) -> float:
    """The slowest rank's timed total (every rank gets it); the local value
    on a single process. NCCL ranks pass their CUDA device, gloo ranks none."""
    if dist is None:
        return local_ms
    import torch
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, samples_per_rank: int, steps: int, total_ms: float) -> float:
    """Whole-job samples/s: every rank's samples over the slowest rank's time."""
    return world * samples_per_rank * steps / (total_ms * 1e-3)


# ---------------------------------------------------------------- reference arm

def run_reference(args, rank, world):
    if rank != 0:
        return 0
    import numpy as np
    import dlrm_synth as synth
    import oracle
    cfg = synth.get_config(args.config)
    if args.batch > 0:
        cfg = cfg.with_batch(args.batch)
    if args.rows > 0:
        cfg = synth.DlrmConfig(cfg.name, cfg.batch, cfg.ln_bot, (args.rows,) * cfg.n_tables,
                               cfg.emb_dim, cfg.bag_size, cfg.ln_top, cfg.table_range,
                               cfg.index_dist, cfg.zipf_s)
    inp = synth.make_inputs(cfg, seed=args.seed)
    lib = oracle.load()
    threads = os.cpu_count() or 1
    probe = np.arange(min(cfg.batch, 32))
    t0 = time.perf_counter()
    oracle.forward(inp, sample_ids=probe, threads=threads, lib=lib)
    per_sample = max((time.perf_counter() - t0) / len(probe), 1e-7)
    budget = 120.0 / max(1, args.steps + args.warmup)       # whole run within ~2 minutes
    n = int(max(1, min(cfg.batch, budget / per_sample)))
    ids = np.arange(n)
    for _ in range(args.warmup):
        oracle.forward(inp, sample_ids=ids, threads=threads, lib=lib)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.forward(inp, sample_ids=ids, threads=threads, lib=lib)
    dt = time.perf_counter() - t0
    value = n * args.steps / dt
    line = dict(metric=METRIC, value=value, unit=UNIT, impl="reference", n_gpus=world,
                steps=args.steps, warmup=args.warmup, ms_per_step=dt * 1e3 / args.steps,
                higher_is_better=True, scaling="weak", vs_baseline=None, dtype="f64",
                data="synthetic (seeded SplitMix64 inputs)",
                config=dict(workload=cfg.name, global_batch=cfg.batch, batch_per_gpu=cfg.batch,
                            tables=cfg.n_tables, rows=cfg.rows[0], emb_dim=cfg.emb_dim,
                            bag_size=cfg.bag_size, ln_bot=list(cfg.ln_bot),
                            ln_top=list(cfg.ln_top), math="fp64 (oracle)",
                            parallelism="rank 0 only"),
                cpu_baseline=dict(kind="oracle", cores=threads, value=value, unit=UNIT,
                                  sample=f"{n} of {cfg.batch} samples per step (fp64 CPU "
                                         f"oracle, {threads} threads)"),
                e2e=dict(value=value, unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0),
                note="reference arm = the CPU oracle; the pages ship no runnable code")
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm

def stage_work(cfg, name, batch):
    """Algorithmic (flops, bytes) of one stage launch."""
    k, d, l = cfg.n_tables, cfg.emb_dim, cfg.bag_size
    f = k + 1
    p = f * (f - 1) // 2
    if name == "gather":
        byts = batch * k * l * d * 4 + batch * k * l * 8 + batch * k * 8 + batch * k * d * 4
        return batch * k * (l - 1) * d, byts
    if name == "interaction":
        return 2 * batch * p * d, batch * f * d * 4 + batch * (d + p) * 4
    if name == "fused":
        return forward_work(cfg, batch)
    widths = cfg.ln_bot if name.startswith("bottom") else cfg.ln_top
    i = int(name[len("bottom"):] if name.startswith("bottom") else name[len("top"):])
    kin, nout = widths[i], widths[i + 1]
    return 2 * batch * kin * nout, 4 * (batch * kin + kin * nout + nout + batch * nout)


def forward_work(cfg, batch):
    """Algorithmic (flops, bytes) of one whole forward: every GEMM's 2*M*N*K, the
    pair dots and bag adds; HBM bytes of the inputs, tables rows, weights and output."""
    k, d, l = cfg.n_tables, cfg.emb_dim, cfg.bag_size
    f = k + 1
    p = f * (f - 1) // 2
    flops = batch * k * (l - 1) * d + 2 * batch * p * d
    w_bytes = 0
    for widths in (cfg.ln_bot, cfg.ln_top):
        for a, b in zip(widths[:-1], widths[1:]):
            flops += 2 * batch * a * b
            w_bytes += 4 * (a * b + b)
    byts = batch * (k * l * d * 4 + k * l * 8 + k * 8 + cfg.n_dense * 4 + 4) + w_bytes
    return flops, byts


def forward_roofline_parts(cfg, plan, math, fp32_peak_tflops, pk):
    """Roofline time of one forward on the pipes its plan uses: the GEMM layers
    the layer-wise plan runs on the tensor cores (plan["tensor_core_layers"])
    at the tensor rate of their arithmetic (split-TF32: three tf32 products per
    fp32 product; TF32 taken as half the measured bf16 peak, the nominal
    ratio), every other flop at the FP32 FFMA peak, against the algorithmic
    HBM bytes: max(tensor + FFMA time, HBM time)."""
    import dlrm_embedding_interaction_gb300 as dl
    flops, byts = forward_work(cfg, cfg.batch)
    layers = list(zip(cfg.ln_bot[:-1], cfg.ln_bot[1:])) + list(zip(cfg.ln_top[:-1], cfg.ln_top[1:]))
    mask = plan["tensor_core_layers"]
    tc_flops = sum(2 * cfg.batch * k * n for g, (k, n) in enumerate(layers) if (mask >> g) & 1)
    if plan["split_tf32"]:
        tc_time, what = 3 * tc_flops / (pk["bf16_tflops"] * 0.5 * 1e12), "split-TF32"
    elif math == dl.MATH_BF16:
        tc_time, what = tc_flops / (pk["bf16_tflops"] * 1e12), "bf16"
    else:
        tc_time, what = tc_flops / (pk["bf16_tflops"] * 0.5 * 1e12), "tf32"
    alu_time = (flops - tc_flops) / (fp32_peak_tflops * 1e12)
    hbm_time = byts / (pk["hbm_gbs"] * 1e9)
    if hbm_time >= tc_time + alu_time:
        bound = "hbm"
    elif tc_flops:
        bound = f"tensor ({what} GEMM layers) + FP32 FFMA (the rest)"
    else:
        bound = "alu (FP32 FFMA)"
    return dict(roofline_us=max(tc_time + alu_time, hbm_time) * 1e6, bound=bound,
                tensor_core_layers=[g for g in range(len(layers)) if (mask >> g) & 1])


def device_tables(torch, synth, cfg, seed, n=None):
    """The workload's first n tables from the seeded generator, filled on the host
    one at a time into a reused pinned buffer and copied to the current device."""
    n = cfg.n_tables if n is None else n
    host = torch.empty((max(cfg.rows[:n]), cfg.emb_dim), dtype=torch.float32).pin_memory()
    out = []
    for t in range(n):
        h = host[:cfg.rows[t]]
        synth.make_table(cfg, seed, t, out=h.numpy())
        out.append(h.to("cuda"))
    del host
    return out


def gather_measure(torch, dl, synth, pk, tables, steps=10, cfg=None):
    """Standalone gather on the 26 x 1M x 128 workload (bags of 20), Zipf and uniform."""
    cfg = cfg or synth.get_config("b65536_k26_zipf")
    off = torch.from_numpy(synth.make_offsets(cfg)).cuda()
    out = torch.empty((cfg.batch, cfg.n_tables, cfg.emb_dim), device="cuda")
    _, byts = stage_work(cfg, "gather", cfg.batch)
    res = {}
    for dist in ("zipf", "uniform"):
        c = cfg if dist == "zipf" else synth.DlrmConfig(
            cfg.name, cfg.batch, cfg.ln_bot, cfg.rows, cfg.emb_dim, cfg.bag_size, cfg.ln_top)
        idx = torch.from_numpy(synth.make_indices(c, 1234)).cuda()
        s = torch.cuda.current_stream()
        for _ in range(3):
            dl.embedding_bag_sum_multi(tables, idx, off, out, cfg.bag_size, stream=s)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        torch.cuda.synchronize()
        for a, b in ev:
            a.record(s)
            dl.embedding_bag_sum_multi(tables, idx, off, out, cfg.bag_size, stream=s)
            b.record(s)
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(b) for a, b in ev) / steps
        gbs = byts / (ms * 1e-3) / 1e9
        # repeated rows are served from L2 (Zipf's hot rows; with uniform indices the
        # repeats within a table's pass): the algorithmic ratio is not an HBM fraction,
        # the DRAM bytes ncu counted on this workload give that
        res[dist] = dict(ms_per_launch=ms, algorithmic_gbs=gbs,
                         algorithmic_over_measured_hbm_l2_served=gbs / pk["hbm_gbs"])
        full = cfg.name == "b65536_k26_zipf" and cfg.rows[0] == 1_000_000
        dram = NCU_GATHER_DRAM.get(dist) if full else None
        if dram is not None:
            dgbs = dram / (ms * 1e-3) / 1e9
            res[dist].update(dram_bytes_ncu=dram, dram_gbs=dgbs,
                             dram_frac_of_measured_hbm=dgbs / pk["hbm_gbs"],
                             dram_frac_of_nominal_8tbs=dgbs / 8000.0)
        del idx
    del out
    torch.cuda.empty_cache()
    return dict(workload=f"{cfg.n_tables} tables x {cfg.rows[0]} x {cfg.emb_dim} fp32 "
                         f"({cfg.n_tables * cfg.rows[0] * cfg.emb_dim * 4 / 1e9:.1f} GB), "
                         f"batch {cfg.batch}, bags of {cfg.bag_size}",
                bytes_per_launch=byts, launches_timed=steps,
                note="inputs far larger than L2; algorithmic bytes = rows + indices + offsets "
                     "+ output; bags run table-major, so rows repeated within a table's "
                     "pass (Zipf's hot rows, and some uniform repeats) are served from L2; "
                     "dram_* from ncu's DRAM byte counters on this workload", **res)


def bag_modes_measure(torch, dl, synth, pk, tables, steps=10, cfg=None):
    """embedding_bag_multi on the 26 x 1M x 128 tables: bags of random lengths 0..40
    (mean 20, empty bags included) over general offsets, sum / mean / max, Zipf and
    uniform indices."""
    cfg = cfg or synth.get_config("b65536_k26_zipf")
    out = torch.empty((cfg.batch, cfg.n_tables, cfg.emb_dim), device="cuda")
    modes = {"sum": dl.BAG_SUM, "mean": dl.BAG_MEAN, "max": dl.BAG_MAX}
    res = {}
    for dist in ("zipf", "uniform"):
        c = cfg if dist == "zipf" else synth.DlrmConfig(
            cfg.name, cfg.batch, cfg.ln_bot, cfg.rows, cfg.emb_dim, cfg.bag_size, cfg.ln_top)
        idx_h, off_h, lens = synth.make_variable_bags(c, 1234, 40)
        n_idx = idx_h.shape[1]
        rows_read = int(lens.sum())
        # algorithmic bytes: rows read + all indices + offsets + the (B, K, D) output
        byts = (rows_read * cfg.emb_dim * 4 + cfg.n_tables * n_idx * 8
                + cfg.n_tables * cfg.batch * 8 + cfg.batch * cfg.n_tables * cfg.emb_dim * 4)
        idx, off = torch.from_numpy(idx_h).cuda(), torch.from_numpy(off_h).cuda()
        del idx_h, off_h
        s = torch.cuda.current_stream()
        per = {}
        for name, mode in modes.items():
            for _ in range(3):
                dl.embedding_bag_multi(tables, idx, off, out, mode, stream=s)
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(steps)]
            torch.cuda.synchronize()
            for a, b in ev:
                a.record(s)
                dl.embedding_bag_multi(tables, idx, off, out, mode, stream=s)
                b.record(s)
            torch.cuda.synchronize()
            ms = sum(a.elapsed_time(b) for a, b in ev) / steps
            gbs = byts / (ms * 1e-3) / 1e9
            per[name] = {"ms_per_launch": ms, "algorithmic_gbs": gbs,
                         "algorithmic_over_measured_hbm_l2_served": gbs / pk["hbm_gbs"]}
        res[dist] = dict(bytes_per_launch=byts, mean_bag=rows_read / (cfg.batch * cfg.n_tables),
                         **per)
        del idx, off
    del out
    torch.cuda.empty_cache()
    return dict(workload=f"{cfg.n_tables} tables x {cfg.rows[0]} x {cfg.emb_dim} fp32, batch "
                         f"{cfg.batch}, bag lengths uniform on 0..40 (general offsets)",
                launches_timed=steps, **res)


def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch

    import dlrm_embedding_interaction_gb300 as dl
    import dlrm_synth as synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    pk = peaks()
    if args.only_gather:
        c4 = synth.get_config("b65536_k26_zipf")
        if args.gather_rows > 0:
            c4 = synth.DlrmConfig(c4.name, c4.batch, c4.ln_bot, (args.gather_rows,) * c4.n_tables,
                                  c4.emb_dim, c4.bag_size, c4.ln_top, c4.table_range,
                                  c4.index_dist, c4.zipf_s)
        tabs = device_tables(torch, synth, c4, args.seed)
        gather = gather_measure(torch, dl, synth, pk, tabs, cfg=c4)
        gather["general_bags"] = bag_modes_measure(torch, dl, synth, pk, tabs, cfg=c4)
        if rank == 0:
            print(json.dumps(dict(metric=METRIC, mode="only-gather",
                                  gather_b65536_k26_zipf=gather)), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return 0
    cfg = synth.get_config(args.config)
    if args.batch > 0:
        cfg = cfg.with_batch(args.batch)
    if args.rows > 0:
        cfg = synth.DlrmConfig(cfg.name, cfg.batch, cfg.ln_bot, (args.rows,) * cfg.n_tables,
                               cfg.emb_dim, cfg.bag_size, cfg.ln_top, cfg.table_range,
                               cfg.index_dist, cfg.zipf_s)
    inp = synth.make_inputs(cfg, seed=args.seed)
    cu = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    maths = {"fp32": dl.MATH_FP32, "fp32_ffma": dl.MATH_FP32_FFMA, "tf32": dl.MATH_TF32,
             "bf16": dl.MATH_BF16,
             "tf32x3": dl.MATH_TF32X3}
    math = maths[args.math]
    config_math = maths[args.config_math]
    plan = {"auto": dl.PATH_AUTO, "fused": dl.PATH_FUSED, "layerwise": dl.PATH_LAYERWISE}[args.path]
    model = dl.DlrmModel(cfg.ln_bot, cfg.ln_top, [cu(t) for t in inp["tables"]],
                         [cu(w) for w in inp["bot_w"]], [cu(b) for b in inp["bot_b"]],
                         [cu(w) for w in inp["top_w"]], [cu(b) for b in inp["top_b"]],
                         cfg.bag_size, cfg.batch, math, plan)
    dense, idx, off = cu(inp["dense"]), cu(inp["indices"]), cu(inp["offsets"])
    out = torch.empty(cfg.batch, device=dev)
    flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    # the kernels the timed forward runs (an AUTO fp32 handle on the fused plan
    # takes the layer-wise plan from its crossover batch)
    kind = model.kernels(cfg.batch)
    path_used = dl.PATH_LAYERWISE if kind == dl.KERNELS_LAYERWISE else dl.PATH_FUSED
    n_stages = (len(cfg.ln_bot) + len(cfg.ln_top)) if path_used == dl.PATH_LAYERWISE else 1

    def barrier():
        if dist is not None:
            dist.barrier()

    def timed(step_fn, k, w):
        with torch.cuda.stream(stream):
            for _ in range(w):
                flush_buf.zero_()
                step_fn()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(k)]
            torch.cuda.synchronize()
            barrier()
            torch.cuda.synchronize()
            t0 = time.time()
            for a, b in ev:
                flush_buf.zero_()
                a.record(stream)
                step_fn()
                b.record(stream)
            torch.cuda.synchronize()
            barrier()
            torch.cuda.synchronize()
            t1 = time.time()
        ms = [a.elapsed_time(b) for a, b in ev]
        return ms, (t0, t1)

    clocks = ClockSampler(local_rank)
    time.sleep(1.0)          # let nvidia-smi start sampling

    # device-resident forward (the headline value)
    ms, win = timed(lambda: model.forward(dense, idx, off, out, stream=stream),
                    args.steps, args.warmup)
    clocks.mark(*win)
    if model.error(stream) != dl.OK:
        raise RuntimeError("device error during the timed forward")
    if args.only_forward:
        clocks.finish()
        model.close()
        if rank == 0:
            print(json.dumps(dict(metric=METRIC, value=cfg.batch * args.steps / (sum(ms) * 1e-3),
                                  unit=UNIT, us_per_batch=sum(ms) * 1e3 / args.steps,
                                  config=dict(workload=cfg.name, math=args.math),
                                  mode="only-forward")))
        return 0
    total_ms = max_over_ranks(sum(ms), dist, dev)
    ms_per_step = total_ms / args.steps
    value = job_throughput(world, cfg.batch, args.steps, total_ms)

    # end to end through the host-buffer C-ABI call
    h_dense = torch.from_numpy(inp["dense"]).pin_memory()
    h_idx = torch.from_numpy(inp["indices"]).pin_memory()
    h_off = torch.from_numpy(inp["offsets"]).pin_memory()
    h_out = torch.empty(cfg.batch).pin_memory()
    e2e_steps = args.steps
    ms_e2e, win = timed(lambda: model.forward_host(h_dense, h_idx, h_off, h_out, stream=stream),
                        e2e_steps, args.warmup)
    clocks.mark(*win)
    if model.error(stream) != dl.OK:
        raise RuntimeError("device error during the e2e forward")
    e2e_total = max_over_ranks(sum(ms_e2e), dist, dev)
    h2d = (inp["dense"].nbytes + inp["indices"].nbytes + inp["offsets"].nbytes)
    e2e = dict(value=job_throughput(world, cfg.batch, e2e_steps, e2e_total), unit=UNIT,
               us_per_batch=e2e_total * 1e3 / e2e_steps, steps=e2e_steps,
               h2d_bytes_per_step=int(h2d), d2h_bytes_per_step=int(cfg.batch * 4),
               api="dlrm_forward_host, pinned host buffers: the kernels read the inputs and "
                   "write the output in host memory over NVLink-C2C (no staging copies)")
    # wall clock of the host-buffer call back to back, as a serving loop makes
    # it: host time around `steps` calls and one final stream sync, no flush
    # (the per-call host cost: binding, ctypes dispatch, pointer-attribute
    # lookups, launch)
    def wall_us(fn, n):
        with torch.cuda.stream(stream):
            for _ in range(max(3, args.warmup)):
                fn()
            stream.synchronize()
            t0 = time.perf_counter()
            for _ in range(n):
                fn()
            stream.synchronize()
            return (time.perf_counter() - t0) * 1e6 / n
    e2e["wall_clock_back_to_back"] = dict(
        us_per_call=wall_us(lambda: model.forward_host(h_dense, h_idx, h_off, h_out,
                                                       stream=stream), args.steps),
        calls=args.steps,
        note="host perf_counter around back-to-back dlrm_forward_host calls and one stream "
             "sync; no L2 flush")
    e2e["wall_clock_device_inputs_back_to_back"] = dict(
        us_per_call=wall_us(lambda: model.forward(dense, idx, off, out, stream=stream),
                            args.steps),
        calls=args.steps, api="dlrm_forward (device buffers)")
    # the same call with pageable buffers: staged host<->device copies each step
    p_dense, p_idx = torch.from_numpy(inp["dense"]).clone(), torch.from_numpy(inp["indices"]).clone()
    p_off, p_out = torch.from_numpy(inp["offsets"]).clone(), torch.empty(cfg.batch)
    ms_st, win = timed(lambda: model.forward_host(p_dense, p_idx, p_off, p_out, stream=stream),
                       max(1, args.steps // 5), max(3, args.warmup // 5))
    clocks.mark(*win)
    if model.error(stream) != dl.OK:
        raise RuntimeError("device error during the staged e2e forward")
    st_total = max_over_ranks(sum(ms_st), dist, dev)
    e2e["staged_copies"] = dict(us_per_batch=st_total * 1e3 / len(ms_st),
                                value=job_throughput(world, cfg.batch, len(ms_st), st_total),
                                api="dlrm_forward_host, pageable host buffers (cudaMemcpyAsync "
                                    "to and from the handle's staging buffers)")

    # CUDA-graph replay of the same forward
    with torch.cuda.stream(stream):
        model.forward(dense, idx, off, out, stream=stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        model.forward(dense, idx, off, out, stream=stream)
    ms_g, win = timed(graph.replay, max(1, args.steps // 5), 3)
    clocks.mark(*win)
    graph_us = statistics.median(ms_g) * 1e3
    clock_info = clocks.finish()

    # per-stage device times (library event profiling, flush before each call)
    model.set_profiling(True)
    with torch.cuda.stream(stream):
        for _ in range(args.profile_steps):
            flush_buf.zero_()
            model.forward(dense, idx, off, out, stream=stream)
    names, totals, calls = model.stage_times()
    model.set_profiling(False)
    stage_us = {n: t * 1e3 / max(calls, 1) for n, t in zip(names, totals)}

    # per-phase device time of the fused kernel (%globaltimer stamps per tile)
    phases_us = None
    if path_used == dl.PATH_FUSED:
        tiles = None
        buf = torch.zeros(((cfg.batch + 3) // 4) * dl.TRACE_SLOTS, dtype=torch.int64, device=dev)
        rows = model.set_phase_trace(buf)
        tiles = (cfg.batch + rows - 1) // rows
        pnames = model.phase_names()
        acc = np.zeros(len(pnames))
        # fp32 kernel: the leader also stamps the end of every GEMM's k-loop
        # (slot 20 + g) while the phase stamps end below slot 20
        n_bot = len(cfg.ln_bot) - 1
        n_gemm = n_bot + len(cfg.ln_top) - 2
        split = args.math == "fp32" and n_gemm + 3 < 20 and n_gemm <= 10
        kacc = np.zeros((n_gemm, 3))
        span = 0.0
        reps = 20
        with torch.cuda.stream(stream):
            for _ in range(reps):
                flush_buf.zero_()
                buf.zero_()
                model.forward(dense, idx, off, out, stream=stream)
                stream.synchronize()
                full = buf.view(-1, dl.TRACE_SLOTS)[:tiles].cpu().numpy()
                t = full[:, :len(pnames) + 1]
                acc += np.diff(t, axis=1).mean(axis=0) / 1e3
                span += (t[:, -1].max() - t[:, 0].min()) / 1e3
                if split:
                    for g in range(n_gemm):
                        first = 1 + g if g < n_bot else 2 + g    # stamp before the layer
                        kend = full[:, 20 + g]
                        kacc[g, 0] += (kend - full[:, first]).mean() / 1e3
                        kacc[g, 1] += (full[:, first + 1] - kend).mean() / 1e3
                        # cycles warp 0 waited for weight stages, as us at the max clock
                        kacc[g, 2] += full[:, 30 + g].mean() / pk["sm_max_mhz"]
        model.set_phase_trace(None)
        phases_us = {n: float(v / reps) for n, v in zip(pnames, acc)}
        phases_us["kernel_span"] = span / reps
        if split:
            names_g = [pnames[1 + g] if g < n_bot else pnames[2 + g] for g in range(n_gemm)]
            phases_us["gemm_kloop_epilogue"] = {
                n: [float(kacc[g, 0] / reps), float(kacc[g, 1] / reps)] for g, n in enumerate(names_g)}
            phases_us["gemm_weight_wait"] = {
                n: float(kacc[g, 2] / reps) for g, n in enumerate(names_g)}
    dom = max(stage_us, key=stage_us.get)
    flops, byts = stage_work(cfg, dom, cfg.batch)
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    smem_optin = getattr(props, "shared_memory_per_block_optin", dl.GB300_SMEM_PER_BLOCK)
    fp32_peak = sms * FP32_LANES_PER_SM * 2 * pk["sm_max_mhz"] * 1e6 / 1e12
    # one launch per step (fused plan): the timed region's own CUDA-event time
    # is that launch's duration; else the library's per-stage event profile
    t_dom = (ms_per_step * 1e-3 if n_stages == 1 else stage_us[dom] * 1e-6)
    if dom in ("gather", "interaction") and byts / (pk["hbm_gbs"] * 1e9) >= flops / (fp32_peak * 1e12):
        ach = byts / t_dom / 1e9
        roof = dict(bound="hbm", achieved=ach, peak=pk["hbm_gbs"], unit="GB/s",
                    frac=ach / pk["hbm_gbs"], traffic=None, kernel=dom,
                    peak_source=f"{pk['source']} (MEASURED_PEAKS hbm_gbs)")
    elif args.math != "fp32" and dom in ("fused",) + tuple(
            f"{w}{i}" for w in ("bottom", "top") for i in range(16)):
        # tensor-pipe work: measured bf16 peak, tf32 at the nominal half rate
        tpeak = pk["bf16_tflops"] * (1.0 if args.math == "bf16" else 0.5)
        ach = flops / t_dom / 1e12
        roof = dict(bound="tensor", achieved=ach, peak=tpeak, unit="TFLOP/s",
                    frac=ach / tpeak, traffic=None, kernel=dom,
                    peak_source=f"{pk['source']} bf16_tflops" +
                    ("" if args.math == "bf16" else " x 0.5 (tf32 nominal ratio)"))
    else:
        ach = flops / t_dom / 1e12
        roof = dict(bound="alu", achieved=ach, peak=fp32_peak, unit="TFLOP/s",
                    frac=ach / fp32_peak, traffic=None, kernel=dom,
                    peak_source=f"FP32 FFMA: {sms} SMs x 128 lanes x 2 x {pk['sm_max_mhz']:.0f} MHz")
    roof["algorithmic_per_launch"] = byts if roof["bound"] == "hbm" else flops
    roof["launch_us"] = t_dom * 1e6
    roof["launch_us_source"] = ("timed region (one launch per step)" if n_stages == 1
                                else "library per-stage event profile")
    roof["traffic"] = NCU_TRAFFIC.get((dom, cfg.name)) if args.math == "fp32" else None
    roof["algorithmic_bytes_per_launch"] = byts

    # whole-forward roofline fraction (slower of HBM bytes and FP32 flops)
    tot_flops, fwd_bytes = forward_work(cfg, cfg.batch)
    t_roof = max(fwd_bytes / (pk["hbm_gbs"] * 1e9), tot_flops / (fp32_peak * 1e12))
    forward_roofline = dict(algorithmic_flops=tot_flops, algorithmic_bytes=fwd_bytes,
                            roofline_us=t_roof * 1e6, frac=t_roof / (ms_per_step * 1e-3),
                            bound="alu (FP32 FFMA)" if tot_flops / (fp32_peak * 1e12) >
                            fwd_bytes / (pk["hbm_gbs"] * 1e9) else "hbm")

    # opt-in tensor-core modes (tcgen05), same inputs and weights, same timing rules
    tc_modes = {}
    for mode_name, mode in (("tf32", dl.MATH_TF32), ("bf16", dl.MATH_BF16),
                            ("tf32x3", dl.MATH_TF32X3)):
        m2 = dl.DlrmModel(cfg.ln_bot, cfg.ln_top, model.tables,
                          [cu(w) for w in inp["bot_w"]], [cu(b) for b in inp["bot_b"]],
                          [cu(w) for w in inp["top_w"]], [cu(b) for b in inp["top_b"]],
                          cfg.bag_size, cfg.batch, mode)
        ms_tc, _ = timed(lambda: m2.forward(dense, idx, off, out, stream=stream),
                         max(1, args.steps // 5), 10)
        if m2.error(stream) != dl.OK:
            raise RuntimeError(f"device error in the {mode_name} forward")
        tot = sum(ms_tc)
        tc_plan = ("fused single launch, tcgen05 MMAs" if m2.path == dl.PATH_FUSED
                   else "layer-wise launches, tcgen05 GEMMs")
        tc_modes[mode_name] = dict(us_per_batch=tot * 1e3 / len(ms_tc),
                                   samples_per_s=cfg.batch * len(ms_tc) / (tot * 1e-3),
                                   plan=tc_plan,
                                   tolerance=("fp32 parity (abs 1e-5, rel 1e-4)"
                                              if mode == dl.MATH_TF32X3
                                              else "rel 2e-2 vs the fp64 oracle"))
        m2.close()

    def forward_point(c, tabs, steps, warmup, math_name=None):
        """One workload's forward through the library, same timing rules as the
        headline: mean and median us per batch, samples/s, the plan taken and the
        whole-forward roofline fraction (forward_roofline_parts: the tensor pipe
        for the GEMMs the plan runs there, the FP32 FFMA peak for the rest, HBM)."""
        math_name = math_name or args.config_math
        ci = synth.make_inputs(c, seed=args.seed, with_tables=False)
        m = dl.DlrmModel(c.ln_bot, c.ln_top, tabs,
                         [cu(w) for w in ci["bot_w"]], [cu(b) for b in ci["bot_b"]],
                         [cu(w) for w in ci["top_w"]], [cu(b) for b in ci["top_b"]],
                         c.bag_size, c.batch, maths[math_name])
        d_, i_, o_ = cu(ci["dense"]), cu(ci["indices"]), cu(ci["offsets"])
        y_ = torch.empty(c.batch, device=dev)
        ms_c, _ = timed(lambda: m.forward(d_, i_, o_, y_, stream=stream), steps, warmup)
        ok = m.error(stream) == dl.OK
        plan = {dl.KERNELS_LAYERWISE: "layer-wise", dl.KERNELS_FUSED: "fused",
                dl.KERNELS_FUSED_CLUSTER: "fused, cluster-split",
                dl.KERNELS_FUSED_TC: "fused, tensor cores"}[m.kernels(c.batch)]
        m.close()
        if not ok:
            raise RuntimeError(f"device error in the {c.name} forward")
        t = sum(ms_c) / len(ms_c) * 1e-3
        plan_info = dl.dlrm_plan_query(c.ln_bot, c.ln_top, c.rows, c.emb_dim, c.bag_size,
                                       c.batch, maths[math_name], dl.PATH_AUTO,
                                       sms, smem_optin)
        rf = forward_roofline_parts(c, plan_info, maths[math_name], fp32_peak, pk)
        r = dict(us_per_batch=t * 1e6, us_median=statistics.median(ms_c) * 1e3,
                 samples_per_s=c.batch / t, steps=len(ms_c), plan=plan,
                 math=math_name, roofline_frac=rf["roofline_us"] * 1e-6 / t,
                 bound=rf["bound"])
        if rf["tensor_core_layers"]:
            r["tensor_core_layers"] = rf["tensor_core_layers"]
        return r

    configs = None
    gather = None
    cpu = None
    if rank == 0 and world == 1:
        if not args.no_configs:
            configs = {cfg.name: "this line"}
            for name in ("tiny_b64_k3", "b2048_k32"):
                if name != cfg.name:
                    c = synth.get_config(name)
                    tabs = device_tables(torch, synth, c, args.seed)
                    configs[name] = forward_point(c, tabs, 200, 10)
                    del tabs
            # batch x tables sweep; table t is the same seeded stream for every K,
            # so one set of 32 tables serves all cells
            tabs = device_tables(torch, synth, synth.sweep_config(1, 32), args.seed)
            sweep = {}
            for k in synth.SWEEP_TABLES:
                for b in synth.SWEEP_BATCHES:
                    r = forward_point(synth.sweep_config(b, k), tabs[:k], 30, 5)
                    sweep[f"b{b}_k{k}"] = {key: r[key] for key in
                                           ("us_per_batch", "samples_per_s", "roofline_frac", "plan")}
            configs["sweep_b1-8192_k1-32"] = sweep
            del tabs
            torch.cuda.empty_cache()
        if not args.no_gather:
            c4 = synth.get_config("b65536_k26_zipf")
            tabs = device_tables(torch, synth, c4, args.seed)
            gather = gather_measure(torch, dl, synth, pk, tabs)
            gather["general_bags"] = bag_modes_measure(torch, dl, synth, pk, tabs)
            if configs is not None:
                configs[c4.name] = forward_point(c4, tabs, 5, 3)
                # the same model with every GEMM on the FP32 FFMA pipe (the fp32
                # layer-wise plan runs its large GEMMs as split-TF32)
                configs[c4.name + "_fp32_ffma"] = forward_point(c4, tabs, 5, 3, "fp32_ffma")
            del tabs
            torch.cuda.empty_cache()
        if not args.no_cpu_baseline:
            cpu = time_oracle(inp, cfg.batch, args.cpu_seconds)
            # the same oracle on one thread, a short sample beside the all-core figure
            one = time_oracle(inp, cfg.batch, min(3.0, args.cpu_seconds), threads=1)
            cpu["single_thread"] = {k: one[k] for k in ("value", "unit", "cores", "sample")}

    model.close()
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0
    line = dict(
        metric=METRIC, value=value, unit=UNIT, n_gpus=world, steps=args.steps,
        warmup=args.warmup, ms_per_step=ms_per_step, us_per_batch=ms_per_step * 1e3,
        us_per_batch_median=statistics.median(ms) * 1e3,
        us_per_batch_p10_p90=[float(np.percentile(ms, 10) * 1e3), float(np.percentile(ms, 90) * 1e3)],
        higher_is_better=True, scaling="weak", vs_baseline=None,
        dtype={"fp32": "f32", "fp32_ffma": "f32", "tf32": "tf32", "bf16": "bf16",
               "tf32x3": "3xtf32"}[args.math],
        data="synthetic: seeded SplitMix64 inputs of the workload's shapes and distributions",
        config=dict(workload=cfg.name, global_batch=cfg.batch * world, batch_per_gpu=cfg.batch,
                    tables=cfg.n_tables, rows=cfg.rows[0], emb_dim=cfg.emb_dim,
                    bag_size=cfg.bag_size, ln_bot=list(cfg.ln_bot), ln_top=list(cfg.ln_top),
                    math=args.math, l2="flushed before every step (256 MB write)",
                    plan={dl.PATH_FUSED: "fused single launch",
                          dl.PATH_LAYERWISE: "layer-wise launches"}[path_used],
                    parallelism="replicas" if world > 1 else "single GPU"),
        e2e=e2e, gpu_launches=args.steps * n_stages, clocks=clock_info,
        roofline=roof, forward_roofline=forward_roofline, stages_us=stage_us,
        fused_phases_us=phases_us, opt_in_tensor_core=tc_modes, configs=configs,
        graph=dict(us_per_batch_median=graph_us, samples_per_s=cfg.batch / (graph_us * 1e-6)),
        cpu_baseline=cpu)
    line["gather_b65536_k26_zipf"] = gather
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    return run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    sys.exit(main())
