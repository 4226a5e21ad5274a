#!/usr/bin/env python
"""Benchmark of the decode-time KV-cache compression event on GB300.

One step = one compression event (all six steps) over every unit of the
workload, inputs resident in HBM.  Default workload: the 28-layer Qwen-7B-shaped
event (L28 B32 H4 G7 d128, 1536 slots -> 1024, W 128), in the state of its
second event (credit carried from the first, 512 fresh slots appended).

Metric: cached tokens scanned per second per compression event
(sum over units of the valid slots, divided by the event time).  The JSON line
also carries the live per-kernel timing (CUDA events on the launch stream), the
roofline of the dominant kernel against MEASURED_PEAKS.json, the event roofline,
the CPU oracle as a baseline, an end-to-end figure through host buffers, and the
SM clocks sampled during the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun every rank runs the same per-GPU workload (weak scaling, no
collective on the data path); rank 0 prints the line.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "cached tokens scanned/s per compression event"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
from eviction_gb300.kvc import ABLATIONS  # noqa: E402  (the pages' ablations as switches)

KERNEL_SOURCES = {
    "compact_paged": "paged.cu",
    "refresh_trigger": "refresh.cu",
    "usage_pass1_rowstats_tcgen05": ("attn_usage.cu", "attn_common.cuh"),
    "usage_pass2_colsum_tcgen05": ("attn_usage.cu", "attn_common.cuh"),
    "mass_pool_ema": ("mass_post.cu", "unit_phases.cuh"),
    "segment_quota": ("segment_quota.cu", "unit_phases.cuh"),
    "select_topk": ("select.cu", "unit_phases.cuh"),
    "mass_segment_select": ("unit_post.cu", "unit_phases.cuh"),
    "gather_compact": "compact.cu",
    "redundancy_score": "redundancy.cu",
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen_28l")
    ap.add_argument("--layers", type=int, default=None,
                    help="the same workload recipe cut to this many layers (small profiling case)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--e2e-layers", type=int, default=2,
                    help="layers per host<->device copy stage of the end-to-end leg")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--paged", action="store_true",
                    help="compact into a paged KV pool (block size 16) instead of dense caches")
    ap.add_argument("--ablation", choices=sorted(ABLATIONS), default="none",
                    help="time one of the method's ablations (the pages' ablation table)")
    ap.add_argument("--attn-kernel", type=int, default=0, choices=[0, 1, 2],
                    help="step-1 tensor-core kernel: 1 = one SM per MMA, 2 = CTA pairs, "
                         "0 = the library's choice")
    ap.add_argument("--grouped", type=int, default=0, metavar="G",
                    help="ragged batch sorted by length and run in groups of G sequences, each "
                         "padded only to its own longest sequence (SkipKV's batch grouping)")
    ap.add_argument("--redundancy", type=float, default=0.0, metavar="SIGMA",
                    help="select on the SkipKV key-redundancy mix with this sigma (0.1 in the "
                         "pages); 0 = the attention score alone")
    return ap.parse_args()


def sched_kw(args):
    """Switches of our arm only that change how, not what, it computes."""
    return {"attn_kernel": args.attn_kernel} if args.attn_kernel else {}


def method_kw(args):
    """Config switches shared by both arms: an ablation and the second base score."""
    kw = dict(ABLATIONS[args.ablation])
    if args.redundancy > 0:
        kw["redundancy_sigma"] = args.redundancy
    return kw



# --------------------------------------------------------------------- helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def unit_work(w, T_valid, T):
    """Algorithmic work of one unit: flops of one QK^T, bytes of the event, and
    per-kernel bytes.  T_valid = valid slots of the unit."""
    G, W, d, Kb = w.group, w.window, w.head_dim, w.budget
    kept = min(Kb, T_valid)
    flops = 2.0 * G * W * T_valid * d
    q_bytes = 2.0 * G * W * d
    k_bytes = 2.0 * T_valid * d
    ev_bytes = (q_bytes + k_bytes + 2.0 * kept * d + 4.0 * kept * d
                + 4.0 * T_valid + 4.0 * kept + 4.0 * kept)
    per_kernel = {
        "usage_pass1_rowstats_tcgen05": ("tensor", flops, q_bytes + k_bytes),
        "usage_pass2_colsum_tcgen05": ("tensor", flops, q_bytes + k_bytes),
        # raw usage, credit in; score, mass, credit out; row statistics
        "mass_pool_ema": ("hbm", 0.0, 4.0 * T * 5 + 8.0 * G * W),
        "segment_quota": ("hbm", 0.0, 4.0 * T),
        "select_topk": ("hbm", 0.0, 4.0 * T + 4.0 * Kb),
        # the three above in one launch: mass's traffic and the kept indices
        # (the mass and the score stay on chip for the later steps)
        "mass_segment_select": ("hbm", 0.0, 4.0 * T * 5 + 8.0 * G * W + 4.0 * Kb),
        # kept K and V rows read, written; credit read/written; indices read
        "gather_compact": ("hbm", 0.0, 8.0 * Kb * d + 12.0 * Kb),
        # the same rows and credit moved into pool blocks; plus indices validated
        "compact_paged": ("hbm", 0.0, 8.0 * Kb * d + 16.0 * Kb),
        # K read once; the score read and the mixed score written
        "redundancy_score": ("hbm", 0.0, 2.0 * T_valid * d + 8.0 * T_valid),
    }
    return flops, ev_bytes, per_kernel


def source_sha(kernel):
    """First 16 hex digits of the sha256 of the kernel's source file(s), concatenated."""
    src = KERNEL_SOURCES.get(kernel)
    if not src:
        return None
    h = hashlib.sha256()
    for name in (src if isinstance(src, tuple) else (src,)):
        with open(os.path.join(ROOT, "eviction_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def read_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, or None if absent or
    taken on a different version of the kernel's source."""
    path = os.path.join(ROOT, "profiles", f"{kernel}__{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_t = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m_s = re.search(r"source_sha:\s*([0-9a-f]+)", text)
    if not m_t or not m_s or m_s.group(1) != source_sha(kernel):
        return None
    return float(m_t.group(1))


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons in the background."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "20"]
            if self.gpu_id is not None:
                cmd += ["-i", str(self.gpu_id)]
            self.proc = subprocess.Popen(cmd, stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return []
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                    rows.append(dict(t=ts + frac, sm=float(parts[2]), sm_max=float(parts[3]),
                                     reasons=parts[5], hw=parts[6], hw_th=parts[7],
                                     sw_th=parts[8], pcap=parts[9]))
                except ValueError:
                    continue
        os.unlink(self.file.name)
        return rows


def summarize_clocks(rows, t0, t1):
    if not rows:
        return None
    inside = [r for r in rows if t0 - 0.05 <= r["t"] <= t1 + 0.05]
    window = "timed"
    if len(inside) < 3:
        inside = [r for r in rows if r["t"] <= t1 + 0.05] or rows
        window = "warmup+timed (timed region shorter than the sampling period)"
    reasons = set()
    for r in inside:
        for key, name in (("hw", "hw_slowdown"), ("hw_th", "hw_thermal_slowdown"),
                          ("sw_th", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
            if r[key].lower() == "active":
                reasons.add(name)
    return {"sm_mhz": statistics.median(r["sm"] for r in inside),
            "sm_max_mhz": max(r["sm_max"] for r in inside),
            "reasons": sorted(reasons), "samples": len(inside), "window": window}


def reduce_over_ranks(elapsed_ms, tokens, device):
    """(max elapsed over ranks, sum of tokens over ranks); identity on one rank.

    Timing only: the ranks exchange two numbers, never any data of the event."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(elapsed_ms), float(tokens)
    t = torch.tensor([float(elapsed_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    n = torch.tensor([float(tokens)], dtype=torch.float64, device=device)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), float(n.item())


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ------------------------------------------------------------ reference arm

def run_reference(args, w):
    """The oracle (the reference implementation of this build) on host cores."""
    import numpy as np

    import oracle
    import workload as wl

    oracle.build()
    sample_w = wl.scaled(w, n_layers=1, batch=1)
    first = wl.generate(sample_w, device="cpu")
    p = oracle.RefParams(group=w.group, head_dim=w.head_dim, window=w.window, budget=w.budget,
                         n_sink=w.n_sink, n_recent=w.n_recent, **method_kw(args))

    def unit_inputs(inp):
        return (wl.bf16_bits(wl.q_units(inp.q, inp.w)), wl.bf16_bits(wl.units_of(inp.k, inp.w)),
                wl.bf16_bits(wl.units_of(inp.v, inp.w)), wl.units_of(inp.credit, inp.w).numpy(),
                wl.unit_pad(inp).numpy(), wl.unit_n_carry(inp).numpy())

    inp = first
    if w.n_events > 1:
        r = oracle.event(p, *unit_inputs(first))
        import torch
        Kb = w.budget
        shape = (1, 1, w.n_kv_heads)
        inp = wl.next_event(sample_w, first,
                            torch.from_numpy(r["k_out"].view(np.int16)).view(torch.bfloat16)
                            .reshape(*shape, Kb, w.head_dim),
                            torch.from_numpy(r["v_out"].view(np.int16)).view(torch.bfloat16)
                            .reshape(*shape, Kb, w.head_dim),
                            torch.from_numpy(r["credit_out"]).reshape(*shape, Kb),
                            torch.from_numpy(r["n_kept"]).reshape(shape), 1)
    q, k, v, c, pad, nc = unit_inputs(inp)
    U = q.shape[0]
    T = k.shape[1]
    cores = host_cores()

    def step(i):
        """One step: `cores` units of the workload at once, one per host core."""
        us = [(i * cores + j) % U for j in range(cores)]
        oracle.event(p, q[us], k[us], v[us], c[us], pad[us], nc[us], threads=cores)
        return sum(T - int(pad[u]) for u in us)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    tokens = 0
    for i in range(args.steps):
        tokens += step(i)
    dt = time.perf_counter() - t0
    value = tokens / dt
    sample = (f"{args.steps} steps, each {cores} units (one sequence x one KV head x one layer, "
              f"T={T}, G={w.group}, W={w.window}, d={w.head_dim}) of the {w.name} workload, "
              f"one unit per host core; C oracle (fp64) through a thread pool")
    world = dist_env()[0]
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": dict(workload_config(w, T, args.ablation, redundancy=args.redundancy),
                       parallelism=f"replicas x{world}"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def workload_config(w, T, ablation="none", paged=False, redundancy=0.0, grouped=0):
    cfg = {"workload": (f"{w.name}: {w.n_layers} layers x batch {w.batch} x {w.n_kv_heads} KV heads"
                         f" (GQA {w.group}), d {w.head_dim}, {T} slots -> budget {w.budget}, "
                         f"window {w.window}" + (", event 2 (credit carried, 512 fresh slots)"
                                                 if w.n_events > 1 else "")),
            "units": w.units, "T": T, "budget": w.budget, "window": w.window,
            "group": w.group, "head_dim": w.head_dim,
            "l2": "inputs larger than L2 (no flush needed)"}
    if ablation != "none":
        cfg["ablation"] = f"{ablation}: {ABLATIONS[ablation]}"
    if redundancy > 0:
        cfg["score"] = (f"SkipKV key-redundancy mix, sigma {redundancy}: "
                        "sigma * score/sum(score) - (1 - sigma) * softmax(mean key cosine)")
    if paged:
        cfg["paged"] = "compaction into a paged pool, block size 16 (stack and table restored per step)"
    if grouped:
        cfg["layout"] = (f"sequences sorted by length, {w.batch // grouped} events of {grouped} "
                         "sequences, each padded to its own longest sequence")
    elif w.prefill is not None:
        cfg["layout"] = f"left-padded to the longest sequence ({T} slots)"
    return cfg


# ------------------------------------------------------------------ our arm

def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_oracle_baseline(args, w, parts):
    """The oracle as it stands, on a bounded random sample of the timed event's
    units: single-threaded for about half of --cpu-seconds, then the units split
    over a thread pool on every host core for about the other half (units are
    independent; ctypes releases the GIL in the C calls).  Unit data are copied
    to the host before each timed part."""
    import numpy as np

    import oracle
    import workload as wl
    oracle.build()
    p = oracle.RefParams(group=w.group, head_dim=w.head_dim, window=w.window, budget=w.budget,
                         n_sink=w.n_sink, n_recent=w.n_recent, **method_kw(args))
    pool = [(j, u) for j, part in enumerate(parts) for u in range(part["w"].units)]
    order = np.random.default_rng(0).permutation(len(pool))
    nxt = 0

    def take(n):
        """Host copies of the next n sampled units (the sample wraps around the
        workload's units when they run out): (inputs, valid tokens)."""
        nonlocal nxt
        chosen = [pool[order[(nxt + i) % len(pool)]] for i in range(n)]
        nxt += len(chosen)
        cols = [[] for _ in range(6)]
        tokens = 0
        for j, u in chosen:
            inp, pw = parts[j]["inp"], parts[j]["w"]
            sl = slice(u, u + 1)
            pad_u = wl.unit_pad(inp)[sl]
            vals = (wl.bf16_bits(wl.q_units(inp.q, pw)[sl]), wl.bf16_bits(wl.units_of(inp.k, pw)[sl]),
                    wl.bf16_bits(wl.units_of(inp.v, pw)[sl]),
                    wl.units_of(inp.credit, pw)[sl].cpu().numpy(), pad_u.cpu().numpy(),
                    wl.unit_n_carry(inp)[sl].cpu().numpy())
            for c, v in zip(cols, vals):
                c.append(v)
            tokens += parts[j]["T"] - int(pad_u.item())
        return cols, tokens

    def run(cols, threads):
        # units of different groups differ in T: one call per unit in that case
        if len({c.shape[1] for c in cols[1]}) == 1:
            arrs = [np.concatenate(c, axis=0) for c in cols]
            t0 = time.perf_counter()
            oracle.event(p, *arrs, threads=threads)
            return time.perf_counter() - t0
        from concurrent.futures import ThreadPoolExecutor
        t0 = time.perf_counter()
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(lambda i: oracle.event(p, *[c[i] for c in cols]), range(len(cols[0]))))
        return time.perf_counter() - t0

    half = args.cpu_seconds / 2
    done1 = tok1 = 0
    dt1 = 0.0
    while dt1 < half or done1 == 0:
        cols, tokens = take(1)
        dt1 += run(cols, 1)
        done1 += 1
        tok1 += tokens
    rate1 = tok1 / dt1
    cores = host_cores()
    per_unit = dt1 / done1
    n_all = int(max(cores, cores * half / per_unit))
    n_all -= n_all % cores
    value, used, sample_all = rate1, 1, None
    if n_all > 0:
        cols, tokens = take(n_all)
        used = min(cores, n_all)
        dtn = run(cols, used)
        value = tokens / dtn
        sample_all = f"{n_all} further units on {used} threads ({dtn:.1f} s)"
    return {"value": value, "unit": UNIT, "cores": used, "kind": "oracle",
            "single_core_value": rate1,
            "sample": (f"random units of the timed event (seed 0, repeated once all {len(pool)} are "
                       f"used), same inputs, C oracle in fp64: "
                       f"{done1} units single-threaded ({dt1:.1f} s, value {rate1:.4g} tokens/s)"
                       + (f"; {sample_all} give the value, cores = threads used"
                          if sample_all else "; value = single-threaded"))}


def run_ours(args, w):
    import numpy as np
    import torch

    import eviction_gb300 as kvc
    import workload as wl

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    assert torch.cuda.is_available(), "bench.py (ours) needs a CUDA GPU"
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    kvc.load_library()

    seed = w.seed + 7919 * rank
    first = wl.generate(w, device=dev, seed=seed)
    T = first.T
    cfg = kvc.Config(w.n_layers, w.batch, w.n_kv_heads, w.group, w.head_dim,
                     max(T, w.budget + w.interval), w.budget, window=w.window, n_sink=w.n_sink,
                     n_recent=w.n_recent, **method_kw(args), **sched_kw(args))
    h = kvc.Handle(cfg)
    inp = first
    if w.n_events > 1:
        o1 = h.outputs(T, dev)
        h.event(first.q, first.k, first.v, T, first.pad, first.n_carry, first.credit,
                o1["k_out"], o1["v_out"], o1["credit_out"], o1["kept_idx"], o1["n_kept"])
        inp = wl.next_event(w, first, o1["k_out"], o1["v_out"], o1["credit_out"], o1["n_kept"],
                            1, seed=seed)
        del o1, first
        torch.cuda.empty_cache()
    T = inp.T
    stream = torch.cuda.current_stream(dev)
    # the timed work: one event per part (one part, or the length-sorted groups)
    if args.grouped:
        assert w.prefill is not None and w.n_events == 1, "--grouped needs a ragged workload"
        assert w.batch % args.grouped == 0, "the batch must split into equal groups"
        lengths = (T - inp.pad.long()).cpu().numpy()
        by_len = np.argsort(lengths, kind="stable")
        gw = wl.scaled(w, batch=args.grouped)
        h.close()
        h = kvc.Handle(kvc.Config(w.n_layers, args.grouped, w.n_kv_heads, w.group, w.head_dim,
                                  T, w.budget, window=w.window, n_sink=w.n_sink,
                                  n_recent=w.n_recent, **method_kw(args), **sched_kw(args)))
        parts = []
        for g0 in range(0, w.batch, args.grouped):
            grp = by_len[g0:g0 + args.grouped]
            Tg = int(lengths[grp].max())
            idx = torch.as_tensor(grp, device=dev, dtype=torch.long)
            pad_g = torch.as_tensor(Tg - lengths[grp], device=dev).to(torch.int32)
            gi = wl.Inputs(gw, Tg, inp.q.index_select(1, idx).contiguous(),
                           inp.k.index_select(1, idx)[:, :, :, T - Tg:].contiguous(),
                           inp.v.index_select(1, idx)[:, :, :, T - Tg:].contiguous(),
                           inp.credit.index_select(1, idx)[:, :, :, T - Tg:].contiguous(),
                           pad_g, (Tg - pad_g).to(torch.int32))
            parts.append({"inp": gi, "T": Tg, "w": gw, "out": h.outputs(Tg, dev)})
        del inp
        torch.cuda.empty_cache()
    else:
        parts = [{"inp": inp, "T": T, "w": w, "out": h.outputs(T, dev)}]
    inp, out = parts[0]["inp"], parts[0]["out"]
    tokens_per_step = float(sum(pt["w"].n_layers * pt["w"].n_kv_heads
                                * (pt["T"] - pt["inp"].pad.long()).sum().item() for pt in parts))

    def step():
        for pt in parts:
            x, o = pt["inp"], pt["out"]
            h.event(x.q, x.k, x.v, pt["T"], x.pad, x.n_carry, x.credit, o["k_out"],
                    o["v_out"], o["credit_out"], o["kept_idx"], o["n_kept"])

    if args.paged:
        args.no_e2e = True  # the host round trip is timed for the dense path only
        # the same cache in a paged pool (block size 16, a random block table);
        # one step = steps 1-5 through the stage entry points, then the paged
        # compaction; the stack and table are restored before each step
        bs = 16
        lens = (T - inp.pad.long()).tolist()
        max_blocks = (T + bs - 1) // bs
        n_old = sum((n + bs - 1) // bs for n in lens)
        n_new = w.batch * ((w.budget + bs - 1) // bs)
        n_blocks = n_old + n_new
        perm = torch.randperm(n_blocks, generator=torch.Generator().manual_seed(0)).to(torch.int32)
        table0 = torch.full((w.batch, max_blocks), -1, dtype=torch.int32)
        at = 0
        for b, n in enumerate(lens):
            nb = (n + bs - 1) // bs
            table0[b, :nb] = perm[at:at + nb]
            at += nb
        free0 = torch.zeros(n_blocks, dtype=torch.int32)
        free0[:n_new] = perm[n_old:]
        table0, free0 = table0.to(dev), free0.to(dev)
        top0 = torch.tensor([n_new], dtype=torch.int32, device=dev)
        L_, H_, d_ = w.n_layers, w.n_kv_heads, w.head_dim
        k_pool = torch.zeros((L_, n_blocks, H_, bs, d_), dtype=torch.bfloat16, device=dev)
        v_pool = torch.zeros_like(k_pool)
        t_idx = torch.arange(T, device=dev)
        for b, n in enumerate(lens):
            pb = T - n
            pos = t_idx[:n]
            blk = table0[b, pos // bs].long()
            k_pool[:, blk, :, pos % bs] = inp.k[:, b, :, pb:].permute(2, 0, 1, 3)
            v_pool[:, blk, :, pos % bs] = inp.v[:, b, :, pb:].permute(2, 0, 1, 3)
        seq_len = torch.tensor(lens, dtype=torch.int32, device=dev)
        stage = h.stage_buffers(T, dev)
        table, free, top = table0.clone(), free0.clone(), top0.clone()
        table_new = torch.empty_like(table0)

        def step():  # noqa: F811
            table.copy_(table0)
            free.copy_(free0)
            top.copy_(top0)
            h.mass_select(inp.q, inp.k, T, inp.pad, inp.n_carry, inp.credit,
                          stage["credit_post"], stage["mass"], stage["score"],
                          stage["seg_start"], stage["seg_len"], stage["quota"], stage["n_seg"],
                          out["kept_idx"], out["n_kept"])
            h.compact_paged(k_pool, v_pool, bs, seq_len, inp.pad, out["kept_idx"], out["n_kept"],
                            stage["credit_post"], T, out["credit_out"], table, table_new, free,
                            top)

    warm = max(3, args.warmup)
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        gpu_id = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        gpu_id = None
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.2)
    for _ in range(warm):
        step()
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    h.profile(True)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    time.sleep(0.1)
    clock_rows = sampler.stop()
    elapsed_ms = e0.elapsed_time(e1)
    kernels = h.profile_read(reset=True)
    h.profile(False)
    status = h.device_status()
    if status:
        raise RuntimeError(f"device status bits {status:#x} after the timed region")

    max_ms, total_tokens = reduce_over_ranks(elapsed_ms, tokens_per_step, dev)
    ms_per_step = max_ms / args.steps
    value = total_tokens / (ms_per_step / 1000.0)

    # ---- roofline of the dominant kernel and of the event
    peaks, peak_src = load_peaks()
    flops_ev = bytes_ev = 0.0
    per_kernel_work = {}
    for pt in parts:
        for Tv in (pt["T"] - pt["inp"].pad.long()).cpu().numpy():
            f, b, pk = unit_work(w, int(Tv), pt["T"])
            n_u = w.n_layers * w.n_kv_heads
            flops_ev += f * n_u
            bytes_ev += b * n_u
            for name, (bound, fl, by) in pk.items():
                acc = per_kernel_work.setdefault(name, [bound, 0.0, 0.0])
                acc[1] += fl * n_u   # per step; divided over the step's launches below
                acc[2] += by * n_u
    total_kernel_ms = sum(k["total_ms"] for k in kernels) or 1.0
    krows = []
    for k in kernels:
        if not k["launches"]:
            continue
        bound, fl, by = per_kernel_work[k["name"]]
        per_step = k["launches"] / args.steps   # launches of this kernel in one step
        fl, by = fl / per_step, by / per_step   # algorithmic work of one launch
        avg_s = k["total_ms"] / k["launches"] / 1000.0
        if bound == "tensor":
            ach, peak, unit = fl / avg_s / 1e12, peaks["bf16_tflops"], "TFLOP/s"
        else:
            ach, peak, unit = by / avg_s / 1e9, peaks["hbm_gbs"], "GB/s"
        krows.append({"name": k["name"], "launches": k["launches"],
                      "avg_ms": 1000.0 * avg_s, "share": k["total_ms"] / total_kernel_ms,
                      "bound": bound, "achieved": ach, "peak": peak, "unit": unit,
                      "frac": ach / peak, "algorithmic_per_launch": fl if bound == "tensor" else by,
                      "launches_per_step": per_step})
    dom = max(krows, key=lambda r: r["avg_ms"] * r["launches"])
    roofline = {"kernel": dom["name"], "bound": dom["bound"], "achieved": dom["achieved"],
                "peak": dom["peak"], "unit": dom["unit"], "frac": dom["frac"],
                "peak_source": f"{'bf16_tflops (burst)' if dom['bound'] == 'tensor' else 'hbm_gbs'}"
                               f" of {peak_src}",
                "traffic": (None if read_traffic(dom["name"], w.name) is None else
                            read_traffic(dom["name"], w.name) / dom["launches_per_step"])}
    t_flop = flops_ev / (peaks["bf16_tflops"] * 1e12)
    t_byte = bytes_ev / (peaks["hbm_gbs"] * 1e9)
    roof_ms = 1000.0 * max(t_flop, t_byte)
    event_roofline = {"bound": "tensor" if t_flop > t_byte else "hbm",
                      "roofline_ms": roof_ms, "achieved_ms": ms_per_step,
                      "frac": roof_ms / ms_per_step, "tensor_ms": 1000.0 * t_flop,
                      "hbm_ms": 1000.0 * t_byte, "flops": flops_ev, "bytes": bytes_ev,
                      "peaks": f"of {peak_src}"}

    # ---- end to end through host buffers
    e2e = None
    if not args.no_e2e:
        lps = args.e2e_layers
        legs = []
        for pt in parts:
            x = pt["inp"]
            host_in = {k: getattr(x, k).cpu().pin_memory() for k in
                       ("q", "k", "v", "credit", "pad", "n_carry")}
            host_out = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
                        for k, v in pt["out"].items()}
            dev_in = {k: torch.empty_like(getattr(x, k))  # staging, as a caller has
                      for k in ("q", "k", "v", "credit", "pad", "n_carry")}
            legs.append((host_in, dev_in, host_out, pt))

        def e2e_step():
            h2d_s = d2h_s = 0
            for host_in, dev_in, host_out, pt in legs:
                a, b = h.event_from_host(host_in, dev_in, host_out, pt["out"], pt["T"],
                                         layers_per_stage=lps)
                h2d_s += a
                d2h_s += b
            return h2d_s, d2h_s

        e2e_step()  # warm-up
        torch.cuda.synchronize(dev)
        # every step as a caller runs it: enqueue, wait for the result and read
        # it on the host (its kept counts), all inside the timed region
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        kept_seen = 0
        for _ in range(args.e2e_steps):
            h2d, d2h = e2e_step()
            torch.cuda.synchronize(dev)
            kept_seen += sum(int(leg[2]["n_kept"][0, 0, 0]) for leg in legs)
        f1.record(stream)
        torch.cuda.synchronize(dev)
        # V is read in place at the kept rows (page-locked host buffer)
        h2d += sum(int(leg[2]["n_kept"].long().sum().item()) for leg in legs) * w.head_dim * 2
        e2e_ms = f0.elapsed_time(f1) / args.e2e_steps
        e2e_ms, _ = reduce_over_ranks(e2e_ms, 0.0, dev)
        e2e = {"value": total_tokens / (e2e_ms / 1000.0), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "steps": args.e2e_steps,
               "path": f"kvc_event_host, pinned host buffers, {lps} layers per copy stage; "
                       "V read in place at the kept rows; each step synchronised and its "
                       "result read on the host"}
        del legs

    # ---- CPU oracle baseline on a bounded sample (rank 0, N = 1)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle_baseline(args, w, parts)
    clocks = summarize_clocks(clock_rows, t_wall0, t_wall1)
    # kernels per traced entry (the paged compaction is four launches)
    launches = sum(r["launches"] * (4 if r["name"] == "compact_paged" else 1) for r in krows)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": warm, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(workload_config(w, T, args.ablation, args.paged, args.redundancy,
                                       args.grouped),
                       parallelism=f"replicas x{world}"),
        "roofline": roofline, "event_roofline": event_roofline,
        "kernels": [{k2: (round(v, 6) if isinstance(v, float) else v) for k2, v in r.items()}
                    for r in krows],
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
        "events_per_s": 1000.0 / ms_per_step,
    }
    if rank == 0:
        print(json.dumps(line))
    h.close()
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    args = parse_args()
    import workload as wl
    w = wl.CONFIGS[args.workload]
    if args.layers:
        w = wl.scaled(w, n_layers=args.layers, name=f"{w.name}_{args.layers}layers")
    if args.impl == "reference":
        world, rank, _ = dist_env()
        if rank != 0:
            return
        run_reference(args, w)
        return
    run_ours(args, w)


if __name__ == "__main__":
    main()
