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
    "usage_pass1_rowstats_tcgen05": "attn_usage.cu",
    "usage_pass2_colsum_tcgen05": "attn_usage.cu",
    "mass_pool_ema": "mass_post.cu",
    "segment_quota": "segment_quota.cu",
    "select_topk": "select.cu",
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
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--e2e-layers", type=int, default=2,
                    help="layers per host<->device copy stage of the end-to-end leg")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--paged", action="store_true",
                    help="compact into a paged KV pool (block size 16) instead of dense caches")
    ap.add_argument("--ablation", choices=sorted(ABLATIONS), default="none",
                    help="time one of the method's ablations (the pages' ablation table)")
    ap.add_argument("--redundancy", type=float, default=0.0, metavar="SIGMA",
                    help="select on the SkipKV key-redundancy mix with this sigma (0.1 in the "
                         "pages); 0 = the attention score alone")
    return ap.parse_args()


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
        # kept K and V rows read, written; credit read/written; indices read
        "gather_compact": ("hbm", 0.0, 8.0 * Kb * d + 12.0 * Kb),
        # the same rows and credit moved into pool blocks; plus indices validated
        "compact_paged": ("hbm", 0.0, 8.0 * Kb * d + 16.0 * Kb),
        # K read once; the score read and the mixed score written
        "redundancy_score": ("hbm", 0.0, 2.0 * T_valid * d + 8.0 * T_valid),
    }
    return flops, ev_bytes, per_kernel


def source_sha(kernel):
    src = KERNEL_SOURCES.get(kernel)
    if not src:
        return None
    with open(os.path.join(ROOT, "eviction_gb300", "csrc", src), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


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

    def step(i):
        u = i % U
        oracle.event(p, q[u:u + 1], k[u:u + 1], v[u:u + 1], c[u:u + 1], pad[u:u + 1], nc[u:u + 1])
        return T - int(pad[u])

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    tokens = 0
    for i in range(args.steps):
        tokens += step(i)
    dt = time.perf_counter() - t0
    value = tokens / dt
    sample = (f"{args.steps} steps, each one unit (one sequence x one KV head x one layer, "
              f"T={T}, G={w.group}, W={w.window}, d={w.head_dim}) of the {w.name} workload; "
              f"single-threaded C oracle (fp64)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(w, T, args.ablation, redundancy=args.redundancy),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def workload_config(w, T, ablation="none", paged=False, redundancy=0.0):
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
    return cfg


# ------------------------------------------------------------------ our arm

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
                     n_recent=w.n_recent, **method_kw(args))
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
    out = h.outputs(T, dev)
    stream = torch.cuda.current_stream(dev)
    tokens_per_step = float(w.n_layers * w.n_kv_heads * (T - inp.pad.long()).sum().item())

    def step():
        h.event(inp.q, inp.k, inp.v, T, inp.pad, inp.n_carry, inp.credit, out["k_out"],
                out["v_out"], out["credit_out"], out["kept_idx"], out["n_kept"])

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
            h.mass(inp.q, inp.k, T, inp.pad, inp.n_carry, inp.credit, stage["credit_post"],
                   stage["mass"], stage["score"])
            h.segment_quota(stage["mass"], T, inp.pad, stage["seg_start"], stage["seg_len"],
                            stage["quota"], stage["n_seg"])
            h.select(stage["score"], T, inp.pad, stage["seg_start"], stage["seg_len"],
                     stage["quota"], stage["n_seg"], out["kept_idx"], out["n_kept"])
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
    lengths = (T - inp.pad.long()).cpu().numpy()
    flops_ev = bytes_ev = 0.0
    per_kernel_work = {}
    for Tv in lengths:
        f, b, pk = unit_work(w, int(Tv), T)
        n_u = w.n_layers * w.n_kv_heads
        flops_ev += f * n_u
        bytes_ev += b * n_u
        for name, (bound, fl, by) in pk.items():
            acc = per_kernel_work.setdefault(name, [bound, 0.0, 0.0])
            acc[1] += fl * n_u
            acc[2] += by * n_u
    total_kernel_ms = sum(k["total_ms"] for k in kernels) or 1.0
    krows = []
    for k in kernels:
        if not k["launches"]:
            continue
        bound, fl, by = per_kernel_work[k["name"]]
        avg_s = k["total_ms"] / k["launches"] / 1000.0
        if bound == "tensor":
            ach, peak, unit = fl / avg_s / 1e12, peaks["bf16_tflops"], "TFLOP/s"
        else:
            ach, peak, unit = by / avg_s / 1e9, peaks["hbm_gbs"], "GB/s"
        krows.append({"name": k["name"], "launches": k["launches"],
                      "avg_ms": 1000.0 * avg_s, "share": k["total_ms"] / total_kernel_ms,
                      "bound": bound, "achieved": ach, "peak": peak, "unit": unit,
                      "frac": ach / peak, "algorithmic_per_launch": fl if bound == "tensor" else by})
    dom = max(krows, key=lambda r: r["avg_ms"] * r["launches"])
    roofline = {"kernel": dom["name"], "bound": dom["bound"], "achieved": dom["achieved"],
                "peak": dom["peak"], "unit": dom["unit"], "frac": dom["frac"],
                "peak_source": f"{'bf16_tflops (burst)' if dom['bound'] == 'tensor' else 'hbm_gbs'}"
                               f" of {peak_src}",
                "traffic": read_traffic(dom["name"], w.name)}
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
        host_in = {k: getattr(inp, k).cpu().pin_memory() for k in
                   ("q", "k", "v", "credit", "pad", "n_carry")}
        host_out = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
                    for k, v in out.items()}
        dev_in = {k: getattr(inp, k) for k in ("q", "k", "v", "credit", "pad", "n_carry")}
        dev_in = {k: torch.empty_like(v) for k, v in dev_in.items()}  # staging, as a caller has
        lps = args.e2e_layers
        h.event_from_host(host_in, dev_in, host_out, out, T, layers_per_stage=lps)  # warm-up
        torch.cuda.synchronize(dev)
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(args.e2e_steps):
            h2d, d2h = h.event_from_host(host_in, dev_in, host_out, out, T, layers_per_stage=lps)
        f1.record(stream)
        torch.cuda.synchronize(dev)
        # V is read in place at the kept rows (page-locked host buffer)
        h2d += int(host_out["n_kept"].long().sum().item()) * w.head_dim * 2
        e2e_ms = f0.elapsed_time(f1) / args.e2e_steps
        e2e_ms, _ = reduce_over_ranks(e2e_ms, 0.0, dev)
        e2e = {"value": total_tokens / (e2e_ms / 1000.0), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "steps": args.e2e_steps,
               "path": f"kvc_event_host, pinned host buffers, {lps} layers per copy stage; "
                       "V read in place at the kept rows"}
        del host_in, host_out

    # ---- CPU oracle baseline on a bounded sample (rank 0, N = 1)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        p = oracle.RefParams(group=w.group, head_dim=w.head_dim, window=w.window,
                             budget=w.budget, n_sink=w.n_sink, n_recent=w.n_recent,
                             **method_kw(args))
        q_u = wl.q_units(inp.q, w)
        k_u = wl.units_of(inp.k, w)
        v_u = wl.units_of(inp.v, w)
        c_u = wl.units_of(inp.credit, w)
        pad_u = wl.unit_pad(inp)
        nc_u = wl.unit_n_carry(inp)
        rng = np.random.default_rng(0)
        order = rng.permutation(w.units)
        t0 = time.perf_counter()
        done = tokens = 0
        while done < len(order) and (time.perf_counter() - t0 < args.cpu_seconds or done == 0):
            u = int(order[done])
            oracle.event(p, wl.bf16_bits(q_u[u:u + 1]), wl.bf16_bits(k_u[u:u + 1]),
                         wl.bf16_bits(v_u[u:u + 1]), c_u[u:u + 1].cpu().numpy(),
                         pad_u[u:u + 1].cpu().numpy(), nc_u[u:u + 1].cpu().numpy())
            tokens += T - int(pad_u[u])
            done += 1
        dt = time.perf_counter() - t0
        cpu = {"value": tokens / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{done} of {w.units} units of the timed event (random, seed 0), "
                         f"same inputs, single-threaded C oracle (fp64); host copies included"}

    clocks = summarize_clocks(clock_rows, t_wall0, t_wall1)
    # kernels per traced entry (the paged compaction is four launches)
    launches = sum(r["launches"] * (4 if r["name"] == "compact_paged" else 1) for r in krows)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": warm, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(workload_config(w, T, args.ablation, args.paged, args.redundancy),
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
