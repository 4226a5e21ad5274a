"""Seeded synthetic workloads for the KV-cache compression event.

This module only draws random inputs; it holds none of the method's arithmetic.
Both the CUDA library's tests/benchmark and the oracle's tests take their inputs
from here.

The pages measure on reasoning traces of DeepSeek-R1-Distill-Qwen-7B / Llama-8B
(MATH-500, AIME, GSM8K). Those models and datasets are not used. The synthetic
caches below take only their shapes (model dimensions, budgets, compression
interval 512, query window 128 -- "Adaptive Mass-Segmented KV Compression for
Long-Form Reasoning", Loss function / training strategy) and plant regions of
keys aligned with the window's query mean so that attention mass is non-uniform.

Recipe (all seeded with torch generators on the target device):
  * Q, K, V ~ N(0, 1), rounded to bf16 (round to nearest even);
  * per unit (layer, sequence, KV head), u_hat = unit mean of the group's G*W
    window queries; each planted region adds a * sqrt(d) * u_hat to its keys,
    a ~ LogNormal(0, 0.7); region starts are uniform in
    [n_sink + pad, T - n_recent - len]; overlaps add up;
  * left padding holds zeros;
  * credit starts at zeros with every valid slot "carried" (first event).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    n_layers: int
    batch: int
    n_kv_heads: int
    group: int
    head_dim: int
    T: int                      # cache slots per unit (padded length)
    window: int
    budget: int
    n_recent: int
    n_sink: int = 4
    regions: tuple = (10, 20)   # inclusive range of planted regions per unit
    region_len: tuple = ("uniform", 16, 128)  # or ("geometric", mean)
    prefill: Optional[tuple] = None  # ragged: prefill ~ U[lo, hi] + `generated`
    generated: int = 512
    n_events: int = 1
    interval: int = 512
    seed: int = 1

    @property
    def units(self) -> int:
        return self.n_layers * self.batch * self.n_kv_heads

    @property
    def n_q_heads(self) -> int:
        return self.n_kv_heads * self.group


# The five workloads, smallest first.
CONFIGS = {
    # 1 layer, 1 sequence, 1 KV head, 1 query head, d 64, 256 + 512 slots, W 32.
    "tiny": Workload("tiny", 1, 1, 1, 1, 64, 768, 32, 256, n_recent=32, regions=(6, 6),
                     seed=0),
    # Qwen-7B-shaped single layer.
    "qwen_1l": Workload("qwen_1l", 1, 8, 4, 7, 128, 768, 128, 256, n_recent=64),
    # Qwen-7B-shaped, 28 layers, 1024 kept + 512 new slots, 4 events.
    "qwen_28l": Workload("qwen_28l", 28, 32, 4, 7, 128, 1536, 128, 1024, n_recent=64,
                         n_events=4),
    # Llama-8B-shaped ragged batch: prefill U[100, 600] + 512 generated, left padded.
    "llama_ragged": Workload("llama_ragged", 32, 64, 8, 4, 128, 0, 128, 512, n_recent=64,
                             prefill=(100, 600)),
    # Long context: 32768 slots -> 4096, 200 regions of geometric length (mean 96).
    "long": Workload("long", 28, 4, 4, 7, 128, 32768, 128, 4096, n_recent=256,
                     regions=(200, 200), region_len=("geometric", 96)),
}


def scaled(w: Workload, **kw) -> Workload:
    """The same recipe at other sizes (parity tests at oracle-friendly sizes)."""
    return replace(w, **kw)


@dataclass
class Inputs:
    """One event's inputs, layer-stacked as the library takes them.

    q [L,B,Hq,W,d] bf16; k, v [L,B,H,T,d] bf16; credit [L,B,H,T] f32;
    pad, n_carry [B] int32.
    """
    w: Workload
    T: int
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    credit: torch.Tensor
    pad: torch.Tensor
    n_carry: torch.Tensor
    lengths: Optional[torch.Tensor] = None  # valid lengths [B]


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def sequence_lengths(w: Workload, device="cpu") -> torch.Tensor:
    """Valid lengths per sequence [B] (int64 on `device`)."""
    if w.prefill is None:
        return torch.full((w.batch,), w.T, dtype=torch.int64, device=device)
    g = _gen("cpu", w.seed * 7919 + 17)
    lo, hi = w.prefill
    pre = torch.randint(lo, hi + 1, (w.batch,), generator=g)
    return (pre + w.generated).to(device)


def _region_profile(w: Workload, g, device, B, H, T, lo, span_end):
    """Amplitude profile amp[B,H,T]: sum of planted region amplitudes per slot.

    lo [B] = first slot a region may start at; span_end = last slot + 1 a region
    may reach (per sequence, [B]).
    """
    rmin, rmax = w.regions
    R = rmax
    count = torch.randint(rmin, rmax + 1, (B, H, 1), generator=g, device=device)
    active = (torch.arange(R, device=device).view(1, 1, R) < count).float()
    if w.region_len[0] == "uniform":
        _, lmin, lmax = w.region_len
        length = torch.randint(lmin, lmax + 1, (B, H, R), generator=g, device=device)
    else:
        mean = w.region_len[1]
        length = torch.empty((B, H, R), device=device).geometric_(1.0 / mean, generator=g)
        length = length.to(torch.int64)
    lo = lo.view(B, 1, 1).to(torch.int64)
    room = (span_end.view(B, 1, 1).to(torch.int64) - lo).clamp(min=0)
    length = torch.minimum(length, room)
    hi = lo + room - length                      # last admissible start
    u = torch.rand((B, H, R), generator=g, device=device)
    start = lo + torch.floor(u * (hi - lo + 1).float()).to(torch.int64)
    start = torch.minimum(start, hi)
    amp = torch.exp(0.7 * torch.randn((B, H, R), generator=g, device=device)) * active
    diff = torch.zeros((B, H, T + 1), device=device)
    diff.scatter_add_(2, start, amp)
    diff.scatter_add_(2, start + length, -amp)
    regions = (start, length, (active > 0) & (length > 0))
    return torch.cumsum(diff, dim=2)[:, :, :T], regions


def _layer(w: Workload, g, device, T, lengths, region_lo_offset=None):
    B, H, G, W, d = w.batch, w.n_kv_heads, w.group, w.window, w.head_dim
    pad = (T - lengths).to(device)
    q = torch.randn((B, H * G, W, d), generator=g, device=device).to(torch.bfloat16)
    k = torch.randn((B, H, T, d), generator=g, device=device)
    v = torch.randn((B, H, T, d), generator=g, device=device)
    u_hat = q.float().view(B, H, G * W, d).mean(dim=2)
    u_hat = u_hat / u_hat.norm(dim=-1, keepdim=True).clamp(min=1e-12)
    if region_lo_offset is None:
        lo = pad + w.n_sink
    else:
        lo = torch.full_like(pad, region_lo_offset)
    amp, regions = _region_profile(w, g, device, B, H, T, lo, torch.full_like(pad, T - w.n_recent))
    k = k + amp.unsqueeze(-1) * math.sqrt(d) * u_hat.unsqueeze(2)
    slot = torch.arange(T, device=device).view(1, 1, T, 1)
    valid = slot >= pad.view(B, 1, 1, 1)
    k = torch.where(valid, k, torch.zeros((), device=device)).to(torch.bfloat16)
    v = torch.where(valid, v, torch.zeros((), device=device)).to(torch.bfloat16)
    return q, k, v, regions


def _stack_regions(regs):
    """[(start, length, active) per layer] -> dict of [L, B, H, R] tensors."""
    return {"start": torch.stack([r[0] for r in regs]), "length": torch.stack([r[1] for r in regs]),
            "active": torch.stack([r[2] for r in regs])}


def generate(w: Workload, device="cpu", seed: Optional[int] = None, return_regions=False):
    """First-event inputs of workload `w` on `device` (and, if asked, the planted
    regions: slot start, length and an active flag, [L, B, H, R] each)."""
    seed = w.seed if seed is None else seed
    lengths = sequence_lengths(w, device)
    T = int(lengths.max().item()) if w.prefill is not None else w.T
    g = _gen(device, seed)
    qs, ks, vs, regs = [], [], [], []
    for _ in range(w.n_layers):
        q, k, v, reg = _layer(w, g, device, T, lengths)
        qs.append(q)
        ks.append(k)
        vs.append(v)
        regs.append(reg)
    q = torch.stack(qs)
    k = torch.stack(ks)
    v = torch.stack(vs)
    pad = (T - lengths).to(torch.int32)
    credit = torch.zeros((w.n_layers, w.batch, w.n_kv_heads, T), dtype=torch.float32,
                         device=device)
    inp = Inputs(w, T, q, k, v, credit, pad, (T - pad).to(torch.int32), lengths)
    return (inp, _stack_regions(regs)) if return_regions else inp


def next_event(w: Workload, prev: Inputs, k_out, v_out, credit_out, n_kept, event_index: int,
               seed: Optional[int] = None, return_regions=False):
    """Inputs of the next event: the compacted cache plus `interval` fresh slots.

    The fresh slots follow the same law (N(0,1) keys with planted regions aligned
    with the new window's query mean); the compacted credit is carried and the
    fresh slots are new (they start at their current mass). Requires every
    sequence to have kept a full budget (no padding after compaction).
    """
    device = k_out.device
    seed = (w.seed if seed is None else seed) * 1000003 + event_index
    g = _gen(device, seed)
    Kb, I = w.budget, w.interval
    assert bool((n_kept == Kb).all()), "next_event needs full-budget compaction"
    T = Kb + I
    fresh_w = replace(w, n_recent=0, n_sink=0)
    qs, ks, vs, regs = [], [], [], []
    lengths_fresh = torch.full((w.batch,), I, dtype=torch.int64, device=device)
    for _ in range(w.n_layers):
        q, kf, vf, reg = _layer(fresh_w, g, device, I, lengths_fresh, region_lo_offset=0)
        qs.append(q)
        ks.append(kf)
        vs.append(vf)
        regs.append((reg[0] + Kb, reg[1], reg[2]))  # slots of the fresh part
    q = torch.stack(qs)
    k = torch.cat([k_out, torch.stack(ks)], dim=3).contiguous()
    v = torch.cat([v_out, torch.stack(vs)], dim=3).contiguous()
    credit = torch.cat([credit_out, torch.zeros(credit_out.shape[:3] + (I,),
                                                device=device)], dim=3).contiguous()
    pad = torch.zeros((w.batch,), dtype=torch.int32, device=device)
    n_carry = torch.full((w.batch,), Kb, dtype=torch.int32, device=device)
    lengths = torch.full((w.batch,), T, dtype=torch.int64, device=device)
    inp = Inputs(w, T, q, k, v, credit, pad, n_carry, lengths)
    return (inp, _stack_regions(regs)) if return_regions else inp


# ---- unit-major views (for the oracle, which works on compact [U, ...]) --------

def unit_index(w: Workload, l: int, b: int, h: int) -> int:
    return (l * w.batch + b) * w.n_kv_heads + h


def units_of(x: torch.Tensor, w: Workload) -> torch.Tensor:
    """[L,B,H,...] -> [U, ...] with U = L*B*H (unit-major, as the oracle takes it)."""
    return x.reshape(w.n_layers * w.batch * w.n_kv_heads, *x.shape[3:])


def q_units(q: torch.Tensor, w: Workload) -> torch.Tensor:
    """Window queries [L,B,Hq,W,d] -> [U,G,W,d]; query head h*G+g belongs to KV head h."""
    return q.reshape(w.n_layers * w.batch * w.n_kv_heads, w.group, w.window, q.shape[-1])


def unit_pad(inp: Inputs) -> torch.Tensor:
    """Per-unit padding [U] from per-sequence padding [B]."""
    w = inp.w
    return inp.pad.view(1, w.batch, 1).expand(w.n_layers, w.batch, w.n_kv_heads).reshape(-1)


def unit_n_carry(inp: Inputs) -> torch.Tensor:
    w = inp.w
    return inp.n_carry.view(1, w.batch, 1).expand(w.n_layers, w.batch,
                                                  w.n_kv_heads).reshape(-1)


def bf16_bits(x: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (on the host)."""
    return x.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")
