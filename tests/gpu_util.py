"""Helpers shared by the GPU parity tests: run library stages on seeded inputs
and bring results back as numpy arrays. Inputs always come from the seeded
generator or from the oracle, never from the CUDA path."""
from __future__ import annotations

import numpy as np
import torch

import eviction_gb300 as kvc
import workload as wl
from tests import e2e_check


def config_for(w: wl.Workload, T: int, **kw) -> kvc.Config:
    return kvc.Config(w.n_layers, w.batch, w.n_kv_heads, w.group, w.head_dim, T, w.budget,
                      window=w.window, n_sink=w.n_sink, n_recent=w.n_recent, **kw)


def ref_params(ref, w: wl.Workload, **kw):
    return ref.RefParams(group=w.group, head_dim=w.head_dim, window=w.window, budget=w.budget,
                         n_sink=w.n_sink, n_recent=w.n_recent, **kw)


def to_device(inp: wl.Inputs, dev="cuda"):
    return {k: getattr(inp, k).to(dev).contiguous()
            for k in ("q", "k", "v", "credit", "pad", "n_carry")}


def oracle_inputs(inp: wl.Inputs):
    w = inp.w
    return (wl.bf16_bits(wl.q_units(inp.q, w)), wl.bf16_bits(wl.units_of(inp.k, w)),
            wl.bf16_bits(wl.units_of(inp.v, w)), wl.units_of(inp.credit, w).cpu().numpy(),
            wl.unit_pad(inp).cpu().numpy(), wl.unit_n_carry(inp).cpu().numpy())


def gpu_mass(h: kvc.Handle, g, T):
    buf = h.stage_buffers(T)
    h.mass(g["q"], g["k"], T, g["pad"], g["n_carry"], g["credit"], buf["credit_post"],
           buf["mass"], buf["score"])
    torch.cuda.synchronize()
    U = h.cfg.units
    return (buf["mass"].reshape(U, T).cpu().numpy(), buf["score"].reshape(U, T).cpu().numpy(),
            buf["credit_post"].reshape(U, T).cpu().numpy())


def gpu_segment_quota(h: kvc.Handle, mass_np, pad_b, T):
    cfg = h.cfg
    L, B, H = cfg.n_layers, cfg.batch, cfg.n_kv_heads
    buf = h.stage_buffers(T)
    mass = torch.from_numpy(np.ascontiguousarray(mass_np, np.float32)).reshape(L, B, H, T).cuda()
    pad = torch.as_tensor(pad_b, dtype=torch.int32).cuda()
    h.segment_quota(mass, T, pad, buf["seg_start"], buf["seg_len"], buf["quota"], buf["n_seg"])
    torch.cuda.synchronize()
    U, S = cfg.units, h.s_max(T)
    return tuple(buf[k].reshape(U, -1).cpu().numpy() if k != "n_seg"
                 else buf[k].reshape(U).cpu().numpy()
                 for k in ("seg_start", "seg_len", "quota", "n_seg"))


def gpu_select(h: kvc.Handle, score_np, pad_b, T, seg_start, seg_len, quota, n_seg):
    cfg = h.cfg
    L, B, H = cfg.n_layers, cfg.batch, cfg.n_kv_heads
    S = h.s_max(T)

    def dev_i(x, shape):
        return torch.from_numpy(np.ascontiguousarray(x, np.int32)).reshape(shape).cuda()

    score = torch.from_numpy(np.ascontiguousarray(score_np, np.float32)).reshape(L, B, H, T).cuda()
    kept = torch.empty((L, B, H, cfg.budget), dtype=torch.int32, device="cuda")
    nk = torch.empty((L, B, H), dtype=torch.int32, device="cuda")
    h.select(score, T, dev_i(pad_b, (B,)), dev_i(seg_start, (L, B, H, S)),
             dev_i(seg_len, (L, B, H, S)), dev_i(quota, (L, B, H, S)), dev_i(n_seg, (L, B, H)),
             kept, nk)
    torch.cuda.synchronize()
    return kept.reshape(cfg.units, -1).cpu().numpy(), nk.reshape(-1).cpu().numpy()


def gpu_event(h: kvc.Handle, g, T):
    out = h.outputs(T)
    h.event(g["q"], g["k"], g["v"], T, g["pad"], g["n_carry"], g["credit"], out["k_out"],
            out["v_out"], out["credit_out"], out["kept_idx"], out["n_kept"])
    torch.cuda.synchronize()
    return out


# the end-to-end checker lives in its own module (CPU-tested in test_e2e_check.py)
mass_close = e2e_check.mass_close
check_unit_e2e = e2e_check.check_unit_e2e
