"""Helpers shared by the GPU parity tests: run library stages on seeded inputs
and bring results back as numpy arrays. Inputs always come from the seeded
generator or from the oracle, never from the CUDA path."""
from __future__ import annotations

import numpy as np
import torch

import eviction_gb300 as kvc
import workload as wl


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


def mass_close(gpu, ref, rtol=1e-4, atol=1e-9):
    """|gpu - ref| <= rtol*|ref| + atol elementwise; returns (ok, worst relative error)."""
    finite = np.isfinite(ref)
    with np.errstate(invalid="ignore"):
        err = np.abs(gpu.astype(np.float64) - ref.astype(np.float64))
    bound = rtol * np.abs(ref.astype(np.float64)) + atol
    ok = bool(np.all(err[finite] <= bound[finite])) and bool(
        np.array_equal(gpu[~finite], ref[~finite]))
    rel = float(np.max(err[finite] / np.maximum(np.abs(ref[finite]), 1e-30))) if finite.any() else 0.0
    return ok, rel


def check_unit_e2e(p, w: wl.Workload, pad_u: int, kept_g, mass_g, score_g, seg_g, r, i):
    """One unit's end-to-end result against oracle run `r` (row i).

    kept_g: the GPU's kept slots (ascending); mass_g / score_g: the GPU's fp32
    m_used and score; seg_g: the GPU's segments for the unit (dict with
    seg_start, seg_len, quota rows and n_seg) from its own segment kernel on its
    own mass.  Nothing from the GPU is fed to the oracle.  Checks:
      1. m_used and score within 1e-4 relative (+1e-9) of the oracle's;
      2. identical kept sets, or, where the GPU's segments and quotas equal the
         oracle's, kept sets that differ only by swapped pairs at score near-ties
         (gap at most 1e-5 of G*W, the total usage scale);
      3. where the segments differ, the oracle's own fp64 cumulative mass lies
         within 1e-5 of a cut threshold k*delta at the first differing boundary
         (a rounding-order shift inside the mass tolerance); where only quotas
         differ, at most two units moved between segments.
    Returns "identical", "near_tie" or "shifted".
    """
    ok_m, rel_m = mass_close(mass_g, r["mass"][i])
    ok_s, rel_s = mass_close(score_g, r["score"][i])
    assert ok_m and ok_s, f"unit row {i}: mass rel {rel_m:.3g}, score rel {rel_s:.3g}"
    kept_r = r["kept_idx"][i, :r["n_kept"][i]]
    if np.array_equal(kept_r, kept_g):
        return "identical"
    ns_g, ns_r = int(seg_g["n_seg"]), int(r["n_seg"][i])
    st_g, st_r = seg_g["seg_start"][:ns_g], r["seg_start"][i, :ns_r]
    same_seg = ns_g == ns_r and np.array_equal(st_g, st_r) and np.array_equal(
        seg_g["seg_len"][:ns_g], r["seg_len"][i, :ns_r])
    a, b = set(kept_g.tolist()), set(kept_r.tolist())
    only_g, only_r = sorted(a - b), sorted(b - a)
    assert len(only_g) == len(only_r)
    if same_seg and np.array_equal(seg_g["quota"][:ns_g], r["quota"][i, :ns_r]):
        s = r["score"][i]
        gap = max(abs(float(s[x]) - float(s[y])) for x, y in zip(only_g, only_r))
        tol = 1e-5 * w.group * w.window
        assert gap <= tol, f"unit row {i}: kept sets differ beyond near-ties ({gap:.3g})"
        return "near_tie"
    if same_seg:
        moved = int(np.abs(seg_g["quota"][:ns_g] - r["quota"][i, :ns_r]).sum())
        assert moved <= 4, f"unit row {i}: quotas differ by {moved} units"
        return "shifted"
    # first differing segment start, in valid-slot offsets
    n = min(ns_g, ns_r)
    k0 = next((k for k in range(n) if st_g[k] != st_r[k]), n)
    cuts = sorted({int(st_g[k0]) if k0 < ns_g else int(mass_g.shape[0]),
                   int(st_r[k0]) if k0 < ns_r else int(mass_g.shape[0])})
    m = r["mass"][i][pad_u:].astype(np.float64)
    cum = np.cumsum(m) / m.sum()
    lo, hi = max(cuts[0] - pad_u - 2, 0), min(cuts[1] - pad_u + 1, len(cum))
    levels = np.arange(1, int(1.0 / p.delta) + 1) * p.delta
    near = np.min(np.abs(cum[lo:hi, None] - levels[None, :])) if hi > lo else 1.0
    assert near <= 1e-5, f"unit row {i}: segments differ away from a cut threshold ({near:.3g})"
    return "shifted"
