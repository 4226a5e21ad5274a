"""The fused per-unit kernel (kvc_mass_select, units of up to 4096 slots) against
the stage entry points chained: mass, credit, score, segments, quotas, kept
indices and counts bit-identical, on every unit, across the shapes that pick
different code (slots per thread 4 / 8 / 16, the selection's gathered-key
search past 2048 slots, ragged padding with an all-padding sequence and a
sequence shorter than the sinks) and the method's ablations.  The whole event
(fused) is compared with kvc_compact after the stage chain the same way."""
import pytest
import torch

import eviction_gb300 as kvc
import workload as wl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

STAGE_KEYS = ("credit_post", "mass", "score", "seg_start", "seg_len", "quota", "n_seg")


def _bits(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t


def _same(a, b):
    return torch.equal(_bits(a), _bits(b))


def _inputs(name, over, pads=None, seed=3):
    w = wl.scaled(wl.CONFIGS[name], **over)
    inp = wl.generate(w, seed=seed)
    g = gu.to_device(inp)
    if pads is not None:
        for i, pv in enumerate(pads):
            g["pad"][i] = min(int(pv), inp.T) if pv is not None else g["pad"][i]
    return w, inp.T, g


def _run_fused(h, g, T):
    buf = h.stage_buffers(T)
    out = h.outputs(T)
    h.mass_select(g["q"], g["k"], T, g["pad"], g["n_carry"], g["credit"], buf["credit_post"],
                  buf["mass"], buf["score"], buf["seg_start"], buf["seg_len"], buf["quota"],
                  buf["n_seg"], out["kept_idx"], out["n_kept"])
    torch.cuda.synchronize()
    return buf, out


def _run_stages(h, g, T):
    buf = h.stage_buffers(T)
    out = h.outputs(T)
    h.mass(g["q"], g["k"], T, g["pad"], g["n_carry"], g["credit"], buf["credit_post"],
           buf["mass"], buf["score"])
    h.segment_quota(buf["mass"], T, g["pad"], buf["seg_start"], buf["seg_len"], buf["quota"],
                    buf["n_seg"])
    h.select(buf["score"], T, g["pad"], buf["seg_start"], buf["seg_len"], buf["quota"],
             buf["n_seg"], out["kept_idx"], out["n_kept"])
    torch.cuda.synchronize()
    return buf, out


def _kernels(h, fn):
    h.profile(True)
    h.profile_read(reset=True)
    fn()
    names = {k["name"]: k["launches"] for k in h.profile_read(reset=True) if k["launches"]}
    h.profile(False)
    return names


CASES = [
    # name, workload overrides, per-sequence pads (None = the generator's), config extras
    ("qwen_1l_T768", "qwen_1l", dict(batch=4), None, {}),           # 4 slots per thread
    ("tiny_d64", "tiny", {}, None, {}),
    ("qwen_T1536", "qwen_28l", dict(n_layers=2, batch=4, n_events=1), None, {}),  # 8 per thread
    ("qwen_T3000", "qwen_1l", dict(batch=3, T=3000, budget=1024), None, {}),      # 16, gathered keys
    ("qwen_T4096", "qwen_1l", dict(batch=2, T=4096, budget=2048), None, {}),
    ("llama_ragged", "llama_ragged", dict(n_layers=2, batch=8), None, {}),
    # an all-padding sequence, one shorter than the sinks, one of 40 slots
    ("edge_pads", "qwen_1l", dict(batch=4), [10 ** 6, 768 - 3, 768 - 40, 0], {}),
] + [(f"ablation_{a}", "qwen_1l", dict(batch=4), None, kw)
     for a, kw in kvc.ABLATIONS.items() if a != "none"]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_fused_matches_stage_chain(case):
    _, name, over, pads, extra = case
    w, T, g = _inputs(name, over, pads)
    h = kvc.Handle(gu.config_for(w, T, **extra))
    try:
        names = _kernels(h, lambda: _run_fused(h, g, T))
        assert names.get("mass_segment_select") == 1 and "segment_quota" not in names, names
        fb, fo = _run_fused(h, g, T)
        sb, so = _run_stages(h, g, T)
        for k in STAGE_KEYS:
            assert _same(fb[k], sb[k]), k
        assert _same(fo["kept_idx"], so["kept_idx"])
        assert _same(fo["n_kept"], so["n_kept"])
        assert int(fo["n_kept"].min()) >= 0
        # repeat: identical bits
        fb2, fo2 = _run_fused(h, g, T)
        for k in STAGE_KEYS:
            assert _same(fb[k], fb2[k]), k
        assert _same(fo["kept_idx"], fo2["kept_idx"])
        assert h.device_status() == 0
    finally:
        h.close()


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_event_fused_equals_stage_chain_and_compact(case):
    """kvc_event on the fused path (mass, segments and selection in one launch,
    then the gather) against the stage entry points and kvc_compact: compacted
    K, V, credit, kept indices and counts bit-identical (zero rows past n_kept,
    the all-padding sequence, head_dim 64 and 128 included)."""
    _, name, over, pads, extra = case
    w, T, g = _inputs(name, over, pads)
    h = kvc.Handle(gu.config_for(w, T, **extra))
    try:
        names = _kernels(h, lambda: gu.gpu_event(h, g, T))
        assert names.get("mass_segment_select") == 1 and names.get("gather_compact") == 1
        ev = gu.gpu_event(h, g, T)
        sb, so = _run_stages(h, g, T)
        out = h.outputs(T)
        h.compact(g["k"], g["v"], sb["credit_post"], T, so["kept_idx"], so["n_kept"],
                  out["k_out"], out["v_out"], out["credit_out"])
        torch.cuda.synchronize()
        for k in ("k_out", "v_out", "credit_out", "kept_idx", "n_kept"):
            src = out if k in ("k_out", "v_out", "credit_out") else so
            assert _same(ev[k], src[k]), k
        assert h.device_status() == 0
    finally:
        h.close()


def test_longer_units_take_the_stage_kernels():
    w, T, g = _inputs("qwen_1l", dict(batch=1, T=5000, budget=1024))
    h = kvc.Handle(gu.config_for(w, T))
    try:
        names = _kernels(h, lambda: _run_fused(h, g, T))
        assert "mass_segment_select" not in names
        assert names.get("segment_quota") == 1 and names.get("select_topk") == 1
        fb, fo = _run_fused(h, g, T)
        sb, so = _run_stages(h, g, T)
        for k in STAGE_KEYS:
            assert _same(fb[k], sb[k]), k
        assert _same(fo["kept_idx"], so["kept_idx"])
    finally:
        h.close()


def test_redundancy_mix_takes_the_stage_kernels():
    w, T, g = _inputs("qwen_1l", dict(batch=2))
    h = kvc.Handle(gu.config_for(w, T, redundancy_sigma=0.1))
    try:
        names = _kernels(h, lambda: _run_fused(h, g, T))
        assert "mass_segment_select" not in names and names.get("redundancy_score") == 1
        fb, fo = _run_fused(h, g, T)
        sb = h.stage_buffers(T)
        so = h.outputs(T)
        h.mass(g["q"], g["k"], T, g["pad"], g["n_carry"], g["credit"], sb["credit_post"],
               sb["mass"], sb["score"])
        h.segment_quota(sb["mass"], T, g["pad"], sb["seg_start"], sb["seg_len"], sb["quota"],
                        sb["n_seg"])
        h.redundancy_score(g["k"], sb["score"], T, g["pad"], sb["score"])
        h.select(sb["score"], T, g["pad"], sb["seg_start"], sb["seg_len"], sb["quota"],
                 sb["n_seg"], so["kept_idx"], so["n_kept"])
        torch.cuda.synchronize()
        for k in STAGE_KEYS:
            assert _same(fb[k], sb[k]), k
        assert _same(fo["kept_idx"], so["kept_idx"])
    finally:
        h.close()
