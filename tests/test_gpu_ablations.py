"""GPU parity of the ablation switches ("Adaptive Mass-Segmented KV Compression for
Long-Form Reasoning", Experiments, ablation table) against the oracle.

Same bars as the main parity tests: segments, quotas and kept sets bit-exact when
both sides get the same fp32 mass / score (the oracle's); end to end, kept sets
equal up to score near-ties.
"""
import numpy as np
import pytest
import torch

import workload as wl

pytestmark = pytest.mark.gpu

from tests import gpu_util as gu  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


SWITCHES = {
    "fixed_segments": dict(seg_fixed=32),
    "no_mass_quota": dict(quota_by_len=1),
    "fixed_and_length_quota": dict(seg_fixed=48, quota_by_len=1),
    "global_topk": dict(global_topk=1),
    "no_credit": dict(beta=1.0),
}

CASES = {
    "qwen_small": (wl.scaled(wl.CONFIGS["qwen_1l"], batch=2, n_kv_heads=2, T=1000), None),
    "ragged": (wl.scaled(wl.CONFIGS["llama_ragged"], n_layers=1, batch=5, n_kv_heads=2, group=4,
                         prefill=(10, 400), generated=300, budget=300), [0, 37, 250, 620, 700]),
}


def _inputs(name):
    w, pads = CASES[name]
    inp = wl.generate(w)
    if pads is not None:
        T = inp.T
        pad = torch.tensor([min(p, T) for p in pads], dtype=torch.int32)
        slot = torch.arange(T).view(1, 1, 1, T, 1)
        valid = slot >= pad.view(1, -1, 1, 1, 1)
        inp.k = torch.where(valid, inp.k, torch.zeros((), dtype=inp.k.dtype))
        inp.v = torch.where(valid, inp.v, torch.zeros((), dtype=inp.v.dtype))
        inp.pad = pad
        inp.n_carry = (T - pad).to(torch.int32)
    return w, inp


@pytest.fixture(scope="module")
def runs(ref):
    out = {}
    for name in CASES:
        w, inp = _inputs(name)
        for sw, kw in SWITCHES.items():
            p = gu.ref_params(ref, w, **kw)
            out[(name, sw)] = (w, inp, kw, ref.event(p, *gu.oracle_inputs(inp)))
    return out


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("sw", list(SWITCHES))
def test_segments_quotas_select_bit_exact(ref, runs, name, sw):
    import eviction_gb300 as kvc
    w, inp, kw, r = runs[(name, sw)]
    p = gu.ref_params(ref, w, **kw)
    T = inp.T
    h = kvc.Handle(gu.config_for(w, T, **kw))
    st, ln, qu, ns = gu.gpu_segment_quota(h, r["mass"], inp.pad.numpy(), T)
    assert np.array_equal(ns, r["n_seg"])
    assert np.array_equal(st, r["seg_start"]) and np.array_equal(ln, r["seg_len"])
    assert np.array_equal(qu, r["quota"])
    kept, nk = gu.gpu_select(h, r["score"], inp.pad.numpy(), T, r["seg_start"], r["seg_len"],
                             r["quota"], r["n_seg"])
    assert np.array_equal(nk, r["n_kept"]) and np.array_equal(kept, r["kept_idx"])
    if sw == "global_topk":
        assert np.all(r["n_seg"][r["n_kept"] > 0] == 1)


@pytest.mark.parametrize("sw", list(SWITCHES))
def test_event_end_to_end(ref, runs, sw):
    """The event under each switch against the oracle's chain through the
    end-to-end checker (GPU segments from the GPU's own mass)."""
    import eviction_gb300 as kvc
    w, inp, kw, r = runs[("qwen_small", sw)]
    p = gu.ref_params(ref, w, **kw)
    T = inp.T
    h = kvc.Handle(gu.config_for(w, T, **kw))
    g = gu.to_device(inp)
    out = gu.gpu_event(h, g, T)
    m, s, _ = gu.gpu_mass(h, g, T)
    st, ln, qu, ns = gu.gpu_segment_quota(h, m, inp.pad.numpy(), T)
    assert h.device_status() == 0
    U = w.units
    kept = out["kept_idx"].reshape(U, -1).cpu().numpy()
    nk = out["n_kept"].reshape(U).cpu().numpy()
    assert np.array_equal(nk, r["n_kept"])
    pads_u = wl.unit_pad(inp).numpy()
    for u in range(U):
        seg = dict(seg_start=st[u], seg_len=ln[u], quota=qu[u], n_seg=int(ns[u]))
        gu.check_unit_e2e(p, w, int(pads_u[u]), kept[u, :nk[u]], m[u], s[u], seg, r, u)


def test_switches_change_the_result(runs):
    """Each switch really changes the segmentation or the quotas (beta = 1 equals the
    method on a first event, whose credit is zero)."""
    for sw in ("fixed_segments", "no_mass_quota", "global_topk"):
        r = runs[("qwen_small", sw)][3]
        r2 = runs[("qwen_small", "no_credit")][3]
        assert not (np.array_equal(r["seg_start"], r2["seg_start"]) and
                    np.array_equal(r["quota"], r2["quota"]))
