"""kvc_mass_noalloc against kvc_mass (collected last on purpose).

kvc_mass_noalloc serves callers that cannot allocate device memory when they
compress (for instance an engine that has reserved all free memory for its KV
pool): it takes no handle and keeps its scratch in a fixed device array. Here
its outputs must match kvc_mass on the same inputs within the mass tolerance
of the parity tests (|a - b| <= 1e-4 |b| + 1e-9), on two calls in a row with
different inputs (so stale scratch from the first call would show), and a
request larger than the fixed scratch must be refused.
"""
import numpy as np
import pytest
import torch

import workload as wl

pytestmark = pytest.mark.gpu


def _close(a, b):
    a = a.cpu().numpy().astype(np.float64)
    b = b.cpu().numpy().astype(np.float64)
    fin = np.isfinite(b)
    assert np.array_equal(a[~fin], b[~fin])
    assert np.all(np.abs(a[fin] - b[fin]) <= 1e-4 * np.abs(b[fin]) + 1e-9)


def _run_both(kvc, w, seed):
    inp = wl.generate(w, device="cuda", seed=seed)
    T = inp.T
    cfg = kvc.Config(w.n_layers, w.batch, w.n_kv_heads, w.group, w.head_dim, T, w.budget,
                     window=w.window, n_recent=w.n_recent)
    h = kvc.Handle(cfg)
    ref = h.stage_buffers(T)
    h.mass(inp.q, inp.k, T, inp.pad, inp.n_carry, inp.credit, ref["credit_post"], ref["mass"],
           ref["score"])
    got = {key: torch.full_like(ref[key], float("nan")) for key in ("mass", "score", "credit_post")}
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = kvc.mass_noalloc(cfg, inp.q, inp.k, T, inp.pad, inp.n_carry, inp.credit,
                          got["credit_post"], got["mass"], got["score"], status=status)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for key in got:
        _close(got[key], ref[key])
    h.close()
    return cfg, inp


def test_noalloc_matches_mass_twice():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import eviction_gb300 as kvc
    # a ragged batch first, then a different shape and seed on the same scratch
    w1 = wl.scaled(wl.CONFIGS["llama_ragged"], n_layers=1, batch=3, n_kv_heads=2, group=4,
                   prefill=(50, 400), generated=300, budget=300)
    w2 = wl.scaled(wl.CONFIGS["qwen_1l"], batch=2, n_kv_heads=2, T=1000)
    _run_both(kvc, w1, seed=5)
    _run_both(kvc, w2, seed=6)


def test_noalloc_rejects_oversize():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import eviction_gb300 as kvc
    # 28 layers x 32 sequences x 4 heads of 1536 slots need ~12M scratch floats > 1M
    w = wl.CONFIGS["qwen_28l"]
    cfg = kvc.Config(w.n_layers, w.batch, w.n_kv_heads, w.group, w.head_dim, w.T, w.budget,
                     window=w.window)
    small = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    i32 = torch.zeros(4, dtype=torch.int32, device="cuda")
    f32 = torch.zeros(4, dtype=torch.float32, device="cuda")
    rc = kvc.mass_noalloc(cfg, small, small, w.T, i32, i32, f32, f32, f32, f32)
    assert rc == -2  # KVC_ERR_SHAPE, nothing launched
