"""kvc_mass_noalloc against kvc_mass (collected last on purpose).

kvc_mass_noalloc serves callers that cannot allocate device memory when they
compress (for instance an engine that has reserved all free memory for its KV
pool): it takes no handle and keeps its scratch in a fixed device array. It
runs the same kernels in the same launch shapes as kvc_mass, so its outputs must
equal kvc_mass's bit for bit on the same inputs, on two calls in a row with
different inputs (so stale scratch from the first call would show); one unit is
also checked against the oracle within the mass tolerance of the parity tests
(|a - b| <= 1e-4 |b| + 1e-9).  A request larger than the fixed scratch, and a
call without a status word, must be refused before anything is launched.
"""
import numpy as np
import pytest
import torch

import workload as wl

pytestmark = pytest.mark.gpu


def _close(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    fin = np.isfinite(b)
    assert np.array_equal(a[~fin], b[~fin])
    assert np.all(np.abs(a[fin] - b[fin]) <= 1e-4 * np.abs(b[fin]) + 1e-9)


def _run_both(kvc, w, seed, oracle=None):
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
        assert torch.equal(got[key], ref[key]), key
    if oracle is not None:
        # one unit (the last sequence's first head of layer 0) against the oracle
        u = (w.batch - 1) * w.n_kv_heads
        p = oracle.RefParams(group=w.group, head_dim=w.head_dim, window=w.window,
                             budget=w.budget, n_recent=w.n_recent)
        sl = slice(u, u + 1)
        m, s, c = oracle.mass(p, wl.bf16_bits(wl.q_units(inp.q, w)[sl]),
                              wl.bf16_bits(wl.units_of(inp.k, w)[sl]),
                              wl.units_of(inp.credit, w)[sl].cpu().numpy(),
                              wl.unit_pad(inp)[sl].cpu().numpy(),
                              wl.unit_n_carry(inp)[sl].cpu().numpy())
        U = w.units
        _close(got["mass"].reshape(U, T)[u].cpu().numpy(), m[0])
        _close(got["score"].reshape(U, T)[u].cpu().numpy(), s[0])
        _close(got["credit_post"].reshape(U, T)[u].cpu().numpy(), c[0])
    h.close()
    return cfg, inp


def test_noalloc_matches_mass_twice(ref):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import eviction_gb300 as kvc
    # a ragged batch first, then a different shape and seed on the same scratch
    w1 = wl.scaled(wl.CONFIGS["llama_ragged"], n_layers=1, batch=3, n_kv_heads=2, group=4,
                   prefill=(50, 400), generated=300, budget=300)
    w2 = wl.scaled(wl.CONFIGS["qwen_1l"], batch=2, n_kv_heads=2, T=1000)
    _run_both(kvc, w1, seed=5, oracle=ref)
    _run_both(kvc, w2, seed=6, oracle=ref)


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
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = kvc.mass_noalloc(cfg, small, small, w.T, i32, i32, f32, f32, f32, f32, status=status)
    assert rc == -2  # KVC_ERR_SHAPE, nothing launched


def test_noalloc_requires_status():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import eviction_gb300 as kvc
    w = wl.CONFIGS["tiny"]
    cfg = kvc.Config(1, 1, 1, w.group, w.head_dim, w.T, w.budget, window=w.window)
    small = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    i32 = torch.zeros(4, dtype=torch.int32, device="cuda")
    f32 = torch.zeros(4, dtype=torch.float32, device="cuda")
    rc = kvc.mass_noalloc(cfg, small, small, w.T, i32, i32, f32, f32, f32, f32)
    assert rc == -1  # KVC_ERR_ARG: the device failure reports need a status word
