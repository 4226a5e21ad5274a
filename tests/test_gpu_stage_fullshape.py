"""Bit-exact stage parity on EVERY unit at the launch shapes the benchmark times.

kvc_segment_quota and kvc_select run on full-size handles (the 28-layer Qwen
event: 3584 units, T = 1536; the long-context event: 448 units, T = 32768; the
Llama-shaped ragged batch: 16384 units, both left-padded to the longest sequence
and regrouped by length in groups of 8), and every unit's segments, quotas,
kept slots and counts must equal the oracle's bit for bit.  Both sides take the
same fp32 masses and scores, drawn by a seeded generator (peaky masses with
planted heavy runs and spikes; scores with many exact ties), so no GPU value is
ever an oracle input.  kvc_compact is checked on every unit of the Qwen shape
against a plain torch gather of the oracle's kept slots.

Sources: "Adaptive Mass-Segmented KV Compression for Long-Form Reasoning",
Method, Key designs 2-4.
"""
import os

import numpy as np
import pytest
import torch

import workload as wl

pytestmark = pytest.mark.gpu

from tests import gpu_util as gu  # noqa: E402

THREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def draw_mass_score(seed, U, T, pads_u):
    """Seeded fp32 masses (non-negative, summing to about 1 over the valid slots,
    zero on padding) and scores (-inf on padding) for U units: a power-law base,
    a few heavy runs and spikes; half the units get scores rounded to 1/64 so that
    exact ties are everywhere."""
    rng = np.random.default_rng(seed)
    slot = np.arange(T)[None, :]
    valid = slot >= pads_u[:, None]
    expo = rng.choice([1.0, 4.0, 12.0], size=(U, 1))
    w = rng.random((U, T)) ** expo
    n = np.maximum(T - pads_u, 1)
    for _ in range(4):                                   # heavy runs
        start = pads_u + (rng.random(U) * n).astype(np.int64)
        length = rng.integers(4, 160, U)
        run = (slot >= start[:, None]) & (slot < (start + length)[:, None])
        w += run * rng.random((U, 1)) * 8.0
    for _ in range(3):                                   # spikes
        at = np.minimum(pads_u + (rng.random(U) * n).astype(np.int64), T - 1)
        w[np.arange(U), at] += rng.random(U) * 0.05 * T
    w = np.where(valid, w, 0.0)
    tot = w.sum(1, keepdims=True)
    mass = np.where(tot > 0, w / np.where(tot > 0, tot, 1.0), 0.0).astype(np.float32)
    s = rng.random((U, T)) * 3.0
    tied = rng.random(U) < 0.5
    s[tied] = np.floor(s[tied] * 64.0) / 64.0
    score = np.where(valid, s, -np.inf).astype(np.float32)
    return mass, score


def _stage_parity(ref, w, T, pad_b, seed):
    import eviction_gb300 as kvc
    p = gu.ref_params(ref, w)
    U = w.units
    pads_u = np.broadcast_to(np.asarray(pad_b, np.int64)[None, :, None],
                             (w.n_layers, w.batch, w.n_kv_heads)).reshape(U)
    mass, score = draw_mass_score(seed, U, T, pads_u)
    h = kvc.Handle(gu.config_for(w, T))
    st, ln, qu, ns = gu.gpu_segment_quota(h, mass, pad_b, T)
    rs, rl, rq, rn = ref.segment_quota(p, mass, pads_u.astype(np.int32), threads=THREADS)
    bad = np.flatnonzero((ns != rn) | np.any(st != rs, 1) | np.any(ln != rl, 1)
                         | np.any(qu != rq, 1))
    assert bad.size == 0, f"{w.name}: segments/quotas differ on {bad.size} of {U} units ({bad[:8]})"
    kept, nk = gu.gpu_select(h, score, pad_b, T, rs, rl, rq, rn)
    kr, nr = ref.select(p, score, pads_u.astype(np.int32), rs, rl, rq, rn, threads=THREADS)
    bad = np.flatnonzero((nk != nr) | np.any(kept != kr, 1))
    assert bad.size == 0, f"{w.name}: kept slots differ on {bad.size} of {U} units ({bad[:8]})"
    assert h.device_status() == 0
    print(f"{w.name} T={T}: {U} units bit-exact (segments, quotas, kept slots)")
    return h, kr, nr


def test_qwen_28l_every_unit(ref):
    import eviction_gb300 as kvc
    w = wl.CONFIGS["qwen_28l"]
    T = w.budget + w.interval
    h, kept, nk = _stage_parity(ref, w, T, np.zeros(w.batch, np.int64), seed=31)
    # compaction of every unit against a plain gather of the oracle's kept slots
    U, d = w.units, w.head_dim
    g = torch.Generator(device="cuda").manual_seed(5)
    k = torch.randn((w.n_layers, w.batch, w.n_kv_heads, T, d), generator=g,
                    device="cuda").to(torch.bfloat16)
    v = torch.randn(k.shape, generator=g, device="cuda").to(torch.bfloat16)
    c = torch.rand((w.n_layers, w.batch, w.n_kv_heads, T), generator=g, device="cuda")
    kept_d = torch.from_numpy(kept).reshape(w.n_layers, w.batch, w.n_kv_heads, -1).cuda()
    nk_d = torch.from_numpy(nk).reshape(w.n_layers, w.batch, w.n_kv_heads).cuda()
    out = h.outputs(T)
    h.compact(k, v, c, T, kept_d, nk_d, out["k_out"], out["v_out"], out["credit_out"])
    torch.cuda.synchronize()
    assert h.device_status() == 0
    idx = kept_d.reshape(U, -1).long()
    live = idx >= 0
    src = idx.clamp(min=0)
    for name, x, y in (("k", k, out["k_out"]), ("v", v, out["v_out"])):
        ref_rows = torch.gather(x.reshape(U, T, d), 1, src[:, :, None].expand(-1, -1, d))
        ref_rows = torch.where(live[:, :, None], ref_rows, torch.zeros((), dtype=x.dtype,
                                                                        device="cuda"))
        assert torch.equal(y.reshape(U, -1, d).view(torch.int16),
                           ref_rows.view(torch.int16)), name
    ref_c = torch.where(live, torch.gather(c.reshape(U, T), 1, src), torch.zeros((), device="cuda"))
    assert torch.equal(out["credit_out"].reshape(U, -1), ref_c)


def test_long_every_unit(ref):
    w = wl.CONFIGS["long"]
    _stage_parity(ref, w, w.T, np.zeros(w.batch, np.int64), seed=32)


def test_llama_ragged_every_unit_padded_and_grouped(ref):
    w = wl.CONFIGS["llama_ragged"]
    lengths = wl.sequence_lengths(w).numpy()
    T = int(lengths.max())
    _stage_parity(ref, w, T, T - lengths, seed=33)
    by_len = np.argsort(lengths, kind="stable")
    for g0 in range(0, w.batch, 8):
        grp = by_len[g0:g0 + 8]
        Tg = int(lengths[grp].max())
        gw = wl.scaled(w, batch=len(grp), name=f"llama_ragged group {g0 // 8}")
        _stage_parity(ref, gw, Tg, Tg - lengths[grp], seed=34 + g0)
