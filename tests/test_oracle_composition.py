"""Pin of the oracle's composition of steps 1-2 (usage -> fill -> score / pools ->
mass -> EMA credit -> mixed mass), the part of ``kvc_ref_mass`` that no per-step pin
covers.

The expected values come from an independent fp64 pipeline written with torch
library routines, in the order the pages give:
  * "Adaptive Mass-Segmented KV Compression for Long-Form Reasoning", Method,
    Key design 1: usage of each cache position by the W most recent queries,
    unseen entries filled with the window maximum, a small average pool, the mass
    equation m = (max(u, 0) + eps) / sum, the EMA credit and the beta mix;
  * "RefreshKV: Updating Small KV Cache During Long-form Generation", A2 and A6:
    the selection score is the attention max-pooled over neighbours, kernel 7;
  * "SkipKV: ...", A2 Method details: query head i reads KV head floor(i/n),
    padding masked out.
Each row's softmax is ``torch.softmax`` over the slots the query sees, the pools
are ``torch.nn.functional.max_pool1d`` / ``avg_pool1d``.  A wiring mistake in the
oracle (score pooled from u instead of a, fill added after pooling, credit mixed
before normalisation, new slots not restarted at their mass) changes these values by far more than the fp32 rounding allowed here,
and ``test_composition_detects_wiring_mistakes`` shows it for each of them.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import workload as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits_to_f64(bits):
    """bf16 bit patterns -> fp64 tensor (exact: bf16 is the top half of an fp32)."""
    f32 = (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)
    return torch.from_numpy(f32.astype(np.float64))


def _torch_pipeline(q, k, c_in, pad, n_carry, lam, beta, eps, scale=None, *,
                    score_from="a", fill_after_pool=False, mix_unnormalised=False,
                    restart_new=True):
    """Steps 1-2 of one unit in fp64 torch: q [G, W, d], k [T, d], c_in [T].

    The keyword switches plant the wiring mistakes the pin must catch; the
    defaults are the method as the pages state it."""
    G, W, d = q.shape
    T = k.shape[0]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    n = T - pad
    rows, seen_mask = [], []
    for h in range(G):
        for j in range(W):
            qpos = T - W + j
            if qpos < pad:
                continue                       # absent query (its slot is padding)
            logits = scale * (k[pad:qpos + 1] @ q[h, j])
            p = torch.zeros(T, dtype=torch.float64)
            p[pad:qpos + 1] = torch.softmax(logits, dim=0)
            rows.append(p)
            m = torch.zeros(T, dtype=torch.bool)
            m[pad:qpos + 1] = True
            seen_mask.append(m)
    P = torch.stack(rows)                      # [R, T]
    S = torch.stack(seen_mask)
    fill = P.max()                             # largest probability over the window
    unseen = (~S) & (torch.arange(T) >= pad)[None, :]
    a_seen = P.sum(0)
    a = a_seen + fill * unseen.sum(0)
    valid = a[pad:]
    pooled_src = a_seen[pad:] if fill_after_pool else valid
    u = F.avg_pool1d(pooled_src[None, None], 5, 1, 2, count_include_pad=True)[0, 0]
    if fill_after_pool:
        u = u + fill * unseen.sum(0)[pad:]
    score_src = valid if score_from == "a" else u
    s_valid = F.max_pool1d(score_src[None, None], 7, 1, 3)[0, 0]
    m_v = (torch.clamp(u, min=0.0) + eps)
    m_v = m_v / m_v.sum()
    c_prior = c_in[pad:].clone()
    if restart_new:
        c_prior[n_carry:] = m_v[n_carry:]
    c_v = lam * c_prior + (1 - lam) * m_v
    c_n = c_v if mix_unnormalised else c_v / c_v.sum()
    mu = beta * m_v + (1 - beta) * c_n
    mu = mu / mu.sum()
    out = {}
    for name, v, fillv in (("mass", mu, 0.0), ("score", s_valid, -math.inf),
                           ("credit_post", c_v, 0.0)):
        full = torch.full((T,), fillv, dtype=torch.float64)
        full[pad:] = v
        out[name] = full.numpy()
    return out


def _cases():
    """Seeded units with planted regions: pads (the last one leaves only 10 valid
    slots, so 14 of the 24 window queries sit in the padding and are absent),
    carried and new credit, GQA groups of 1 and 3."""
    tiny = wl.generate(wl.scaled(wl.CONFIGS["tiny"], T=200, budget=64, window=16,
                                 regions=(3, 3)))
    grp = wl.generate(wl.scaled(wl.CONFIGS["qwen_1l"], batch=3, n_kv_heads=1, group=3,
                                head_dim=32, T=150, window=24, budget=50, regions=(2, 4)))
    out = []
    for inp, pads, carry in ((tiny, [0], [200]), (grp, [0, 37, 140], [100, 13, 5])):
        w = inp.w
        q = wl.bf16_bits(wl.q_units(inp.q, w))
        k = wl.bf16_bits(wl.units_of(inp.k, w))
        U, T = k.shape[0], k.shape[1]
        rng = np.random.default_rng(5)
        credit = (rng.random((U, T)) * 2e-3).astype(np.float32)
        for u in range(U):
            b = (u // w.n_kv_heads) % w.batch
            pad = pads[b]
            k[u, :pad] = 0
            credit[u, :pad] = 0
            out.append((w, q[u], k[u], credit[u], pad, min(carry[b], T - pad)))
    return out


@pytest.mark.parametrize("case", range(4))
def test_mass_composition_matches_torch_pipeline(ref, case):
    """m_used, score and post-EMA credit of kvc_ref_mass against the torch pipeline,
    elementwise within fp32 rounding (the oracle returns fp32)."""
    w, q, k, credit, pad, n_carry = _cases()[case]
    p = ref.RefParams(group=w.group, head_dim=w.head_dim, window=w.window, budget=w.budget,
                      lam=0.9, beta=0.9, eps=1e-6)
    m, s, c = ref.mass(p, q[None], k[None], credit[None], np.array([pad], np.int32),
                       np.array([n_carry], np.int32))
    exp = _torch_pipeline(_bits_to_f64(q), _bits_to_f64(k),
                          torch.from_numpy(credit.astype(np.float64)), pad, n_carry,
                          float(np.float32(0.9)), float(np.float32(0.9)),
                          float(np.float32(1e-6)))
    for name, got in (("mass", m[0]), ("score", s[0]), ("credit_post", c[0])):
        e = exp[name]
        fin = np.isfinite(e)
        assert np.array_equal(np.isfinite(got), fin), name
        assert np.all(got[~fin] == e[~fin]), name
        np.testing.assert_allclose(got[fin].astype(np.float64), e[fin], rtol=2e-7, atol=1e-30,
                                   err_msg=name)


@pytest.mark.parametrize("mistake", ["score_from_u", "fill_after_pool", "mix_unnormalised",
                                     "no_restart"])
def test_composition_detects_wiring_mistakes(ref, mistake):
    """The pin has teeth: each plausible wiring mistake, planted in the torch
    pipeline, moves some value far outside the tolerance the pin uses."""
    w, q, k, credit, pad, n_carry = _cases()[1]
    p = ref.RefParams(group=w.group, head_dim=w.head_dim, window=w.window, budget=w.budget)
    m, s, c = ref.mass(p, q[None], k[None], credit[None], np.array([pad], np.int32),
                       np.array([n_carry], np.int32))
    kw = {"score_from_u": dict(score_from="u"), "fill_after_pool": dict(fill_after_pool=True),
          "mix_unnormalised": dict(mix_unnormalised=True),
          "no_restart": dict(restart_new=False)}[mistake]
    bad = _torch_pipeline(_bits_to_f64(q), _bits_to_f64(k),
                          torch.from_numpy(credit.astype(np.float64)), pad, n_carry,
                          float(np.float32(0.9)), float(np.float32(0.9)),
                          float(np.float32(1e-6)), **kw)
    worst = 0.0
    for name, got in (("mass", m[0]), ("score", s[0]), ("credit_post", c[0])):
        e = bad[name]
        fin = np.isfinite(e) & np.isfinite(got)
        rel = np.abs(got[fin] - e[fin]) / np.maximum(np.abs(e[fin]), 1e-30)
        worst = max(worst, float(rel.max()))
    assert worst > 1e-3, f"{mistake}: planted mistake not detected ({worst:.3g})"


def _golden(name):
    vals = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *rest = line.split()
        vals[key] = [Fraction(x) for x in rest]
    return vals


def test_credit_mix_closed_form_beta_09(ref):
    """A hand-derived case at lambda = beta = 0.9 with partly carried, nonzero
    credit (tests/golden/credit_mix_case.txt): every value is an exact fraction."""
    g = _golden("credit_mix_case.txt")
    m = np.array([float(x) for x in g["m"]])
    c_in = np.array([float(x) for x in g["c_in"]])
    n_carry = int(g["n_carry"][0])
    c, mu = ref.credit(m, c_in, pad=0, n_carry=n_carry, lam=0.9, beta=0.9)
    np.testing.assert_allclose(c, [float(x) for x in g["expected_c"]], rtol=1e-14)
    np.testing.assert_allclose(mu, [float(x) for x in g["expected_m_used"]], rtol=1e-14)
