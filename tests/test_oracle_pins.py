"""Pins of the CPU oracle against what the pages and mathematics fix.

Nothing here compares the oracle with itself: every expected value comes from a
closed form, a library routine (torch softmax / pooling / index_select, numpy
sort), exact rational arithmetic, Python's own IEEE doubles, brute-force
enumeration or the worked example
of "Adaptive Mass-Segmented KV Compression for Long-Form Reasoning" (section
"A complete example").
"""
import itertools
import math
import os
import zlib
from fractions import Fraction

import numpy as np
import pytest
import torch

from tests import threshold_cases

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    cases, cur = {}, None
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        if key == "case":
            cur = cases.setdefault(vals[0], {})
            continue
        tgt = cur if cur is not None else cases
        tgt[key] = [float(v) if "." in v else int(v) for v in vals]
    return cases


# ---------------------------------------------------------------- step 1: usage

def test_usage_single_query_is_softmax(ref):
    """W = 1, G = 1: the last query sees every slot, a = softmax(q K^T / sqrt(d))."""
    rng = np.random.default_rng(1)
    for pad in (0, 5):
        q = rng.standard_normal((1, 1, 16))
        k = rng.standard_normal((40, 16))
        a, fill = ref.usage(q, k, pad=pad)
        logits = torch.tensor(k[pad:] @ q[0, 0]) / math.sqrt(16)
        expect = torch.softmax(logits, dim=0).numpy()
        np.testing.assert_allclose(a[pad:], expect, rtol=1e-13, atol=0)
        assert np.all(a[:pad] == 0)
        assert fill == pytest.approx(expect.max(), rel=1e-14)


def test_usage_explicit_scale(ref):
    """The scale multiplies the logits: scale s on q equals scale 1 on s*q."""
    rng = np.random.default_rng(2)
    q = rng.standard_normal((2, 3, 8))
    k = rng.standard_normal((20, 8))
    a1, _ = ref.usage(q, k, scale=0.37)
    a2, _ = ref.usage(0.37 * q, k, scale=1.0)
    np.testing.assert_allclose(a1, a2, rtol=1e-12)


def _uniform_closed_form(G, W, T, pad):
    """Zero queries attend uniformly: query j sees n_j = T-W+j-pad+1 slots, p = 1/n_j.

    fill = largest p = 1/min n_j over present queries; a_i = sum over present
    queries that see i of 1/n_j + fill * #(present (h, j) that do not see i).
    """
    present = [j for j in range(W) if T - W + j >= pad]
    n_seen = {j: T - W + j - pad + 1 for j in present}
    fill = 1.0 / min(n_seen.values())
    a = np.zeros(T)
    for i in range(pad, T):
        for j in present:
            if i <= T - W + j:
                a[i] += G * (1.0 / n_seen[j])
            else:
                a[i] += G * fill
    return a, fill


@pytest.mark.parametrize("G,W,T,pad", [(3, 5, 12, 2), (1, 6, 8, 4), (2, 4, 4, 0), (4, 1, 9, 3)])
def test_usage_uniform_closed_form(ref, G, W, T, pad):
    q = np.zeros((G, W, 4))
    k = np.random.default_rng(3).standard_normal((T, 4))
    a, fill = ref.usage(q, k, pad=pad)
    expect, efill = _uniform_closed_form(G, W, T, pad)
    np.testing.assert_allclose(a, expect, rtol=1e-13, atol=1e-15)
    assert fill == pytest.approx(efill, rel=1e-14)


def test_usage_mass_conservation(ref):
    """Each present softmax row sums to 1, so sum_i a_i = #rows + fill * #unseen entries."""
    rng = np.random.default_rng(4)
    G, W, T, pad = 3, 7, 50, 6
    q = rng.standard_normal((G, W, 16)) * 2
    k = rng.standard_normal((T, 16))
    a, fill = ref.usage(q, k, pad=pad)
    unseen = G * sum(W - 1 - j for j in range(W))  # query j misses slots T-W+j+1..T-1
    assert a.sum() == pytest.approx(G * W + fill * unseen, rel=1e-13)


def test_usage_invariances(ref):
    """Permuting the group's heads, or adding one vector to every key (a per-row
    constant on the logits), leaves a unchanged."""
    rng = np.random.default_rng(5)
    q = rng.standard_normal((4, 5, 8))
    k = rng.standard_normal((30, 8))
    a, _ = ref.usage(q, k, pad=2)
    a_perm, _ = ref.usage(q[[2, 0, 3, 1]], k, pad=2)
    np.testing.assert_allclose(a_perm, a, rtol=1e-13)
    x = rng.standard_normal(8)
    a_x, _ = ref.usage(q, k + x[None, :], pad=2)
    np.testing.assert_allclose(a_x, a, rtol=1e-11)


def test_usage_fill_counts_unseen(ref):
    """Slot T-W+m is unseen by the m earlier window queries of every head."""
    rng = np.random.default_rng(6)
    G, W, T = 2, 6, 20
    q = rng.standard_normal((G, W, 8))
    k = rng.standard_normal((T, 8))
    a, fill = ref.usage(q, k)
    # drop the last query's contribution: it sees everything, so the fill term of
    # slot T-1 equals G*(W-1)*fill, and a[T-1] - that is the sum of seen p.
    seen = a[T - 1] - G * (W - 1) * fill
    logits = (q[:, W - 1] @ k.T) / math.sqrt(8)
    p_last = torch.softmax(torch.tensor(logits), dim=1).numpy()[:, T - 1]
    assert seen == pytest.approx(p_last.sum(), rel=1e-12)


# ------------------------------------------------------------- pools and mass

@pytest.mark.parametrize("pad", [0, 3])
def test_maxpool_matches_torch(ref, pad):
    a = np.random.default_rng(7).random(60)
    s = ref.maxpool(a, pad=pad, kernel=7)
    expect = torch.nn.functional.max_pool1d(torch.tensor(a[pad:])[None, None], 7, 1, 3)[0, 0]
    np.testing.assert_array_equal(s[pad:], expect.numpy())
    assert np.all(np.isneginf(s[:pad]))


@pytest.mark.parametrize("pad", [0, 4])
def test_avgpool_matches_torch(ref, pad):
    a = np.random.default_rng(8).random(45)
    u = ref.avgpool(a, pad=pad, kernel=5)
    expect = torch.nn.functional.avg_pool1d(torch.tensor(a[pad:])[None, None], 5, 1, 2,
                                            count_include_pad=True)[0, 0]
    np.testing.assert_allclose(u[pad:], expect.numpy(), rtol=1e-14)
    assert np.all(u[:pad] == 0)


def test_mass_normalize(ref):
    """Mass sums to 1 and is proportional to max(u, 0) + eps."""
    u = np.random.default_rng(9).random(30) - 0.2
    m = ref.mass_normalize(u, pad=2, eps=1e-3)
    assert m[2:].sum() == pytest.approx(1.0, abs=1e-14)
    assert np.all(m[:2] == 0)
    w = np.maximum(u[2:], 0) + 1e-3
    np.testing.assert_allclose(m[2:] / m[2], w / w[0], rtol=1e-13)


# ---------------------------------------------------------------- credit (EMA)

def _mass(n, seed):
    r = np.random.default_rng(seed).random(n) + 0.05
    return r / r.sum()


def test_credit_from_zero(ref):
    """c_in = 0, all carried: c = (1-lambda) m and m_used = m exactly."""
    m = _mass(40, 10)
    c, mu = ref.credit(m, np.zeros(40), lam=0.9, beta=0.9)
    np.testing.assert_allclose(c, 0.1 * m, rtol=1e-14)
    np.testing.assert_allclose(mu, m, rtol=1e-13)


def test_credit_repeated_events(ref):
    """n identical events from zero credit give c = (1 - lambda^n) m."""
    m = _mass(25, 11)
    c = np.zeros(25)
    for n in range(1, 6):
        c, mu = ref.credit(m, c, lam=0.9, beta=0.9)
        np.testing.assert_allclose(c, (1 - 0.9 ** n) * m, rtol=1e-13)
        np.testing.assert_allclose(mu, m, rtol=1e-12)


def test_credit_special_cases(ref):
    m = _mass(30, 12)
    c_in = _mass(30, 13)
    # beta = 1: the history is ignored in the mix
    _, mu = ref.credit(m, c_in, lam=0.9, beta=1.0)
    np.testing.assert_allclose(mu, m, rtol=1e-13)
    # nothing carried: every slot starts at its current mass -> c = m, m_used = m
    c, mu = ref.credit(m, c_in, n_carry=0, lam=0.9, beta=0.9)
    np.testing.assert_allclose(c, m, rtol=1e-14)
    np.testing.assert_allclose(mu, m, rtol=1e-13)
    # lambda = 1 keeps the credit; beta = 0 uses only the normalised history
    c, mu = ref.credit(m, c_in, lam=1.0, beta=0.0)
    np.testing.assert_allclose(c, c_in, rtol=0)
    np.testing.assert_allclose(mu, c_in / c_in.sum(), rtol=1e-13)
    # partial carry with padding: new slots restart, padding is zero
    c, mu = ref.credit(np.r_[0, 0, m[2:] / m[2:].sum()], c_in, pad=2, n_carry=10, lam=0.5,
                       beta=0.9)
    assert np.all(c[:2] == 0) and np.all(mu[:2] == 0)
    mm = m[2:] / m[2:].sum()
    np.testing.assert_allclose(c[12:], mm[10:], rtol=1e-14)
    np.testing.assert_allclose(c[2:12], 0.5 * c_in[2:12] + 0.5 * mm[:10], rtol=1e-14)
    assert mu.sum() == pytest.approx(1.0, abs=1e-14)


# ---------------------------------------------------------------- segmentation

def _exact_boundaries(m32, delta32, normalise):
    """b_k from the definition with exact rationals of the fp32 masses."""
    m = [Fraction(float(x)) for x in m32]
    C = list(itertools.accumulate(m))
    total = C[-1]
    d = Fraction(float(np.float32(delta32)))
    out, k = [], 1
    while k * d < 1:
        thr = k * d * (total if normalise else 1)
        out.append(next(t + 1 for t, c in enumerate(C) if c >= thr) if C[-1] >= thr else None)
        k += 1
    return out, C, total


@pytest.mark.parametrize("seed,n", [(20, 300), (21, 1536), (22, 77), (23, 4000)])
def test_boundaries_match_exact_rule(ref, seed, n):
    """Fixed-point cut points equal b_k = min{t : C(t) >= k Delta} computed exactly.

    The fixed-point rule normalises by the total; it agrees with the exact
    normalised rule except when C(t)/C(n) is within 1e-7 of k*Delta, and with the
    page's un-normalised rule except within the fp32 rounding of the total.
    """
    rng = np.random.default_rng(seed)
    w = rng.random(n) ** 4 + 1e-3
    m32 = (w / w.sum()).astype(np.float32)
    b, _ = ref.boundaries(m32, delta=0.1)
    exact, C, total = _exact_boundaries(m32, 0.1, normalise=True)
    raw, _, _ = _exact_boundaries(m32, 0.1, normalise=False)
    assert len(b) == len(exact) == 9
    d = Fraction(float(np.float32(0.1)))
    for k, (bk, ek, rk) in enumerate(zip(b, exact, raw), start=1):
        near = any(abs(c / total - k * d) < Fraction(1, 10 ** 7) for c in C)
        if not near:
            assert bk == ek, (k, bk, ek)
        near_raw = any(abs(c - k * d) < abs(total - 1) + Fraction(1, 10 ** 7) for c in C)
        if rk is not None and not near_raw:
            assert bk == rk, (k, bk, rk)


@pytest.mark.parametrize("delta", [0.1, 0.07, 0.013])
@pytest.mark.parametrize("kind", threshold_cases.KINDS)
def test_boundaries_round_thresholds_as_double(ref, delta, kind):
    """The reading that fixes the cut points bit for bit: tau_k =
    ceil(fl(fl(k*Delta) * S)) in IEEE double, ties to even.  On masses whose
    prefix sums sit on tau_k - 1 and tau_k where that rounding decides (the
    double threshold one below the exact ceiling for "below" and "tie_even"),
    the oracle cuts exactly where Python's doubles put the threshold, and a
    threshold one off either way would cut elsewhere."""
    rng = np.random.default_rng(zlib.crc32(f"{delta}/{kind}".encode()))
    K = threshold_cases.threshold_count(delta)
    ks = [k for k in range(1, K + 1) if threshold_cases.usable(k, delta)]
    for k in sorted({ks[0], ks[-1], ks[len(ks) // 2], int(rng.choice(ks))}):
        c = threshold_cases.craft(rng, int(rng.integers(1536, 4097)), k, delta, kind)
        m = c.mass_f32()
        b, total = ref.boundaries(m, 0, delta)
        assert total == c.S and len(b) == K
        assert b[k - 1] == c.t0
        C = np.cumsum(c.mu)
        cut = lambda tau: int(np.searchsorted(C, tau)) + 1  # min{t : C(t) >= tau}
        assert cut(c.tau - 1) == c.t0 - 1 and cut(c.tau + 1) == c.t0 + 1
        exact = threshold_cases.tau_exact(k, delta, c.S)
        assert cut(exact) == (c.t0 + 1 if kind in ("below", "tie_even") else c.t0)


def test_segmentation_golden(ref):
    cases = _golden("segmentation_cases.txt")
    # spike
    n = 600
    m = np.full(n, 0.09 / 599, np.float64)
    m[100] = 0.91
    m32 = m.astype(np.float32)
    b, _ = ref.boundaries(m32)
    assert list(b) == cases["spike"]["boundaries"]
    st, ln, M = ref.segments(m32)
    assert list(st) == cases["spike"]["seg_start"] and list(ln) == cases["spike"]["seg_len"]
    # merge
    n = 100
    m = np.zeros(n)
    spikes = [5, 10, 30, 50, 60, 65, 70, 90, 95, 100]
    wts = [0.105] + [0.1] * 8 + [0.095]
    for t, wt in zip(spikes, wts):
        m[t - 1] = wt
    b, _ = ref.boundaries(m.astype(np.float32))
    assert list(b) == cases["merge"]["boundaries"]
    st, ln, M = ref.segments(m.astype(np.float32))
    assert list(st) == cases["merge"]["seg_start"] and list(ln) == cases["merge"]["seg_len"]
    # merge before split
    n = 400
    m = np.full(n, 0.05 / 398)
    m[9], m[269] = 0.15, 0.80
    b, _ = ref.boundaries(m.astype(np.float32))
    assert list(b) == cases["merge_then_split"]["boundaries"]
    st, ln, M = ref.segments(m.astype(np.float32))
    assert list(st) == cases["merge_then_split"]["seg_start"]
    assert list(ln) == cases["merge_then_split"]["seg_len"]
    # uniform
    n = 997
    b, _ = ref.boundaries(np.full(n, 1.0 / n, np.float32))
    assert list(b) == cases["uniform"]["boundaries"]
    assert list(b) == [math.ceil(k * 0.1 * n) for k in range(1, 10)]


@pytest.mark.parametrize("seed,n,pad", [(30, 1536, 0), (31, 862, 250), (32, 20, 3),
                                        (33, 10, 0), (34, 32768, 0), (35, 5000, 17)])
def test_segment_invariants(ref, seed, n, pad):
    """Contiguous cover of the valid slots, lengths in [16, 256] (one segment if n < 16),
    masses recounted: sum of segment masses = fixed-point total."""
    rng = np.random.default_rng(seed)
    T = n + pad
    w = np.zeros(T)
    w[pad:] = rng.random(n) ** 6
    if n > 100:
        w[pad + rng.integers(0, n, 3)] += 50 * w.sum() / n  # a few spikes
    m32 = (w / w.sum()).astype(np.float32)
    st, ln, M = ref.segments(m32, pad=pad)
    assert st[0] == 0 and ln.sum() == n
    assert np.all(st[1:] == st[:-1] + ln[:-1])
    if n >= 16:
        assert ln.min() >= 16 and ln.max() <= 256
    else:
        assert len(ln) == 1
    _, total = ref.boundaries(m32, pad=pad)
    assert int(M.astype(object).sum()) == total
    fixed = np.array([int(np.ldexp(np.float64(x), 40)) for x in m32[pad:]], dtype=object)
    for s, l, mm in zip(st, ln, M):
        assert int(mm) == int(fixed[s:s + l].sum())


def test_single_segment_when_delta_ge_1(ref):
    m32 = _mass(200, 40).astype(np.float32)
    st, ln, _ = ref.segments(m32, delta=1.0, seg_max=256)
    assert list(st) == [0] and list(ln) == [200]


# ---------------------------------------------------------------------- quotas

def test_quota_worked_example(ref):
    g = _golden("ams_worked_example.txt")
    M = np.array([int(np.ldexp(x, 40)) for x in g["seg_mass"]], np.uint64)
    q = ref.quotas(g["seg_len"], M, g["budget"][0], g["q_min"][0])
    assert list(q) == g["expected_quota"]


def test_worked_example_selection(ref):
    """With the first and last positions must-keep, each segment still keeps 2."""
    g = _golden("ams_worked_example.txt")
    n = g["n_positions"][0]
    st = np.array([0, 4, 8, 12], np.int32)
    ln = np.array(g["seg_len"], np.int32)
    q = np.array(g["expected_quota"], np.int32)
    score = np.random.default_rng(41).random(n).astype(np.float32)
    kept = ref.select_unit(score, 0, st, ln, q, g["budget"][0],
                           n_sink=g["must_keep_first"][0], n_recent=g["must_keep_last"][0])
    per_seg = [int(((kept >= s) & (kept < s + 4)).sum()) for s in st]
    assert per_seg == g["expected_kept_per_segment"]
    assert 0 in kept and n - 1 in kept


@pytest.mark.parametrize("seed", range(8))
def test_quota_invariants_and_apportionment(ref, seed):
    """Sum = budget, q_i <= L_i, q_i >= min(q_min, L_i); without clipping every
    quota is within 1 of its ideal share q_i^min + T_rem M_i / sum M."""
    rng = np.random.default_rng(50 + seed)
    ns = int(rng.integers(1, 40))
    L = rng.integers(16, 257, ns).astype(np.int32)
    M = (rng.random(ns) ** 3 * 2 ** 36).astype(np.uint64) + np.uint64(1)
    n = int(L.sum())
    budget = int(rng.integers(ns, max(ns + 1, n)))
    q = ref.quotas(L, M, budget, 1)
    assert q.sum() == budget
    assert np.all(q <= L) and np.all(q >= 1)
    qmin = np.minimum(1, L)
    t_rem = budget - qmin.sum()
    ideal = qmin + t_rem * M.astype(np.float64) / M.astype(np.float64).sum()
    if np.all(ideal <= L - 1):
        assert np.all(np.abs(q - ideal) < 1.0 + 1e-9)


@pytest.mark.parametrize("seed", range(6))
def test_quota_correction_is_the_best_bids(ref, seed):
    """Reading 10's correction, one unit at a time on the exact remainders, as a
    sort.  Giving a segment one unit lowers its remainder by the mass total, so
    the greedy picks are a merge of per-segment decreasing sequences.  When
    short, the units taken are the best D of all bids rem_s - k*sum(M)
    (k < L_s - q_s) by value, ties to the lower index.  When over, they are the
    worst D of rem_s + k*sum(M) (k < q_s - q_min_s), ties to the higher index.
    A quarter of the cases have infeasible minimums, handed out by a stable sort
    on descending mass.  Tiny tie-heavy cases (masses from {0..3}, some all
    zero), exact integers."""
    rng = np.random.default_rng(60 + seed)
    for _ in range(300):
        ns = int(rng.integers(1, 9))
        L = rng.integers(1, 13, ns).astype(np.int32)
        M = rng.integers(0, 4, ns).astype(np.uint64) * np.uint64(rng.choice([1, 7, 1 << 30]))
        q_min = int(rng.choice([1, 2, 4]))
        floor = np.minimum(q_min, L).astype(np.int64)
        if rng.random() < 0.25 and floor.sum() > 1:
            # infeasible minimums: they go to the heaviest segments first (ties:
            # lower index), a stable sort by descending mass, until the budget
            # runs out
            budget = int(rng.integers(1, int(floor.sum())))
            left = budget
            for s in sorted(range(ns), key=lambda i: -int(M[i])):
                give = min(int(floor[s]), left)
                floor[s] = give
                left -= give
        else:
            budget = int(rng.integers(int(floor.sum()), int(L.sum()) + 1))
        Mt = int(M.sum())
        t_rem = budget - int(floor.sum())
        q0 = np.array([min(int(L[s]), int(floor[s]) + ((2 * t_rem * int(M[s]) + Mt) // (2 * Mt)
                                                      if Mt > 0 else 0)) for s in range(ns)])
        rem = [int(floor[s]) * Mt + t_rem * int(M[s]) - int(q0[s]) * Mt for s in range(ns)]
        D = budget - int(q0.sum())
        q = q0.copy()
        if D > 0:
            bids = [(rem[s] - k * Mt, s) for s in range(ns) for k in range(int(L[s] - q0[s]))]
            bids.sort(key=lambda b: (-b[0], b[1]))
            for _, s in bids[:D]:
                q[s] += 1
        elif D < 0:
            bids = [(rem[s] + k * Mt, s) for s in range(ns) for k in range(int(q0[s] - floor[s]))]
            bids.sort(key=lambda b: (b[0], -b[1]))
            for _, s in bids[:-D]:
                q[s] -= 1
        assert list(ref.quotas(L, M, budget, q_min)) == list(q), (L, M, budget, q_min)


def test_quota_infeasible_minimums(ref):
    """More segments than budget: the heaviest segments get their minimum, sum = budget."""
    L = np.full(10, 16, np.int32)
    M = np.array([5, 9, 1, 7, 7, 3, 8, 2, 6, 4], np.uint64) * np.uint64(1000)
    q = ref.quotas(L, M, 4, 1)
    assert q.sum() == 4
    assert list(np.nonzero(q)[0]) == [1, 3, 4, 6]  # masses 9, 8, 7, 7 (tie: lower index)


def test_quota_budget_ge_length_keeps_all(ref):
    L = np.array([20, 30, 16], np.int32)
    M = np.array([1, 100, 7], np.uint64)
    q = ref.quotas(L, M, int(L.sum()), 1)
    np.testing.assert_array_equal(q, L)


def test_quota_clipping_redistributes(ref):
    """A heavy short segment is clipped to its length; the excess goes elsewhere."""
    L = np.array([16, 200, 200], np.int32)
    M = np.array([90, 5, 5], np.uint64) * np.uint64(2 ** 30)
    q = ref.quotas(L, M, 100, 1)
    assert q.sum() == 100 and q[0] == 16 and q[1] + q[2] == 84 and abs(int(q[1]) - int(q[2])) <= 1


# ------------------------------------------------------------------- selection

def _order_key(score, v):
    return (-float(score[v]), v)


@pytest.mark.parametrize("seed", range(12))
def test_selection_brute_force(ref, seed):
    """On tiny segments, each segment's picks are the best subset of its
    non-must-keep slots under (score desc, slot asc), found by enumeration; if
    must-keep overflows the budget, the globally worst picks are the ones dropped."""
    rng = np.random.default_rng(60 + seed)
    lens = rng.integers(3, 9, 3)
    n = int(lens.sum())
    st = np.r_[0, np.cumsum(lens)[:-1]].astype(np.int32)
    score = rng.integers(0, 4, n).astype(np.float32)  # many exact ties
    budget = int(rng.integers(4, n))
    n_recent = int(rng.integers(0, 6))
    q = ref.quotas(lens.astype(np.int32), np.full(3, 1000, np.uint64), budget, 1)
    kept = ref.select_unit(score, 0, st, lens.astype(np.int32), q, budget, n_sink=1,
                           n_recent=n_recent)
    n_s = min(1, budget)
    n_r = min(n_recent, budget - n_s)
    must = set(range(n_s)) | set(range(n - n_r, n))
    picks = []
    for s, l, qq in zip(st, lens, q):
        seg = list(range(s, s + l))
        cand = [v for v in seg if v not in must]
        want = max(0, int(qq) - (l - len(cand)))
        best = min(itertools.combinations(cand, want),
                   key=lambda sub: sorted(_order_key(score, v) for v in sub))
        picks += list(best)
    excess = len(must) + len(picks) - budget
    assert excess >= 0
    worst_first = sorted(picks, key=lambda v: _order_key(score, v), reverse=True)
    expect = sorted(must | set(worst_first[excess:]))
    assert list(kept) == expect
    assert len(kept) == min(budget, n)


def test_selection_over_budget_drops_worst_picks(ref):
    """Must-keep beyond a segment's quota forces removals: the globally worst
    picks go first (score ascending, ties: higher slot first)."""
    n = 40
    st = np.array([0, 20], np.int32)
    ln = np.array([20, 20], np.int32)
    q = np.array([5, 5], np.int32)          # budget 10
    score = np.arange(n, dtype=np.float32)[::-1].copy()  # earlier = better
    kept = ref.select_unit(score, 0, st, ln, q, 10, n_sink=0, n_recent=8)
    # segment 2 holds 8 must-keep > quota 5: picks are only from segment 1 (5 best:
    # slots 0..4); size 13 > 10 -> drop the 3 worst picks (slots 4, 3, 2).
    assert list(kept) == [0, 1] + list(range(32, 40))


def test_selection_one_segment_is_global_topk(ref):
    """Delta >= 1 and seg_max >= n: one segment, so selection = global top-k of the
    non-must-keep slots (numpy stable sort) plus the must-keep set."""
    rng = np.random.default_rng(70)
    n, budget = 200, 60
    score = rng.integers(0, 50, n).astype(np.float32)
    m32 = _mass(n, 71).astype(np.float32)
    st, ln, M = ref.segments(m32, delta=1.0, seg_max=256)
    q = ref.quotas(ln, M, budget, 1)
    kept = ref.select_unit(score, 0, st, ln, q, budget, n_sink=4, n_recent=10)
    must = set(range(4)) | set(range(n - 10, n))
    cand = np.array([v for v in range(n) if v not in must])
    order = cand[np.argsort(-score[cand], kind="stable")]
    expect = sorted(must | set(order[: budget - len(must)].tolist()))
    assert list(kept) == expect


def test_selection_streaming_llm_special_case(ref):
    """Constant scores and n_recent = budget - 4: the result is StreamingLLM,
    4 sinks plus the budget-4 most recent slots."""
    n, budget, pad = 700, 256, 9
    T = n + pad
    m32 = np.zeros(T, np.float32)
    m32[pad:] = 1.0 / n
    st, ln, M = ref.segments(m32, pad=pad)
    q = ref.quotas(ln, M, budget, 1)
    kept = ref.select_unit(np.ones(T, np.float32), pad, st, ln, q, budget, n_sink=4,
                           n_recent=budget - 4)
    assert list(kept) == list(range(pad, pad + 4)) + list(range(T - (budget - 4), T))


# ------------------------------------------------------------------ compaction

def test_compaction_is_index_select(ref):
    rng = np.random.default_rng(80)
    U, T, d = 3, 50, 8
    p = ref.RefParams(group=1, head_dim=d, window=4, budget=20)
    k = rng.integers(0, 2 ** 16, (U, T, d)).astype(np.uint16)
    v = rng.integers(0, 2 ** 16, (U, T, d)).astype(np.uint16)
    c = rng.random((U, T)).astype(np.float32)
    kept = np.full((U, 20), -1, np.int32)
    nk = np.array([20, 13, 0], np.int32)
    for u in range(U):
        kept[u, :nk[u]] = np.sort(rng.choice(T, nk[u], replace=False))
    ko, vo, co = ref.compact(p, k, v, c, kept, nk)
    for u in range(U):
        idx = torch.tensor(kept[u, :nk[u]], dtype=torch.long)
        for got, src in ((ko, k), (vo, v)):
            want = torch.index_select(torch.tensor(src[u].astype(np.int32)), 0, idx).numpy()
            assert np.array_equal(got[u, :nk[u]], want)
        assert np.array_equal(co[u, :nk[u]], c[u, kept[u, :nk[u]]])
        assert not ko[u, nk[u]:].any() and not vo[u, nk[u]:].any() and not co[u, nk[u]:].any()
