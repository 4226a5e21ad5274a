"""CPU tests of the end-to-end checker (tests/e2e_check.py).

The checker decides whether a kept set that differs from the oracle's differs
only at a knife edge of the method's discrete decisions.  Here the "GPU" side is
simulated by the oracle's own stages run on slightly perturbed masses or scores
(within the 1e-4 tolerance of the mass/score comparison), which produces each
legitimate kind of difference on purpose; planted mistakes must be rejected.
"""
import types

import numpy as np
import pytest

from tests import e2e_check as ec

T, PAD, BUDGET = 520, 20, 150
W = types.SimpleNamespace(budget=BUDGET, n_sink=4, n_recent=32, group=1, window=8)


def _params(ref):
    return ref.RefParams(group=1, head_dim=64, window=8, budget=BUDGET, n_sink=4, n_recent=32)


def _stages(ref, mass, score, pad=PAD):
    """Oracle steps 3-5 on one unit's fp32 mass and score -> a run dict (row 0)."""
    p = _params(ref)
    m = np.asarray(mass, np.float32)[None]
    s = np.asarray(score, np.float32)[None]
    pads = np.array([pad], np.int32)
    st, ln, qu, ns = ref.segment_quota(p, m, pads)
    kept, nk = ref.select(p, s, pads, st, ln, qu, ns)
    return dict(mass=m, score=s, seg_start=st, seg_len=ln, quota=qu, n_seg=ns, kept_idx=kept,
                n_kept=nk)


def _gpu_view(r):
    """The GPU-side arguments of check_unit_e2e taken from a run dict."""
    seg = {k: r[k][0] for k in ("seg_start", "seg_len", "quota")}
    seg["n_seg"] = int(r["n_seg"][0])
    return r["kept_idx"][0, :r["n_kept"][0]], r["mass"][0], r["score"][0], seg


def _check(ref, r_gpu, r_ref):
    kept, m, s, seg = _gpu_view(r_gpu)
    return ec.check_unit_e2e(_params(ref), W, PAD, kept, m, s, seg, r_ref, 0)


def _random_unit(seed):
    rng = np.random.default_rng(seed)
    w = np.zeros(T)
    w[PAD:] = rng.random(T - PAD) ** 3 + 1e-3
    mass = (w / w.sum()).astype(np.float32)
    score = np.full(T, -np.inf, np.float32)
    score[PAD:] = (rng.random(T - PAD) * 2 + 0.5).astype(np.float32)
    return mass, score


def test_identical(ref):
    mass, score = _random_unit(1)
    r = _stages(ref, mass, score)
    assert _check(ref, r, r) == "identical"


def _cutoff_pair(r):
    """(last pick, first unpicked candidate) of the first segment that has both."""
    kept = set(r["kept_idx"][0, :r["n_kept"][0]].tolist())
    s = r["score"][0]
    mk, _ = ec.must_keep(PAD, T, BUDGET, 4, 32)
    for a, l in zip(r["seg_start"][0, :r["n_seg"][0]], r["seg_len"][0, :r["n_seg"][0]]):
        cand = [v for v in range(a, a + l) if not mk[v]]
        order = sorted(cand, key=lambda v: (-float(s[v]), v))
        picks = [v for v in order if v in kept]
        if picks and len(picks) < len(order):
            return picks[-1], order[len(picks)]
    raise AssertionError("no segment with a cut-off")


def test_near_tie_swap_accepted(ref):
    mass, score = _random_unit(2)
    y, x = _cutoff_pair(_stages(ref, mass, score))
    score[x] = np.float32(score[y] * (1 - 1e-6))      # the oracle: y just above x
    r = _stages(ref, mass, score)
    g_score = score.copy()
    g_score[x] = np.float32(score[y] * (1 + 1e-6))    # the "GPU": x just above y
    g = _stages(ref, mass, g_score)
    assert not np.array_equal(g["kept_idx"], r["kept_idx"])
    assert _check(ref, g, r) == "near_tie"


def test_far_swap_rejected(ref):
    """A swap whose slots sit far from the cut-off fails even with consistent
    GPU scores: the GPU's score of the demoted pick moved by far more than 1e-4."""
    mass, score = _random_unit(3)
    r = _stages(ref, mass, score)
    y, x = _cutoff_pair(r)
    kept = r["kept_idx"][0, :r["n_kept"][0]]
    best = max((v for v in kept if v not in (y,) and v >= PAD + 4 and v < T - 32),
               key=lambda v: score[v])
    g_score = score.copy()
    g_score[best] = score[x] * 0.5
    g = _stages(ref, mass, g_score)
    with pytest.raises(AssertionError, match="score rel"):
        _check(ref, g, r)


def test_planted_wrong_pick_rejected(ref):
    """A kept set that is not the rule's result for the GPU's own scores fails
    the property check, whatever the oracle says."""
    mass, score = _random_unit(4)
    r = _stages(ref, mass, score)
    g = {k: v.copy() for k, v in r.items()}
    y, x = _cutoff_pair(r)
    kept = g["kept_idx"][0, :g["n_kept"][0]]
    mk, _ = ec.must_keep(PAD, T, BUDGET, 4, 32)
    # drop the segment's best pick instead of its worst, keep x
    seg_picks = [v for v in kept if not mk[v]]
    best = max(seg_picks, key=lambda v: score[v])
    new = sorted((set(kept.tolist()) - {best}) | {x})
    g["kept_idx"][0, :len(new)] = new
    with pytest.raises(AssertionError, match="not the rule's result"):
        _check(ref, g, r)


def _tie_quota_unit():
    """Ten segments, each a run of 39 light slots ending in a heavy one (the last
    also takes the 100 zero-mass slots after it); segments 1-9 hold identical
    masses, so their quota remainders tie exactly and the correction to the
    budget decides between them by the tie rule."""
    m = np.zeros(T)
    seg_mass = [0.101] * 9 + [1 - 0.909]
    for k in range(10):
        lo = PAD + 40 * k
        m[lo:lo + 39] = 1e-5
        m[lo + 39] = seg_mass[k] - 39e-5
    assert abs(m.sum() - 1) < 1e-12
    rng = np.random.default_rng(6)
    score = np.full(T, -np.inf, np.float32)
    score[PAD:] = (rng.random(T - PAD) + 0.5).astype(np.float32)
    return m, score


def test_quota_remainder_tie_accepted(ref):
    m, score = _tie_quota_unit()
    m32 = m.astype(np.float32)
    r = _stages(ref, m32, score)
    assert r["n_seg"][0] == 10
    moved = None
    for seed in range(20):
        rng = np.random.default_rng(100 + seed)
        g_m = (m32 * (1 + 2e-6 * rng.standard_normal(T))).astype(np.float32)
        g = _stages(ref, g_m, score)
        if (np.array_equal(g["seg_start"], r["seg_start"])
                and not np.array_equal(g["quota"], r["quota"])):
            moved = g
            break
    assert moved is not None, "no perturbation moved a tied quota"
    assert _check(ref, moved, r) in ("quota_shift", "identical")
    assert _check(ref, moved, r) == "quota_shift" or np.array_equal(
        moved["kept_idx"], r["kept_idx"])


def test_quota_move_without_tie_rejected(ref):
    """Moving a unit of quota between segments whose remainders are far apart,
    with a kept set consistent with the moved quotas, is rejected."""
    mass, score = _random_unit(7)
    r = _stages(ref, mass, score)
    ns = int(r["n_seg"][0])
    q = r["quota"][0, :ns].astype(np.int64)
    ln = r["seg_len"][0, :ns]
    m = r["mass"][0].astype(np.float64)
    M = np.array([m[a:a + l].sum() for a, l in zip(r["seg_start"][0, :ns], ln)])
    ideal = 1 + (BUDGET - ns) * M / M.sum()
    p = _params(ref)
    tried = 0
    for i in range(ns):
        for j in range(ns):
            if i == j or q[i] >= ln[i] or q[j] <= 1:
                continue
            if abs((ideal[j] - q[j]) + 1 - (ideal[i] - q[i])) < 1e-2:
                continue            # a genuine near-tie: not a planted mistake
            g = {k: v.copy() for k, v in r.items()}
            g["quota"][0, i] += 1
            g["quota"][0, j] -= 1
            kept, nk = ref.select(p, r["score"], np.array([PAD], np.int32), g["seg_start"],
                                  g["seg_len"], g["quota"], g["n_seg"])
            if np.array_equal(kept, r["kept_idx"]):
                continue            # the over-budget removal absorbed the move
            g["kept_idx"], g["n_kept"] = kept, nk
            with pytest.raises(AssertionError, match="remainder tie"):
                _check(ref, g, r)
            tried += 1
    assert tried >= 3


def test_cut_at_threshold_accepted(ref):
    """Uniform mass puts the cumulative mass exactly on k*Delta at every tenth of
    the cache; a GPU mass 5e-5 heavier at the slot before moves that cut by one
    slot, which shifts one unit of mass and so possibly of quota between the two
    segments beside it."""
    n = T - PAD
    mass = np.zeros(T, np.float32)
    mass[PAD:] = np.float32(1.0 / n)
    verdicts = []
    for seed in range(8, 14):
        _, score = _random_unit(seed)
        r = _stages(ref, mass, score)
        for k in range(1, 10):
            g_m = mass.copy()
            g_m[PAD + k * n // 10 - 1] *= np.float32(1 + 5e-5)
            g = _stages(ref, g_m, score)
            if np.array_equal(g["seg_start"], r["seg_start"]):
                continue        # this threshold's fixed-point margin exceeds the nudge
            verdicts.append(_check(ref, g, r))
    assert set(verdicts) <= {"identical", "cut_shift"}
    assert verdicts.count("cut_shift") >= 3, verdicts


def test_cut_away_from_threshold_rejected(ref):
    """Segments that differ where no cumulative mass is near a threshold fail,
    even when the kept set is the rule's result for those segments."""
    mass, score = _random_unit(9)
    r = _stages(ref, mass, score)
    p = _params(ref)
    ns = int(r["n_seg"][0])
    tried = 0
    for j in range(1, ns):
        for shift in (3, -3, 6):
            g = {k: v.copy() for k, v in r.items()}
            g["seg_start"][0, j] += shift       # move the cut between segments j-1 and j
            g["seg_len"][0, j - 1] += shift
            g["seg_len"][0, j] -= shift
            if min(g["seg_len"][0, j - 1], g["seg_len"][0, j]) < 16:
                continue
            kept, nk = ref.select(p, r["score"], np.array([PAD], np.int32), g["seg_start"],
                                  g["seg_len"], g["quota"], g["n_seg"])
            if np.array_equal(kept, r["kept_idx"]):
                continue
            g["kept_idx"], g["n_kept"] = kept, nk
            with pytest.raises(AssertionError, match="away from every cut threshold"):
                _check(ref, g, r)
            tried += 1
    assert tried >= 3


def test_selection_walk_over_budget(ref):
    """A large recent suffix overflows the last segment's quota: the walk finds
    the removal, and a kept set that removed a better pick is flagged."""
    mass, score = _random_unit(10)
    p = ref.RefParams(group=1, head_dim=64, window=8, budget=BUDGET, n_sink=4, n_recent=120)
    m = mass[None]
    pads = np.array([PAD], np.int32)
    st, ln, qu, ns = ref.segment_quota(p, m, pads)
    kept, nk = ref.select(p, score[None], pads, st, ln, qu, ns)
    k0 = kept[0, :nk[0]]
    probs, info = ec.selection_walk(k0, score, PAD, T, st[0, :ns[0]], ln[0, :ns[0]],
                                    qu[0, :ns[0]], BUDGET, 4, 120)
    assert probs == [] and info["removal_cutoffs"], "the over-budget path should run"
    # swap the best removed pick back in for the worst kept pick
    mk, _ = ec.must_keep(PAD, T, BUDGET, 4, 120)
    removed = []
    for sg in info["segs"]:
        removed += sg["order"][sg["k"]:sg["want"]].tolist()
    best_removed = max(removed, key=lambda v: (score[v], -v))
    picks = [v for v in k0 if not mk[v]]
    best_pick = max(picks, key=lambda v: (score[v], -v))
    bad = np.array(sorted((set(k0.tolist()) - {best_pick}) | {best_removed}))
    probs, _ = ec.selection_walk(bad, score, PAD, T, st[0, :ns[0]], ln[0, :ns[0]],
                                 qu[0, :ns[0]], BUDGET, 4, 120)
    assert probs
