"""End-to-end agreement between a compression event's kept set and the oracle's.

The GPU and the oracle compute the mass and the score in different precisions
(fp32 accumulation against fp64), so their kept sets may legitimately differ where
the method's discrete decisions sit on a knife edge: two candidates whose scores
are nearly equal at a segment's cut-off, a cumulative mass within rounding of a
cut threshold k*Delta, or two segments whose quota remainders are nearly equal.
This module decides, for one unit, whether a difference is of that kind, without
ever feeding a GPU value to the oracle:

  1. the GPU's fp32 mass and score are within 1e-4 relative (+1e-9) of the
     oracle's;
  2. the GPU's kept set is exactly what the selection rule gives on the GPU's
     own segments, quotas and scores (a property check: must-keep kept, each
     segment's picks a prefix of its order, the over-budget removal took the
     globally worst picks), and the GPU's segments and quotas are well formed;
  3. against the oracle, segment by segment:
       * a segment both sides cut identically and gave the same quota keeps the
         same picks, or picks that differ only at the segment's cut-off score
         (every swapped slot within the near-tie tolerance of it, by its rank in
         the oracle's own order);
       * a segment with the same cut but a different quota differs by one unit
         at most, the two quota moves pair up at nearly equal remainders of the
         ideal shares (when the segmentation is the same), and its picks are the
         other side's picks plus or minus the next candidates in the oracle's
         order, up to near-ties;
       * segments cut differently lie in blocks that each contain a slot where
         the oracle's fp64 cumulative mass is within 1e-5 of a cut threshold.
     Across segments, a different number of picks in a segment is allowed only
     where its quota moved or where the slots involved sit at the over-budget
     removal's cut-off score.

Verdicts: "identical", "near_tie" (same segments and quotas), "quota_shift" (same
segments, quotas moved), "cut_shift" (segments differ).

Sources: "Adaptive Mass-Segmented KV Compression for Long-Form Reasoning",
Method, Key designs 2-4 (cut points, quotas, must-keep, in-segment selection,
over-budget fix-up).
"""
from __future__ import annotations

import numpy as np

VERDICTS = ("identical", "near_tie", "quota_shift", "cut_shift")


def mass_close(gpu, ref, rtol=1e-4, atol=1e-9):
    """|gpu - ref| <= rtol*|ref| + atol elementwise (non-finite values equal);
    returns (ok, worst relative error)."""
    gpu = np.asarray(gpu)
    ref = np.asarray(ref)
    finite = np.isfinite(ref)
    with np.errstate(invalid="ignore"):
        err = np.abs(gpu.astype(np.float64) - ref.astype(np.float64))
    bound = rtol * np.abs(ref.astype(np.float64)) + atol
    ok = bool(np.all(err[finite] <= bound[finite])) and bool(
        np.array_equal(gpu[~finite], ref[~finite]))
    rel = float(np.max(err[finite] / np.maximum(np.abs(ref[finite]), 1e-30))) if finite.any() else 0.0
    return ok, rel


def must_keep(pad, T, budget, n_sink, n_recent):
    """(must-keep slots as a boolean mask over [0, T), effective budget)."""
    n = T - pad
    B = min(budget, n)
    ns = min(n_sink, B)
    nr = min(n_recent, B - ns)
    mk = np.zeros(T, bool)
    mk[pad:pad + ns] = True
    if nr > 0:
        mk[T - nr:] = True
    return mk, B


def _order(cand, s):
    """Candidates best first: score descending, ties to the lower slot."""
    cand = np.asarray(cand, np.int64)
    if cand.size == 0:
        return cand
    return cand[np.lexsort((cand, -s[cand].astype(np.float64)))]


def _good(s, v):
    """Goodness key for the over-budget removal: lower score is worse, and among
    equal scores the higher slot is worse."""
    return (float(s[v]), -int(v))


def selection_walk(kept, s, pad, T, starts, lens, quotas, budget, n_sink, n_recent):
    """Walk the segments the way the selection rule does.

    Returns (problems, info): problems lists every way `kept` differs from the
    rule's result for these segments (absolute starts), quotas and scores (empty
    when it is the rule's result); info holds per segment the candidates' order,
    the wanted and the kept number of picks, and the removal cut-off scores."""
    probs = []
    kept = np.asarray(kept, np.int64)
    s = np.asarray(s, np.float64)
    n = T - pad
    info = {"segs": [], "removal_cutoffs": []}
    if kept.size and (np.any(np.diff(kept) <= 0) or kept[0] < pad or kept[-1] >= T):
        probs.append("kept slots not ascending, unique and valid")
    if n <= 0:
        if kept.size:
            probs.append("an all-padding unit keeps nothing")
        return probs, info
    if n <= budget:
        if not np.array_equal(kept, np.arange(pad, T)):
            probs.append("a cache no longer than the budget keeps every valid slot")
        return probs, info
    mk, B = must_keep(pad, T, budget, n_sink, n_recent)
    if kept.size != B:
        probs.append(f"{kept.size} kept, budget {B}")
    inK = np.zeros(T, bool)
    inK[kept[(kept >= 0) & (kept < T)]] = True
    if np.any(mk & ~inK):
        probs.append("a must-keep slot is missing")
    starts = np.asarray(starts, np.int64)
    lens = np.asarray(lens, np.int64)
    quotas = np.asarray(quotas, np.int64)
    if (starts.size == 0 or starts[0] != pad or np.any(starts[1:] != starts[:-1] + lens[:-1])
            or lens.sum() != n or np.any(lens <= 0)):
        probs.append("segments do not tile the valid slots")
        return probs, info
    if quotas.sum() != B or np.any(quotas > lens) or np.any(quotas < 0):
        probs.append("quotas do not sum to the budget within the segment lengths")
    kept_picks, removed, n_mk, sum_want = [], [], int(mk.sum()), 0
    for a, l, q in zip(starts, lens, quotas):
        seg = np.arange(a, a + l)
        cand = seg[~mk[seg]]
        want = max(0, int(q) - int(l - cand.size))
        order = _order(cand, s)
        k = int(inK[cand].sum())
        if k > want:
            probs.append(f"segment at {a}: {k} picks, quota allows {want}")
        elif not np.all(inK[order[:k]]):
            probs.append(f"segment at {a}: picks are not the segment's best candidates")
        kept_picks += order[:k].tolist()
        removed += order[k:want].tolist()
        sum_want += want
        info["segs"].append({"start": int(a), "len": int(l), "order": order, "want": want,
                             "k": k})
    excess = max(0, n_mk + sum_want - B)
    if len(removed) != excess:
        probs.append(f"{len(removed)} picks removed, the excess over the budget is {excess}")
    if removed and kept_picks:
        best_removed = max(removed, key=lambda v: _good(s, v))
        worst_kept = min(kept_picks, key=lambda v: _good(s, v))
        if _good(s, best_removed) > _good(s, worst_kept):
            probs.append("the over-budget removal dropped a pick better than one it kept")
        info["removal_cutoffs"] = [float(s[best_removed]), float(s[worst_kept])]
    return probs, info


def _segments_of(seg_start, seg_len, quota, n_seg):
    ns = int(n_seg)
    return (np.asarray(seg_start[:ns], np.int64), np.asarray(seg_len[:ns], np.int64),
            np.asarray(quota[:ns], np.int64))


def _near_threshold_blocks(blocks, mass_r, pad, delta, tol=1e-5):
    """Every block [lo, hi) of slots (absolute) contains, within two slots, a
    position where the oracle's fp64 cumulative mass lies within `tol` of a cut
    threshold k*delta; returns the first block that does not, else None."""
    m = np.asarray(mass_r[pad:], np.float64)
    cum = np.cumsum(m) / m.sum()
    K = int(np.floor((1.0 - 1e-12) / float(np.float32(delta))))
    levels = np.arange(1, K + 1) * float(np.float32(delta))
    for lo, hi in blocks:
        a, b = max(lo - pad - 2, 0), min(hi - pad + 2, cum.size)
        if b <= a or levels.size == 0:
            return (lo, hi)
        if np.min(np.abs(cum[a:b, None] - levels[None, :])) > tol:
            return (lo, hi)
    return None


def _blocks(mask_slots):
    """Contiguous [lo, hi) runs of True in a boolean array."""
    idx = np.flatnonzero(mask_slots)
    if idx.size == 0:
        return []
    cuts = np.flatnonzero(np.diff(idx) > 1)
    los = np.r_[idx[0], idx[cuts + 1]]
    his = np.r_[idx[cuts] + 1, idx[-1] + 1]
    return list(zip(los.tolist(), his.tolist()))


def check_unit_e2e(p, w, pad_u, kept_g, mass_g, score_g, seg_g, r, i):
    """One unit's GPU result against oracle run `r` (row i); see the module
    docstring.  seg_g: dict with the GPU's seg_start, seg_len, quota rows and
    n_seg.  Raises AssertionError on a difference that is not a knife-edge case;
    returns the verdict."""
    T = int(np.asarray(mass_g).shape[0])
    ok_m, rel_m = mass_close(mass_g, r["mass"][i])
    ok_s, rel_s = mass_close(score_g, r["score"][i])
    assert ok_m and ok_s, f"unit row {i}: mass rel {rel_m:.3g}, score rel {rel_s:.3g}"
    kept_g = np.asarray(kept_g, np.int64)
    kept_r = np.asarray(r["kept_idx"][i, :r["n_kept"][i]], np.int64)
    st_g, ln_g, q_g = _segments_of(seg_g["seg_start"], seg_g["seg_len"], seg_g["quota"],
                                   seg_g["n_seg"])
    st_r, ln_r, q_r = _segments_of(r["seg_start"][i], r["seg_len"][i], r["quota"][i],
                                   r["n_seg"][i])
    probs_g, info_g = selection_walk(kept_g, score_g, pad_u, T, st_g, ln_g, q_g, w.budget,
                                     w.n_sink, w.n_recent)
    assert not probs_g, f"unit row {i}: GPU selection is not the rule's result: {probs_g}"
    if np.array_equal(kept_r, kept_g):
        return "identical"
    s = np.asarray(r["score"][i], np.float64)
    probs_r, info_r = selection_walk(kept_r, s, pad_u, T, st_r, ln_r, q_r, w.budget, w.n_sink,
                                     w.n_recent)
    assert not probs_r, f"unit row {i}: oracle selection walk failed: {probs_r}"
    tol = 1e-5 * w.group * w.window
    mk, B = must_keep(pad_u, T, w.budget, w.n_sink, w.n_recent)
    inG = np.zeros(T, bool)
    inG[kept_g] = True
    inR = np.zeros(T, bool)
    inR[kept_r] = True

    # ---- segments: common ones, and blocks of slots cut differently
    seg_r = {(int(a), int(l)): (int(q), j) for j, (a, l, q) in enumerate(zip(st_r, ln_r, q_r))}
    seg_gd = {(int(a), int(l)): int(q) for a, l, q in zip(st_g, ln_g, q_g)}
    common = [key for key in seg_r if key in seg_gd]
    differ = np.zeros(T, bool)
    for a, l in set(seg_r) ^ set(seg_gd):
        differ[a:a + l] = True
    blocks = _blocks(differ)
    bad = _near_threshold_blocks(blocks, r["mass"][i], pad_u, p.delta)
    assert bad is None, (f"unit row {i}: segments differ in slots {bad} away from every cut "
                         "threshold")

    # ---- quotas of common segments
    moved = {key: seg_gd[key] - seg_r[key][0] for key in common if seg_gd[key] != seg_r[key][0]}
    assert all(abs(dq) == 1 for dq in moved.values()), f"unit row {i}: quota moves {moved}"
    assert sum(abs(dq) for dq in moved.values()) <= 4, f"unit row {i}: quota moves {moved}"
    if moved and not blocks:
        # same segmentation: every move pairs with an opposite one at nearly equal
        # remainders of the ideal shares (from the oracle's own masses)
        m = np.asarray(r["mass"][i], np.float64)
        M = np.array([m[a:a + l].sum() for a, l in zip(st_r, ln_r)])
        qmin = np.minimum(p.q_min, ln_r)
        t_rem = B - int(qmin.sum())
        ideal = qmin + t_rem * M / M.sum()
        slack = {key: ideal[seg_r[key][1]] - seg_r[key][0] for key in moved}
        ups = [key for key, dq in moved.items() if dq > 0]
        downs = [key for key, dq in moved.items() if dq < 0]
        assert len(ups) == len(downs), f"unit row {i}: unbalanced quota moves {moved}"
        for key in ups:
            x_i = ideal[seg_r[key][1]]
            ok = any(abs(slack[dn] + 1.0 - slack[key])
                     <= 2e-4 * (x_i + ideal[seg_r[dn][1]]) + 1e-6 for dn in downs)
            assert ok, (f"unit row {i}: quota of the segment at {key[0]} moved away from a "
                        f"remainder tie ({ {k: round(v, 6) for k, v in slack.items()} })")

    # ---- kept picks, segment by segment, over the common segments
    cut_r = info_r["removal_cutoffs"]
    cut_g = [float(x) for x in info_g["removal_cutoffs"]]
    removal_cuts = cut_r + cut_g
    segs_r = {(sg["start"], sg["len"]): sg for sg in info_r["segs"]}
    segs_g = {(sg["start"], sg["len"]): sg for sg in info_g["segs"]}
    for key in common:
        sr, sg = segs_r[key], segs_g[key]
        order = sr["order"]              # the oracle's order of the candidates
        pg = set(order[inG[order]].tolist())
        pr = set(order[inR[order]].tolist())
        if pg == pr:
            continue
        k_g, k_r = len(pg), len(pr)
        if k_g:
            c = s[order[k_g - 1]]
            for x in pg ^ set(order[:k_g].tolist()):
                assert abs(s[x] - c) <= tol, (
                    f"unit row {i}: segment at {key[0]}: slot {x} (score {s[x]:.6g}) "
                    f"swapped at cut-off {c:.6g}, beyond the near-tie tolerance {tol:.3g}")
        if k_g != k_r:
            lo, hi = min(k_g, k_r), max(k_g, k_r)
            by_quota = abs(k_g - k_r) <= abs(sg["want"] - sr["want"])
            at_removal = all(any(abs(s[x] - c) <= tol for c in removal_cuts)
                             for x in order[lo:hi].tolist())
            assert by_quota or at_removal, (
                f"unit row {i}: segment at {key[0]} keeps {k_g} picks on the GPU and {k_r} "
                "in the oracle, with neither a quota move nor a removal near-tie to explain it")
    if blocks:
        return "cut_shift"
    return "quota_shift" if moved else "near_tie"


def cutoff_distance(kept_g, kept_r, s, pad, T, seg_start, seg_len, budget, n_sink, n_recent):
    """Largest distance, in score, between a slot kept by only one side and the
    cut-off of its segment in the oracle's order (segments from the oracle, as
    absolute starts).  For a selection on a score other than the attention usage
    (the redundancy mix), where both sides cut the cache identically."""
    s = np.asarray(s, np.float64)
    mk, _ = must_keep(pad, T, budget, n_sink, n_recent)
    inG = np.zeros(T, bool)
    inG[np.asarray(kept_g, np.int64)] = True
    inR = np.zeros(T, bool)
    inR[np.asarray(kept_r, np.int64)] = True
    worst = 0.0
    for a, l in zip(seg_start, seg_len):
        seg = np.arange(a, a + l)
        order = _order(seg[~mk[seg]], s)
        pg = order[inG[order]]
        pr = order[inR[order]]
        if np.array_equal(np.sort(pg), np.sort(pr)):
            continue
        k = pr.size
        c = s[order[k - 1]] if k else s[order[0]]
        diff = np.setxor1d(pg, pr)
        worst = max(worst, float(np.max(np.abs(s[diff] - c))))
    return worst
