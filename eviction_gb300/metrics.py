"""Selection-quality measurements on synthetic caches: region wipe-out rate and
kept-set IoU across compression events.

"Adaptive Mass-Segmented KV Compression for Long-Form Reasoning", key findings
(Appendix C): the region wipe-out rate falls with the method and the IoU of the
kept sets rises (more stable history selection).  The pages name both measures
without defining them; the readings used here:
  * a token is identified by its position in the generated sequence; compaction
    moves tokens between cache slots but keeps their identity;
  * region wipe-out rate of an event = among the planted regions that still have
    at least one token in the cache before the event, the fraction with none
    left after it;
  * kept-set IoU of an event = per unit, |K_prev & K| / |K_prev | K| of the
    token identities kept by the previous event and by this one, averaged over
    units (undefined for the first event).
The events run through the library (the CUDA path); only the set arithmetic on
the kept indices is done here, on the host.

    python -m eviction_gb300.metrics --workload qwen_1l --events 4 [--ablation global_topk]
"""
from __future__ import annotations

import argparse
import json

import numpy as np


def region_tokens(start, length, active):
    """Planted regions as lists of token-identity ranges: [(unit, lo, hi)]."""
    out = []
    U, R = start.shape
    for u in range(U):
        for r in range(R):
            if active[u, r] and length[u, r] > 0:
                out.append((u, int(start[u, r]), int(start[u, r] + length[u, r])))
    return out


def wipe_out_rate(regions, ids_before, ids_after):
    """Fraction of regions present in `ids_before` (per unit: token ids in the cache
    before the event, -1 = empty slot) with no token in `ids_after`.
    Returns (rate, n_present)."""
    present = wiped = 0
    for u, lo, hi in regions:
        b = ids_before[u]
        if not np.any((b >= lo) & (b < hi)):
            continue
        present += 1
        a = ids_after[u]
        if not np.any((a >= lo) & (a < hi)):
            wiped += 1
    return (wiped / present if present else 0.0), present


def kept_set_iou(ids_prev, ids_now):
    """Mean over units of |A & B| / |A | B| for the kept token ids (-1 ignored)."""
    vals = []
    for a, b in zip(ids_prev, ids_now):
        A = set(int(x) for x in a if x >= 0)
        B = set(int(x) for x in b if x >= 0)
        if A or B:
            vals.append(len(A & B) / len(A | B))
    return float(np.mean(vals)) if vals else 0.0


def compact_ids(ids, kept_idx, n_kept):
    """Token ids of the compacted cache: ids[u, kept_idx[u, r]] for r < n_kept."""
    U, budget = kept_idx.shape
    out = np.full((U, budget), -1, np.int64)
    for u in range(U):
        n = int(n_kept[u])
        out[u, :n] = ids[u, kept_idx[u, :n]]
    return out


def run_chain(workload="qwen_1l", events=4, ablation="none", seed=None):
    """Run `events` compression events of a workload through the library and
    return one record per event."""
    import torch

    import eviction_gb300 as kvc
    import workload as wl

    w = wl.CONFIGS[workload]
    dev = torch.device("cuda")
    inp, reg = wl.generate(w, device=dev, seed=seed, return_regions=True)
    U = w.units
    T = inp.T
    h = kvc.Handle(kvc.Config(w.n_layers, w.batch, w.n_kv_heads, w.group, w.head_dim,
                              max(T, w.budget + w.interval), w.budget, window=w.window,
                              n_sink=w.n_sink, n_recent=w.n_recent, **kvc.ABLATIONS[ablation]))
    pad = wl.unit_pad(inp).cpu().numpy()
    ids = np.tile(np.arange(T, dtype=np.int64), (U, 1))
    ids[np.arange(T)[None, :] < pad[:, None]] = -1
    regions = region_tokens(*(reg[k].reshape(U, -1).cpu().numpy() for k in ("start", "length",
                                                                               "active")))
    next_id = T
    prev_kept = None
    records = []
    for e in range(events):
        out = h.outputs(inp.T)
        h.event(inp.q, inp.k, inp.v, inp.T, inp.pad, inp.n_carry, inp.credit, out["k_out"],
                out["v_out"], out["credit_out"], out["kept_idx"], out["n_kept"])
        torch.cuda.synchronize()
        kept = compact_ids(ids, out["kept_idx"].reshape(U, -1).cpu().numpy(),
                           out["n_kept"].reshape(U).cpu().numpy())
        rate, n_reg = wipe_out_rate(regions, ids, kept)
        rec = {"event": e + 1, "ablation": ablation, "wipe_out_rate": rate, "regions": n_reg}
        if prev_kept is not None:
            rec["kept_iou"] = kept_set_iou(prev_kept, kept)
        records.append(rec)
        prev_kept = kept
        if e + 1 == events:
            break
        inp, reg = wl.next_event(w, inp, out["k_out"], out["v_out"], out["credit_out"],
                                 out["n_kept"], e + 1, seed=seed, return_regions=True)
        I = w.interval
        ids = np.concatenate([kept, next_id + np.tile(np.arange(I, dtype=np.int64), (U, 1))], axis=1)
        start = reg["start"].reshape(U, -1).cpu().numpy() - w.budget + next_id  # slot -> id
        regions += region_tokens(start, reg["length"].reshape(U, -1).cpu().numpy(),
                                 reg["active"].reshape(U, -1).cpu().numpy())
        next_id += I
    return records


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--workload", default="qwen_1l")
    ap.add_argument("--events", type=int, default=4)
    ap.add_argument("--ablation", default="none")
    a = ap.parse_args()
    for rec in run_chain(a.workload, a.events, a.ablation):
        print(json.dumps(rec))


if __name__ == "__main__":
    main()
