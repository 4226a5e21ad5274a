"""End-to-end invariants of the oracle's event on the synthetic workloads.

These check the properties the pages state for a whole event (mass sums to 1,
quotas sum to the budget, sinks and the recent suffix are kept, the kept set is
sorted and unique and never touches padding, compaction is a gather) on inputs
from the seeded generator, at sizes the oracle finishes in seconds.
"""
import numpy as np
import pytest

import workload as wl


def _params(ref, w):
    return ref.RefParams(group=w.group, head_dim=w.head_dim, window=w.window,
                         budget=w.budget, n_sink=w.n_sink, n_recent=w.n_recent)


def _run(ref, w):
    inp = wl.generate(w)
    p = _params(ref, w)
    out = ref.event(p, wl.bf16_bits(wl.q_units(inp.q, w)), wl.bf16_bits(wl.units_of(inp.k, w)),
                    wl.bf16_bits(wl.units_of(inp.v, w)), wl.units_of(inp.credit, w).numpy(),
                    wl.unit_pad(inp).numpy(), wl.unit_n_carry(inp).numpy())
    return inp, p, out


CASES = {
    "tiny": wl.CONFIGS["tiny"],
    "qwen_small": wl.scaled(wl.CONFIGS["qwen_1l"], batch=2, n_kv_heads=1),
    "ragged_small": wl.scaled(wl.CONFIGS["llama_ragged"], n_layers=1, batch=4, n_kv_heads=1,
                              group=2, prefill=(10, 300), generated=200, budget=256),
}


@pytest.mark.parametrize("name", list(CASES))
def test_event_invariants(ref, name):
    w = CASES[name]
    inp, p, out = _run(ref, w)
    T = inp.T
    pads = wl.unit_pad(inp).numpy()
    S = ref.s_max(p, T)
    for u, pad in enumerate(pads):
        n = T - pad
        m = out["mass"][u].astype(np.float64)
        assert abs(m[pad:].sum() - 1.0) < 1e-5 and np.all(m[:pad] == 0)
        assert np.all(np.isneginf(out["score"][u][:pad]))
        ns = out["n_seg"][u]
        st, ln, q = out["seg_start"][u][:ns], out["seg_len"][u][:ns], out["quota"][u][:ns]
        assert st[0] == pad and ln.sum() == n and ns <= S
        assert np.all(st[1:] == st[:-1] + ln[:-1])
        assert ln.min() >= min(16, n) and ln.max() <= 256
        B = min(w.budget, n)
        assert q.sum() == B and np.all(q <= ln) and np.all(q >= np.minimum(1, ln))
        nk = out["n_kept"][u]
        kept = out["kept_idx"][u][:nk]
        assert nk == B and np.all(out["kept_idx"][u][nk:] == -1)
        assert np.all(np.diff(kept) > 0) and kept[0] >= pad and kept[-1] < T
        n_s = min(w.n_sink, B)
        n_r = min(w.n_recent, B - n_s)
        assert set(range(pad, pad + n_s)) <= set(kept.tolist())
        assert set(range(T - n_r, T)) <= set(kept.tolist())
        kb = wl.bf16_bits(wl.units_of(inp.k, w))[u]
        assert np.array_equal(out["k_out"][u][:nk], kb[kept])
        assert np.array_equal(out["credit_out"][u][:nk], out["credit_post"][u][kept])


def test_event_keeps_everything_when_short(ref):
    """A cache no longer than the budget keeps every valid slot."""
    w = wl.scaled(wl.CONFIGS["tiny"], T=200, budget=256, regions=(2, 2))
    inp, p, out = _run(ref, w)
    assert out["n_kept"][0] == 200
    assert list(out["kept_idx"][0][:200]) == list(range(200))


def test_event_all_padding(ref):
    """A sequence with no valid slot produces nothing and keeps nothing."""
    w = wl.CONFIGS["tiny"]
    inp = wl.generate(w)
    p = _params(ref, w)
    T = inp.T
    out = ref.event(p, wl.bf16_bits(wl.q_units(inp.q, w)), wl.bf16_bits(wl.units_of(inp.k, w)),
                    wl.bf16_bits(wl.units_of(inp.v, w)), np.zeros((1, T), np.float32),
                    np.array([T], np.int32), np.array([0], np.int32))
    assert out["n_kept"][0] == 0 and out["n_seg"][0] == 0
    assert np.all(out["kept_idx"][0] == -1) and not out["k_out"].any()
    assert not out["mass"].any()


def test_thread_split_is_the_same_computation(ref):
    """The batched calls split over host threads (units are independent, the C code
    runs unit by unit) give exactly the single-threaded results."""
    w = wl.scaled(wl.CONFIGS["llama_ragged"], n_layers=1, batch=5, n_kv_heads=2, group=2,
                  head_dim=64, prefill=(20, 200), generated=100, budget=120)
    inp = wl.generate(w)
    p = ref.RefParams(group=w.group, head_dim=w.head_dim, window=w.window, budget=w.budget,
                      n_sink=w.n_sink, n_recent=w.n_recent)
    args = (wl.bf16_bits(wl.q_units(inp.q, w)), wl.bf16_bits(wl.units_of(inp.k, w)),
            wl.bf16_bits(wl.units_of(inp.v, w)), wl.units_of(inp.credit, w).numpy(),
            wl.unit_pad(inp).numpy(), wl.unit_n_carry(inp).numpy())
    one = ref.event(p, *args)
    many = ref.event(p, *args, threads=3)
    assert one.keys() == many.keys()
    for k in one:
        assert np.array_equal(one[k], many[k]), k
