"""Pins of the oracle's ablation switches ("Adaptive Mass-Segmented KV Compression
for Long-Form Reasoning", Experiments, ablation table: fixed-length segments, no
mass-weighted quota, no EMA credit, global head-only top-k).

Each switch is pinned against something other than the oracle itself:
closed-form segment shapes, totals from the independent boundary routine, the
closed-form apportionment of equal-length segments, and a plain numpy sort for
the global top-k.  ("No EMA credit" is beta = 1: pinned in test_oracle_pins.)
"""
import numpy as np
import pytest

pytestmark = pytest.mark.filterwarnings("ignore")


def _mass(rng, T, pad, peaky=4):
    m = np.zeros(T, np.float32)
    w = rng.random(T - pad) ** peaky
    m[pad:] = (w / w.sum()).astype(np.float32)
    return m


@pytest.mark.parametrize("T,pad,L", [(300, 0, 16), (301, 7, 16), (1536, 0, 64), (40, 30, 16),
                                     (1000, 1, 250)])
def test_fixed_segments_shape(ref, T, pad, L):
    rng = np.random.default_rng(T + pad)
    m = _mass(rng, T, pad)
    st, ln, M = ref.segments_ablation(m, pad, seg_fixed=L)
    n = T - pad
    ns = max(1, n // L)
    assert len(st) == ns
    assert np.array_equal(st, np.arange(ns) * L)
    assert ln.sum() == n
    if ns > 1:
        assert np.all(ln[:-1] == L)
    assert L <= ln[-1] < 2 * L or ns == 1
    # the recounted masses add up to the fixed-point total of the boundary routine
    _, total = ref.boundaries(m, pad, 0.1)
    assert int(M.sum()) == total


def test_global_one_segment(ref):
    rng = np.random.default_rng(3)
    m = _mass(rng, 777, 12)
    st, ln, M = ref.segments_ablation(m, 12, global_=1)
    assert list(st) == [0] and list(ln) == [765]
    assert int(M[0]) == ref.boundaries(m, 12, 0.1)[1]


@pytest.mark.parametrize("n,L,budget", [(512, 16, 100), (1536, 64, 1024), (1024, 128, 250),
                                        (96, 16, 7)])
def test_quota_by_length_equal_segments(ref, n, L, budget):
    """Equal lengths: the extra units go to the lowest segments, whatever the mass."""
    rng = np.random.default_rng(n + budget)
    p = ref.RefParams(group=1, head_dim=64, window=8, budget=budget, seg_fixed=L,
                      quota_by_len=1)
    ns = n // L
    expect = np.array([budget // ns + (1 if i < budget % ns else 0) for i in range(ns)])
    if budget < ns:  # infeasible minimums: the heaviest segments get them
        pytest.skip("covered by the mass-ordered rule")
    for peaky in (1, 8):
        m = _mass(rng, n, 0, peaky).reshape(1, n)
        st, sl, q, ns_out = ref.segment_quota(p, m, np.zeros(1, np.int32))
        assert ns_out[0] == ns
        assert np.array_equal(q[0, :ns], expect)


def test_quota_by_length_ignores_mass(ref):
    rng = np.random.default_rng(9)
    T = 700
    p = ref.RefParams(group=1, head_dim=64, window=8, budget=300, seg_fixed=48, quota_by_len=1)
    outs = []
    for peaky in (1, 3, 12):
        m = _mass(rng, T, 5, peaky).reshape(1, T)
        outs.append(ref.segment_quota(p, m, np.full(1, 5, np.int32))[2])
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
    # the mass-weighted rule does depend on the mass
    p2 = ref.RefParams(group=1, head_dim=64, window=8, budget=300, seg_fixed=48)
    q_mass = [ref.segment_quota(p2, _mass(np.random.default_rng(s), T, 5, 12).reshape(1, T),
                                np.full(1, 5, np.int32))[2] for s in (1, 2)]
    assert not np.array_equal(q_mass[0], q_mass[1])


@pytest.mark.parametrize("seed,T,pad,budget,n_recent", [(0, 400, 0, 100, 16), (1, 900, 33, 256, 64),
                                                        (2, 64, 10, 60, 8), (3, 300, 0, 299, 32)])
def test_global_topk_is_plain_topk(ref, seed, T, pad, budget, n_recent):
    """One segment: must-keep (4 sinks, recent suffix) plus the best other slots by
    score, ties to the lower slot -- a numpy lexsort, independently."""
    rng = np.random.default_rng(seed)
    p = ref.RefParams(group=1, head_dim=64, window=8, budget=budget, n_recent=n_recent,
                      global_topk=1)
    m = _mass(rng, T, pad).reshape(1, T)
    score = np.full((1, T), -np.inf, np.float32)
    score[0, pad:] = np.round(rng.random(T - pad) * 20).astype(np.float32)  # many ties
    pads = np.full(1, pad, np.int32)
    st, ln, q, ns = ref.segment_quota(p, m, pads)
    assert ns[0] == 1 and q[0, 0] == min(budget, T - pad)
    kept, nk = ref.select(p, score, pads, st, ln, q, ns)
    n = T - pad
    B = min(budget, n)
    n_s = min(4, B)
    n_r = min(n_recent, B - n_s)
    must = set(range(pad, pad + n_s)) | set(range(T - n_r, T))
    cand = np.array([i for i in range(pad, T) if i not in must])
    order = np.lexsort((cand, -score[0, cand]))  # score descending, then slot ascending
    picks = set(cand[order[:B - len(must)]].tolist())
    expect = sorted(must | picks)
    assert nk[0] == B
    assert kept[0, :B].tolist() == expect
