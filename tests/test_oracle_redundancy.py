"""Pins of the oracle's second base score ("SkipKV: Selective Skipping of KV
Generation and Storage for Efficient Inference with Large Reasoning Models", A2
Method details, 4.1: token redundancy score after R-KV, and the sigma mix of the
final eviction score): closed forms
on keys whose cosines are known exactly (parallel, antipodal, orthogonal
clusters at arbitrary scales), the mask, zero keys, the softmax and the
normalised importance, and the sign of the mix seen through the selection."""
import numpy as np
import pytest


def _bits(x):
    """fp32 values that are exact in bf16 -> bf16 bit patterns."""
    x = np.asarray(x, np.float32)
    b = (x.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((b.astype(np.uint32) << 16).view(np.float32), x), "not bf16-exact"
    return b


def _unit(vectors, pad_rows=0, d=None, garbage=0.0):
    """[T, d] keys: pad_rows rows of `garbage` then the given vectors."""
    v = np.asarray(vectors, np.float32)
    d = d or v.shape[1]
    out = np.full((pad_rows + len(v), d), garbage, np.float32)
    out[pad_rows:] = v
    return _bits(out)


def _axis(d, i, scale=1.0):
    e = np.zeros(d, np.float32)
    e[i] = scale
    return e


def test_two_orthogonal_clusters_any_scale(ref):
    """m keys along e0 and n-m along e1, every key at its own power-of-two
    scale: r = (m-1)/(n-1) in the first cluster and (n-m-1)/(n-1) in the
    second (self excluded, keys normalised, mean over the others)."""
    d, m, n = 16, 5, 12
    scales = [2.0 ** (i % 7 - 3) for i in range(n)]
    keys = [_axis(d, 0 if i < m else 1, scales[i]) for i in range(n)]
    k = _unit(keys)
    r = ref.mean_cosine_rows(k, 0, np.arange(n))
    want = np.array([(m - 1) / (n - 1)] * m + [(n - m - 1) / (n - 1)] * (n - m))
    assert np.array_equal(r, want)


def test_antipodal_keys_count_negative(ref):
    """cos = -1 between opposite keys: r_i = (same - 1 - opposite) / (n - 1)."""
    d = 8
    signs = [1, 1, -1, 1, -1, -1, -1]
    k = _unit([_axis(d, 3, s * 0.5) for s in signs])
    n = len(signs)
    r = ref.mean_cosine_rows(k, 0, np.arange(n))
    for i, s in enumerate(signs):
        same = sum(1 for t in signs if t == s)
        assert r[i] == (same - 1 - (n - same)) / (n - 1)


def test_general_angle_closed_form(ref):
    """Keys (1, 0), (1, 1), (0, 1) (scaled): cosines 1/sqrt2, 0, 1/sqrt2."""
    k = _unit([[3.0, 0.0], [0.5, 0.5], [0.0, 0.25]])
    r = ref.mean_cosine_rows(k, 0, np.arange(3))
    c = 1 / np.sqrt(2)
    assert np.allclose(r, [c / 2, c, c / 2], rtol=0, atol=1e-15)


def test_mask_and_zero_keys(ref):
    """Padding rows (huge keys) never count; a zero key has cosine 0 with all
    keys but still counts in the mean's denominator."""
    d = 8
    keys = [_axis(d, 0), _axis(d, 0, 2.0), np.zeros(d), _axis(d, 1)]
    k_clean = _unit(keys)
    k_pad = _unit(keys, pad_rows=5, garbage=1024.0)
    r_clean = ref.mean_cosine_rows(k_clean, 0, np.arange(4))
    r_pad = ref.mean_cosine_rows(k_pad, 5, np.arange(5, 9))
    assert np.array_equal(r_clean, r_pad)
    assert r_clean.tolist() == [1 / 3, 1 / 3, 0.0, 0.0]


def test_fewer_than_two_valid(ref):
    k = _unit([_axis(4, 0), _axis(4, 1), _axis(4, 2)])
    assert ref.mean_cosine_rows(k, 2, [2]).tolist() == [0.0]
    f, R, r = ref.redundancy_score(k[None], np.array([[0, 0, 5.0]], np.float32), [2], 0.1)
    assert r[0, 2] == 0.0 and R[0, 2] == 1.0
    assert f[0, 2] == pytest.approx(0.1 * 1.0 - 0.9 * 1.0, abs=1e-15)
    assert np.all(np.isneginf(f[0, :2])) and not R[0, :2].any()


def test_softmax_importance_and_mix(ref):
    """R = softmax(r) over valid slots, I = s / sum s, f = sigma I - (1-sigma) R,
    checked on the two-cluster closed form with integer scores."""
    d, m, n, pad = 8, 3, 7, 2
    keys = [_axis(d, 0)] * m + [_axis(d, 1)] * (n - m)
    k = _unit(keys, pad_rows=pad, garbage=3.0)
    score = np.array([-np.inf, -np.inf, 1, 2, 3, 4, 5, 6, 7], np.float32)
    sigma = 0.25
    f, R, r = ref.redundancy_score(k[None], score[None], [pad], sigma)
    ra, rb = (m - 1) / (n - 1), (n - m - 1) / (n - 1)
    z = m * np.exp(ra) + (n - m) * np.exp(rb)
    R_want = np.array([np.exp(ra) / z] * m + [np.exp(rb) / z] * (n - m))
    I_want = np.arange(1, 8) / 28.0
    assert np.allclose(R[0, pad:], R_want, rtol=1e-14, atol=0)
    assert abs(R[0, pad:].sum() - 1.0) < 1e-14
    assert np.allclose(f[0, pad:], sigma * I_want - (1 - sigma) * R_want, rtol=1e-13, atol=1e-16)
    # sigma = 1: the importance alone
    f1, _, _ = ref.redundancy_score(k[None], score[None], [pad], 1.0)
    assert np.allclose(f1[0, pad:], I_want, rtol=1e-15, atol=0)
    # all-zero scores: I = 0, the order is the redundancy's alone
    f0, R0, _ = ref.redundancy_score(k[None], np.where(np.isinf(score), score, 0)[None], [pad],
                                     sigma)
    assert np.allclose(f0[0, pad:], -(1 - sigma) * R0[0, pad:], rtol=1e-15, atol=0)


def test_selection_prefers_non_redundant_keys(ref):
    """Equal scores everywhere; half the candidates share one key direction,
    the other half are mutually orthogonal.  With a small sigma the kept
    non-must-keep slots are all orthogonal ones (more redundant -> evicted
    first); with sigma = 1 the ties fall to the lower slots (the score order)."""
    d, n = 64, 48
    rng = np.random.default_rng(0)
    red = rng.permutation(n)[: n // 2]
    keys = np.zeros((n, d), np.float32)
    axis = 0
    for i in range(n):
        if i in red:
            keys[i, 0] = 1.0
        else:
            axis += 1
            keys[i, axis] = 1.0
    k = _unit(keys)
    score = np.ones(n, np.float32)
    budget, n_sink, n_recent = 20, 2, 2
    st = np.array([0], np.int32)
    ln = np.array([n], np.int32)
    qu = np.array([budget], np.int32)
    for sigma, want_orth in ((0.1, True), (1.0, False)):
        f, _, _ = ref.redundancy_score(k[None], score[None], [0], sigma)
        kept = ref.select_unit(f[0].astype(np.float32), 0, st, ln, qu, budget, n_sink, n_recent)
        free = [v for v in kept if n_sink <= v < n - n_recent]
        assert len(kept) == budget
        if want_orth:
            assert all(v not in red for v in free)
        else:
            assert free == list(range(n_sink, n_sink + len(free)))


def test_event_with_sigma_uses_mixed_score(ref):
    """The event with sigma > 0 keeps exactly what select keeps on the mixed
    score, and its segments and quotas are those of sigma = 0."""
    import workload as wl
    w = wl.scaled(wl.CONFIGS["tiny"], n_recent=16)
    inp = wl.generate(w)
    from tests import gpu_util as gu  # input marshalling only (no GPU calls)
    q, k, v, c, pad, nc = gu.oracle_inputs(inp)
    p0 = gu.ref_params(ref, w)
    p1 = gu.ref_params(ref, w, redundancy_sigma=0.1)
    r0 = ref.event(p0, q, k, v, c, pad, nc)
    r1 = ref.event(p1, q, k, v, c, pad, nc)
    for key in ("mass", "seg_start", "seg_len", "quota", "n_seg"):
        assert np.array_equal(r0[key], r1[key])
    f, _, _ = ref.redundancy_score(k, r0["score"], pad, 0.1)
    kept, nk = ref.select(p1, f.astype(np.float32), pad, r0["seg_start"], r0["seg_len"],
                          r0["quota"], r0["n_seg"])
    assert np.array_equal(kept, r1["kept_idx"]) and np.array_equal(nk, r1["n_kept"])
    assert not np.array_equal(r0["kept_idx"], r1["kept_idx"])
