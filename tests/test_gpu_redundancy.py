"""GPU parity of the second base score ("SkipKV: Selective Skipping of KV
Generation and Storage for Efficient Inference with Large Reasoning Models", A2
Method details, 4.1: token redundancy score after R-KV, and the sigma mix of the
final eviction score) against the oracle.

The oracle computes the pairwise definition (every cosine, fp64); the kernel
uses sum_j cos(k_i, k_j) = k^_i . sum_j k^_j - 1 in fp32.  Tolerances follow
from fp32 rounding (unit roundoff u = 2^-24) along the kernel's longest
accumulation chains, for a unit with n valid slots:
  r (mean cosine): |dr| <= 2 m u with m = ceil(n / 16) + 32 (per-thread sums
      over the rows of a CTA, the 8-term dot, the lane and warp trees);
  R = softmax(r):  relative error <= 2 |dr| + (n / 256 + 16) u (the exponent
      error plus the sum of e^r);
  f = sigma I - (1 - sigma) R: |df| <= sigma I (n / 256 + 20) u
      + (1 - sigma) R (rel. error of R) + 2 u |f|.
At sizes where the oracle's O(n^2 d) definition is too slow (32768 slots), r
is checked on sampled rows (exact differences log R_i - log R_j = r_i - r_j),
and sum R = 1 and the mix are checked as identities."""
import math

import numpy as np
import pytest
import torch

import workload as wl

pytestmark = pytest.mark.gpu

from tests import e2e_check as ec  # noqa: E402
from tests import gpu_util as gu  # noqa: E402

U32 = 2.0 ** -24


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _tol_r(n):
    return 2 * (math.ceil(n / 16) + 32) * U32


def _tol_R_rel(n):
    return 2 * _tol_r(n) + (n / 256 + 16) * U32


def _keys(rng, L, B, H, T, d, pads, zero_rows=True):
    """Keys with planted redundant regions (a shared direction added to a run of
    rows), zero rows and huge values in the padding (which must never count)."""
    k = rng.standard_normal((L, B, H, T, d)).astype(np.float32)
    for l in range(L):
        for b in range(B):
            for h in range(H):
                n = T - pads[b]
                for _ in range(4):
                    if n < 8:
                        break
                    ln = int(rng.integers(4, max(5, n // 4)))
                    st = pads[b] + int(rng.integers(0, n - ln + 1))
                    k[l, b, h, st:st + ln] += rng.lognormal(0, 0.7) * 3 * rng.standard_normal(d)
                if zero_rows and n > 3:
                    k[l, b, h, pads[b] + int(rng.integers(0, n))] = 0.0
                k[l, b, h, :pads[b]] = 4096.0
    return wl.bf16_bits(torch.from_numpy(k).to(torch.bfloat16))


def _scores(rng, L, B, H, T, pads):
    s = rng.gamma(0.5, 1.0, (L, B, H, T)).astype(np.float32)
    for b, p in enumerate(pads):
        s[:, b, :, :p] = -np.inf
    return s


def _run(kvc, L, B, H, T, d, pads, k_bits, score, sigma, out_red=True):
    cfg = kvc.Config(L, B, H, 1, d, T, 16, window=8, redundancy_sigma=sigma)
    h = kvc.Handle(cfg)
    k = torch.from_numpy(k_bits.view(np.int16)).view(torch.bfloat16).cuda()
    s = torch.from_numpy(score).cuda()
    sel = torch.full_like(s, 7.0)
    red = torch.full_like(s, 7.0) if out_red else None
    pad = torch.tensor(pads, dtype=torch.int32).cuda()
    h.redundancy_score(k, s, T, pad, sel, red)
    torch.cuda.synchronize()
    assert h.device_status() == 0
    return sel.cpu().numpy(), (red.cpu().numpy() if out_red else None), h


def _check_unit(f_g, R_g, f_o, R_o, s, pad, sigma):
    n = len(s) - pad
    assert np.all(np.isneginf(f_g[:pad])) and not R_g[:pad].any()
    if n == 0:
        return
    tr = _tol_R_rel(n)
    rel = np.abs(R_g[pad:].astype(np.float64) - R_o[pad:]) / R_o[pad:]
    assert rel.max() <= tr, f"R rel error {rel.max():.3g} > {tr:.3g}"
    sv = s[pad:].astype(np.float64)
    I = sv / sv.sum() if sv.sum() > 0 else np.zeros_like(sv)
    tol_f = sigma * I * (n / 256 + 20) * U32 + (1 - sigma) * R_o[pad:] * tr + \
        2 * U32 * np.abs(f_o[pad:])
    err = np.abs(f_g[pad:].astype(np.float64) - f_o[pad:])
    assert np.all(err <= tol_f), f"f error {(err / tol_f).max():.3g} x tolerance"


@pytest.mark.parametrize("L,B,H,T,d,pads", [
    (1, 3, 2, 300, 64, [0, 17, 299]),            # d 64, ragged, one valid slot
    (2, 12, 4, 700, 128, [0, 650, 3, 699, 7, 100, 0, 0, 42, 512, 9, 1]),
                                                 # 96 units: CTAs walk several units each
                                                 # only when the grid is smaller; ragged tails
    (1, 2, 2, 2500, 128, [0, 900]),              # many chunks per unit
    (1, 4, 2, 1536, 128, [0, 1, 700, 1536]),     # the 28-layer shape, an empty unit
    (1, 2, 1, 1112, 64, [5, 1000]),              # d 64, chunk tails
])
def test_redundancy_matches_oracle(ref, L, B, H, T, d, pads):
    import eviction_gb300 as kvc
    rng = np.random.default_rng(T + d)
    kb = _keys(rng, L, B, H, T, d, pads)
    sc = _scores(rng, L, B, H, T, pads)
    sigma = 0.1
    f_g, R_g, _ = _run(kvc, L, B, H, T, d, pads, kb, sc, sigma)
    U = L * B * H
    pad_u = np.array([pads[(u // H) % B] for u in range(U)])
    f_o, R_o, _ = ref.redundancy_score(kb.reshape(U, T, d), sc.reshape(U, T), pad_u, sigma)
    for u in range(U):
        _check_unit(f_g.reshape(U, T)[u], R_g.reshape(U, T)[u], f_o[u], R_o[u],
                    sc.reshape(U, T)[u], pad_u[u], sigma)


def test_degenerate_keys_and_scores(ref):
    """All keys parallel (r = 1, R uniform), all keys zero (r = 0), scores all 0
    (I = 0), sigma = 1 (the importance alone)."""
    import eviction_gb300 as kvc
    L, B, H, T, d = 1, 3, 1, 520, 128
    pads = [0, 8, 100]
    k = np.zeros((L, B, H, T, d), np.float32)
    k[0, 0, 0] = np.arange(1, d + 1) / d                  # parallel keys
    k[0, 0, 0] *= (2.0 ** (np.arange(T) % 5))[:, None]    # at power-of-two scales
    k[0, 1, 0] = 0.0                                      # all zero
    k[0, 2, 0] = np.random.default_rng(3).standard_normal((T, d))
    kb = wl.bf16_bits(torch.from_numpy(k).to(torch.bfloat16))
    sc = _scores(np.random.default_rng(4), L, B, H, T, pads)
    sc[0, 1, 0, pads[1]:] = 0.0
    for sigma in (0.1, 1.0):
        f_g, R_g, _ = _run(kvc, L, B, H, T, d, pads, kb, sc, sigma)
        f_o, R_o, _ = ref.redundancy_score(kb.reshape(B, T, d), sc.reshape(B, T),
                                           np.array(pads), sigma)
        for u in range(B):
            _check_unit(f_g.reshape(B, T)[u], R_g.reshape(B, T)[u], f_o[u], R_o[u],
                        sc.reshape(B, T)[u], pads[u], sigma)
        n0 = T - pads[0]
        assert np.allclose(R_g[0, 0, 0], 1.0 / n0, rtol=_tol_R_rel(n0), atol=0)


def test_in_place_equals_out_of_place():
    import eviction_gb300 as kvc
    L, B, H, T, d = 1, 2, 2, 900, 128
    pads = [0, 333]
    rng = np.random.default_rng(9)
    kb = _keys(rng, L, B, H, T, d, pads)
    sc = _scores(rng, L, B, H, T, pads)
    f_g, _, h = _run(kvc, L, B, H, T, d, pads, kb, sc, 0.1, out_red=False)
    k = torch.from_numpy(kb.view(np.int16)).view(torch.bfloat16).cuda()
    s = torch.from_numpy(sc).cuda()
    h.redundancy_score(k, s, T, torch.tensor(pads, dtype=torch.int32).cuda(), s)
    torch.cuda.synchronize()
    assert np.array_equal(s.cpu().numpy(), f_g)


@pytest.mark.parametrize("T,d,pads", [(32768, 128, [0, 20000]), (65536, 64, [123])])
def test_streamed_long_cache_sampled(ref, T, d, pads):
    """Slices too long to stay in shared memory (streamed twice): sampled rows
    against the oracle's single-row definition, sum R = 1, and the mix."""
    import eviction_gb300 as kvc
    L, H, B = 1, 1, len(pads)
    rng = np.random.default_rng(T)
    kb = _keys(rng, L, B, H, T, d, pads)
    sc = _scores(rng, L, B, H, T, pads)
    sigma = 0.1
    f_g, R_g, _ = _run(kvc, L, B, H, T, d, pads, kb, sc, sigma)
    for b, pad in enumerate(pads):
        n = T - pad
        R = R_g[0, b, 0].astype(np.float64)
        f = f_g[0, b, 0].astype(np.float64)
        assert abs(R[pad:].sum() - 1.0) <= (2 * (n / 256 + 16) + 4) * U32
        rows = np.unique(np.concatenate([[pad, T - 1], rng.integers(pad, T, 40)]))
        r_o = ref.mean_cosine_rows(kb[0, b, 0], pad, rows)
        lr = np.log(R[rows])
        d_g = lr - lr.mean()
        d_o = r_o - r_o.mean()
        assert np.abs(d_g - d_o).max() <= 2 * _tol_r(n) + 8 * U32
        s = sc[0, b, 0, pad:].astype(np.float64)
        want = sigma * s / s.sum() - (1 - sigma) * R[pad:]
        tol = sigma * s / s.sum() * (n / 256 + 20) * U32 + (1 - sigma) * R[pad:] * 4 * U32 + \
            2 * U32 * np.abs(want)
        assert np.all(np.abs(f[pad:] - want) <= tol)
        assert np.all(np.isneginf(f[:pad]))


def test_bench_shape_sampled(ref):
    """The 28-layer workload's keys (3584 units, T 1536, the launch the event
    times), a seeded score, 6 sampled units against the oracle."""
    import eviction_gb300 as kvc
    w = wl.CONFIGS["qwen_28l"]
    inp = wl.generate(w, device="cuda")
    T, U = inp.T, w.units
    rng = np.random.default_rng(28)
    score = torch.from_numpy(rng.gamma(0.5, 1.0, (w.n_layers, w.batch, w.n_kv_heads, T))
                             .astype(np.float32)).cuda()
    sigma = 0.1
    h = kvc.Handle(gu.config_for(w, T, redundancy_sigma=sigma))
    sel = torch.empty_like(score)
    red = torch.empty_like(score)
    h.redundancy_score(inp.k, score, T, inp.pad, sel, red)
    torch.cuda.synchronize()
    assert h.device_status() == 0
    units = rng.choice(U, 6, replace=False)
    idx = torch.as_tensor(units, device="cuda", dtype=torch.long)
    kb = wl.bf16_bits(wl.units_of(inp.k, w).index_select(0, idx))
    sc = score.reshape(U, T).index_select(0, idx).cpu().numpy()
    pad_u = wl.unit_pad(inp).to("cuda").index_select(0, idx).cpu().numpy()
    f_o, R_o, _ = ref.redundancy_score(kb, sc, pad_u, sigma)
    f_g = sel.reshape(U, T).index_select(0, idx).cpu().numpy()
    R_g = red.reshape(U, T).index_select(0, idx).cpu().numpy()
    for i in range(len(units)):
        _check_unit(f_g[i], R_g[i], f_o[i], R_o[i], sc[i], int(pad_u[i]), sigma)


def test_repeat_runs_identical():
    import eviction_gb300 as kvc
    L, B, H, T, d = 1, 2, 2, 1536, 128
    pads = [0, 50]
    rng = np.random.default_rng(1)
    kb = _keys(rng, L, B, H, T, d, pads)
    sc = _scores(rng, L, B, H, T, pads)
    a, ra, _ = _run(kvc, L, B, H, T, d, pads, kb, sc, 0.1)
    b, rb, _ = _run(kvc, L, B, H, T, d, pads, kb, sc, 0.1)
    assert np.array_equal(a, b) and np.array_equal(ra, rb)


def test_sigma_zero_refused():
    import eviction_gb300 as kvc
    h = kvc.Handle(kvc.Config(1, 1, 1, 1, 64, 64, 16, window=8))
    z = torch.zeros((1, 1, 1, 64), device="cuda")
    k = torch.zeros((1, 1, 1, 64, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kvc.KvcError):
        h.redundancy_score(k, z, 64, torch.zeros(1, dtype=torch.int32, device="cuda"), z.clone())


def test_event_with_sigma_end_to_end(ref):
    """The event with sigma = 0.1 against the oracle's event: kept sets equal up
    to near-ties of the mixed score (the GPU score is within 1e-4 relative of
    the oracle's, so I moves by at most 2e-4 I; R as above)."""
    import eviction_gb300 as kvc
    w = wl.scaled(wl.CONFIGS["qwen_1l"], batch=2, n_kv_heads=2, T=1000)
    inp = wl.generate(w)
    T = inp.T
    sigma = 0.1
    p = gu.ref_params(ref, w, redundancy_sigma=sigma)
    r = ref.event(p, *gu.oracle_inputs(inp))
    h = kvc.Handle(gu.config_for(w, T, redundancy_sigma=sigma))
    out = gu.gpu_event(h, gu.to_device(inp), T)
    assert h.device_status() == 0
    U = w.units
    kept = out["kept_idx"].reshape(U, -1).cpu().numpy()
    nk = out["n_kept"].reshape(U).cpu().numpy()
    assert np.array_equal(nk, r["n_kept"])
    pad_u = gu.oracle_inputs(inp)[4]
    for u in range(U):
        a = set(kept[u, :nk[u]].tolist())
        b = set(r["kept_idx"][u, :nk[u]].tolist())
        if a == b:
            continue
        pu = pad_u[u]
        s = r["score"][u][pu:].astype(np.float64)
        I = s / s.sum()
        tol = 4e-4 * sigma * I.max() + 1e-4 * (1 - sigma) * r["redundancy"][u][pu:].max()
        f = r["sel_score"][u]
        ns = int(r["n_seg"][u])
        gap = ec.cutoff_distance(kept[u, :nk[u]], r["kept_idx"][u, :nk[u]], f, int(pu), T,
                                 r["seg_start"][u, :ns], r["seg_len"][u, :ns], w.budget,
                                 w.n_sink, w.n_recent)
        assert gap <= tol, (f"unit {u}: a slot kept by one side only lies {gap:.3g} from its "
                            f"segment's cut-off (tolerance {tol:.3g})")
    # sigma really changes the selection
    r0 = ref.event(gu.ref_params(ref, w), *gu.oracle_inputs(inp))
    assert not np.array_equal(r0["kept_idx"], r["kept_idx"])


@pytest.mark.parametrize("seed", range(8))
def test_redundancy_random_shapes(ref, seed):
    """Seeded random small shapes (T from 1, both head sizes, units that are all
    padding, one or two valid slots) against the oracle's pairwise definition."""
    import eviction_gb300 as kvc
    rng = np.random.default_rng(500 + seed)
    d = int(rng.choice([64, 128]))
    T = int(rng.integers(1, 3000))
    B, H = int(rng.integers(1, 4)), int(rng.integers(1, 3))
    pads = [int(x) for x in rng.integers(0, T + 1, B)]
    pads[0] = [0, T, max(T - 1, 0), max(T - 2, 0)][seed % 4]
    kb = _keys(rng, 1, B, H, T, d, pads)
    sc = _scores(rng, 1, B, H, T, pads)
    sigma = float(rng.choice([0.1, 0.5, 1.0]))
    f_g, R_g, _ = _run(kvc, 1, B, H, T, d, pads, kb, sc, sigma)
    U = B * H
    pad_u = np.array([pads[(u // H) % B] for u in range(U)])
    f_o, R_o, _ = ref.redundancy_score(kb.reshape(U, T, d), sc.reshape(U, T), pad_u, sigma)
    for u in range(U):
        _check_unit(f_g.reshape(U, T)[u], R_g.reshape(U, T)[u], f_o[u], R_o[u],
                    sc.reshape(U, T)[u], pad_u[u], sigma)
