"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Bars (floating point from the benchmark spec's tolerance, integers bit-exact):
  * mass / credit: |gpu - ref| <= 1e-4 |ref| + 1e-9 per element; the score (max-
    pooled usage) uses the same bound; padding holds exactly 0 / -inf;
  * segmentation, quotas, kept sets: bit-exact when both sides get the same fp32
    mass / score (taken from the oracle or the seeded generator);
  * compaction: bit-exact;
  * end to end: identical kept sets except swapped pairs at score near-ties
    (|s_a - s_b| below 1e-5 of the unit's total usage, at least G*W), and
    boundary shifts only where the oracle's cumulative mass sits within 1e-5
    of a cut threshold.
Sizes: several 128-row / 128-slot tiles with a ragged tail, left padding, a
sequence shorter than the window, an all-padding sequence, d = 64 and 128.
"""
import zlib

import numpy as np
import pytest
import torch

import workload as wl

pytestmark = pytest.mark.gpu

from tests import gpu_util as gu  # noqa: E402
from tests import threshold_cases  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


CASES = {
    # d 64, G 1, W 32, one unit (the tiny single-event configuration)
    "tiny": (wl.CONFIGS["tiny"], None),
    # Qwen shapes at oracle-friendly size: T not a multiple of 128
    "qwen_small": (wl.scaled(wl.CONFIGS["qwen_1l"], batch=2, n_kv_heads=2, T=1000), None),
    # ragged: left padding, incl. a sequence shorter than W and one fully padded
    "ragged": (wl.scaled(wl.CONFIGS["llama_ragged"], n_layers=1, batch=5, n_kv_heads=2,
                         group=4, prefill=(10, 400), generated=300, budget=300),
               [0, 37, 250, 620, 700]),
}


def _inputs(name):
    w, pads = CASES[name]
    inp = wl.generate(w)
    if pads is not None:
        T = inp.T
        pad = torch.tensor([min(p, T) for p in pads], dtype=torch.int32)
        slot = torch.arange(T).view(1, 1, 1, T, 1)
        valid = slot >= pad.view(1, -1, 1, 1, 1)
        inp.k = torch.where(valid, inp.k, torch.zeros((), dtype=inp.k.dtype))
        inp.v = torch.where(valid, inp.v, torch.zeros((), dtype=inp.v.dtype))
        inp.pad = pad
        inp.n_carry = (T - pad).to(torch.int32)
    return w, inp


@pytest.fixture(scope="module")
def oracle_runs(ref):
    out = {}
    for name in CASES:
        w, inp = _inputs(name)
        p = gu.ref_params(ref, w)
        out[name] = (w, inp, ref.event(p, *gu.oracle_inputs(inp)))
    return out


@pytest.mark.parametrize("name", list(CASES))
def test_mass_score_credit(oracle_runs, name):
    import eviction_gb300 as kvc
    w, inp, r = oracle_runs[name]
    h = kvc.Handle(gu.config_for(w, inp.T))
    m, s, c = gu.gpu_mass(h, gu.to_device(inp), inp.T)
    assert h.device_status() == 0
    ok_m, rel_m = gu.mass_close(m, r["mass"])
    ok_s, rel_s = gu.mass_close(s, r["score"])
    ok_c, rel_c = gu.mass_close(c, r["credit_post"])
    assert ok_m and ok_s and ok_c, (f"mass rel {rel_m:.3g}, score rel {rel_s:.3g}, "
                                    f"credit rel {rel_c:.3g}")


@pytest.mark.parametrize("name", list(CASES))
def test_segment_quota_bit_exact(ref, oracle_runs, name):
    """Same fp32 mass (the oracle's) on both sides -> identical integers."""
    import eviction_gb300 as kvc
    w, inp, r = oracle_runs[name]
    p = gu.ref_params(ref, w)
    h = kvc.Handle(gu.config_for(w, inp.T))
    st, ln, qu, ns = gu.gpu_segment_quota(h, r["mass"], inp.pad.numpy(), inp.T)
    assert np.array_equal(ns, r["n_seg"])
    assert np.array_equal(st, r["seg_start"])
    assert np.array_equal(ln, r["seg_len"])
    assert np.array_equal(qu, r["quota"])


def _random_masses(rng, U, T, pads):
    m = np.zeros((U, T), np.float32)
    for u in range(U):
        p = pads[u]
        n = T - p
        if n <= 0:
            continue
        w = rng.random(n) ** rng.choice([1, 4, 12])
        for _ in range(rng.integers(0, 4)):
            w[rng.integers(0, n)] += rng.random() * w.sum()
        m[u, p:] = (w / w.sum()).astype(np.float32)
    return m


@pytest.mark.parametrize("seed,T,budget,delta,seg_min,seg_max", [
    (1, 1536, 1024, 0.1, 16, 256), (2, 900, 64, 0.05, 16, 64), (3, 4000, 512, 0.1, 16, 256),
    (4, 300, 6, 0.02, 8, 16), (5, 32768, 4096, 0.1, 16, 256)])
def test_segment_quota_random_masses(ref, seed, T, budget, delta, seg_min, seg_max):
    """Peaky random masses, infeasible minimums (budget < #segments), long T."""
    import eviction_gb300 as kvc
    rng = np.random.default_rng(seed)
    B, H = 3, 2
    pads = rng.integers(0, T // 2, B).astype(np.int32)
    pads[0] = 0
    mass = _random_masses(rng, B * H, T, np.repeat(pads, H))
    cfg = kvc.Config(1, B, H, 1, 64, T, budget, window=8, delta=delta, seg_min=seg_min,
                     seg_max=seg_max)
    h = kvc.Handle(cfg)
    st, ln, qu, ns = gu.gpu_segment_quota(h, mass, pads, T)
    p = ref.RefParams(group=1, head_dim=64, window=8, budget=budget, delta=delta,
                      seg_min=seg_min, seg_max=seg_max)
    rs, rl, rq, rn = ref.segment_quota(p, mass, np.repeat(pads, H))
    assert np.array_equal(ns, rn)
    assert np.array_equal(st, rs) and np.array_equal(ln, rl) and np.array_equal(qu, rq)


def _adversarial_masses(rng, U, T, pads, kind):
    """Masses that drive the quota correction through its cases: peaky ones
    (heavy short segments clipped to their length, so the rounding leaves the
    budget over or short by many units), uniform ones (equal remainders: the
    index tie rules decide), two-level ones (many exact ties)."""
    m = np.zeros((U, T), np.float32)
    for u in range(U):
        n = T - pads[u]
        if n <= 0:
            continue
        if kind == "uniform":
            w = np.ones(n)
        elif kind == "two_level":
            w = np.where(rng.random(n) < 0.5, 1.0, 3.0)
        else:
            w = rng.random(n) ** 8
            hot = rng.integers(0, n, rng.integers(1, 6))
            w[hot] += rng.random(hot.size) * 50 * w.sum()
        m[u, pads[u]:] = (w / w.sum()).astype(np.float32)
    return m


@pytest.mark.parametrize("kind", ["peaky", "uniform", "two_level"])
@pytest.mark.parametrize("T,budget,delta,q_min,seg_min,seg_max", [
    (1536, 1024, 0.1, 4, 16, 256), (1536, 200, 0.02, 8, 16, 64), (777, 700, 0.05, 4, 8, 32),
    (2100, 2000, 0.01, 2, 4, 16)])
def test_quota_correction_many_units(ref, kind, T, budget, delta, q_min, seg_min, seg_max):
    """512 units per case against the oracle's one-unit-at-a-time correction,
    bit-exact: segments, lengths and quotas."""
    import eviction_gb300 as kvc
    rng = np.random.default_rng(zlib.crc32(f"{kind}/{T}/{budget}".encode()))
    B, H = 64, 8
    pads = rng.integers(0, T // 3, B).astype(np.int32)
    pads[:4] = 0
    mass = _adversarial_masses(rng, B * H, T, np.repeat(pads, H), kind)
    cfg = kvc.Config(1, B, H, 1, 64, T, budget, window=8, delta=delta, q_min=q_min,
                     seg_min=seg_min, seg_max=seg_max)
    h = kvc.Handle(cfg)
    st, ln, qu, ns = gu.gpu_segment_quota(h, mass, pads, T)
    p = ref.RefParams(group=1, head_dim=64, window=8, budget=budget, delta=delta, q_min=q_min,
                      seg_min=seg_min, seg_max=seg_max)
    rs, rl, rq, rn = ref.segment_quota(p, mass, np.repeat(pads, H))
    assert np.array_equal(ns, rn)
    assert np.array_equal(st, rs) and np.array_equal(ln, rl) and np.array_equal(qu, rq)


@pytest.mark.parametrize("delta", [0.1, 0.07, 0.013])
def test_segment_thresholds_on_rounding_cases(ref, delta):
    """Masses whose cut points sit on tau_k - 1 and tau_k exactly, with tau_k
    where the double rounding of k*Delta*S decides it (below half of the last
    bit, ties to even and odd, exact, just under a bit): the segments, lengths
    and quotas bit-identical to the oracle's, and every crafted cut where the
    double threshold puts it (a threshold one off either way moves it)."""
    import eviction_gb300 as kvc
    rng = np.random.default_rng(zlib.crc32(f"thresholds/{delta}".encode()))
    T, B, H, budget = 4096, 10, 4, 700
    K = threshold_cases.threshold_count(delta)
    ks = [k for k in range(1, K + 1) if threshold_cases.usable(k, delta)]
    pads = rng.integers(0, T - 1536 + 1, B).astype(np.int32)
    pads[0] = 0
    mass = np.zeros((B * H, T), np.float32)
    crafted = []
    for u in range(B * H):
        pad = int(pads[u // H])
        c = threshold_cases.craft(rng, T - pad, int(rng.choice(ks)), delta,
                                  threshold_cases.KINDS[u % len(threshold_cases.KINDS)])
        mass[u, pad:] = c.mass_f32()
        crafted.append((pad, c))
    cfg = kvc.Config(1, B, H, 1, 64, T, budget, window=8, delta=delta, seg_min=1, seg_max=4096)
    h = kvc.Handle(cfg)
    st, ln, qu, ns = gu.gpu_segment_quota(h, mass, pads, T)
    p = ref.RefParams(group=1, head_dim=64, window=8, budget=budget, delta=delta, seg_min=1,
                      seg_max=4096)
    rs, rl, rq, rn = ref.segment_quota(p, mass, np.repeat(pads, H))
    assert np.array_equal(ns, rn)
    assert np.array_equal(st, rs) and np.array_equal(ln, rl) and np.array_equal(qu, rq)
    for u, (pad, c) in enumerate(crafted):  # no merging or splitting here: raw cuts
        assert pad + c.t0 in set(st[u, :ns[u]].tolist()), (u, c.kind, c.k)


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("scores", ["oracle", "ties"])
def test_select_bit_exact(ref, oracle_runs, name, scores):
    """Same fp32 scores and segments on both sides -> identical kept indices."""
    import eviction_gb300 as kvc
    w, inp, r = oracle_runs[name]
    p = gu.ref_params(ref, w)
    T = inp.T
    score = r["score"].copy()
    if scores == "ties":  # integer scores: plateaus and exact ties everywhere
        rng = np.random.default_rng(7)
        fin = np.isfinite(score)
        score[fin] = rng.integers(0, 5, fin.sum()).astype(np.float32)
    pads_u = wl.unit_pad(inp).numpy()
    kept_ref, nk_ref = ref.select(p, score, pads_u, r["seg_start"], r["seg_len"], r["quota"],
                                  r["n_seg"])
    h = kvc.Handle(gu.config_for(w, T))
    kept, nk = gu.gpu_select(h, score, inp.pad.numpy(), T, r["seg_start"], r["seg_len"],
                             r["quota"], r["n_seg"])
    assert np.array_equal(nk, nk_ref)
    assert np.array_equal(kept, kept_ref)


@pytest.mark.parametrize("T,budget", [(6000, 700), (8192, 900), (32768, 4096)])
def test_select_over_budget_long(ref, T, budget):
    """Long cache, large recent suffix: must-keep overflows the last segments'
    quotas and the global removal path runs (asserted on the oracle's
    segments), on the wide CTAs of units past 4096 slots: at most 8 slots per
    thread (6000, 8192) and 32 (32768)."""
    import eviction_gb300 as kvc
    rng = np.random.default_rng(11 + T)
    B, H, n_recent = 2, 2, 300
    pads = np.array([0, 1234], np.int32)
    mass = _random_masses(rng, B * H, T, np.repeat(pads, H))
    p = ref.RefParams(group=1, head_dim=64, window=8, budget=budget, n_recent=n_recent)
    st, ln, qu, ns = ref.segment_quota(p, mass, np.repeat(pads, H))
    over = 0
    for u in range(B * H):  # picks past the budget, by the selection's own counting
        n = T - int(pads[u // H])
        Bk = min(budget, n)
        n_s = min(4, Bk)
        n_r = min(n_recent, Bk - n_s)
        picks = 0
        for s in range(ns[u]):
            a, L = st[u, s] - pads[u // H], ln[u, s]
            mk = max(0, min(a + L, n_s) - a) + max(0, a + L - max(a, n - n_r))
            picks += max(0, min(qu[u, s] - mk, L - mk))
        over += n_s + n_r + picks - Bk > 0
    assert over > 0
    score = np.where(mass > 0, rng.random(mass.shape) * 3, -np.inf).astype(np.float32)
    score[mass > 0] = np.round(score[mass > 0], 1)  # ties
    kept_ref, nk_ref = ref.select(p, score, np.repeat(pads, H), st, ln, qu, ns)
    h = kvc.Handle(kvc.Config(1, B, H, 1, 64, T, budget, window=8, n_recent=n_recent))
    kept, nk = gu.gpu_select(h, score, pads, T, st, ln, qu, ns)
    assert np.array_equal(nk, nk_ref) and np.array_equal(kept, kept_ref)


def test_compact_bit_exact(ref):
    import eviction_gb300 as kvc
    rng = np.random.default_rng(12)
    L, B, H, T, d, budget = 2, 2, 2, 700, 128, 300
    U = L * B * H
    k = torch.randint(-32768, 32767, (L, B, H, T, d), dtype=torch.int16).view(torch.bfloat16)
    v = torch.randint(-32768, 32767, (L, B, H, T, d), dtype=torch.int16).view(torch.bfloat16)
    c = torch.rand((L, B, H, T))
    kept = np.full((U, budget), -1, np.int32)
    nk = rng.integers(0, budget + 1, U).astype(np.int32)
    nk[0], nk[1] = budget, 0
    for u in range(U):
        kept[u, :nk[u]] = np.sort(rng.choice(T, nk[u], replace=False))
    h = kvc.Handle(kvc.Config(L, B, H, 1, d, T, budget, window=8))
    out = h.outputs(T)
    h.compact(k.cuda(), v.cuda(), c.cuda(), T, torch.from_numpy(kept).reshape(L, B, H, -1).cuda(),
              torch.from_numpy(nk).reshape(L, B, H).cuda(), out["k_out"], out["v_out"],
              out["credit_out"])
    torch.cuda.synchronize()
    p = ref.RefParams(group=1, head_dim=d, window=8, budget=budget)
    ko, vo, co = ref.compact(p, wl.bf16_bits(k.reshape(U, T, d)), wl.bf16_bits(v.reshape(U, T, d)),
                             c.reshape(U, T).numpy(), kept, nk)
    assert np.array_equal(wl.bf16_bits(out["k_out"].reshape(U, budget, d)), ko)
    assert np.array_equal(wl.bf16_bits(out["v_out"].reshape(U, budget, d)), vo)
    assert np.array_equal(out["credit_out"].reshape(U, budget).cpu().numpy(), co)


@pytest.mark.parametrize("name", list(CASES))
def test_event_end_to_end(ref, oracle_runs, name):
    """kvc_event against the oracle's whole chain, unit by unit, through the
    end-to-end checker (the GPU's own segments come from kvc_segment_quota on
    the GPU's own mass; nothing of the GPU's reaches the oracle)."""
    import eviction_gb300 as kvc
    w, inp, r = oracle_runs[name]
    T = inp.T
    p = gu.ref_params(ref, w)
    h = kvc.Handle(gu.config_for(w, T))
    g = gu.to_device(inp)
    out = gu.gpu_event(h, g, T)
    m, s, _ = gu.gpu_mass(h, g, T)
    st, ln, qu, ns = gu.gpu_segment_quota(h, m, inp.pad.numpy(), T)
    assert h.device_status() == 0
    U = w.units
    kept = out["kept_idx"].reshape(U, -1).cpu().numpy()
    nk = out["n_kept"].reshape(U).cpu().numpy()
    assert np.array_equal(nk, r["n_kept"])
    pads_u = wl.unit_pad(inp).numpy()
    verdicts = []
    for u in range(U):
        seg = dict(seg_start=st[u], seg_len=ln[u], quota=qu[u], n_seg=int(ns[u]))
        verdicts.append(gu.check_unit_e2e(p, w, int(pads_u[u]), kept[u, :nk[u]], m[u], s[u],
                                          seg, r, u))
        assert np.all(kept[u, nk[u]:] == -1)
    print(f"{name}: verdicts", {v: verdicts.count(v) for v in set(verdicts)})
    assert verdicts.count("identical") >= U - max(1, U // 10)
    # compaction is exact for the GPU's own indices
    kd = out["k_out"].reshape(U, w.budget, -1)
    ks = g["k"].reshape(U, T, -1)
    for u in range(U):
        idx = torch.from_numpy(kept[u, :nk[u]]).long().cuda()
        assert torch.equal(kd[u, :nk[u]], ks[u].index_select(0, idx))
        assert not kd[u, nk[u]:].any()


def test_repeat_runs_identical():
    """Same inputs, same bits (fixed reduction orders, no atomics in the math)."""
    import eviction_gb300 as kvc
    w, inp = _inputs("qwen_small")
    h = kvc.Handle(gu.config_for(w, inp.T))
    g = gu.to_device(inp)
    o1 = {k: v.clone() for k, v in gu.gpu_event(h, g, inp.T).items()}
    o2 = gu.gpu_event(h, g, inp.T)
    for k in o1:
        assert torch.equal(o1[k].view(torch.int8) if o1[k].dtype == torch.bfloat16 else o1[k],
                           o2[k].view(torch.int8) if o2[k].dtype == torch.bfloat16 else o2[k]), k


def test_host_validation_errors():
    import eviction_gb300 as kvc
    w, inp = _inputs("tiny")
    h = kvc.Handle(gu.config_for(w, inp.T))
    g = gu.to_device(inp)
    out = h.outputs(inp.T)
    with pytest.raises(kvc.KvcError) as e:
        h.event(g["q"], g["k"], g["v"], inp.T + 1, g["pad"], g["n_carry"], g["credit"],
                out["k_out"], out["v_out"], out["credit_out"], out["kept_idx"], out["n_kept"])
    assert e.value.code == -2
    # a view that starts 2 bytes in is not 16-byte aligned
    kk = torch.empty(g["k"].numel() + 8, dtype=torch.bfloat16, device="cuda")[1:1 + g["k"].numel()]
    with pytest.raises(kvc.KvcError) as e:
        h.event(g["q"], kk, g["v"], inp.T, g["pad"], g["n_carry"], g["credit"],
                out["k_out"], out["v_out"], out["credit_out"], out["kept_idx"], out["n_kept"])
    assert e.value.code == -3
