"""CPU oracle of the decode-time KV-cache compression event (test infrastructure).

This package is TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import it. The CUDA library never
calls it, and it never calls the CUDA library: the two share no code.

The arithmetic lives in ``kvc_ref.c`` (plain C, fp64, one unit at a time). This
module only compiles it with gcc and marshals numpy arrays through ctypes.

Sources: "Adaptive Mass-Segmented KV Compression for Long-Form Reasoning"
(Method, Key designs 1-4; the complete example), "RefreshKV: Updating Small KV
Cache During Long-form Generation" (A2 max pooling; A6 kernel size 7) and
"SkipKV: Selective Skipping of KV Generation and Storage for Efficient Inference
with Large Reasoning Models" (A2 Method details, 4.1: token importance score, GQA
mapping and mask; token redundancy score and the sigma mix of the final score).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvc_ref.c")
_HDR = os.path.join(_HERE, "kvc_ref.h")
_LIB = os.path.join(_HERE, "libkvc_ref.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no GPU needed). Returns the library path."""
    stale = (not os.path.exists(_LIB)) or any(
        os.path.getmtime(p) > os.path.getmtime(_LIB) for p in (_SRC, _HDR))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared",
               "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


class _Cfg(ctypes.Structure):
    _fields_ = [
        ("group", ctypes.c_int), ("head_dim", ctypes.c_int), ("window", ctypes.c_int),
        ("budget", ctypes.c_int), ("avg_pool", ctypes.c_int), ("max_pool", ctypes.c_int),
        ("delta", ctypes.c_float), ("seg_min", ctypes.c_int), ("seg_max", ctypes.c_int),
        ("q_min", ctypes.c_int), ("n_sink", ctypes.c_int), ("n_recent", ctypes.c_int),
        ("lambda_", ctypes.c_float), ("beta", ctypes.c_float), ("eps", ctypes.c_float),
        ("softmax_scale", ctypes.c_float), ("seg_fixed", ctypes.c_int),
        ("quota_by_len", ctypes.c_int), ("global_topk", ctypes.c_int),
        ("redundancy_sigma", ctypes.c_float),
    ]


@dataclass
class RefParams:
    """The method's parameters, in the types the library takes them."""
    group: int
    head_dim: int
    window: int
    budget: int
    avg_pool: int = 5
    max_pool: int = 7
    delta: float = 0.1
    seg_min: int = 16
    seg_max: int = 256
    q_min: int = 1
    n_sink: int = 4
    n_recent: int = 32
    lam: float = 0.9
    beta: float = 0.9
    eps: float = 1e-6
    softmax_scale: float = 0.0
    seg_fixed: int = 0       # ablation: fixed-length segments
    quota_by_len: int = 0    # ablation: quotas by length
    global_topk: int = 0     # ablation: one segment per unit
    redundancy_sigma: float = 0.0  # > 0: select on the redundancy-mixed score

    def c(self) -> _Cfg:
        return _Cfg(self.group, self.head_dim, self.window, self.budget, self.avg_pool,
                    self.max_pool, self.delta, self.seg_min, self.seg_max, self.q_min,
                    self.n_sink, self.n_recent, self.lam, self.beta, self.eps,
                    self.softmax_scale, self.seg_fixed, self.quota_by_len, self.global_topk,
                    self.redundancy_sigma)


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        _declare(_lib)
    return _lib


_P = ctypes.c_void_p
_I = ctypes.c_int


def _declare(L):
    L.kvc_ref_usage.argtypes = [_P, _P, _I, _I, _I, _I, _I, ctypes.c_double, _P, _P]
    L.kvc_ref_maxpool.argtypes = [_P, _I, _I, _I, _P]
    L.kvc_ref_avgpool.argtypes = [_P, _I, _I, _I, _P]
    L.kvc_ref_mass_normalize.argtypes = [_P, _I, _I, ctypes.c_double, _P]
    L.kvc_ref_credit.argtypes = [_P, _P, _I, _I, _I, ctypes.c_double, ctypes.c_double, _P, _P]
    L.kvc_ref_boundaries.argtypes = [_P, _I, _I, ctypes.c_float, _P, _P]
    L.kvc_ref_boundaries.restype = _I
    L.kvc_ref_segments.argtypes = [_P, _I, _I, ctypes.c_float, _I, _I, _P, _P, _P]
    L.kvc_ref_segments.restype = _I
    L.kvc_ref_segments_ablation.argtypes = [_P, _I, _I, _I, _I, _P, _P, _P]
    L.kvc_ref_segments_ablation.restype = _I
    L.kvc_ref_quotas.argtypes = [_P, _P, _I, _I, _I, _P]
    L.kvc_ref_select_unit.argtypes = [_P, _I, _I, _P, _P, _P, _I, _I, _I, _I, _P]
    L.kvc_ref_select_unit.restype = _I
    L.kvc_ref_s_max.argtypes = [_P, _I]
    L.kvc_ref_s_max.restype = _I
    L.kvc_ref_mass.argtypes = [_P, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P]
    L.kvc_ref_segment_quota.argtypes = [_P, _I, _I, _P, _P, _P, _P, _P, _P]
    L.kvc_ref_select.argtypes = [_P, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P]
    L.kvc_ref_compact.argtypes = [_P, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P]
    L.kvc_ref_refresh_decision.argtypes = [_I, _I, _I, _P, _P, ctypes.c_double, _P, _P]
    L.kvc_ref_compact_paged.argtypes = [_I] * 8 + [_P] * 10
    L.kvc_ref_compact_paged.restype = _I
    L.kvc_ref_mean_cosine_rows.argtypes = [_P, _I, _I, _I, _P, _I, _P]
    L.kvc_ref_redundancy_score.argtypes = [_P, _P, _I, _I, _I, ctypes.c_double, _P, _P, _P]


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _over_units(fn, p, arrays, threads):
    """Run ``fn(p, *chunk)`` on contiguous chunks of units in a thread pool and
    join the results along the unit axis.  Every array in ``arrays`` is unit-major
    ([U, ...]).  Units are independent, and ctypes releases the GIL for the
    duration of each C call, so the chunks run on separate cores; the arithmetic
    is the same single-unit code either way."""
    U = len(arrays[0])
    threads = max(1, min(int(threads), U))
    bounds = np.linspace(0, U, threads + 1).astype(int)

    def run(i):
        return fn(p, *[np.asarray(a)[bounds[i]:bounds[i + 1]] for a in arrays])

    with ThreadPoolExecutor(threads) as ex:
        parts = list(ex.map(run, range(threads)))
    if isinstance(parts[0], dict):
        return {k: np.concatenate([q[k] for q in parts], axis=0) for k in parts[0]}
    return tuple(np.concatenate([q[j] for q in parts], axis=0) for j in range(len(parts[0])))


# ---- per-unit fp64 steps (used by the pins) ---------------------------------

def usage(q: np.ndarray, k: np.ndarray, pad: int = 0, scale: float | None = None):
    """Step 1 for one unit. q: [G, W, d] float, k: [T, d] float -> (a[T], fill)."""
    q = _c(q, np.float64)
    k = _c(k, np.float64)
    G, W, d = q.shape
    T = k.shape[0]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    a = np.zeros(T, np.float64)
    fill = np.zeros(1, np.float64)
    lib().kvc_ref_usage(_ptr(q), _ptr(k), G, W, d, T, pad, float(scale), _ptr(a), _ptr(fill))
    return a, float(fill[0])


def maxpool(a: np.ndarray, pad: int = 0, kernel: int = 7) -> np.ndarray:
    a = _c(a, np.float64)
    s = np.zeros_like(a)
    lib().kvc_ref_maxpool(_ptr(a), a.shape[0], pad, kernel, _ptr(s))
    return s


def avgpool(a: np.ndarray, pad: int = 0, kernel: int = 5) -> np.ndarray:
    a = _c(a, np.float64)
    u = np.zeros_like(a)
    lib().kvc_ref_avgpool(_ptr(a), a.shape[0], pad, kernel, _ptr(u))
    return u


def mass_normalize(u: np.ndarray, pad: int = 0, eps: float = 1e-6) -> np.ndarray:
    u = _c(u, np.float64)
    m = np.zeros_like(u)
    lib().kvc_ref_mass_normalize(_ptr(u), u.shape[0], pad, float(eps), _ptr(m))
    return m


def credit(m, c_in, pad=0, n_carry=None, lam=0.9, beta=0.9):
    m = _c(m, np.float64)
    c_in = _c(c_in, np.float64)
    T = m.shape[0]
    if n_carry is None:
        n_carry = T - pad
    c = np.zeros_like(m)
    mu = np.zeros_like(m)
    lib().kvc_ref_credit(_ptr(m), _ptr(c_in), T, pad, n_carry, float(lam), float(beta),
                         _ptr(c), _ptr(mu))
    return c, mu


def boundaries(m_used: np.ndarray, pad: int = 0, delta: float = 0.1):
    """Raw cut points b_k (k = 1..K, counted in valid slots) and the fixed-point total."""
    m = _c(m_used, np.float32)
    b = np.zeros(int(1.0 / np.float32(delta)) + 2, np.int64)
    tot = np.zeros(1, np.uint64)
    K = lib().kvc_ref_boundaries(_ptr(m), m.shape[0], pad, float(delta), _ptr(b), _ptr(tot))
    return b[:K].copy(), int(tot[0])


def segments(m_used, pad=0, delta=0.1, seg_min=16, seg_max=256):
    """(starts as valid offsets, lengths, fixed-point masses)."""
    m = _c(m_used, np.float32)
    T = m.shape[0]
    cap = max(1, T)
    st = np.zeros(cap, np.int32)
    ln = np.zeros(cap, np.int32)
    M = np.zeros(cap, np.uint64)
    ns = lib().kvc_ref_segments(_ptr(m), T, pad, float(delta), seg_min, seg_max,
                                _ptr(st), _ptr(ln), _ptr(M))
    return st[:ns].copy(), ln[:ns].copy(), M[:ns].copy()


def segments_ablation(m_used, pad=0, seg_fixed=0, global_=0):
    """Fixed-length (seg_fixed > 0) or single-segment (global_) segmentation:
    (starts as valid offsets, lengths, fixed-point masses)."""
    m = _c(m_used, np.float32)
    T = m.shape[0]
    cap = max(1, T)
    st = np.zeros(cap, np.int32)
    ln = np.zeros(cap, np.int32)
    M = np.zeros(cap, np.uint64)
    ns = lib().kvc_ref_segments_ablation(_ptr(m), T, pad, int(seg_fixed), int(global_),
                                         _ptr(st), _ptr(ln), _ptr(M))
    return st[:ns].copy(), ln[:ns].copy(), M[:ns].copy()


def quotas(seg_len, seg_mass, budget_eff, q_min=1) -> np.ndarray:
    ln = _c(seg_len, np.int32)
    M = _c(seg_mass, np.uint64)
    q = np.zeros(ln.shape[0], np.int32)
    lib().kvc_ref_quotas(_ptr(ln), _ptr(M), ln.shape[0], int(budget_eff), int(q_min), _ptr(q))
    return q


def select_unit(score, pad, seg_start, seg_len, quota, budget, n_sink=4, n_recent=32):
    """seg_start as valid offsets; returns the kept absolute slots (ascending)."""
    s = _c(score, np.float32)
    st = _c(seg_start, np.int32)
    ln = _c(seg_len, np.int32)
    qu = _c(quota, np.int32)
    T = s.shape[0]
    kept = np.zeros(max(1, T), np.int32)
    nk = lib().kvc_ref_select_unit(_ptr(s), T, pad, _ptr(st), _ptr(ln), _ptr(qu), st.shape[0],
                                   int(budget), int(n_sink), int(n_recent), _ptr(kept))
    return kept[:nk].copy()


# ---- batched mirrors on compact unit-major arrays ----------------------------

def s_max(p: RefParams, T: int) -> int:
    cfg = p.c()
    return lib().kvc_ref_s_max(ctypes.byref(cfg), T)


def mass(p: RefParams, q_bits, k_bits, credit_in, pad, n_carry, threads: int = 1):
    """q_bits [U,G,W,d] uint16, k_bits [U,T,d] uint16, credit_in [U,T] f32, pad/n_carry [U].
    threads > 1 splits the units over that many host threads."""
    if threads > 1:
        return _over_units(mass, p, (q_bits, k_bits, credit_in, pad, n_carry), threads)
    q_bits = _c(q_bits, np.uint16)
    k_bits = _c(k_bits, np.uint16)
    U, T = k_bits.shape[0], k_bits.shape[1]
    credit_in = _c(credit_in, np.float32).reshape(U, T)
    pad = _c(pad, np.int32)
    n_carry = _c(n_carry, np.int32)
    m = np.zeros((U, T), np.float32)
    s = np.zeros((U, T), np.float32)
    c = np.zeros((U, T), np.float32)
    cfg = p.c()
    lib().kvc_ref_mass(ctypes.byref(cfg), U, T, _ptr(q_bits), _ptr(k_bits), _ptr(credit_in),
                       _ptr(pad), _ptr(n_carry), _ptr(m), _ptr(s), _ptr(c))
    return m, s, c


def segment_quota(p: RefParams, mass_f32, pad, threads: int = 1):
    if threads > 1:
        return _over_units(segment_quota, p, (mass_f32, pad), threads)
    mass_f32 = _c(mass_f32, np.float32)
    U, T = mass_f32.shape
    pad = _c(pad, np.int32)
    S = s_max(p, T)
    st = np.zeros((U, S), np.int32)
    ln = np.zeros((U, S), np.int32)
    qu = np.zeros((U, S), np.int32)
    ns = np.zeros(U, np.int32)
    cfg = p.c()
    lib().kvc_ref_segment_quota(ctypes.byref(cfg), U, T, _ptr(mass_f32), _ptr(pad), _ptr(st),
                                _ptr(ln), _ptr(qu), _ptr(ns))
    return st, ln, qu, ns


def select(p: RefParams, score_f32, pad, seg_start, seg_len, quota, n_seg, threads: int = 1):
    if threads > 1:
        return _over_units(select, p, (score_f32, pad, seg_start, seg_len, quota, n_seg), threads)
    score_f32 = _c(score_f32, np.float32)
    U, T = score_f32.shape
    kept = np.zeros((U, p.budget), np.int32)
    nk = np.zeros(U, np.int32)
    cfg = p.c()
    lib().kvc_ref_select(ctypes.byref(cfg), U, T, _ptr(score_f32), _ptr(_c(pad, np.int32)),
                         _ptr(_c(seg_start, np.int32)), _ptr(_c(seg_len, np.int32)),
                         _ptr(_c(quota, np.int32)), _ptr(_c(n_seg, np.int32)), _ptr(kept), _ptr(nk))
    return kept, nk


def compact(p: RefParams, k_bits, v_bits, credit_post, kept_idx, n_kept):
    k_bits = _c(k_bits, np.uint16)
    v_bits = _c(v_bits, np.uint16)
    U, T, d = k_bits.shape
    ko = np.zeros((U, p.budget, d), np.uint16)
    vo = np.zeros((U, p.budget, d), np.uint16)
    co = np.zeros((U, p.budget), np.float32)
    cfg = p.c()
    lib().kvc_ref_compact(ctypes.byref(cfg), U, T, _ptr(k_bits), _ptr(v_bits),
                          _ptr(_c(credit_post, np.float32)), _ptr(_c(kept_idx, np.int32)),
                          _ptr(_c(n_kept, np.int32)), _ptr(ko), _ptr(vo), _ptr(co))
    return ko, vo, co


def mean_cosine_rows(k_bits, pad, rows):
    """SkipKV token redundancy of single rows: k_bits [T, d] uint16 (one unit),
    rows: absolute slots.  Returns r [len(rows)] fp64 (mean cosine to the other
    valid keys)."""
    k_bits = _c(k_bits, np.uint16)
    T, d = k_bits.shape
    rows = _c(rows, np.int32)
    out = np.zeros(len(rows), np.float64)
    lib().kvc_ref_mean_cosine_rows(_ptr(k_bits), T, d, int(pad), _ptr(rows), len(rows), _ptr(out))
    return out


def redundancy_score(k_bits, score, pad, sigma):
    """SkipKV redundancy-mixed score for U units: k_bits [U, T, d] uint16, score
    [U, T] f32, pad [U].  Returns (f, R, r), each [U, T] fp64: the final score,
    the softmax-normalised redundancy and the mean cosine."""
    k_bits = _c(k_bits, np.uint16)
    U, T, d = k_bits.shape
    score = _c(score, np.float32).reshape(U, T)
    pad = np.asarray(pad, np.int64).reshape(U)
    f = np.zeros((U, T))
    R = np.zeros((U, T))
    r = np.zeros((U, T))
    for u in range(U):
        lib().kvc_ref_redundancy_score(_ptr(k_bits[u]), _ptr(score[u]), T, d, int(pad[u]),
                                       float(sigma), _ptr(r[u]), _ptr(R[u]), _ptr(f[u]))
    return f, R, r


def event(p: RefParams, q_bits, k_bits, v_bits, credit_in, pad, n_carry, threads: int = 1):
    """The whole event, steps 1-6, for U units. Returns a dict of numpy arrays.
    With p.redundancy_sigma > 0 step 5 selects on the SkipKV redundancy-mixed
    score (rounded to fp32, the score's own precision); "sel_score" holds it.
    threads > 1 splits the units over that many host threads."""
    if threads > 1:
        return _over_units(event, p, (q_bits, k_bits, v_bits, credit_in, pad, n_carry), threads)
    m, s, c = mass(p, q_bits, k_bits, credit_in, pad, n_carry)
    st, ln, qu, ns = segment_quota(p, m, pad)
    sel = s
    extra = {}
    if p.redundancy_sigma > 0:
        f, R, r = redundancy_score(k_bits, s, pad, p.redundancy_sigma)
        sel = f.astype(np.float32)
        extra = dict(sel_score=sel, redundancy=R, mean_cos=r)
    kept, nk = select(p, sel, pad, st, ln, qu, ns)
    ko, vo, co = compact(p, k_bits, v_bits, c, kept, nk)
    return dict(mass=m, score=s, credit_post=c, seg_start=st, seg_len=ln, quota=qu, n_seg=ns,
                kept_idx=kept, n_kept=nk, k_out=ko, v_out=vo, credit_out=co, **extra)


def refresh_decision(q_bits, q_ref, threshold):
    """RefreshKV query-similarity trigger for LB (layer, sequence) rows.
    q_bits [LB, Hq, d] uint16, q_ref [LB, d] (copied; the updated copy is
    returned).  Returns (flag [LB] int32, sim [LB] fp64, q_ref_new [LB, d])."""
    q_bits = _c(q_bits, np.uint16)
    LB, Hq, d = q_bits.shape
    ref = np.array(q_ref, dtype=np.float64, copy=True, order="C").reshape(LB, d)
    flag = np.zeros(LB, np.int32)
    sim = np.zeros(LB, np.float64)
    lib().kvc_ref_refresh_decision(LB, Hq, d, _ptr(q_bits), _ptr(ref), float(threshold),
                                   _ptr(flag), _ptr(sim))
    return flag, sim, ref


def compact_paged(k_pool, v_pool, seq_len, pad, kept_idx, n_kept, table_old, free_list,
                  free_top, block_size):
    """Paged compaction on copies of the pools and the free list.  k_pool, v_pool
    [L, n_blocks, H, bs, d] uint16; kept_idx [L, B, H, budget]; n_kept [L, B, H];
    table_old [B, max_blocks].  Returns (rc, k_pool, v_pool, table_new,
    free_list, free_top)."""
    kp = np.array(k_pool, dtype=np.uint16, copy=True, order="C")
    vp = np.array(v_pool, dtype=np.uint16, copy=True, order="C")
    L, n_blocks, H, bs, d = kp.shape
    assert bs == block_size
    kept = _c(kept_idx, np.int32)
    budget = kept.shape[-1]
    B = kept.shape[1]
    told = _c(table_old, np.int32)
    max_blocks = told.shape[1]
    tnew = np.full((B, max_blocks), -1, np.int32)
    fl = np.array(free_list, dtype=np.int32, copy=True, order="C")
    top = np.array([free_top], np.int32)
    rc = lib().kvc_ref_compact_paged(L, B, H, d, bs, n_blocks, max_blocks, budget, _ptr(kp),
                                     _ptr(vp), _ptr(_c(seq_len, np.int32)),
                                     _ptr(_c(pad, np.int32)), _ptr(kept),
                                     _ptr(_c(n_kept, np.int32)), _ptr(told), _ptr(tnew),
                                     _ptr(fl), _ptr(top))
    return rc, kp, vp, tnew, fl, int(top[0])
