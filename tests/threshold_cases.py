"""Masses whose cut points sit on a rounding decision of the segmentation's
thresholds.

The cut points of AMS, Method, Key design 2 are b_k = min{t : C(t) >= k*Delta}
on the cumulative mass; this library (and the oracle) fix the comparison
exactly: the fp32 mass becomes 40-bit fixed point mu = m * 2^40, S is the
unit's fixed-point total, and the threshold is
tau_k = ceil(fl(fl(k*Delta) * S)) in IEEE double (round to nearest, ties to
even).  A random mass almost never makes that rounding matter: a prefix sum
lands on tau exactly once in about 2^30 draws.  The cases here do it on
purpose.  S is chosen so that the exact product k*Delta*S lies just above an
integer j: by its smallest step, well below half of the double's last kept bit
("below"); by exactly half of that bit with an even kept part ("tie_even"); by
one and a half of it, a tie with an odd kept part ("tie_odd"); by one step
less than the whole bit ("above"); or on j itself ("exact").  In "below" and
"tie_even" the double rounds down to j and tau is j, one less than the exact
ceiling.  The masses are then shaped so
that C(t0 - 1) = tau - 1 and C(t0) = tau: a threshold one too high moves the
cut point to t0 + 1, one too low to t0 - 1.

These are test inputs, written from the definition above with Python's own
floats (IEEE double) and integers; nothing here calls the library or the
oracle."""
from __future__ import annotations

import math
from dataclasses import dataclass
from fractions import Fraction

import numpy as np

KINDS = ("below", "tie_even", "tie_odd", "exact", "above")


def delta_parts(delta: float) -> tuple[int, int]:
    """The fp32 Delta as m * 2^e with m odd."""
    fr = Fraction(float(np.float32(delta)))
    return fr.numerator, -(fr.denominator.bit_length() - 1)


def threshold_count(delta: float) -> int:
    d = float(np.float32(delta))
    K = 0
    while (K + 1) * d < 1.0:
        K += 1
    return K


def tau_double(k: int, delta: float, S: int) -> int:
    """ceil(fl(fl(k*Delta) * S)) with Python floats (IEEE double)."""
    return math.ceil((k * float(np.float32(delta))) * float(S))


def tau_exact(k: int, delta: float, S: int) -> int:
    return math.ceil(Fraction(k) * Fraction(float(np.float32(delta))) * S)


@dataclass
class Case:
    mu: np.ndarray  # int64 fixed-point masses of the unit's valid slots
    k: int          # threshold index, 1-based
    kind: str
    S: int
    tau: int        # the double threshold
    t0: int         # its cut point: C(t0 - 1) = tau - 1, C(t0) = tau

    def mass_f32(self) -> np.ndarray:
        """mu * 2^-40 as fp32, exact (every mu is below 2^24)."""
        return np.ldexp(self.mu.astype(np.float32), -40).astype(np.float32)


def _total(rng, A: int, e: int, kind: str) -> int | None:
    """A total S in [2^32, 2^33) with A*S = j*2^-e + d, d as `kind` asks."""
    mod_full = 1 << (-e)
    S_hi = int(rng.integers(1 << 32, 1 << 33))
    r = (A * S_hi).bit_length() - 53  # bits the double drops from A*S
    if r < 2:
        return None
    a = (A & -A).bit_length() - 1  # A = 2^a * A_odd: A*S moves in steps of 2^a
    if a + 1 >= r:
        return None
    # the kept part's last bit is bit r of N: 0 for a tie at 2^(r-1), 1 at 3*2^(r-1)
    d = {"below": 1 << a, "tie_even": 1 << (r - 1), "tie_odd": 3 << (r - 1), "exact": 0,
         "above": (1 << r) - (1 << a)}[kind]
    mod = mod_full >> a
    S = S_hi - S_hi % mod + (d >> a) * pow(A >> a, -1, mod) % mod
    N = A * S
    if N.bit_length() - 53 != r or N % mod_full != d or not (1 << 32) <= S < (1 << 33):
        return None
    q = N >> r
    if (kind == "tie_even" and q % 2) or (kind == "tie_odd" and q % 2 == 0):
        return None
    return S


def usable(k: int, delta: float) -> bool:
    """Whether fl(k*Delta) has the 24 significant bits that make the double
    round products with totals in [2^32, 2^33) (otherwise they are exact)."""
    return (k * delta_parts(delta)[0]).bit_length() >= 24


def craft(rng: np.random.Generator, n: int, k: int, delta: float, kind: str) -> Case:
    """One unit of n >= 1536 valid slots whose k-th cut point sits on tau_k
    (the total S in [2^32, 2^33), so that every fixed-point mass, and the sum
    of two, stays below 2^24 and is exact in fp32)."""
    if n < 1536 or not usable(k, delta):
        raise ValueError("needs n >= 1536 and usable(k, delta)")
    m, e = delta_parts(delta)
    A = k * m
    for _ in range(10000):
        S = _total(rng, A, e, kind)
        if S is None:
            continue
        tau, ex = tau_double(k, delta, S), tau_exact(k, delta, S)
        if tau != (ex - 1 if kind in ("below", "tie_even") else ex):
            continue
        w = rng.uniform(0.8, 1.2, n)
        mu = np.floor(w / w.sum() * S).astype(np.int64)
        extra = S - int(mu.sum())
        mu[rng.choice(n, extra, replace=False)] += 1
        C = np.cumsum(mu)
        s = int(np.searchsorted(C, tau))  # slot completing the first prefix >= tau
        if s < 2 or s + 1 >= n:
            continue
        before = int(C[s - 2])  # C(s - 1): the first s - 1 slots
        mu[s - 1] = tau - 1 - before
        mu[s + 1] += int(C[s]) - tau
        mu[s] = 1
        C = np.cumsum(mu)
        if (int(C[-1]) != S or mu.min() < 1 or mu.max() >= (1 << 24) or
                int(C[s - 1]) != tau - 1 or int(C[s]) != tau):
            continue
        return Case(mu, k, kind, S, tau, s + 1)
    raise RuntimeError(f"no {kind} case for k={k}, delta={delta}")
