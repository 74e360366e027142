"""The arithmetic argument behind the quantizers' fast code path, checked on
the CPU with a numpy model of it (no GPU, no oracle).

A weight code is roundf(RN(a / D)) (round half away from zero of the IEEE
quotient).  The kernels compute it from an approximate reciprocal r of D
(within 1 ulp): k = the integer nearest the exact product a r (the low bits of
RN(a r + 1.5 * 2^23)) and d = RN(a r - k).  A code is kept unless |d| reaches
the guard 0.5 - g (g = 2^-15 for Q8_0 codes, |Q| <= 127.5; 2^-18 for Q4_K
codes, which matter only for |Q| <= 15.5); a flagged code is decided exactly:
roundf(RN(a / D)) lies beyond the half-step h = k + sign(d) / 2 exactly when
|a| / D exceeds the midpoint m between |h| and its float predecessor, a
comparison that is exact in double precision.  The model draws quotients on
and a few ulps around half-steps, perturbs the reciprocal by one ulp either
way, and requires every code to equal the IEEE one; a guard that is too
narrow must fail the same check.
"""
import numpy as np

MAGIC = 12582912.0  # 1.5 * 2^23


def _rn32(x):
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def _tie_code(a, D, k, d):
    h = k + np.copysign(0.5, d)
    ah = np.abs(h)
    ulp = ah - np.nextafter(ah.astype(np.float32), np.float32(0)).astype(np.float64)
    m = ah - 0.5 * ulp
    far = np.abs(a) > D * m  # float64: D (24 bits) x m (25 bits) is exact
    return np.copysign(np.where(far, ah + 0.5, ah - 0.5), h)


def _mismatches(a, D, guard, lo, hi, rcp_ulps):
    a = a.astype(np.float32).astype(np.float64)
    D = D.astype(np.float32).astype(np.float64)
    r = (1.0 / D).astype(np.float32)
    r = np.where(rcp_ulps > 0, np.nextafter(r, np.float32(np.inf)),
                 np.where(rcp_ulps < 0, np.nextafter(r, np.float32(0)), r)).astype(np.float64)
    p = a * r                      # the exact product (24 x 24 bits)
    k = _rn32(p + MAGIC) - MAGIC   # nearest integer of a r
    d = _rn32(p - k)
    code = np.clip(np.where(np.abs(d) >= guard, _tie_code(a, D, k, d), k), lo, hi)
    q = (a.astype(np.float32) / D.astype(np.float32)).astype(np.float64)  # IEEE quotient
    want = np.clip(np.sign(q) * np.floor(np.abs(q) + 0.5), lo, hi)
    return int(np.count_nonzero(code != want))


def _cases(rng, n, kmax, f16_scales):
    D = _rn32(np.ldexp(1 + rng.random(n), rng.integers(-20, 5, n)))
    if f16_scales:
        D = D.astype(np.float16).astype(np.float64)
        D = np.where(D == 0, 1.0, D)
    a = ((rng.integers(-kmax - 2, kmax + 2, n) + 0.5) * D).astype(np.float32)
    steps = rng.integers(-40, 41, n)  # float32 ulps away from the half-step
    for s in range(40):
        up, dn = steps > s, -steps > s
        a[up] = np.nextafter(a[up], np.float32(np.inf))
        a[dn] = np.nextafter(a[dn], np.float32(-np.inf))
    near = a.astype(np.float64)
    rand = (rng.random(n) * 2 - 1) * (kmax + 3) * D
    return D, near, rand, rng.integers(-1, 2, n)


def test_q8_0_codes_with_guard_2_pow_minus_15():
    rng = np.random.default_rng(1)
    D, near, rand, rcp = _cases(rng, 400_000, 127, True)
    g = 0.5 - 2.0 ** -15
    assert _mismatches(near, D, g, -127, 127, rcp) == 0
    assert _mismatches(rand, D, g, -127, 127, rcp) == 0
    # a guard much narrower than the reciprocal's error misrounds
    assert _mismatches(near, D, 0.5 - 2.0 ** -22, -127, 127, rcp) > 0


def test_q4_k_codes_with_guard_2_pow_minus_18():
    rng = np.random.default_rng(2)
    D, near, rand, rcp = _cases(rng, 400_000, 15, False)
    g = 0.5 - 2.0 ** -18
    assert _mismatches(near, D, g, 0, 15, rcp) == 0
    assert _mismatches(rand, D, g, 0, 15, rcp) == 0
    assert _mismatches(near, D, 0.5 - 2.0 ** -23, 0, 15, rcp) > 0


def test_exact_half_steps_round_away_from_zero():
    # a = (k + 1/2) D exactly: the IEEE quotient is the half-step itself and
    # roundf goes away from zero, which the nearest-even k alone would not
    D = np.array([2.0 ** -7, 0.375, 3.0], dtype=np.float64)
    for k in (-4, -1, 0, 1, 2, 7):
        a = (k + 0.5) * D
        assert _mismatches(a, D, 0.5 - 2.0 ** -15, -127, 127, np.zeros(3)) == 0
