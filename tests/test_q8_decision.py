"""The q8_1 quant decision the kernels use, against its definition.

The definition (the activation format the K-quant GEMVs consume,
moe_v41.rs module doc): q = round-half-away(fl(v / d)) with d = fl(amax /
127), an IEEE f32 division. The kernels form z = fl(v * fl(1 / d)) instead
and fall back to the division only when z is within 2^-15 of a
half-integer: z is within 381 * 2^-24 < 2^-15 of fl(v / d) for |v| <= amax,
so elsewhere both round to the same integer. This restates that rule in
numpy f32 (IEEE, correctly rounded like the device intrinsics) and checks it
against the definition on random blocks and on values a few ulps from every
half-integer quotient."""
import numpy as np

F = np.float32


def _round_half_away(x):
    return np.where(x >= 0, np.floor(x + F(0.5)), -np.floor(-x + F(0.5)))


def _definition(v, d):
    return _round_half_away((v / d).astype(F))


def _rule(v, d):
    with np.errstate(over="ignore", invalid="ignore"):  # 1 / d overflows for subnormal d
        r = (F(1) / d).astype(F)
        z = (v * r).astype(F)
        a = np.abs(z)
        f = (a - np.floor(a)).astype(F)
        near = ~(np.abs((f - F(0.5)).astype(F)) >= F(2.0 ** -15))
        return np.where(near, _definition(v, d), _round_half_away(z)), near


def test_rule_matches_division_on_random_blocks():
    rng = np.random.default_rng(7)
    scale = (F(10.0) ** rng.uniform(-30, 30, size=(40000, 1)).astype(F)).astype(F)
    v = (rng.standard_normal((40000, 32)).astype(F) * scale).astype(F)
    amax = np.abs(v).max(axis=1, keepdims=True)
    d = (amax / F(127)).astype(F)
    got, near = _rule(v, d)
    assert np.array_equal(got, _definition(v, d))
    assert near.mean() < 1e-3  # the division is the rare case


def test_rule_matches_division_next_to_half_integers():
    rng = np.random.default_rng(8)
    n = 100000
    d = (F(10.0) ** rng.uniform(-30, 30, size=n).astype(F)).astype(F)
    k = rng.integers(-127, 127, size=n).astype(F)
    v = ((k + F(0.5)) * d).astype(F)
    steps = rng.integers(-4, 5, size=n)
    for s in range(1, 5):
        move = np.abs(steps) >= s
        v = np.where(move, np.nextafter(v, np.where(steps > 0, np.inf, -np.inf).astype(F)), v).astype(F)
    keep = np.abs(v) <= F(127) * d  # |v| <= amax = 127 d (up to rounding)
    got, near = _rule(v[keep], d[keep])
    assert np.array_equal(got, _definition(v[keep], d[keep]))
    assert near.any()  # the fallback is exercised


def test_rule_falls_back_when_the_reciprocal_overflows():
    d = np.array([F(1e-39), F(2.0 ** -149)], dtype=F)  # subnormal: 1 / d overflows
    v = (d * F(100.5)).astype(F)
    got, near = _rule(v, d)
    assert near.all()
    assert np.array_equal(got, _definition(v, d))
