"""Pins of the oracle's number conversions (no GPU).

bf16: the hand-derived fixture tests/golden/bf16_rne.txt (rule of page
spark_model/layers/moe_v41.rs, fn bf16_bytes) and torch's round-to-nearest-
even bfloat16 conversion. f16: numpy's IEEE binary16 conversion.
"""
import os

import numpy as np
import pytest
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _f32_from_bits(bits):
    return np.array(bits, dtype=np.uint32).view(np.float32)


def test_bf16_golden_fixture():
    rows = []
    with open(os.path.join(GOLD, "bf16_rne.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                a, b = line.split()[:2]
                rows.append((int(a, 16), int(b, 16)))
    x = _f32_from_bits([r[0] for r in rows])
    got = oracle.bf16_from_f32(x)
    assert [int(v) for v in got] == [r[1] for r in rows]


def test_bf16_matches_torch_rne():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2 ** 32, size=4000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    x = np.concatenate([x, rng.standard_normal(2000).astype(np.float32)])
    want = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_from_f32(x)
    np.testing.assert_array_equal(got, want)


def test_bf16_to_f64_is_exact_widening():
    h = np.arange(0, 65536, 97, dtype=np.uint16)
    want = (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    got = oracle.bf16_to_f64(h)
    fin = np.isfinite(want)
    np.testing.assert_array_equal(got[fin], want[fin])


def test_f16_from_f32_matches_numpy():
    rng = np.random.default_rng(2)
    parts = [
        rng.standard_normal(3000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-5).astype(np.float32),     # f16 subnormal range
        (rng.standard_normal(1000) * 3e-8).astype(np.float32),     # underflow edge
        (rng.standard_normal(1000) * 4e4).astype(np.float32),      # overflow edge
        np.array([0.0, -0.0, 65504.0, 65519.0, 65520.0, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26,
                  np.inf, -np.inf], dtype=np.float32),
    ]
    x = np.concatenate(parts)
    want = x.astype(np.float16).view(np.uint16)
    got = oracle.f16_from_f32(x)
    np.testing.assert_array_equal(got, want)


def test_f16_to_f64_matches_numpy():
    h = np.arange(0, 65536, dtype=np.uint16)
    want = h.view(np.float16).astype(np.float64)
    fin = np.isfinite(want)
    got = oracle.f16_to_f64(h[fin])
    np.testing.assert_array_equal(got, want[fin])


def _rn32(mp, x):
    """The f32 nearest to the mpmath value x (ties cannot occur for these
    transcendental values), and whether x lies within 2^-56 of a midpoint."""
    c = np.float32(float(x))
    best = None
    for cand in (np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))):
        d = abs(mp.mpf(float(cand)) - x)
        if best is None or d < best[0]:
            best = (d, cand)
    r = best[1]
    nb = np.nextafter(r, np.float32(np.inf) if x > mp.mpf(float(r)) else np.float32(-np.inf))
    mid = (mp.mpf(float(r)) + mp.mpf(float(nb))) / 2
    near = x != 0 and abs(x - mid) <= abs(x) * mp.mpf(2) ** -56
    return r, near


def _chain(mp, t):
    """Page moe_v41.rs fn softplus / fn route_from_logits in f32, each operation
    correctly rounded: e = f32(e^t), sp = f32(ln(1 + e)) (sp = t for t > 20),
    s = f32(sqrt(sp)); also the exact value rounded once, for contrast."""
    tm = mp.mpf(float(t))
    if t > 20:
        sp, n1 = t, False
        once = mp.sqrt(tm)
    else:
        e, n0 = _rn32(mp, mp.exp(tm))
        sp, n1 = _rn32(mp, mp.log1p(mp.mpf(float(e))))
        n1 = n1 or n0
        once = mp.sqrt(mp.log1p(mp.exp(tm)))
    s, n2 = _rn32(mp, mp.sqrt(mp.mpf(float(sp))))
    return s, n1 or n2, _rn32(mp, once)[0]


@pytest.mark.parametrize("temp", [1.0, 0.7])
def test_scores_match_60_digit_arithmetic(temp):
    """score = f32(sqrt(f32(ln(1 + f32(e^t))))), t = f32(l / temp), and
    f32(sqrt(t)) for t > 20: every step checked against 60-digit arithmetic.
    The inputs include values where this chain and the once-rounded exact
    sqrt(softplus(t)) differ, so the test tells the two readings apart."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 60
    vals = [-200.0, -104.0, -103.97, -103.9, -90.0, -87.5, -30.0, -17.3, -5.25, -1.0, -1e-3, 0.0,
            1e-3, 0.5, 1.0, 2.75, 10.0, 19.999, 20.0, 20.001, 25.0, 88.0, 1e6]
    rng = np.random.default_rng(3)
    vals += list(rng.standard_normal(600) * 2.0)
    vals += list(rng.uniform(-104.0, -16.0, 200))
    differ = 0
    for v in vals:
        l = np.float32(v)
        t = np.float32(l / np.float32(temp))
        want, near, once = _chain(mp, t)
        s, onear = oracle.score(float(l), temp)
        if near:
            assert onear, v  # the oracle flags what it cannot certify
            continue
        assert np.float32(s).view(np.uint32) == want.view(np.uint32), (v, s, want)
        differ += int(want != once)
    assert differ > 0  # some inputs separate the chain from the once-rounded value


def test_score_chain_hand_worked_values():
    """Closed forms: t = 0 gives e = 1, sp = f32(ln 2), s = f32(sqrt(f32(ln 2)));
    t > 20 gives sqrt(t) (exact for t = 25, 100); t = -inf gives 0; a t
    below -150 ln 2 makes f32(e^t) = 0 and the score 0."""
    ln2_f32 = np.float32(0.6931471805599453)  # ln 2 = 0.69314718055994530942...
    assert oracle.score(0.0, 1.0)[0] == np.sqrt(ln2_f32)  # numpy's f32 sqrt is IEEE
    assert oracle.score(25.0, 1.0)[0] == 5.0
    assert oracle.score(200.0, 2.0)[0] == 10.0
    assert oracle.score(float("-inf"), 1.0)[0] == 0.0
    assert oracle.score(-104.0, 1.0)[0] == 0.0
    assert oracle.score(-103.9, 1.0)[0] > 0.0  # e^-103.9 > 2^-150: one subnormal unit
    assert oracle.score(-103.9, 1.0)[0] == np.float32(np.sqrt(np.float32(2.0 ** -149)))

