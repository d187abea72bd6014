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


@pytest.mark.parametrize("temp", [1.0, 0.7])
def test_scores_match_60_digit_arithmetic(temp):
    """score = f32 rounding of sqrt(softplus(f32(l / temp))), softplus(x) = x for x > 20."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 60
    vals = [-200.0, -104.0, -87.5, -30.0, -5.25, -1.0, -1e-3, 0.0, 1e-3, 0.5, 1.0, 2.75, 10.0,
            19.999, 20.0, 20.001, 25.0, 88.0, 1e6]
    rng = np.random.default_rng(3)
    vals += list(rng.standard_normal(200) * 2.0)
    for v in vals:
        l = np.float32(v)
        t = np.float32(l / np.float32(temp))
        tm = mp.mpf(float(t))
        sp = tm if t > 20 else mp.log1p(mp.exp(tm))
        exact = mp.sqrt(sp)
        s, near = oracle.score(float(l), temp)
        if near:
            continue
        # s must be a nearest f32 to the exact value
        lo = np.nextafter(s, np.float32(-np.inf))
        hi = np.nextafter(s, np.float32(np.inf))
        d = abs(mp.mpf(float(s)) - exact)
        assert d <= abs(mp.mpf(float(lo)) - exact) and d <= abs(mp.mpf(float(hi)) - exact), (v, s)
