"""The constants of the device's float-float score (page moe_v41.rs fn
softplus: the score is evaluated as e^t against expm1(m^2)): each 1/n! pair
is the exact rational rounded to f32 twice, and the three parts of ln 2
(Cody and Waite's reduction) add up to ln 2 with the first part short
enough for k * part exact. Read from the kernel source, checked against
exact arithmetic."""
import math
import os
import re
import struct
from fractions import Fraction

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "moe_decode_quantized_gb300", "csrc", "moe_route.cuh")


def _f32(x):
    return struct.unpack("f", struct.pack("f", float(x)))[0]


def _ln2():
    return sum(Fraction(1, k * 2 ** k) for k in range(1, 300))  # ln 2 = sum 1 / (k 2^k)


def test_inverse_factorials_are_exact_float_float_pairs():
    src = open(SRC).read()
    body = src[src.index("c_inv_fact[15] = {"):]
    body = body[:body.index("};")]
    pairs = [(float.fromhex(a), float.fromhex(b))
             for a, b in re.findall(r"\{([-0-9a-fx.p]+)f, ([-0-9a-fx.p]+)f\}", body)]
    assert len(pairs) == 15
    for n in range(15):
        c = Fraction(1, math.factorial(n))
        hi = _f32(c)
        assert pairs[n] == (hi, _f32(c - Fraction(hi))), n


def test_ln2_over_32_parts():
    """Tang's reduction x = k ln2 / 32 + r: the three parts add up to ln 2 / 32
    and the first is short enough that k times it is exact for |k| < 4096."""
    src = open(SRC).read()
    m = re.search(r"P1 = ([0-9a-fx.p-]+)f, P2 = ([0-9a-fx.p-]+)f, P3 = ([0-9a-fx.p-]+)f", src)
    p1, p2, p3 = (Fraction(float.fromhex(g)) for g in m.groups())
    assert abs(p1 + p2 + p3 - _ln2() / 32) < Fraction(1, 2 ** 70)  # x 4096 still below 2^-58
    for k in (-4095, -3001, -17, 1, 2047, 4095):
        assert Fraction(_f32(k * float(p1))) == k * p1
    assert p1.numerator.bit_length() <= 12 and p1.denominator & (p1.denominator - 1) == 0


def test_exp2_table():
    """2^(j/32), j = 0..31, as float-float pairs within 2^-48 relative."""
    from decimal import Decimal, getcontext
    getcontext().prec = 60
    src = open(SRC).read()
    body = src[src.index("c_exp2_32[32] = {"):]
    body = body[:body.index("};")]
    pairs = re.findall(r"\{([-0-9a-fx.p+]+)f, ([-0-9a-fx.p+]+)f\}", body)
    assert len(pairs) == 32
    for j, (hi, lo) in enumerate(pairs):
        exact = Decimal(2) ** (Decimal(j) / Decimal(32))
        got = Decimal(float.fromhex(hi)) + Decimal(float.fromhex(lo))
        assert abs(got - exact) / exact < Decimal(2) ** -48, j
        assert float.fromhex(hi) == _f32(float(exact)), j
