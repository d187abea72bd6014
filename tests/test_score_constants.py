"""The constants of the device's score chain (page moe_v41.rs fn softplus:
e^t and ln(1 + e) rounded to f32, decided against e^t and e^m - 1 at
midpoints m): each 1/n! pair is the exact rational rounded to f32 twice; the
float-float parts of ln 2 / 32 and the double-double parts of ln 2 (Cody and
Waite's reduction) add up to the constant, the first double part short enough
for k times it to be exact. Read from the kernel source, checked against
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
    return sum(Fraction(1, k * 2 ** k) for k in range(1, 400))  # ln 2 = sum 1 / (k 2^k)


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
    """Tang's reduction x = k ln2 / 32 + r (|k| <= 5100 for |x| <= 110): the
    three f32 parts add up to ln 2 / 32 within 2^-70, so k times the error
    stays below 2^-57 (k P1 and k P2 are formed as exact float-float
    products)."""
    src = open(SRC).read()
    m = re.search(r"P1 = ([0-9a-fx.p-]+)f, P2 = ([0-9a-fx.p-]+)f, P3 = ([0-9a-fx.p-]+)f", src)
    p1, p2, p3 = (Fraction(float.fromhex(g)) for g in m.groups())
    assert abs(p1 + p2 + p3 - _ln2() / 32) < Fraction(1, 2 ** 70)
    for p in (p1, p2, p3):
        assert Fraction(_f32(float(p))) == p


def test_ln2_double_double_parts():
    """The level-3 reduction x = k ln2 + r (|k| <= 160): L1 + L2 + L3 = ln 2
    within 2^-130, and L1 has at most 32 significant bits, so k L1 is an
    exact double for |k| < 2^21."""
    src = open(SRC).read()
    m = re.search(r"L1 = ([0-9a-fx.p+-]+), L2 = ([0-9a-fx.p+-]+), L3 = ([0-9a-fx.p+-]+);", src)
    l1, l2, l3 = (Fraction(float.fromhex(g)) for g in m.groups())
    assert abs(l1 + l2 + l3 - _ln2()) < Fraction(1, 2 ** 130)
    num = l1.numerator
    while num % 2 == 0:
        num //= 2
    assert num.bit_length() <= 32
    assert l1.denominator & (l1.denominator - 1) == 0


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
