"""The quantizer kernels compute x / s as RN(x * RN(1/s)) followed by one
exact-remainder fma correction (Markstein's method). This checks, on the CPU, that the
sequence gives the IEEE binary32 quotient for the operand classes the kernels use:
binary16 by binary16, any positive binary32 by 2^b - 1, and binary16 by 2048 - 2^b. Each fma is emulated
exactly: the products and sums involved fit the 64-bit significand of the x87
extended type, so rounding the extended result once to binary32 is the fma's rounding.
"""

import numpy as np
import pytest

LD = np.longdouble
pytestmark = pytest.mark.skipif(np.finfo(LD).nmant < 60, reason="needs an extended-precision long double")


def _fma32(a, b, c):
    return (a.astype(LD) * b.astype(LD) + c.astype(LD)).astype(np.float32)


def markstein(a, b, rb):
    q0 = (a.astype(LD) * rb.astype(LD)).astype(np.float32)
    r = _fma32(-b, q0, a)
    return _fma32(r, rb, q0)


def _f16_all():
    v = np.arange(0x10000, dtype=np.uint32).astype(np.uint16).view(np.float16)
    with np.errstate(invalid="ignore"):
        return v[np.isfinite(v)].astype(np.float32)


def test_binary16_by_binary16():
    rng = np.random.default_rng(5)
    xs = _f16_all()
    pos = xs[xs > 0]
    for s in np.concatenate([rng.choice(pos, 300, replace=False), pos[:8], pos[-8:]]):
        s = np.float32(s)
        sv = np.full(xs.shape, s, np.float32)
        rs = np.float32(1) / sv  # IEEE binary32 division: RN(1/s)
        got = markstein(xs, sv, rs)
        ref = xs / sv
        nz = xs != 0  # -0 / s comes out as +0; the kernels only round it and add integers
        assert np.array_equal(got[nz].view(np.uint32), ref[nz].view(np.uint32)), float(s)
        assert np.all(got[~nz] == 0)


@pytest.mark.parametrize("bits", [8, 4, 2])
def test_binary32_by_levels(bits):
    rng = np.random.default_rng(bits)
    n = np.float32((1 << bits) - 1)
    # ranges of binary16 groups: differences of two binary16 values, plus random binary32
    xs = _f16_all()
    a = np.abs(rng.choice(xs, 2_000_000) - rng.choice(xs, 2_000_000)).astype(np.float32)
    a = np.concatenate([a, rng.uniform(1e-7, 1e5, 2_000_000).astype(np.float32)])
    a = a[a > 0]
    nv = np.full(a.shape, n, np.float32)
    rn = np.float32(1) / nv
    got = markstein(a, nv, rn)
    ref = a / nv
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("bits", [8, 4, 2])
def test_binary16_by_far_divisors(bits):
    """max|x| / (2048 - 2^b), the scale floor of groups far from zero: every positive
    binary16 numerator (exhaustive)."""
    xs = _f16_all()
    a = xs[xs > 0]
    n = np.full(a.shape, np.float32(2048 - (1 << bits)), np.float32)
    rn = np.float32(1) / n
    got = markstein(a, n, rn)
    ref = a / n
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_reciprocal_constants():
    """The kernels' constants RN(1/(2^b - 1)) and RN(1/(2048 - 2^b)) as binary32 bit patterns."""
    for bits, pat in ((8, 0x3B808081), (4, 0x3D888889), (2, 0x3EAAAAAB)):
        v = np.float32(1) / np.float32((1 << bits) - 1)
        assert int(v.view(np.uint32)) == pat
    for bits, pat in ((8, 0x3A124925), (4, 0x3A010204), (2, 0x3A004020)):
        v = np.float32(1) / np.float32(2048 - (1 << bits))
        assert int(v.view(np.uint32)) == pat
