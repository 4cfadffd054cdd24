"""The published-K rounding test of the RoPE/publish kernel, restated in numpy.

The kernel decides most rotated K pairs in fp32 and sends the rest to the exact
fp64 expressions of the published-K contract (RNE_bf16(fl64(fl64(a c) -+ fl64(b s))),
Ziv's rounding test).  This test re-evaluates its fast path step by step —
r0 = fma(-b, s32, a c32), r1 = fma(b, c32, a s32); m = |a||u32| + |b||w32|
rounded up; e = 2^-22 m + 2^-140 rounded up; interval ends r -+ e rounded
outward; accept when both ends give the same bf16 pair and m < 2^126 — and
checks that every accepted pair equals the oracle's contract value, and that
the fallback stays rare.  Fused operations are evaluated in extended precision
and rounded once; directed roundings step to the neighbouring float.
"""
import numpy as np

from oracle import ff_oracle as fo

LD = np.longdouble


def _round32(x, mode):
    x = np.asarray(x, LD)
    f = x.astype(np.float32)
    back = f.astype(LD)
    if mode == "down":
        f = np.where(back > x, np.nextafter(f, np.float32(-np.inf)), f)
    elif mode == "up":
        f = np.where(back < x, np.nextafter(f, np.float32(np.inf)), f)
    return f


def _fma(a, b, c, mode="nearest"):
    return _round32(LD(a) * LD(b) + LD(c), mode)


def _mul(a, b, mode="nearest"):
    return _round32(LD(a) * LD(b), mode)


def _bf16_of_f32(x):
    return fo.f64_to_bf16_bits(np.asarray(x, np.float64))


def fast_path(a, b, c64, s64):
    """Returns (accepted mask, bf16 bits of the two components) of the fp32 path."""
    with np.errstate(over="ignore", invalid="ignore"):  # special inputs overflow or are NaN by design
        return _fast_path(a, b, c64, s64)


def _fast_path(a, b, c64, s64):
    c32, s32 = c64.astype(np.float32), s64.astype(np.float32)
    r0 = _fma(-b, s32, _mul(a, c32))
    r1 = _fma(b, c32, _mul(a, s32))
    aa, ab, ac, as_ = np.abs(a), np.abs(b), np.abs(c32), np.abs(s32)
    m0 = _fma(aa, ac, _mul(ab, as_, "up"), "up")
    m1 = _fma(aa, as_, _mul(ab, ac, "up"), "up")
    e0 = _fma(m0, np.float32(2.0 ** -22), np.float32(2.0 ** -140), "up")
    e1 = _fma(m1, np.float32(2.0 ** -22), np.float32(2.0 ** -140), "up")
    lo0, hi0 = _bf16_of_f32(_fma(e0, -1, r0, "down")), _bf16_of_f32(_fma(e0, 1, r0, "up"))
    lo1, hi1 = _bf16_of_f32(_fma(e1, -1, r1, "down")), _bf16_of_f32(_fma(e1, 1, r1, "up"))
    ok = (lo0 == hi0) & (lo1 == hi1) & (m0 < 2.0 ** 126) & (m1 < 2.0 ** 126)
    return ok, lo0, lo1


def contract(a, b, c64, s64):
    a64, b64 = a.astype(np.float64), b.astype(np.float64)
    return fo.f64_to_bf16_bits(a64 * c64 - b64 * s64), fo.f64_to_bf16_bits(a64 * s64 + b64 * c64)


def test_accepted_pairs_equal_the_contract():
    rng = np.random.default_rng(5)
    n = 400_000
    scale = np.where(rng.random(n) < 0.1, 50.0, 1.0)
    a = fo.bf16_bits_to_f64(fo.f64_to_bf16_bits(rng.standard_normal(n) * scale)).astype(np.float32)
    b = fo.bf16_bits_to_f64(fo.f64_to_bf16_bits(rng.standard_normal(n) * scale[::-1])).astype(np.float32)
    ang = rng.random(n) * 260.0  # positions up to the longest axis times the largest frequency
    c64, s64 = np.cos(ang), np.sin(ang)
    ok, x, y = fast_path(a, b, c64, s64)
    ex, ey = contract(a, b, c64, s64)
    assert np.all(x[ok] == ex[ok]) and np.all(y[ok] == ey[ok])
    rate = 1.0 - ok.mean()
    assert 0.0 < rate < 0.003, rate


def test_special_inputs_take_the_exact_path():
    a = np.array([np.nan, np.inf, 0.0, 3.0e38, -3.0e38, 1.0], np.float32)
    b = np.array([1.0, 1.0, np.nan, 3.0e38, 1.0, -np.inf], np.float32)
    c64 = np.full(a.shape, np.cos(0.3))
    s64 = np.full(a.shape, np.sin(0.3))
    ok, _, _ = fast_path(a, b, c64, s64)
    assert not ok.any()


def test_identity_rotation_and_zero_pair():
    # the rotation at position 0 (c = 1, s = 0) keeps nonzero pairs and decides them in fp32
    a = np.array([1.5, -2.25, 3.0e-3], np.float32)
    b = np.array([-0.5, 4.0, 7.0], np.float32)
    ok, x, y = fast_path(a, b, np.ones(3), np.zeros(3))
    ex, ey = contract(a, b, np.ones(3), np.zeros(3))
    assert ok.all() and np.all(x == ex) and np.all(y == ey)
    assert np.all(x == fo.f64_to_bf16_bits(a.astype(np.float64)))
    # a zero result: the interval straddles -0 and +0 (different bf16 patterns), so
    # the pair goes to the exact path
    ok0, _, _ = fast_path(np.zeros(1, np.float32), np.zeros(1, np.float32), np.ones(1), np.zeros(1))
    assert not ok0.any()
