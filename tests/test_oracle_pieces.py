"""Pins for the oracle's rounding and the stack's pointwise / row pieces (CPU only).

These functions are the checkers the GPU stack tests lean on, so each is held
to something the mathematics fixes rather than to a retyped formula:

- bf16 rounding of a double (every bf16 storage point of the oracle): an
  independent round-to-nearest-even written here with exact rational
  arithmetic over the bf16 value lattice, on exact midpoints of both
  parities, one double-ulp either side of them, subnormals, signed zeros
  and the overflow edge;
- SwiGLU (SiLU(g) * u): its zero, its odd-part identity
  SiLU(g) - SiLU(-g) = g, exact linearity in u, the saturated limit, and
  the logistic function's value at 1 and 2;
- RMSNorm forward: rows whose normalisation is known in closed form (a
  constant row, the row (3, 4)), which fix the mean and where eps enters,
  and exact scale invariance at eps = 0;
- the backward pieces the stack uses (RMSNorm, SwiGLU, the kv-head repeat):
  central differences of the forward pieces, and the adjoint identity
  <repeat(v), w> = <v, repeat^T(w)> in exact integer arithmetic.
"""
import math
from fractions import Fraction

import numpy as np

from weight_streaming_nf4_gb300 import synth


# ------------------------------------------------------------------------ bf16 rounding
def _bf16_value(b: int) -> Fraction:
    """Exact value of a finite non-negative bf16 bit pattern (0 <= b < 0x7F80)."""
    e = (b >> 7) & 0xFF
    m = b & 0x7F
    if e == 0:
        return Fraction(m, 1) * Fraction(1, 2 ** 133)
    return Fraction(128 + m, 1) * Fraction(2) ** (e - 127 - 7)


def _ref_round(d: float) -> int:
    """Round-to-nearest-even of a double to bf16 bits, by search over the
    ordered lattice of bf16 values (ties to the even bit pattern; past the
    largest finite value the next lattice point is 2^128, i.e. infinity)."""
    if d == 0.0:
        return 0x8000 if math.copysign(1.0, d) < 0 else 0
    sign = 0x8000 if d < 0 else 0
    a = Fraction(abs(d))
    lo, hi = 0, 0x7F7F
    if a >= _bf16_value(hi):
        below, above_v, above_b = hi, Fraction(2) ** 128, 0x7F80
    else:
        while hi - lo > 1:  # invariant: value(lo) <= a < value(hi)
            mid = (lo + hi) // 2
            if _bf16_value(mid) <= a:
                lo = mid
            else:
                hi = mid
        below, above_v, above_b = lo, _bf16_value(hi), hi
    dlo = a - _bf16_value(below)
    dhi = above_v - a
    if dlo < dhi or (dlo == dhi and below % 2 == 0):
        return sign | below
    return sign | above_b


def _cases():
    rng = np.random.default_rng(5)
    vals = [0.0, -0.0, 1.0, -1.0, 3.0, 1e-45, -1e-45, 3.4e38, -3.3e38]
    # exact midpoints between neighbours, both parities, normal and subnormal
    for b in list(rng.integers(1, 0x7F7E, 60)) + list(rng.integers(1, 0x7E, 20)) + [0x7E, 0x7F, 0x80]:
        b = int(b)
        for bb in (b, b + 1):
            m = (_bf16_value(bb) + _bf16_value(bb + 1)) / 2
            mf = float(m)
            assert Fraction(mf) == m  # 9 significant bits: exact in double
            vals += [mf, -mf, float(np.nextafter(mf, np.inf)), float(np.nextafter(mf, -np.inf))]
    # the overflow edge: halfway between the largest finite value and 2^128
    top = (_bf16_value(0x7F7F) + Fraction(2) ** 128) / 2
    vals += [float(top), float(np.nextafter(float(top), 0.0))]
    # random magnitudes across the range, and the subnormal range
    vals += list(rng.normal(0, 1, 100) * 10.0 ** rng.integers(-30, 30, 100))
    vals += list(rng.uniform(-1, 1, 40) * 2.0 ** -127)
    vals += list(rng.uniform(-1, 1, 40) * 2.0 ** -132)
    return vals


def test_f64_to_bf16_is_single_round_to_nearest_even(orc):
    vals = _cases()
    got = orc.f64_to_bf16(np.array(vals))
    for v, g in zip(vals, got):
        assert int(g) == _ref_round(v), (v, hex(int(g)), hex(_ref_round(v)))


def test_f64_to_bf16_ties_go_to_even_both_ways(orc):
    # 1 + 2^-8 lies halfway between 1 (even pattern 0x3F80) and 1 + 2^-7 (odd): rounds down;
    # 1 + 3 * 2^-8 lies halfway between 1 + 2^-7 (odd) and 1 + 2^-6 (even): rounds up.
    assert int(orc.f64_to_bf16(np.array([1.0 + 2.0 ** -8]))[0]) == 0x3F80
    assert int(orc.f64_to_bf16(np.array([1.0 + 3 * 2.0 ** -8]))[0]) == 0x3F82
    assert int(orc.f64_to_bf16(np.array([-(1.0 + 3 * 2.0 ** -8)]))[0]) == 0xBF82
    # a hair above a tie rounds up, a hair below rounds down
    assert int(orc.f64_to_bf16(np.array([1.0 + 2.0 ** -8 + 2.0 ** -40]))[0]) == 0x3F81
    assert int(orc.f64_to_bf16(np.array([1.0 + 3 * 2.0 ** -8 - 2.0 ** -40]))[0]) == 0x3F81


def test_f32_to_bf16_agrees_with_f64_path_on_floats(orc):
    """For an fp32 input both roundings are a single RNE rounding."""
    x = np.random.default_rng(3).normal(0, 1, 400).astype(np.float32)
    assert np.array_equal(orc.f32_to_bf16(x), orc.f64_to_bf16(x.astype(np.float64)))
    assert np.array_equal(orc.f32_to_bf16(x), synth.to_bf16_bits(x))


# ------------------------------------------------------------------------ SwiGLU
def _bits(vals):
    return synth.to_bf16_bits(np.asarray(vals, dtype=np.float32))


def _f(b):
    return synth.bf16_bits_to_f32(b).astype(np.float64)


def test_silu_mul_closed_forms(orc):
    u = _bits([1.0, -2.5, 0.375, 7.0])
    zero = _bits([0.0] * 4)
    assert np.all(_f(orc.silu_mul_bf16(zero, u)) == 0.0)          # SiLU(0) = 0
    # saturation: sigmoid(64) = 1 - 1.6e-28, so SiLU(64) u rounds to 64 u exactly
    g64 = _bits([64.0] * 4)
    assert np.array_equal(_f(orc.silu_mul_bf16(g64, u)), 64.0 * _f(u))
    gm = _bits([-64.0] * 4)
    neg = _f(orc.silu_mul_bf16(gm, _bits([1.0] * 4)))
    assert np.all(neg < 0) and np.all(np.abs(neg) < 1e-25)
    # the logistic function at 1 and 2: sigma(1) = e / (1 + e), sigma(2) = e^2 / (1 + e^2)
    one = orc.silu_mul_bf16(_bits([1.0]), _bits([1.0]))
    two = orc.silu_mul_bf16(_bits([2.0]), _bits([1.0]))
    assert int(one[0]) == _ref_round(0.7310585786300049)
    assert int(two[0]) == _ref_round(2.0 * 0.8807970779778823)


def test_silu_mul_odd_part_and_linearity(orc):
    rng = np.random.default_rng(11)
    g = _bits(rng.normal(0, 3, 300))
    one = _bits(np.ones(300))
    ng = g ^ np.uint16(0x8000)
    a = _f(orc.silu_mul_bf16(g, one))
    b = _f(orc.silu_mul_bf16(ng, one))
    # SiLU(g) - SiLU(-g) = g (sigmoid(g) + sigmoid(-g) = 1), up to two bf16 roundings
    # (each at most half an ulp, i.e. 2^-8 of the value)
    assert np.all(np.abs((a - b) - _f(g)) <= 2.0 ** -8 * (np.abs(a) + np.abs(b)) + 1e-30)
    # exact linearity in u: scaling u by a power of two scales the rounded product exactly
    u = _bits(rng.normal(0, 1, 300))
    u4 = _bits(4.0 * _f(u))
    assert np.array_equal(4.0 * _f(orc.silu_mul_bf16(g, u)), _f(orc.silu_mul_bf16(g, u4)))
    # unrounded form agrees with the rounded one to half a bf16 ulp
    exact = orc.silu_mul_f64(_f(g), _f(u))
    assert np.array_equal(orc.f64_to_bf16(exact), orc.silu_mul_bf16(g, u))


# ------------------------------------------------------------------------ RMSNorm forward
def test_rmsnorm_forward_closed_forms(orc):
    # constant row c: rstd = 1 / sqrt(c^2 + eps)
    x = np.full((1, 64), 1.5)
    y, r = orc.rmsnorm_f64(x, eps=0.25)
    assert abs(r[0] - 0.6324555320336759) <= 1e-15          # 1 / sqrt(2.5)
    assert np.all(np.abs(y - 0.9486832980505138) <= 1e-15)   # 1.5 / sqrt(2.5)
    yb, rb = orc.rmsnorm_bf16(x, eps=0.25)
    assert np.all(yb == _ref_round(0.9486832980505138)) and rb[0] == r[0]
    # the row (3, 4): mean of squares 12.5
    y, r = orc.rmsnorm_f64(np.array([[3.0, 4.0]]), eps=0.0)
    assert abs(r[0] - 0.28284271247461906) <= 1e-16         # 1 / sqrt(12.5)
    assert np.allclose(y, [[0.848528137423857, 1.131370849898476]], rtol=0, atol=2e-16)
    # eps enters under the root beside the mean: (3, 4) with eps 0.25 -> 1 / sqrt(12.75)
    _, r = orc.rmsnorm_f64(np.array([[3.0, 4.0]]), eps=0.25)
    assert abs(r[0] - 0.28005601680560194) <= 1e-16


def test_rmsnorm_scale_invariance_at_eps_zero(orc):
    x = np.random.default_rng(2).normal(0, 1, (5, 48))
    y1, r1 = orc.rmsnorm_f64(x, eps=0.0)
    y2, r2 = orc.rmsnorm_f64(8.0 * x, eps=0.0)
    assert np.array_equal(y1, y2) and np.array_equal(r1, 8.0 * r2)


# ------------------------------------------------------------------------ backward pieces
def test_rmsnorm_backward_central_differences(orc):
    rng = np.random.default_rng(4)
    M, H, eps = 3, 16, 0.1
    x = rng.normal(0, 1, (M, H))
    dy = rng.normal(0, 1, (M, H))
    _, rstd = orc.rmsnorm_f64(x, eps=eps)
    base = rng.normal(0, 1, (M, H))
    g = orc.rmsnorm_bwd(x, rstd, dy, dx=base) - base       # the backward adds into dx
    h = 1e-6
    for m in range(M):
        for i in range(H):
            xp, xm = x.copy(), x.copy()
            xp[m, i] += h
            xm[m, i] -= h
            lp = np.sum(dy * orc.rmsnorm_f64(xp, eps=eps)[0])
            lm = np.sum(dy * orc.rmsnorm_f64(xm, eps=eps)[0])
            assert abs((lp - lm) / (2 * h) - g[m, i]) <= 1e-8 * (1 + abs(g[m, i]))


def test_silu_mul_backward_central_differences(orc):
    rng = np.random.default_rng(6)
    n = 64
    g = rng.normal(0, 2, n)
    u = rng.normal(0, 1, n)
    d = rng.normal(0, 1, n)
    dg, du = orc.silu_mul_bwd(d, g, u, round_bf16=False)
    h = 1e-6
    fd_g = d * (orc.silu_mul_f64(g + h, u) - orc.silu_mul_f64(g - h, u)) / (2 * h)
    fd_u = d * (orc.silu_mul_f64(g, u + h) - orc.silu_mul_f64(g, u - h)) / (2 * h)
    assert np.allclose(dg, fd_g, rtol=1e-7, atol=1e-9)
    assert np.allclose(du, fd_u, rtol=1e-7, atol=1e-9)
    # the stored (bf16) form is the rounding of the exact one
    dgb, dub = orc.silu_mul_bwd(d, g, u, round_bf16=True)
    assert np.array_equal(dgb, _f(orc.f64_to_bf16(dg)))
    assert np.array_equal(dub, _f(orc.f64_to_bf16(du)))


def test_repeat_kv_backward_is_the_adjoint(orc):
    rng = np.random.default_rng(8)
    M, H, KV, hd = 6, 128, 32, 16
    v_int = rng.integers(-50, 50, (M, KV)).astype(np.float64)
    w = rng.integers(-50, 50, (M, H)).astype(np.float64)
    vr = _f(orc.repeat_kv(_bits(v_int), H, hd))
    dv = orc.repeat_kv_bwd(w, KV, hd, round_bf16=False)
    assert np.sum(vr * w) == np.sum(v_int * dv)              # exact in integers
    # every query head reads exactly one kv head: the repeat of ones is ones, and the
    # adjoint of ones counts the H / KV query heads per kv head
    assert np.all(orc.repeat_kv_bwd(np.ones((M, H)), KV, hd, round_bf16=False) == H // KV)
