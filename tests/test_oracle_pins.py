"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these re-types the oracle's own formula: each check is a closed form,
an invariant, an exact-rational brute force on a tiny input, a hand-derived
worked example, or a constant the pages print (tests/golden/page_constants.txt).
They are chosen so that a plausible slip in the oracle (a dropped abs, a wrong
divisor, round-half-away instead of half-even, a transposed operand, a wrong
bit order in the packing) fails at least one of them.
"""
from __future__ import annotations

import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_constants.txt")


def golden():
    out = {}
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].strip()
        if line:
            k, v = (t.strip() for t in line.split("=", 1))
            out[k] = v
    return out


def f32(x) -> np.float32:
    return np.float32(x)


def f32_bits(x: float) -> int:
    return struct.unpack("<I", struct.pack("<f", float(x)))[0]


def frac_to_f32_rne(x: Fraction) -> np.float32:
    """Exact rational -> nearest fp32, ties to even.  Written from the IEEE-754
    definition (binary32: 24-bit significand, emin = -126, subnormal quantum
    2^-149); used only as an independent check."""
    if x == 0:
        return np.float32(0.0)
    sign = -1 if x < 0 else 1
    x = abs(x)
    e = x.numerator.bit_length() - x.denominator.bit_length()
    if Fraction(2) ** e > x:
        e -= 1
    # now 2^e <= x < 2^(e+1)
    q = max(e - 23, -149)
    scaled = x / (Fraction(2) ** q)
    fl = scaled.numerator // scaled.denominator
    rem = scaled - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    val = Fraction(fl) * Fraction(2) ** q
    if val >= Fraction(2) ** 128:
        return np.float32(sign * np.inf)
    return np.float32(sign * float(val))  # exact: val has <= 24 significant bits


def exact_mean_abs(W) -> Fraction:
    vals = [Fraction(float(abs(float(w)))) for w in np.asarray(W, dtype=np.float32).reshape(-1)]
    return sum(vals, Fraction(0)) / len(vals)


# ---------------------------------------------------------------- constants

def test_page_constants_packing_density():
    g = golden()
    per_byte = int(g["weights_per_byte"])
    bits = 8 / per_byte
    assert per_byte == 4
    assert abs(math.log2(3) - float(g["log2_3"])) < 5e-6
    # 2 bits per weight is above the information bound log2(3) ~ 1.58496 and
    # below 3 bits: four ternary codes fit one byte, five would not at 2 bits.
    assert float(g["log2_3"]) <= bits < 3
    q = np.array([[-1, 0, 1, 1] * 16] * 3, dtype=np.int8)
    assert oracle.pack(q).nbytes * per_byte == q.size
    # a 70B-class 8192 x 28672 matrix packs to N*K/4 bytes
    assert 8192 * 28672 // per_byte == 58_720_256


# ---------------------------------------------------------------- gamma (R1)

@pytest.mark.parametrize("c", [0.02, -0.02, 1.0, 3.0e38, 1e-45, -7.5, 2.0**-140])
def test_gamma_constant_matrix_is_abs_c(c):
    W = np.full((3, 8), c, dtype=np.float32)
    assert oracle.absmean(W) == abs(f32(c))


@pytest.mark.parametrize("K,c", [(4, 1.0), (7, 0.3), (64, -0.05), (1000, 2.5)])
def test_gamma_scaled_identity(K, c):
    W = (np.eye(K, dtype=np.float32) * f32(c)).astype(np.float32)
    want = frac_to_f32_rne(Fraction(float(abs(f32(c)))) / K)
    assert oracle.absmean(W) == want


def test_gamma_round_half_even_ties():
    one, u = 1.0, 2.0**-23
    # mean = 1 + 2^-24: halfway between 1 (even) and 1+2^-23 (odd) -> 1
    assert oracle.absmean(np.array([one, one + u], np.float32)) == f32(1.0)
    # mean = 1 + 1.5*2^-23: halfway between 1+2^-23 (odd) and 1+2^-22 (even) -> 1+2^-22
    assert oracle.absmean(np.array([one + u, one + 2 * u], np.float32)) == f32(one + 2 * u)
    # one more tiny term breaks the first tie upwards
    w = np.array([one, one + u, 2.0**-100, 0.0], np.float32)
    assert oracle.absmean(w) == frac_to_f32_rne(exact_mean_abs(w))


def test_gamma_brute_force_fraction_random():
    rng = np.random.default_rng(7)
    for trial in range(40):
        n = int(rng.integers(1, 60))
        scale = 10.0 ** rng.uniform(-42, 37)
        W = (rng.standard_normal(n) * scale).astype(np.float32)
        if trial % 5 == 0:
            W[rng.integers(0, n)] = np.float32(1e-45)  # a subnormal
        assert oracle.absmean(W) == frac_to_f32_rne(exact_mean_abs(W)), (trial, n, scale)


def test_gamma_mixed_exponents_brute_force():
    # values spread across the whole fp32 range, where a plain float sum loses bits
    W = np.array([3e38, 1.0, 1e-30, -2.5e-38, 1e-45, 7.0, -1e20, 5e-3] * 5, dtype=np.float32)
    assert oracle.absmean(W) == frac_to_f32_rne(exact_mean_abs(W))


def test_gamma_is_order_independent_and_sign_blind():
    rng = np.random.default_rng(3)
    W = (rng.standard_normal(4096) * 0.02).astype(np.float32)
    g = oracle.absmean(W)
    assert oracle.absmean(rng.permutation(W)) == g
    assert oracle.absmean(-W) == g
    assert oracle.absmean(W * np.float32(8.0)) == g * np.float32(8.0)  # power-of-two scaling is exact


def test_gamma_gaussian_closed_form():
    # E|W| for W ~ N(0, sigma) is sigma*sqrt(2/pi)
    rng = np.random.default_rng(11)
    sigma = 0.02
    W = (rng.standard_normal(2_000_000) * sigma).astype(np.float32)
    g = float(oracle.absmean(W))
    assert abs(g / (sigma * math.sqrt(2 / math.pi)) - 1) < 2e-3


def test_gamma_nonfinite_is_nan():
    assert np.isnan(oracle.absmean(np.array([1.0, np.inf], np.float32)))
    assert np.isnan(oracle.absmean(np.array([np.nan, 1.0], np.float32)))


# ---------------------------------------------------------------- ternarize (R2)

def test_ternarize_alphabet_and_gaussian_zero_fraction():
    rng = np.random.default_rng(5)
    W = (rng.standard_normal((1000, 1000)) * 0.02).astype(np.float32)
    g = oracle.absmean(W)
    q = oracle.ternarize(W, g)
    assert set(np.unique(q).tolist()) <= {-1, 0, 1}
    # zero iff |W| <= (gamma+eps)/2 (up to fp32 rounding): P(|Z| <= sqrt(2/pi)/2)
    p0 = math.erf(math.sqrt(2 / math.pi) / 2 / math.sqrt(2))
    assert abs(p0 - 0.3101) < 1e-4
    assert abs((q == 0).mean() - p0) < 3e-3
    # sign agreement wherever the weight is kept
    nz = q != 0
    assert np.all(np.sign(W[nz]) == q[nz])


def test_ternarize_half_even_ties_and_clip():
    gamma = f32(1.0)
    d = f32(gamma + f32(1e-5))
    half = f32(d * f32(0.5))  # exact
    vals = np.array([half, -half, np.nextafter(half, np.float32(1)), f32(1.5) * d, f32(2.5) * d, -f32(7) * d,
                     f32(0.0), f32(-0.0)], dtype=np.float32)
    q = oracle.ternarize(vals, gamma, f32(1e-5))
    # 0.5 -> 0 (half to even), -0.5 -> 0, just above 0.5 -> 1, 1.5 -> 2 -> clipped 1, 2.5 -> 2 -> 1, -7 -> -1
    assert q.tolist() == [0, 0, 1, 1, 1, -1, 0, 0]


def test_ternarize_threshold_characterisation_exact():
    # IEEE rounding fixes where the zero band ends: fl(|w|/d) <= 1/2 exactly when the
    # real quotient |w|/d <= 1/2 + 2^-25 (the midpoint between 0.5 and its fp32 successor,
    # a tie that goes to the even 0.5).  Check the oracle against that rational bound.
    rng = np.random.default_rng(9)
    for gamma in (f32(0.0123), f32(1.0), f32(3.7e-3), f32(0.0)):
        d = Fraction(float(f32(gamma + f32(1e-5))))
        bound = d * (Fraction(1, 2) + Fraction(1, 2**25))
        centre = np.float32(float(d / 2))
        w = centre
        ws = [w]
        for _ in range(40):
            w = np.nextafter(w, np.float32(np.inf))
            ws.append(w)
        w = centre
        for _ in range(40):
            w = np.nextafter(w, np.float32(0))
            ws.append(w)
        ws = np.array(ws + list((rng.standard_normal(200) * float(d)).astype(np.float32)), dtype=np.float32)
        q = oracle.ternarize(ws, gamma, f32(1e-5))
        for wi, qi in zip(ws.tolist(), q.tolist()):
            want = 0 if Fraction(abs(wi)) <= bound else (1 if wi > 0 else -1)
            assert qi == want, (gamma, wi)


def test_ternarize_closed_forms():
    # constant matrix: every entry is sign(c) because |c|/(|c|+eps) > 1/2
    W = np.full((4, 16), -0.02, np.float32)
    assert np.all(oracle.ternarize(W, oracle.absmean(W)) == -1)
    # scaled identity: gamma = c/K, diagonal c/(c/K+eps) > 1 -> 1, off-diagonal 0
    K = 32
    W = np.eye(K, dtype=np.float32) * np.float32(0.5)
    assert np.array_equal(oracle.ternarize(W, oracle.absmean(W)), np.eye(K, dtype=np.int8))
    # all zero: gamma = 0, d = eps, everything 0
    Z = np.zeros((3, 8), np.float32)
    assert oracle.absmean(Z) == 0 and np.all(oracle.ternarize(Z, 0.0) == 0)


# ---------------------------------------------------------------- packing (R3)

def test_pack_known_bytes():
    # code = q + 1, weight k at bits 2*(k % 4) of byte k/4
    q = np.array([[-1, 0, 1, 1], [1, 1, 1, 1], [0, 0, 0, 0], [-1, -1, -1, -1], [1, -1, 0, -1]], np.int8)
    assert oracle.pack(q).reshape(-1).tolist() == [0xA4, 0xAA, 0x55, 0x00, 0b00_01_00_10]


def test_pack_roundtrip_and_no_code3():
    rng = np.random.default_rng(1)
    q = rng.integers(-1, 2, size=(37, 128)).astype(np.int8)
    p = oracle.pack(q)
    assert p.shape == (37, 32)
    codes = np.stack([(p >> (2 * j)) & 3 for j in range(4)])
    assert not np.any(codes == 3)
    back, bad = oracle.unpack(p, 128)
    assert bad == 0 and np.array_equal(back, q)
    # row-major: row n of q only touches bytes [n*K/4, (n+1)*K/4)
    q2 = q.copy()
    q2[5] = 0
    p2 = oracle.pack(q2)
    diff_rows = np.nonzero(np.any(p2 != p, axis=1))[0].tolist()
    assert diff_rows == [5] or np.all(q[5] == 0)


def test_unpack_flags_code3():
    _, bad = oracle.unpack(np.array([[0xFF, 0x00]], np.uint8), 8)
    assert bad == 4


# ---------------------------------------------------------------- activations (R4, R5)

def test_quant_act_power_of_two_worked_example():
    # a = max|x| = 1 so s = 127 exactly and x*s is exact; then half-to-even rounding.
    x = np.array([[1.0, 0.5, -0.5, 0.25, 0.75, -1.0, 1 / 256, 3 / 254]], np.float32)
    xq, s = oracle.quant_act(x)
    assert s.tolist() == [127.0]
    # 127, 63.5->64, -63.5->-64, 31.75->32, 95.25->95, -127, 0.496->0, 1.5->2
    assert xq.tolist() == [[127, 64, -64, 32, 95, -127, 0, 2]]
    # a = 127/64 so s = 64 exactly; the ties 0.5, 2.5, 62.5 separate half-to-even from half-away
    x = np.array([[127 / 64, 2.5 / 64, 0.5 / 64, -2.5 / 64, 3.5 / 64, -127 / 64, 62.5 / 64, -0.5 / 64]], np.float32)
    xq, s = oracle.quant_act(x)
    assert s.tolist() == [64.0]
    assert xq.tolist() == [[127, 2, 0, -2, 4, -127, 62, 0]]


def test_quant_act_range_and_max_code():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((50, 300)).astype(np.float32)
    x[3] *= 1e6
    x[4] *= 1e-3
    xq, s = oracle.quant_act(x)
    assert xq.min() >= -127 and xq.max() <= 127  # |x*s| <= 127 (+rounding) never reaches -128
    assert np.all(np.abs(xq).max(axis=1) == 127)
    # sign agreement and monotonicity within a row
    for m in range(50):
        order = np.argsort(x[m], kind="stable")
        assert np.all(np.diff(xq[m][order].astype(int)) >= 0)
        big = np.abs(x[m]) * s[m] >= 0.5
        assert np.all(np.sign(xq[m][big]) == np.sign(x[m][big]))
    # error bound: |x_q - x*127/a| <= 1/2 + a few fp32 ulps of 127
    a = np.abs(x).max(axis=1, keepdims=True).astype(np.float64)
    err = np.abs(xq - x.astype(np.float64) * 127 / a)
    assert err.max() <= 0.5 + 64 * 2.0**-23 * 127


def test_quant_act_zero_and_tiny_rows_use_clamp():
    x = np.zeros((3, 16), np.float32)
    x[1, 3] = 1e-7  # below the 1e-5 clamp
    x[2, :] = -2e-6
    xq, s = oracle.quant_act(x)
    assert np.all(s == f32(127.0) / f32(1e-5))
    assert xq[0].tolist() == [0] * 16
    assert xq[1, 3] == round(1e-7 * 127 / 1e-5)  # 1.27 -> 1
    assert np.all(xq[2] == -25)  # -2e-6*1.27e7 = -25.4 -> -25


def test_quant_act_power_of_two_scale_invariance():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((8, 64)).astype(np.float32)
    xq1, s1 = oracle.quant_act(x)
    xq2, s2 = oracle.quant_act(x * np.float32(16))
    assert np.array_equal(xq1, xq2) and np.array_equal(s1, s2 * np.float32(16))


def test_bf16_widening_bit_patterns():
    bits = np.array([0x3F80, 0xC000, 0x0001, 0x7F7F, 0x8000], np.uint16)
    out = oracle.bf16_bits_to_f32(bits)
    assert out[0] == 1.0 and out[1] == -2.0 and out[2] == np.float32(2.0**-133)
    assert out[3] == np.float32(3.3895313892515355e38) and f32_bits(out[4]) == 0x80000000


# ---------------------------------------------------------------- product and dequant (R6)

def test_matmul_int_brute_force_python():
    rng = np.random.default_rng(6)
    M, N, K = 3, 5, 12
    q = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    xq = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    acc = oracle.matmul_int(q, xq)
    for m in range(M):
        for n in range(N):
            assert acc[m, n] == sum(int(q[n, k]) * int(xq[m, k]) for k in range(K))


def test_matmul_int_closed_forms():
    rng = np.random.default_rng(8)
    K = 64
    xq = rng.integers(-127, 128, size=(4, K)).astype(np.int8)
    # identity weights reproduce x_q
    assert np.array_equal(oracle.matmul_int(np.eye(K, dtype=np.int8), xq), xq.astype(np.int32))
    # constant weights give the row sums, with the weight's sign
    for c in (1, -1):
        acc = oracle.matmul_int(np.full((7, K), c, np.int8), xq)
        assert np.array_equal(acc, c * np.repeat(xq.astype(np.int32).sum(1, keepdims=True), 7, 1))
    # one +1 at (n=2, k=17) picks column 17 of x_q into output column 2
    q = np.zeros((5, K), np.int8)
    q[2, 17] = 1
    acc = oracle.matmul_int(q, xq)
    assert np.array_equal(acc[:, 2], xq[:, 17].astype(np.int32)) and np.count_nonzero(acc[:, [0, 1, 3, 4]]) == 0
    # worst-case magnitude stays exact: 127 * K
    big = oracle.matmul_int(np.ones((1, 28672), np.int8), np.full((1, 28672), 127, np.int8))
    assert big[0, 0] == 127 * 28672


def test_dequant_exact_and_bounded():
    acc = np.array([[0, 1, -3, 127 * 2560, -1000]], np.int32)
    y = oracle.dequant(acc, f32(0.25), np.array([f32(4.0)], np.float32))
    assert y.tolist() == [[0.0, 0.0625, -0.1875, 127 * 2560 / 16, -62.5]]  # powers of two: exact
    rng = np.random.default_rng(10)
    acc = rng.integers(-300000, 300000, size=(6, 50)).astype(np.int32)
    s = (rng.uniform(0.5, 200, size=6)).astype(np.float32)
    g = f32(0.0157)
    y = oracle.dequant(acc, g, s)
    for m in range(6):
        for n in range(50):
            exact = Fraction(int(acc[m, n])) * Fraction(float(g)) / Fraction(float(s[m]))
            if exact != 0:
                assert abs(Fraction(float(y[m, n])) - exact) <= abs(exact) * Fraction(1, 2**22)  # two roundings
            else:
                assert y[m, n] == 0


def test_forward_end_to_end_tiny():
    rng = np.random.default_rng(12)
    M, N, K = 8, 48, 256
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    x = rng.standard_normal((M, K)).astype(np.float32)
    packed, g = oracle.pack_weights(W)
    xq, s = oracle.quant_act(x)
    y, acc = oracle.forward(packed, g, xq, s, K)
    q = oracle.ternarize(W, g)
    for m in range(M):
        for n in range(N):
            assert acc[m, n] == sum(int(q[n, k]) * int(xq[m, k]) for k in range(K))
    # the quantised layer tracks the float layer: for Gaussian weights the ternary
    # code correlates with W at 2*phi(t)/sqrt(P(|Z|>t)) ~ 0.887 (t = sqrt(2/pi)/2);
    # a mismatched weight row (a transposed or shifted operand) gives ~0.
    def cos(a, b):
        return (a * b).sum() / np.sqrt((a * a).sum() * (b * b).sum())
    yf = x.astype(np.float64) @ W.astype(np.float64).T
    assert cos(y, yf) > 0.8
    assert abs(cos(y, np.roll(yf, 1, axis=1))) < 0.3
    with pytest.raises(ValueError):
        oracle.forward(np.full((N, K // 4), 0xFF, np.uint8), g, xq, s, K)


# ---------------------------------------------------------------- sub-layer RMS norm and squared ReLU (R9, R10)

def sqrt_f32_rne(v: Fraction) -> np.float32:
    """The fp32 nearest to sqrt(v), v >= 0 exact: the candidate c whose
    neighbouring midpoints bracket sqrt(v), compared through squares (exact).
    sqrt of a rational is never exactly half-way between two fp32 values
    unless it is itself an fp32 value, so no tie rule is needed."""
    if v == 0:
        return np.float32(0.0)
    c = np.float32(math.sqrt(float(v)))
    for _ in range(4):
        lo = np.nextafter(c, np.float32(0))
        hi = np.nextafter(c, np.float32(np.inf))
        m_lo = (Fraction(float(lo)) + Fraction(float(c))) / 2
        m_hi = (Fraction(float(c)) + Fraction(float(hi))) / 2
        if v < m_lo * m_lo:
            c = lo
        elif v > m_hi * m_hi:
            c = hi
        else:
            return c
    raise AssertionError("sqrt search did not settle")


def rint_half_even(x: Fraction) -> int:
    fl = x.numerator // x.denominator
    rem = x - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return fl


def rmsnorm_quant_exact(x, g, eps):
    """Reading R9 evaluated in exact rationals, each fp32 step rounded with
    the IEEE rules written out above; tiny rows only."""
    x = [Fraction(float(v)) for v in np.asarray(x, np.float32)]
    g = [Fraction(1)] * len(x) if g is None else [Fraction(float(v)) for v in np.asarray(g, np.float32)]
    ms = frac_to_f32_rne(sum((v * v for v in x), Fraction(0)) / len(x))
    v = frac_to_f32_rne(Fraction(float(ms)) + Fraction(float(np.float32(eps))))
    r = Fraction(float(sqrt_f32_rne(Fraction(float(v)))))
    xn = [Fraction(float(frac_to_f32_rne(Fraction(float(frac_to_f32_rne(xi * gi))) / r))) for xi, gi in zip(x, g)]
    a = max(abs(t) for t in xn)
    a = max(a, Fraction(float(np.float32(1e-5))))
    s = frac_to_f32_rne(127 / a)
    codes = [min(127, max(-128, rint_half_even(Fraction(float(frac_to_f32_rne(t * Fraction(float(s)))))))) for t in xn]
    return codes, s


def exact_mean_sq(x) -> Fraction:
    vals = [Fraction(float(v)) ** 2 for v in np.asarray(x, dtype=np.float32).reshape(-1)]
    return sum(vals, Fraction(0)) / len(vals)


def test_mean_sq_brute_force_fraction():
    rng = np.random.default_rng(17)
    for trial in range(60):
        n = int(rng.integers(1, 40))
        x = (rng.standard_normal(n) * 10.0 ** rng.uniform(-25, 18)).astype(np.float32)
        if trial % 6 == 0:
            x[rng.integers(0, n)] = np.float32(1e-45)
        if trial % 7 == 0:
            x[rng.integers(0, n)] = np.float32(3e18)  # square near the top of fp32
        assert oracle.mean_sq(x) == frac_to_f32_rne(exact_mean_sq(x)), (trial, n)
    # values spread over the whole range, where an fp32 or fp64 sum drops bits
    x = np.array([1.8e19, 1.0, 1e-20, -2.5e-38, 1e-45, 7.0, -1e10, 5e-3] * 3, np.float32)
    assert oracle.mean_sq(x) == frac_to_f32_rne(exact_mean_sq(x))


def test_mean_sq_closed_forms_and_ties():
    assert oracle.mean_sq(np.array([3.0, -4.0, 0.0, 0.0], np.float32)) == np.float32(6.25)
    assert oracle.mean_sq(np.full(1000, -0.5, np.float32)) == np.float32(0.25)
    # squares above the fp32 range: the mean rounds to +inf; far below it: to 0
    assert oracle.mean_sq(np.array([2.0**70, 0.0], np.float32)) == np.float32(np.inf)
    assert oracle.mean_sq(np.array([2.0**-80], np.float32)) == np.float32(0.0)
    # 2^-75 squared is 2^-150, half the smallest subnormal: a tie, to even (0);
    # with a second, larger term the mean goes above the midpoint
    assert oracle.mean_sq(np.array([2.0**-75], np.float32)) == np.float32(0.0)
    assert oracle.mean_sq(np.array([2.0**-74, 2.0**-74], np.float32)) == np.float32(2.0**-148)
    # 297^2 + 5785^2 = 2 * (2^24 + 1): the mean 2^24 + 1 lies half-way between
    # the fp32 neighbours 2^24 and 2^24 + 2, and rounds to the even one, 2^24;
    # a third, tiny square pushes it above the midpoint (to 2^24 + 2 for
    # K = 2 terms scaled to K = 3: checked against the exact fraction)
    assert oracle.mean_sq(np.array([297.0, 5785.0], np.float32)) == np.float32(2.0**24)
    x = np.array([297.0, 5785.0, 1e-30], np.float32)
    assert oracle.mean_sq(x) == frac_to_f32_rne(exact_mean_sq(x))
    assert oracle.mean_sq(np.array([1.0, 1.0, 0.0, 0.0], np.float32)) == np.float32(0.5)


def test_rmsnorm_quant_worked_example_exact_sqrt():
    # x = [3, -4, 0, 0], eps = 2.75: mean(x^2) = 25/4, v = 9, r = 3 exactly;
    # x_n = [1, fp32(-4/3)], max|x_n| = fp32(4/3) = 11184811 * 2^-23,
    # s = fp32(127 / that) = fp32(95.2499972...) = 95.25 (fp32 spacing 2^-17 there);
    # codes: rint(1 * 95.25) = 95, rint(-127.0000...) = -127
    xq, s = oracle.rmsnorm_quant_act(np.array([[3.0, -4.0, 0.0, 0.0]], np.float32), eps=np.float32(2.75))
    assert xq.tolist() == [[95, -127, 0, 0]]
    assert s.tolist() == [95.25]


def test_rmsnorm_quant_near_tie_normalise_then_quantise():
    # x = [2, 1], eps = 2^-9.  mean(x^2) = 2.5, v = 2.501953125 (exact),
    # r = fp32(sqrt(v)) = 0x1.94edfcp+0, x_n = [0x1.43b0dap+0, 0x1.43b0dap-1]
    # (1/r and 2/r round to the same significand), s = fp32(127 / x_n[0]) =
    # 0x1.91c41ep+6, and x_n[1] * s = 63.4999977... rounds to 0x1.fbfffep+5 =
    # 63.49999619, so the code is 63.  Quantising x itself and moving the RMS
    # factor into s instead would give 1 * 63.5 = 63.5, which rounds (half to
    # even) to 64: this case tells the two orders apart.
    xq, s = oracle.rmsnorm_quant_act(np.array([[2.0, 1.0]], np.float32), eps=np.float32(2.0**-9))
    assert xq.tolist() == [[127, 63]]
    assert float(s[0]) == float.fromhex("0x1.91c41ep+6")
    xq_fold, _ = oracle.quant_act(np.array([[2.0, 1.0]], np.float32))
    assert xq_fold.tolist() == [[127, 64]]


def test_rmsnorm_quant_brute_force_exact_rationals():
    rng = np.random.default_rng(23)
    for trial in range(80):
        K = int(rng.integers(1, 7))
        x = (rng.standard_normal(K) * 10.0 ** rng.uniform(-6, 6)).astype(np.float32)
        if trial % 5 == 0:
            x[0] = x[-1] * np.float32(0.5)  # ratios that land near half-way codes
        g = None if trial % 3 == 0 else rng.uniform(0.1, 3.0, size=K).astype(np.float32)
        eps = np.float32(10.0 ** rng.uniform(-8, 0))
        codes, s_ref = rmsnorm_quant_exact(x, g, eps)
        xq, s = oracle.rmsnorm_quant_act(x[None, :], gain=g, eps=eps)
        assert xq[0].tolist() == codes, (trial, x, g, eps)
        assert s[0] == s_ref, (trial, s[0], s_ref)


def test_rmsnorm_quant_is_invariant_to_token_scale():
    # RMS normalisation makes the BitLinear input independent of a per-token
    # scale: with eps far below mean(x^2), multiplying a row by 2^k scales the
    # exact mean of squares by 4^k and r by 2^k exactly, so x_n, x_q and s stay
    # the same bit for bit (plain absmax quantisation would divide s by 2^k)
    rng = np.random.default_rng(9)
    X = rng.standard_normal((5, 96)).astype(np.float32)
    eps = np.float32(2.0**-100)
    xq0, s0 = oracle.rmsnorm_quant_act(X, eps=eps)
    for k in (-3, 1, 6):
        xq1, s1 = oracle.rmsnorm_quant_act(X * np.float32(2.0 ** k), eps=eps)
        assert np.array_equal(xq0, xq1)
        assert np.array_equal(s0, s1)
    _, sp0 = oracle.quant_act(X)
    _, sp1 = oracle.quant_act(X * np.float32(8.0))
    assert np.array_equal(sp1 * np.float32(8.0), sp0)


def test_rmsnorm_quant_gain():
    rng = np.random.default_rng(10)
    X = rng.standard_normal((3, 64)).astype(np.float32)
    xq0, s0 = oracle.rmsnorm_quant_act(X)
    # a uniform gain of 2 doubles every normalised value exactly: same codes, half the scale
    xq2, s2 = oracle.rmsnorm_quant_act(X, gain=np.full(64, 2.0, np.float32))
    assert np.array_equal(xq0, xq2) and np.array_equal(s2 * np.float32(2.0), s0)
    # channels with zero gain quantise to zero; the others keep their sign
    g = np.ones(64, np.float32)
    g[::4] = 0.0
    xqg, _ = oracle.rmsnorm_quant_act(X, gain=g)
    assert np.all(xqg[:, ::4] == 0)
    nz = (xqg != 0)
    assert np.all(np.sign(xqg[nz]) == np.sign(X[nz]))


def test_rmsnorm_quant_constant_and_zero_rows():
    # constant row c = -0.5: mean(x^2) = 0.25, r = 0.5 (eps far below), x_n = -1,
    # so every code is -127 and s = 127
    xq, s = oracle.rmsnorm_quant_act(np.full((2, 40), -0.5, np.float32), eps=np.float32(2.0**-100))
    assert np.all(xq == -127) and np.all(s == 127.0)
    # an all-zero token normalises to zeros, and the absmax clamp keeps s finite
    xq, s = oracle.rmsnorm_quant_act(np.zeros((1, 16), np.float32))
    assert np.all(xq == 0) and s[0] == np.float32(127.0) / np.float32(1e-5)
    with pytest.raises(ValueError):
        oracle.rmsnorm_quant_act(np.ones((1, 4), np.float32), eps=np.float32(0.0))


def test_rmsnorm_quant_close_to_fp64_normalisation():
    # normalising in fp64 and quantising must land on the same codes away from
    # half-way points, and x_q / s must reconstruct x_n to half a step
    rng = np.random.default_rng(11)
    K = 300
    X = (rng.standard_normal((6, K)) * rng.uniform(0.01, 50.0, size=(6, 1))).astype(np.float32)
    g = rng.uniform(0.2, 2.0, size=K).astype(np.float32)
    eps = 1e-5
    xq, s = oracle.rmsnorm_quant_act(X, gain=g, eps=np.float32(eps))
    x64 = X.astype(np.float64)
    xn = x64 * g.astype(np.float64) / np.sqrt((x64 ** 2).mean(axis=1, keepdims=True) + np.float32(eps))
    sc = 127.0 / np.abs(xn).max(axis=1, keepdims=True)
    t = xn * sc
    far = np.abs(np.abs(t - np.floor(t)) - 0.5) > 1e-3
    codes = np.clip(np.rint(t), -127, 127).astype(np.int8)
    assert np.array_equal(xq[far], codes[far])
    assert np.allclose(s, sc[:, 0], rtol=1e-6, atol=0)
    assert np.all(np.abs(xq / s[:, None].astype(np.float64) - xn) <= 0.5 / s[:, None] * (1 + 1e-5))


def test_relu2_values():
    y = np.array([-1.5, -0.0, 0.0, 2.5, 3.0e20, np.float32(1e-23)], np.float32)
    out = oracle.relu2(y)
    assert out[:4].tolist() == [0.0, 0.0, 0.0, 6.25]
    assert np.isinf(out[4]) and out[4] > 0          # overflows to +inf in fp32
    assert out[5] == np.float32(np.float32(1e-23) * np.float32(1e-23))  # rounds to the nearest fp32 (a subnormal)


# ---------------------------------------------------------------- base-3 packing, five weights per byte (R11)

def test_tq5_hand_computed_bytes():
    # q = [1, 0, -1, 1, 1] -> digits [2, 1, 0, 2, 2] -> 2 + 1*3 + 0*9 + 2*27 + 2*81 = 221
    # all -1 -> 0, all 0 -> 1 + 3 + 9 + 27 + 81 = 121, all +1 -> 2 * 121 = 242
    q = np.array([[1, 0, -1, 1, 1, -1, -1, -1, -1, -1, 0, 0, 0, 0, 0, 1, 1, 1, 1, 1]], np.int8)
    p = oracle.pack_tq5(q)
    assert p.shape == (1, 16)
    assert p[0, :4].tolist() == [221, 0, 121, 242]
    assert np.all(p[0, 4:] == 121)  # padding: five zero codes


def test_tq5_enumerates_every_code_in_order():
    # row v holds the little-endian base-3 digits of v: the byte must be v itself,
    # so the 243 patterns map one to one, in order, onto 0..242
    v = np.arange(243)
    digits = np.stack([(v // 3 ** i) % 3 for i in range(5)], axis=1)
    p = oracle.pack_tq5((digits - 1).astype(np.int8))
    assert p[:, 0].tolist() == v.tolist()
    q, bad = oracle.unpack_tq5(p, 5)
    assert bad == 0 and np.array_equal(q, (digits - 1).astype(np.int8))


def test_tq5_ragged_row_padding():
    # K = 7: byte 0 holds k = 0..4, byte 1 holds k = 5, 6 and three zero codes
    q = np.array([[0, 0, 0, 0, 0, 1, -1]], np.int8)
    p = oracle.pack_tq5(q)
    assert p[0, 0] == 121
    assert p[0, 1] == 2 + 0 * 3 + 1 * 9 + 1 * 27 + 1 * 81  # = 119
    assert np.all(p[0, 2:] == 121) and p.shape == (1, 16)


def test_tq5_round_trip_and_invalid_bytes():
    rng = np.random.default_rng(12)
    for K in (1, 5, 80, 6912, 2563):
        q = rng.integers(-1, 2, size=(9, K)).astype(np.int8)
        p = oracle.pack_tq5(q)
        assert p.shape == (9, oracle.tq5_row_bytes(K)) and p.max() <= 242
        q2, bad = oracle.unpack_tq5(p, K)
        assert bad == 0 and np.array_equal(q, q2)
    p = oracle.pack_tq5(np.zeros((1, 5), np.int8))
    p[0, 0] = 243  # not a five-digit base-3 value
    p[0, 1] = 120  # a padding byte whose digits are not all zero codes
    _, bad = oracle.unpack_tq5(p, 5)
    assert bad == 2


def test_tq5_bits_per_weight():
    # 8 / 5 = 1.6 bits per weight when K is a multiple of 80, above the
    # information bound log2(3) = 1.58496 (page constant) and below the 2-bit code
    for K in (80, 2560, 6912):
        bits = oracle.tq5_row_bytes(K) * 8 / K
        assert math.isclose(bits, 1.6) if K % 80 == 0 else bits < 2.0
        assert bits >= math.log2(3)
    assert oracle.tq5_row_bytes(2560) == 512 and oracle.tq5_row_bytes(6912) == 1392


def test_tq5_forward_equals_two_bit_forward():
    # two independent encodings of the same ternary weights give the same
    # integer products and outputs
    rng = np.random.default_rng(13)
    N, K, M = 33, 320, 3
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    p2, g2 = oracle.pack_weights(W)
    p5, g5 = oracle.pack_weights_tq5(W)
    assert g2 == g5
    xq, s = oracle.quant_act(rng.standard_normal((M, K)).astype(np.float32))
    y2, a2 = oracle.forward(p2, g2, xq, s, K)
    y5, a5 = oracle.forward_tq5(p5, g5, xq, s, K)
    assert np.array_equal(a2, a5) and np.array_equal(y2.view(np.uint32), y5.view(np.uint32))
