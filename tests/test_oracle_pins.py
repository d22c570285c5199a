"""Pins of the CPU oracle against facts outside itself.

Each check ties an oracle function to something it does not compute: numpy's
binary16 conversion, hand-worked fixtures under tests/golden, brute-force
dequantise-then-dense products in f64 (numpy matmul), exact rational sums,
closed-form special cases and invariants of the encodings.  A dropped term,
a wrong sign or index, or a transposed operand in the oracle fails at least
one of them.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

from conftest import read_golden
from q8_quantized_projection_gb300 import synth

QK = 32


# ----------------------------------------------------------------- binary16

def test_f16_to_f32_all_patterns(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([orc.f16_to_f32(int(b)) for b in bits], dtype=np.float32)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite].view(np.uint32), ref[finite].view(np.uint32))
    assert np.all(np.isnan(got[np.isnan(ref)]))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


def test_f32_to_f16_matches_numpy(orc):
    rng = np.random.default_rng(1)
    mags = np.exp2(rng.uniform(-30, 17, size=4000)).astype(np.float32)
    vals = np.concatenate([mags, -mags])
    # exact midpoints between neighbouring binary16 values (ties to even)
    h = rng.integers(1, 0x7bff, size=1000, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    mids = ((lo + hi) / 2).astype(np.float32)
    special = np.array([0.0, -0.0, 65504.0, 65519.996, 65520.0, 65536.0, 1e9,
                        2.0**-24, 2.0**-25, 2.0**-25 * 3, 2.0**-26, 2.0**-14,
                        2.0**-14 - 2.0**-25, 6.1e-5, 5.96e-8], dtype=np.float32)
    vals = np.concatenate([vals, mids[np.isfinite(mids)], special, -special])
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = orc.f32_to_f16_array(vals)
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------ pack

def test_pack_hand_block(orc):
    rows = read_golden("pack_block.txt")
    scale_bits = int(rows[0][0], 16)
    w = np.array([int(r[0]) * 2.0**-8 for r in rows[1:]], dtype=np.float32)
    qexp = np.array([int(r[1]) for r in rows[1:]], dtype=np.int8)
    assert w.size == QK
    q, s, ov = orc.q8_pack(w.reshape(1, QK))
    assert ov == 0
    assert int(s[0, 0]) == scale_bits
    assert np.array_equal(q[0], qexp)


def test_pack_roundtrip_bound_and_idempotence(orc):
    rng = np.random.default_rng(2)
    w = synth.f32_weights(rng, 37, 96 * 2)
    w[3, :QK] = 0.0                       # an all-zero block
    w[5, QK:2 * QK] *= 1e-6               # scale rounds to binary16 zero
    w[6, QK:2 * QK] *= 1e-3               # subnormal binary16 scale
    q, s, ov = orc.q8_pack(w)
    assert ov == 0
    sf = s.view(np.float16).astype(np.float32)
    sfe = np.repeat(sf, QK, axis=1)
    err = np.abs(w.astype(np.float64) - sfe.astype(np.float64) * q)
    # normal scales (relative rounding <= 2^-11): |w - s q| <= s/2
    normal = sfe >= 2.0**-14
    assert np.all((err <= sfe * 0.5 * (1 + 2.0**-20))[normal])
    # subnormal scales may clamp: the error is then amax - 127 s at most
    amax_e = np.repeat(np.abs(w.reshape(37, -1, QK)).max(axis=2), QK, axis=1)
    sub = (sfe > 0) & ~normal
    assert sub.any()
    assert np.all((err <= np.maximum(sfe * 0.5 * (1 + 2.0**-20), amax_e - 127.0 * sfe))[sub])
    assert s[5, 1] == 0 and np.all(q[5, QK:2 * QK] == 0)
    assert np.all(q[3, :QK] == 0) and s[3, 0] == 0
    assert np.all(np.abs(q.astype(np.int32)) <= 127)
    # the largest |w| of every non-zero block maps to +-127
    blocks = np.abs(q.reshape(37, -1, QK).astype(np.int32)).max(axis=2)
    normal_blk = s.view(np.float16).astype(np.float32) >= 2.0**-14
    assert np.all((blocks == 127)[normal_blk])
    # pack(dequant(pack(w))) == pack(w)
    w2 = (sfe * q).astype(np.float32)
    q2, s2, _ = orc.q8_pack(w2)
    nb = np.repeat(normal_blk, QK, axis=1)
    assert np.array_equal(q2[nb], q[nb]) and np.array_equal(s2[normal_blk], s[normal_blk])
    # the stored scale is the binary16 rounding of amax/127 (numpy's rounding)
    amax = np.abs(w.reshape(37, -1, QK)).max(axis=2)
    assert np.array_equal(s, (amax / np.float32(127)).astype(np.float16).view(np.uint16))


def test_pack_overflow_counted(orc):
    w = np.zeros((1, 64), np.float32)
    w[0, 0] = 65504.0 * 127 * 2     # scale overflows binary16
    w[0, 40] = 1.0
    q, s, ov = orc.q8_pack(w)
    assert ov == 1
    assert s[0, 0] == 0x7C00 and np.all(q[0, :QK] == 0)
    assert q[0, 40] == 127


# --------------------------------------------------------- activation codes

def test_act_i8_hand_block(orc):
    rows = read_golden("act_i8_block.txt")
    d = float(rows[0][0])
    x = np.array([float(r[0]) for r in rows[1:]], dtype=np.float32)
    qexp = np.array([int(r[1]) for r in rows[1:]], dtype=np.int8)
    xq, xd = orc.act_quant_i8(x.reshape(1, QK))
    assert xd[0, 0] == np.float32(d)
    assert np.array_equal(xq[0], qexp)


def test_act_i8_bound_and_monotone(orc):
    rng = np.random.default_rng(3)
    x = synth.activations(rng, 5, 4 * QK)
    x[1, :QK] = 0.0
    xq, xd = orc.act_quant_i8(x)
    de = np.repeat(xd, QK, axis=1).astype(np.float64)
    err = np.abs(x - de * xq)
    assert np.all(err <= de * (0.5 + 1e-5))
    assert np.all(xq[1, :QK] == 0) and xd[1, 0] == 0
    for m in range(5):
        for b in range(4):
            xb, qb = x[m, b * QK:(b + 1) * QK], xq[m, b * QK:(b + 1) * QK]
            order = np.argsort(xb, kind="stable")
            assert np.all(np.diff(qb[order].astype(np.int32)) >= 0)
            if xd[m, b] > 0:
                assert np.abs(qb.astype(np.int32)).max() == 127


def test_i8x2_split_table(orc):
    table = [(int(a), int(b), int(c)) for a, b, c in read_golden("i8x2_split.txt")]
    # d = 8191 / 8191 = 1 when the block holds 8191, so each code is its own x.
    codes = [t[0] for t in table]
    x = np.zeros(((len(codes) + QK - 2) // (QK - 1)) * QK, np.float32)
    blocks = x.reshape(-1, QK)
    where = {}
    for i, c in enumerate(codes):
        b, j = divmod(i, QK - 1)
        blocks[b, 0] = 8191.0
        blocks[b, j + 1] = c
        where[c] = (b, j + 1)
    xh, xl, xd = orc.act_quant_i8x2(x.reshape(1, -1))
    assert np.all(xd == 1.0)
    hb, lb = xh.reshape(-1, QK), xl.reshape(-1, QK)
    for q, hi, lo in table:
        b, j = where[q]
        assert (int(hb[b, j]), int(lb[b, j])) == (hi, lo), q


def test_i8x2_identity_ranges_bound(orc):
    rng = np.random.default_rng(4)
    x = synth.activations(rng, 7, 6 * QK) * np.float32(3.0)
    x[2, QK:2 * QK] = 0.0
    xh, xl, xd = orc.act_quant_i8x2(x)
    Q = 128 * xh.astype(np.int32) + xl.astype(np.int32)
    assert xh.min() >= -64 and xh.max() <= 64
    assert xl.min() >= -64 and xl.max() <= 63
    assert np.abs(Q).max() <= 8191
    de = np.repeat(xd, QK, axis=1).astype(np.float64)
    assert np.all(np.abs(x - de * Q) <= de * (0.5 + 1e-3))
    assert np.all(xl[Q % 128 == 0] == 0)
    for m in range(7):
        for b in range(6):
            xb, qb = x[m, b * QK:(b + 1) * QK], Q[m, b * QK:(b + 1) * QK]
            order = np.argsort(xb, kind="stable")
            assert np.all(np.diff(qb[order]) >= 0)
            if xd[m, b] > 0:
                assert np.abs(qb).max() == 8191


# ----------------------------------------------------------- block dots

@pytest.mark.parametrize("two_word", [False, True])
def test_block_dots_order_invariance(orc, two_word):
    rng = np.random.default_rng(5)
    n, k, rows = 11, 5 * QK, 3
    q, _ = synth.q8_weights(rng, n, k)
    x = synth.activations(rng, rows, k)
    if two_word:
        xh, xl, _ = orc.act_quant_i8x2(x)
        a = 128 * xh.astype(np.int64) + xl.astype(np.int64)
        isum = orc.block_dots(q, xh, xl)
    else:
        xh, _ = orc.act_quant_i8(x)
        a = xh.astype(np.int64)
        isum = orc.block_dots(q, xh)
    # independent contraction: numpy int64 einsum over (m, n, b, i)
    ref = np.einsum("nbi,mbi->mnb", q.astype(np.int64).reshape(n, -1, QK), a.reshape(rows, -1, QK))
    assert np.array_equal(isum.astype(np.int64), ref)
    # reversed element order within each block gives the same integers
    rev = np.einsum("nbi,mbi->mnb", q.astype(np.int64).reshape(n, -1, QK)[:, :, ::-1],
                    a.reshape(rows, -1, QK)[:, :, ::-1])
    assert np.array_equal(isum.astype(np.int64), rev)


# --------------------------------------------------- projections vs brute force

def _dense(q, s):
    sf = s.view(np.float16).astype(np.float64)
    return q.astype(np.float64) * np.repeat(sf, QK, axis=1)


@pytest.mark.parametrize("n,k,rows", [(1, 32, 1), (3, 64, 2), (5, 96, 3), (4, 160, 1)])
@pytest.mark.parametrize("mode", ["i8", "i8x2"])
def test_proj_q_brute_force(orc, n, k, rows, mode):
    rng = np.random.default_rng(100 + n * 7 + k + rows)
    q, s = synth.q8_weights(rng, n, k)
    x = synth.activations(rng, rows, k)
    act = orc.quantize(mode, x)
    y, norm = orc.project(mode, q, s, act)
    if mode == "i8":
        xq, xd = act
        a = xq.astype(np.float64)
    else:
        xh, xl, xd = act
        a = 128.0 * xh.astype(np.float64) + xl.astype(np.float64)
    xdq = a * np.repeat(xd.astype(np.float64), QK, axis=1)      # dequantised activation
    ref = xdq @ _dense(q, s).T                                   # [rows, n]
    assert y.shape == (rows, n)
    assert np.all(np.abs(y - ref) <= 1e-6 * norm + 1e-30)
    # the tolerance scale is the sum over blocks of |block dot * scales|
    wd = _dense(q, s)
    nref = sum(np.abs(xdq[:, b * QK:(b + 1) * QK] @ wd[:, b * QK:(b + 1) * QK].T)
               for b in range(k // QK))
    assert np.allclose(norm, nref, rtol=1e-12, atol=0)


@pytest.mark.parametrize("n,k,rows", [(1, 32, 1), (3, 64, 2), (2, 96, 3)])
def test_proj_f64_exact_rational(orc, n, k, rows):
    rng = np.random.default_rng(200 + n + k + rows)
    q, s = synth.q8_weights(rng, n, k)
    x = synth.activations(rng, rows, k)
    y, norm = orc.proj_f64(q, s, x)
    w = _dense(q, s)
    for m in range(rows):
        for j in range(n):
            exact = sum(Fraction(float(w[j, kk])) * Fraction(float(x[m, kk])) for kk in range(k))
            nexact = sum(abs(Fraction(float(w[j, kk])) * Fraction(float(x[m, kk]))) for kk in range(k))
            assert abs(Fraction(float(y[m, j])) - exact) <= Fraction(k) * Fraction(2) ** -53 * nexact
            assert math.isclose(float(norm[m, j]), float(nexact), rel_tol=1e-12)
            fs = math.fsum(float(w[j, kk]) * float(x[m, kk]) for kk in range(k))
            assert abs(y[m, j] - fs) <= k * 2.0**-53 * norm[m, j]


def test_one_hot_activation(orc):
    rng = np.random.default_rng(6)
    n, k = 9, 4 * QK
    q, s = synth.q8_weights(rng, n, k)
    kk, v = 77, np.float32(-1.75)
    x = np.zeros((1, k), np.float32)
    x[0, kk] = v
    sw = s.view(np.float16).astype(np.float32)[:, kk // QK]
    # f32 activations: exactly S * Q * v
    y64, _ = orc.proj_f64(q, s, x)
    assert np.array_equal(y64[0], sw.astype(np.float64) * q[:, kk] * np.float64(v))
    # one word: code -127, d = 1.75 / 127 (the sign of v is in the code)
    xq, xd = orc.act_quant_i8(x)
    assert xq[0, kk] == -127 and np.count_nonzero(xq) == 1
    yb, _ = orc.proj_q(q, s, xq, None, xd)
    ref = sw.astype(np.float64) * q[:, kk] * np.float64(v)
    assert np.all(np.abs(yb[0] - ref) <= 2 * 2.0**-24 * np.abs(ref) + 1e-30)
    # two words: code -8191
    xh, xl, xd2 = orc.act_quant_i8x2(x)
    assert 128 * int(xh[0, kk]) + int(xl[0, kk]) == -8191
    yc, _ = orc.proj_q(q, s, xh, xl, xd2)
    assert np.all(np.abs(yc[0] - ref) <= 3 * 2.0**-24 * np.abs(ref) + 1e-30)


def test_zero_blocks_and_identity(orc):
    # identity-like weights: row j has a single 127 at column 32*j with scale 1/127
    n, k = 4, 4 * QK
    q = np.zeros((n, k), np.int8)
    s = np.zeros((n, k // QK), np.uint16)
    one = np.float16(1.0 / 127).view(np.uint16)
    for j in range(n):
        q[j, QK * j] = 127
        s[j, j] = one
    x = np.zeros((1, k), np.float32)
    x[0, ::QK] = np.array([1.0, -2.0, 0.5, 4.0], np.float32)
    y64, _ = orc.proj_f64(q, s, x)
    sf = np.float64(np.float32(np.float16(1.0 / 127)))
    assert np.array_equal(y64[0], sf * 127 * x[0, ::QK].astype(np.float64))
    xq, xd = orc.act_quant_i8(x)
    yb, _ = orc.proj_q(q, s, xq, None, xd)
    assert np.allclose(yb[0], x[0, ::QK], rtol=2e-3)
    # all-zero activation gives exact zeros in every mode
    z = np.zeros((2, k), np.float32)
    for mode in ("f32", "i8", "i8x2"):
        y, nrm = orc.project(mode, q, s, orc.quantize(mode, z))
        assert np.all(y == 0) and np.all(nrm == 0)


# ---------------------------------------------------------------- RMSNorm

def test_rmsnorm_power_of_two_constant(orc):
    g = synth.gain(np.random.default_rng(7), 96)
    for c in (0.25, -4.0, 1.0, 2.0**-10):
        h = np.full((1, 96), c, np.float32)
        x, r = orc.rmsnorm(h, g, eps=0.0)
        assert r[0] == 1.0 / abs(c)
        assert np.array_equal(x[0], np.sign(c).astype(np.float32) * g)


def _round_bin64(v: Fraction) -> Fraction:
    """An exact positive rational rounded to binary64 (53-bit significand),
    ties to even."""
    e = v.numerator.bit_length() - v.denominator.bit_length()
    if Fraction(2) ** e > v:
        e -= 1
    q = Fraction(2) ** (e - 52)
    m = v / q
    n = m.numerator // m.denominator
    rem = m - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return n * q


def test_rmsnorm_rounding_order_golden(orc):
    """The producer rounds h * rf first, then multiplies by the gain: a block
    where h * (rf * g) rounds one ulp apart, and where that ulp moves a
    one-word code from 64 to 63 (tests/golden/rmsnorm_order.txt).

    The projection's scale product has the same kind of freedom: the oracle
    rounds (s_w * d_x) first, then multiplies by float(isum), and no pin tells
    that from s_w * (d_x * isum); both stay within the float tolerance, so
    they change no verdict."""
    fx = {r[0]: r[1] for r in read_golden("rmsnorm_order.txt")}
    hx = lambda k: float.fromhex(fx[k])
    g0 = np.float32(hx("g0"))
    h = np.zeros((1, QK), np.float32)
    h[0, :2] = 3.0
    g = np.ones(QK, np.float32)
    g[0], g[1] = g0, g0 / np.float32(2)
    # the fixture against exact rationals, both orders
    r = _round_bin64(Fraction(4, 3))
    rf = Fraction(_round_f32(r))
    hrf = Fraction(_round_f32(3 * rf))
    x0 = _round_f32(hrf * Fraction(float(g0)))
    alt = _round_f32(3 * Fraction(_round_f32(rf * Fraction(float(g0)))))
    assert (float(r), float(rf), float(hrf)) == (hx("r"), hx("rf"), hx("hrf"))
    assert (x0, alt) == (hx("x0"), hx("x0_alt")) and x0 != alt
    assert _round_f32(Fraction(x0) / 127) == hx("d_i8")
    assert _round_f32(Fraction(alt) / 127) == hx("d_alt")
    # the oracle takes the first order
    x, rr = orc.rmsnorm(h, g, eps=0.0)
    assert rr[0] == hx("r")
    assert float(x[0, 0]) == hx("x0") and float(x[0, 1]) == hx("x1")
    assert not np.any(x[0, 2:])
    xq, xd = orc.act_quant_i8(x)
    assert float(xd[0, 0]) == hx("d_i8")
    assert (int(xq[0, 0]), int(xq[0, 1])) == (int(fx["code0"]), int(fx["code1"]))
    # the code depends on the order: the other order's x gives the other code
    xa = x.copy()
    xa[0, 0], xa[0, 1] = np.float32(hx("x0_alt")), np.float32(hx("x0_alt") / 2)
    xqa, _ = orc.act_quant_i8(xa)
    assert int(xqa[0, 1]) == int(fx["code1_alt"])


def test_rmsnorm_matches_f64_formula(orc):
    rng = np.random.default_rng(8)
    h = synth.activations(rng, 6, 4096)
    g = synth.gain(rng, 4096)
    x, r = orc.rmsnorm(h, g, eps=1e-5)
    hd = h.astype(np.float64)
    ref_r = 1.0 / np.sqrt(np.mean(hd * hd, axis=1) + np.float64(np.float32(1e-5)))
    assert np.allclose(r, ref_r, rtol=1e-14, atol=0)
    ref = hd * ref_r[:, None] * g.astype(np.float64)
    assert np.all(np.abs(x - ref) <= 3 * 2.0**-24 * np.abs(ref))
    x1, _ = orc.rmsnorm(h, None, eps=1e-5)
    assert np.all(np.abs(x1 - hd * ref_r[:, None]) <= 2 * 2.0**-24 * np.abs(hd * ref_r[:, None]))


# ---------------------------------------------------------------- residual

def _round_f32(v: Fraction) -> float:
    """An exact rational rounded to the nearest binary32, ties to even (an
    independent restatement of IEEE rounding: scale to a 24-bit integer
    significand, round, rescale)."""
    if v == 0:
        return 0.0
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)                      # subnormal range: fixed quantum 2^-149
    q = Fraction(2) ** (e - 23)           # the quantum at this binade
    m = a / q
    n = m.numerator // m.denominator
    rem = m - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    r = n * q
    if r >= Fraction(2) ** 128:
        return sign * float("inf")
    return sign * float(r)


def test_residual_add_exact_rational(orc):
    # s = h + r rounded once: against exact rationals, over wide exponent gaps
    rng = np.random.default_rng(21)
    rows, k = 3, 256
    h = (rng.standard_normal((rows, k)) * np.exp2(rng.integers(-30, 30, (rows, k)))).astype(np.float32)
    r = (rng.standard_normal((rows, k)) * np.exp2(rng.integers(-30, 30, (rows, k)))).astype(np.float32)
    s = orc.residual_add(h, r)
    for i in range(rows):
        for j in range(k):
            want = _round_f32(Fraction(float(h[i, j])) + Fraction(float(r[i, j])))
            assert float(s[i, j]) == want, (h[i, j], r[i, j], s[i, j], want)


def test_residual_add_hand_cases(orc):
    # hand-worked binary32 sums: ties to even at 2^24 and at 1, cancellation,
    # overflow, and the identities r = 0 and r = -h
    two24 = float(2 ** 24)
    cases = [
        (two24, 1.0, two24),                      # 2^24 + 1: a tie, stays even
        (two24, 3.0, two24 + 4.0),                # 2^24 + 3: a tie, rounds up to even
        (1.0, 2.0 ** -24, 1.0),                   # 1 + half an ulp: tie to even
        (1.0, 3 * 2.0 ** -25, 1.0 + 2.0 ** -23),  # just above the tie
        (1e30, -1e30, 0.0),
        (3.0e38, 3.0e38, float("inf")),
    ]
    h = np.array([[c[0] for c in cases]], np.float32)
    r = np.array([[c[1] for c in cases]], np.float32)
    s = orc.residual_add(h, r)
    assert [float(v) for v in s[0]] == [c[2] for c in cases]
    x = synth.activations(np.random.default_rng(22), 2, 64)
    assert np.array_equal(orc.residual_add(x, np.zeros_like(x)), x)
    assert not np.any(orc.residual_add(x, -x))


# ---------------------------------------------------------------- SwiGLU

def _ulps(a: float, b: float) -> int:
    ia = int(np.float32(a).view(np.int32))
    ib = int(np.float32(b).view(np.int32))
    return abs(ia - ib)


def test_exp_f32_within_one_ulp(orc):
    # against the double-precision exponential rounded to binary32, over the
    # whole finite range and its edges
    xs = np.concatenate([np.linspace(-103.9, 88.7, 40001, dtype=np.float64),
                         [1e-30, -1e-30, 0.5, -0.5, 1.0, -1.0, 10.0, -10.0]])
    for x in xs.astype(np.float32):
        want = math.exp(float(x))
        assert _ulps(orc.exp_f32(float(x)), want) <= 1, x
    assert orc.exp_f32(0.0) == 1.0
    assert orc.exp_f32(89.0) == math.inf and orc.exp_f32(-105.0) == 0.0
    assert orc.exp_f32(-math.inf) == 0.0 and orc.exp_f32(math.inf) == math.inf
    assert math.isnan(orc.exp_f32(math.nan))
    assert 0.0 < orc.exp_f32(-100.0) < 2.0 ** -126       # subnormal results exist


def test_swiglu_special_values_and_layout(orc):
    f = 4
    gu = np.array([[0.0, 1.0, 20.0, -100.0,   # gate
                    5.0, 2.0, 3.0, 7.0]],      # up
                  np.float32)
    x = orc.swiglu(gu)[0]
    assert x[0] == 0.0                                  # silu(0) = 0
    assert _ulps(x[1], 2.0 / (1.0 + math.exp(-1.0))) <= 2
    assert x[2] == np.float32(60.0)                     # 1 + e^-20 rounds to 1
    assert x[3] == 0.0                                  # e^100 overflows: silu -> -0
    swapped = orc.swiglu(np.concatenate([gu[:, f:], gu[:, :f]], axis=1))[0]
    assert not np.array_equal(swapped, x)               # gate first, then up


def test_swiglu_matches_f64_formula(orc):
    rng = np.random.default_rng(31)
    f = 512
    gu = (rng.standard_normal((3, 2 * f)) * 3.0).astype(np.float32)
    x = orc.swiglu(gu)
    g = gu[:, :f].astype(np.float64)
    u = gu[:, f:].astype(np.float64)
    ref = g / (1.0 + np.exp(-g)) * u
    # four roundings of binary32 (exp, 1 + e, the division, the product)
    assert np.all(np.abs(x - ref) <= 6 * 2.0 ** -24 * np.abs(ref) + 1e-38)


# ---------------------------------------------------------------- KV rows

def test_kv_write_hand_example(orc):
    # two sequences, N = 10 outputs: q = columns 0..3, K = 4..6, V = 7..9
    y = np.arange(20, dtype=np.float32).reshape(2, 10) + 0.5
    kc = np.full((2, 4, 3), -1.0, np.float32)
    vc = np.full((2, 4, 3), -1.0, np.float32)
    bad = orc.kv_write(y, [2, 0], 4, 3, kc, vc)
    assert bad == 0
    assert kc[0, 2].tolist() == [4.5, 5.5, 6.5] and vc[0, 2].tolist() == [7.5, 8.5, 9.5]
    assert kc[1, 0].tolist() == [14.5, 15.5, 16.5] and vc[1, 0].tolist() == [17.5, 18.5, 19.5]
    untouched = np.ones((2, 4), bool)
    untouched[0, 2] = untouched[1, 0] = False
    assert np.all(kc[untouched] == -1.0) and np.all(vc[untouched] == -1.0)
    # a position out of range writes nothing and is counted
    kc2, vc2 = kc.copy(), vc.copy()
    assert orc.kv_write(y, [4, -1], 4, 3, kc2, vc2) == 2
    assert np.array_equal(kc2, kc) and np.array_equal(vc2, vc)


# ---------------------------------------------------------------- arg-max

def test_argmax_hand_vectors(orc):
    cases = [
        ([1.0, 3.0, 3.0, 2.0], 1),
        ([-0.0, 0.0], 0),
        ([0.0, -0.0, 0.0], 0),
        ([5.0], 0),
        ([-1.0, -1.0, -1.0], 0),
        ([-3.0, -2.0, -2.5], 1),
        ([1.0, 2.0, 4.0, 4.0, 8.0], 4),
        ([np.float32(1.0) + np.float32(2**-23), 1.0], 0),
        ([-np.inf, -np.inf, -np.inf], 0),
        ([-np.inf, -3.0e38, -np.inf], 1),
        ([np.inf, 1.0, np.inf], 0),
    ]
    for vals, want in cases:
        for dt in (np.float32, np.float64):
            tok, best = orc.argmax(np.array([vals], dt))
            assert tok[0] == want, (vals, dt)
            assert best[0] == max(vals)
    # NaN is no candidate; a row of NaN only gives index 0 and the value NaN
    nan = np.nan
    nan_cases = [
        ([nan, 1.0, 2.0, 2.0], 2, 2.0),
        ([1.0, nan, 0.5], 0, 1.0),
        ([nan, -np.inf, nan], 1, -np.inf),
        ([nan, nan, nan], 0, nan),
        ([-1.0, nan, -1.0], 0, -1.0),
    ]
    for vals, want, wbest in nan_cases:
        for dt in (np.float32, np.float64):
            tok, best = orc.argmax(np.array([vals], dt))
            assert tok[0] == want, (vals, dt)
            assert (np.isnan(best[0]) and np.isnan(wbest)) or best[0] == wbest, (vals, dt)


def test_planted_head_margin(orc):
    n, k, rows = 3000, 256, 16
    q, s, h, pos = synth.planted_head(9, n, k, rows)
    x, _ = orc.rmsnorm(h)
    for mode in ("f32", "i8", "i8x2"):
        tok, best, y = orc.head_argmax(mode, q, s, orc.quantize(mode, x))
        assert np.array_equal(tok, pos[np.arange(rows) % 8])
        top2 = np.sort(y, axis=1)[:, -2]
        assert np.all(best - top2 > 0.5 * best)


# --------------------------------------------------- RMSNorm near-tie report

def test_near_tie_classifier_at_known_distances(orc):
    # binary32 neighbours f and f + ulp; their midpoint is the rounding boundary
    for f in (1.0, 1.5 - 2.0**-23, 0.7390851, 3.0e-5, 1234.5):
        f = float(np.float32(f))
        ulp = float(np.spacing(np.float32(f)))
        mid = f + ulp / 2                           # exact in binary64
        assert orc.near_tie([mid])[0]
        for rel in (2.0**-45, 2.0**-41):
            assert orc.near_tie([mid * (1 + rel)])[0] and orc.near_tie([mid * (1 - rel)])[0]
        for rel in (2.0**-38, 2.0**-30):
            assert not orc.near_tie([mid * (1 + rel)])[0]
            assert not orc.near_tie([mid * (1 - rel)])[0]
        assert not orc.near_tie([f])[0]             # an f32 value: half an ulp away
    # across a binade boundary the midpoint below 2^k uses the smaller ulp
    mid_below = 2.0 - 2.0**-24
    assert orc.near_tie([mid_below])[0] and not orc.near_tie([2.0 - 2.0**-23])[0]
    assert not orc.near_tie([0.0])[0] and not orc.near_tie([np.inf])[0]


def test_near_tie_constructed_row(orc):
    # K = 32, eps = 0, h = (1 - 2^-19, 1, ..., 1): sum h^2 = 32 - 2^-18 + 2^-38
    # exactly, so r = (1 - 2^-23 + 2^-43)^(-1/2) = 1 + 2^-24 - 2^-44 + O(2^-46):
    # 2^-44 from the boundary 1 + 2^-24 between 1 and 1 + 2^-23
    h = np.ones((2, QK), np.float32)
    h[0, 0] = np.float32(1 - 2.0**-19)
    h[1, 0] = np.float32(1.25)                      # a row far from any boundary
    _, r = orc.rmsnorm(h, None, eps=0.0)
    ss = Fraction(float(h[0, 0])) ** 2 + 31
    m = ss / 32
    mid = 1 + Fraction(1, 2**24)
    # r lies between the two bounds 1/sqrt(m) is squeezed into
    assert abs(Fraction(float(r[0])) - mid) < Fraction(1, 2**43)
    assert (1 / (mid * mid) - m) != 0
    flags = orc.near_tie(r)
    assert flags[0] and not flags[1]
    # random RMSNorm rows are almost never near ties (about 2^-16 each)
    hr = synth.activations(np.random.default_rng(17), 64, 4096)
    _, rr = orc.rmsnorm(hr)
    assert orc.near_tie(rr).sum() == 0
