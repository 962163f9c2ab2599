"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test is chosen so that a plausible slip in the oracle (a wrong nibble
order, a dropped ``-8``, a swapped operand, a transposed index, ``sum``
instead of ``mean`` in RMSNorm, ``eps`` outside the square root, ``silu`` on
the wrong factor, a tie going to the wrong index) fails at least one of them:

* exhaustive decodes of every fp16 and bf16 bit pattern against numpy's own
  conversions (a library routine);
* the golden layout fixtures in ``tests/golden/`` and their closed forms;
* exact rational arithmetic (``fractions.Fraction``) on tiny products;
* a brute-force numpy decode with correctly rounded sums (``math.fsum``);
* one-hot activations, all-zero weights, power-of-two scalings;
* closed forms for RMSNorm of a constant vector and for the affine group-sum
  identity, and scipy's logistic function for SiLU.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import q4_workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_fixture(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split(":", 1)
            out[key.strip()] = val.split()
    return out


def _q4_0_weight(blocks, n, k):
    return oracle.HostWeight.q4_0(blocks, n, k)


def _aff_weight(a):
    return oracle.HostWeight.affine(a.nib, a.s, a.m, a.n, a.k)


# ------------------------------------------------------------------ decoders

def test_half_decode_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert math.copysign(1.0, oracle.half_to_f64(0x8000)) == -1.0


def test_bf16_decode_exhaustive():
    bits = np.arange(65536, dtype=np.uint32)
    ref = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    got = np.array([oracle.bf16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# ------------------------------------------------------------- layout pins

def test_q4_0_block_fixture_closed_form():
    fx = _read_fixture("q4_0_block.txt")
    blk = np.array([int(b, 16) for b in fx["bytes"]], dtype=np.uint8)
    assert blk.size == 18                       # 18 bytes per 32 weights
    w = oracle.dequant_row(_q4_0_weight(blk, 1, 32), 0)
    expect = [2.0 * (i - 8) for i in range(16)] + [2.0 * (7 - i) for i in range(16)]
    assert w.tolist() == expect


def test_affine_group_fixture_closed_form():
    fx = _read_fixture("affine_group.txt")
    nib = np.array([int(b, 16) for b in fx["nibbles"]], dtype=np.uint8)
    s = np.array([int(fx["s"][0], 16)], dtype=np.uint16)
    m = np.array([int(fx["m"][0], 16)], dtype=np.uint16)
    w = oracle.dequant_row(oracle.HostWeight.affine(nib, s, m, 1, 32), 0)
    expect = []
    for i in range(16):
        expect += [i - 0.5, 14.5 - i]
    assert w.tolist() == expect


def test_generator_layout_matches_fixture_reading():
    # The generator's packing puts element i and i+16 in byte i (Q4_0) and
    # elements 2i, 2i+1 in byte i (affine): decode of a known q gives it back.
    rng = np.random.default_rng(11)
    q = rng.integers(0, 16, size=(3, 64), dtype=np.uint8)
    d = np.full((3, 2), 0x3C00, dtype=np.uint16)           # d = 1.0
    W = _q4_0_weight(wl.pack_q4_0(q, d), 3, 64)
    assert np.array_equal(oracle.dequant(W), q.astype(np.float64) - 8.0)
    s = np.full((3, 2), 0x3F80, dtype=np.uint16)           # s = 1.0
    m = np.zeros((3, 2), dtype=np.uint16)                  # m = 0
    Wa = oracle.HostWeight.affine(wl.pack_affine_nibbles(q), s, m, 3, 64)
    assert np.array_equal(oracle.dequant(Wa), q.astype(np.float64))


# ------------------------------------------------------------ dot products

def _frac_half(bits):
    return Fraction(float(np.uint16(bits).view(np.float16)))


def _frac_bf16(bits):
    return Fraction(float(np.uint32(int(bits) << 16).view(np.float32)))


@pytest.mark.parametrize("n,k", [(1, 32), (2, 64), (3, 96)])
def test_q4_0_exact_rationals(n, k):
    rng = np.random.default_rng(100 + n)
    W = wl.draw_q4_0(rng, n, k)
    x = wl.draw_x(rng, 2, k)
    y, S = oracle.q4_gemv(_q4_0_weight(W.blocks, n, k), x)
    for r in range(2):
        for i in range(n):
            exact = Fraction(0)
            for b in range(k // 32):
                blk = W.blocks[i, b]
                d = _frac_half(int(blk[0]) | (int(blk[1]) << 8))
                for j in range(32):
                    q = (blk[2 + j] & 15) if j < 16 else (blk[2 + j - 16] >> 4)
                    exact += d * (int(q) - 8) * Fraction(float(x[r, b * 32 + j]))
            err = abs(Fraction(y[r, i]) - exact)
            assert err <= Fraction(k) * Fraction(2) ** -52 * Fraction(S[r, i])


@pytest.mark.parametrize("n,k", [(1, 32), (2, 64), (3, 96)])
def test_affine_exact_rationals(n, k):
    rng = np.random.default_rng(200 + n)
    A = wl.draw_affine(rng, n, k)
    x = wl.draw_x(rng, 2, k)
    y, S = oracle.q4_gemv(_aff_weight(A), x)
    for r in range(2):
        for i in range(n):
            exact = Fraction(0)
            for e in range(k):
                byte = int(A.nib[i, e // 2])
                q = (byte >> 4) if (e & 1) else (byte & 15)
                w = _frac_bf16(A.s[i, e // 32]) * q + _frac_bf16(A.m[i, e // 32])
                exact += w * Fraction(float(x[r, e]))
            err = abs(Fraction(y[r, i]) - exact)
            assert err <= Fraction(k) * Fraction(2) ** -52 * Fraction(S[r, i])


def _numpy_decode_q4_0(blocks):
    n, nbk, _ = blocks.shape
    d = blocks[:, :, 0].astype(np.uint16) | (blocks[:, :, 1].astype(np.uint16) << 8)
    dv = d.view(np.float16).astype(np.float64)
    lo = (blocks[:, :, 2:] & 0x0F).astype(np.int64)
    hi = (blocks[:, :, 2:] >> 4).astype(np.int64)
    q = np.concatenate([lo, hi], axis=2) - 8
    return (q * dv[:, :, None]).reshape(n, nbk * 32)


def _numpy_decode_affine(A):
    q = np.empty((A.n, A.k), dtype=np.int64)
    q[:, 0::2] = A.nib & 0x0F
    q[:, 1::2] = A.nib >> 4
    s = (A.s.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    m = (A.m.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return q * np.repeat(s, 32, axis=1) + np.repeat(m, 32, axis=1)


@pytest.mark.parametrize("fmt", ["q4_0", "affine"])
@pytest.mark.parametrize("n,k", [(16, 256), (7, 96), (5, 32)])
def test_brute_force_numpy_fsum(fmt, n, k):
    rng = np.random.default_rng(7 * n + k)
    if fmt == "q4_0":
        H = wl.draw_q4_0(rng, n, k)
        W = _q4_0_weight(H.blocks, n, k)
        wd = _numpy_decode_q4_0(H.blocks)
    else:
        H = wl.draw_affine(rng, n, k)
        W = _aff_weight(H)
        wd = _numpy_decode_affine(H)
    # every nibble value is present somewhere
    assert len(np.unique(np.rint(wd * 1e6))) > 16
    x = wl.draw_x(rng, 3, k)
    y, S = oracle.q4_gemv(W, x)
    for r in range(3):
        for i in range(n):
            ref = math.fsum(wd[i] * x[r].astype(np.float64))
            assert abs(y[r, i] - ref) <= k * 2.0 ** -53 * S[r, i]
            assert S[r, i] == pytest.approx(math.fsum(np.abs(wd[i] * x[r])), rel=1e-12)


@pytest.mark.parametrize("fmt", ["q4_0", "affine"])
def test_one_hot_picks_the_column(fmt):
    # N != K and nb rows with different one-hots catch transposed operands
    # and a wrong row order.
    n, k = 48, 96
    rng = np.random.default_rng(5)
    W = (_q4_0_weight(wl.draw_q4_0(rng, n, k).blocks, n, k) if fmt == "q4_0"
         else _aff_weight(wl.draw_affine(rng, n, k)))
    dense = oracle.dequant(W)
    cols = [0, 17, 31, 32, 95]
    x = np.zeros((len(cols), k), dtype=np.float32)
    for r, c in enumerate(cols):
        x[r, c] = 1.0
    y, _ = oracle.q4_gemv(W, x)
    for r, c in enumerate(cols):
        assert np.array_equal(y[r], dense[:, c])


def test_q4_0_all_eight_is_exact_zero():
    rng = np.random.default_rng(6)
    n, k = 9, 128
    q = np.full((n, k), 8, dtype=np.uint8)
    d = rng.uniform(0.005, 0.02, size=(n, k // 32)).astype(np.float16).view(np.uint16)
    W = _q4_0_weight(wl.pack_q4_0(q, d), n, k)
    y, S = oracle.q4_gemv(W, wl.draw_x(rng, 2, k))
    assert np.all(y == 0.0) and np.all(S == 0.0)


def test_q4_0_power_of_two_scalings_are_exact():
    rng = np.random.default_rng(8)
    n, k = 11, 160
    H = wl.draw_q4_0(rng, n, k)
    x = wl.draw_x(rng, 2, k)
    y, _ = oracle.q4_gemv(_q4_0_weight(H.blocks, n, k), x)
    b2 = H.blocks.copy()
    d = (b2[:, :, 0].astype(np.uint16) | (b2[:, :, 1].astype(np.uint16) << 8)) + 0x0400  # exponent + 1
    b2[:, :, 0] = (d & 0xFF).astype(np.uint8)
    b2[:, :, 1] = (d >> 8).astype(np.uint8)
    y2, _ = oracle.q4_gemv(_q4_0_weight(b2, n, k), x)
    assert np.array_equal(y2, 2.0 * y)
    y4, _ = oracle.q4_gemv(_q4_0_weight(H.blocks, n, k), 4.0 * x)
    assert np.array_equal(y4, 4.0 * y)


def test_q4_0_additive_in_x():
    rng = np.random.default_rng(9)
    n, k = 6, 64
    W = _q4_0_weight(wl.draw_q4_0(rng, n, k).blocks, n, k)
    x1, x2 = wl.draw_x(rng, 1, k), wl.draw_x(rng, 1, k)
    y1, S1 = oracle.q4_gemv(W, x1)
    y2, S2 = oracle.q4_gemv(W, x2)
    y12, _ = oracle.q4_gemv(W, x1.astype(np.float64) + x2.astype(np.float64))
    assert np.allclose(y12, y1 + y2, rtol=0, atol=1e-12 * (S1 + S2).max())


def test_affine_group_sum_identities():
    # w = s*q + m  =>  y = sum_g s_g * sum_j q_j x_j + m_g * gsum_g.
    rng = np.random.default_rng(10)
    n, k, G = 4, 128, 4
    x = wl.draw_x(rng, 2, k).astype(np.float64)
    gs = np.array([[math.fsum(x[r, 32 * g:32 * g + 32]) for g in range(G)] for r in range(2)])
    s = wl.f32_to_bf16_bits(rng.uniform(0.005, 0.02, (n, G)).astype(np.float32))
    m = wl.f32_to_bf16_bits(rng.uniform(-0.1, 0.0, (n, G)).astype(np.float32))
    sv = (s.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    mv = (m.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    # all q = 0 -> sum_g m_g gsum_g
    W0 = oracle.HostWeight.affine(np.zeros((n, k // 2), np.uint8), s, m, n, k)
    y0, _ = oracle.q4_gemv(W0, x)
    ref0 = gs @ mv.T
    assert np.allclose(y0, ref0, rtol=1e-13, atol=1e-14)
    # s = 0 gives the same whatever q is
    Ws = oracle.HostWeight.affine(rng.integers(0, 256, (n, k // 2), dtype=np.uint8),
                                  np.zeros_like(s), m, n, k)
    ys, _ = oracle.q4_gemv(Ws, x)
    assert np.allclose(ys, ref0, rtol=1e-13, atol=1e-14)
    # q = c in every group: sum_g (s_g c + m_g) gsum_g
    for c in (1, 7, 15):
        byte = np.uint8(c | (c << 4))
        Wc = oracle.HostWeight.affine(np.full((n, k // 2), byte, np.uint8), s, m, n, k)
        yc, _ = oracle.q4_gemv(Wc, x)
        refc = gs @ (sv * c + mv).T
        assert np.allclose(yc, refc, rtol=1e-12, atol=1e-13)
    # m = 0: pure scale, y = sum_g s_g * sum_j q_j x_j
    nib = rng.integers(0, 256, (n, k // 2), dtype=np.uint8)
    Wm = oracle.HostWeight.affine(nib, s, np.zeros_like(m), n, k)
    ym, _ = oracle.q4_gemv(Wm, x)
    q = np.empty((n, k)); q[:, 0::2] = nib & 15; q[:, 1::2] = nib >> 4
    refm = np.array([[sum(sv[i, g] * math.fsum(q[i, 32 * g:32 * g + 32] * x[r, 32 * g:32 * g + 32])
                          for g in range(G)) for i in range(n)] for r in range(2)])
    assert np.allclose(ym, refm, rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------------ RMSNorm

@pytest.mark.parametrize("eps", [1e-6, 0.5])
@pytest.mark.parametrize("k", [32, 2048])
def test_rmsnorm_constant_vector(eps, k):
    rng = np.random.default_rng(12)
    gamma = wl.draw_gamma(rng, k).astype(np.float64)
    for c in (3.0, -0.25, 1e-3):
        xh = oracle.rmsnorm(np.full((1, k), c), gamma, eps)
        ref = gamma * (c / math.sqrt(c * c + eps))
        assert np.allclose(xh[0], ref, rtol=1e-14, atol=0)


def test_rmsnorm_two_elements_and_scale_invariance():
    g = np.array([1.5, -2.0])
    xh = oracle.rmsnorm(np.array([[3.0, 4.0]]), g, 0.0)
    rms = math.sqrt((9.0 + 16.0) / 2.0)
    assert np.allclose(xh[0], [3.0 / rms * 1.5, 4.0 / rms * -2.0], rtol=1e-15)
    rng = np.random.default_rng(13)
    x = wl.draw_x(rng, 2, 256)
    gamma = wl.draw_gamma(rng, 256)
    a = oracle.rmsnorm(x, gamma, 1e-12)
    b = oracle.rmsnorm(1000.0 * x.astype(np.float64), gamma, 1e-12)
    assert np.allclose(a, b, rtol=1e-12, atol=0)


def test_nrm_gemv_constant_vector_closed_form():
    rng = np.random.default_rng(14)
    n, k, c, eps = 8, 64, 0.75, 1e-6
    W = _q4_0_weight(wl.draw_q4_0(rng, n, k).blocks, n, k)
    gamma = wl.draw_gamma(rng, k).astype(np.float64)
    y, _ = oracle.q4_nrm_gemv(W, np.full((1, k), c), gamma, eps)
    y2, _ = oracle.q4_gemv(W, gamma * (c / math.sqrt(c * c + eps)))
    assert np.allclose(y, y2, rtol=1e-13, atol=1e-15)


# ----------------------------------------------------------- SiLU, residual

def test_silu_against_logistic():
    scipy_special = pytest.importorskip("scipy.special")
    t = np.concatenate([np.linspace(-30, 30, 601), [0.0, 1e-8, -1e-8, 50.0, -50.0]])
    got = np.array([oracle.silu(v) for v in t])
    ref = t * scipy_special.expit(t)
    assert np.allclose(got, ref, rtol=1e-14, atol=1e-300)
    assert oracle.silu(0.0) == 0.0


def test_swiglu_factor_order():
    g = np.array([2.0, -1.0, 0.0])
    u = np.array([-3.0, 5.0, 7.0])
    h = oracle.swiglu(g, u)
    ref = [2.0 / (1.0 + math.exp(-2.0)) * -3.0, -1.0 / (1.0 + math.exp(1.0)) * 5.0, 0.0]
    assert np.allclose(h, ref, rtol=1e-15)


def test_gus_zero_gate_or_up_gives_zero():
    rng = np.random.default_rng(15)
    n, k = 16, 64
    zeros = _q4_0_weight(wl.pack_q4_0(np.full((n, k), 8, np.uint8),
                                      np.full((n, k // 32), 0x3C00, np.uint16)), n, k)
    W = _q4_0_weight(wl.draw_q4_0(rng, n, k).blocks, n, k)
    x = wl.draw_x(rng, 1, k)
    gamma = wl.draw_gamma(rng, k)
    h, *_ = oracle.q4_gus_nrm(zeros, W, x, gamma, 1e-6)
    assert np.all(h == 0.0)
    h, *_ = oracle.q4_gus_nrm(W, zeros, x, gamma, 1e-6)
    assert np.all(h == 0.0)


def test_residual_cases():
    rng = np.random.default_rng(16)
    n, k = 12, 96
    H = wl.draw_q4_0(rng, n, k)
    W = _q4_0_weight(H.blocks, n, k)
    x = wl.draw_x(rng, 2, k)
    y0, _ = oracle.q4_gemv(W, x)
    y, _ = oracle.q4_res_gemv(W, x, np.zeros((2, n)))
    assert np.array_equal(y, y0)
    r = wl.draw_x(rng, 2, n)
    zero = _q4_0_weight(wl.pack_q4_0(np.full((n, k), 8, np.uint8),
                                     np.full((n, k // 32), 0x3C00, np.uint16)), n, k)
    yz, _ = oracle.q4_res_gemv(zero, x, r)
    assert np.array_equal(yz, r.astype(np.float64))


def test_dual_is_two_gemvs():
    rng = np.random.default_rng(17)
    k = 64
    Wa = _q4_0_weight(wl.draw_q4_0(rng, 16, k).blocks, 16, k)
    Wb = _q4_0_weight(wl.draw_q4_0(rng, 8, k).blocks, 8, k)
    x = wl.draw_x(rng, 1, k)
    gamma = wl.draw_gamma(rng, k)
    ya, _, yb, _ = oracle.q4_dual_gemv(Wa, Wb, x, gamma, 1e-6)
    ra, _ = oracle.q4_nrm_gemv(Wa, x, gamma, 1e-6)
    rb, _ = oracle.q4_nrm_gemv(Wb, x, gamma, 1e-6)
    assert np.array_equal(ya, ra) and np.array_equal(yb, rb)


# ------------------------------------------------------------------- argmax

def test_argmax_matches_numpy_first_max():
    rng = np.random.default_rng(18)
    cases = [rng.standard_normal(1000),
             np.array([1.0, 3.0, 3.0, 2.0]),
             np.full(17, -4.0),
             np.array([-np.inf, -1e300, -1e300]),
             np.concatenate([np.zeros(50), [5.0], np.zeros(50), [5.0]])]
    for v in cases:
        assert oracle.argmax(v) == int(np.argmax(v))


def test_argmax_planted_unique_max():
    rng = np.random.default_rng(19)
    n, k = 64, 32
    q = rng.integers(0, 16, (n, k), dtype=np.uint8)
    q[41, :] = 15                         # row 41 dominates for a positive x
    d = np.full((n, 1), 0x3C00, np.uint16)
    W = _q4_0_weight(wl.pack_q4_0(q, d), n, k)
    idx, logits, _ = oracle.q4_argmax(W, np.ones((1, k), np.float32))
    assert idx[0] == 41 == int(np.argmax(logits[0]))


@pytest.mark.parametrize("fmt", ["q4_0", "affine"])
def test_threaded_rows_give_the_same_bits(fmt):
    # the CPU baseline runs the oracle's rows on several threads: every
    # output must be the same bits as the single-threaded walk
    rng = np.random.default_rng(5)
    H = wl.draw_q4_0(rng, 333, 256) if fmt == "q4_0" else wl.draw_affine(rng, 333, 256)
    W = oracle._hw(H)
    x = wl.draw_x(rng, 3, 256)
    y1, S1 = oracle.gemv(W, x)
    old = oracle.set_threads(7)
    try:
        y7, S7 = oracle.gemv(W, x)
    finally:
        oracle.set_threads(old)
    assert np.array_equal(y1, y7) and np.array_equal(S1, S7)


def test_halfset_rows_interleave_and_decode():
    # HalfSet reading: element 2i of a row from the even stream, 2i+1 from
    # the odd one; every f16 bit pattern decodes as numpy's float16 does
    rng = np.random.default_rng(6)
    bits = rng.integers(0, 1 << 16, size=(4, 256), dtype=np.uint16)
    bits[(bits & 0x7C00) == 0x7C00] = 0x3C00          # finite values only (no inf / NaN)
    x = oracle.halfset_rows(bits[:, 0::2], bits[:, 1::2])
    assert np.array_equal(x, bits.view(np.float16).astype(np.float64))


def test_halfset_gemv_one_hot_and_equivalence():
    rng = np.random.default_rng(7)
    n, k = 40, 128
    H = wl.draw_q4_0(rng, n, k)
    W = oracle._hw(H)
    dense = oracle.dequant(W)
    # a one in the even stream at i is column 2i, in the odd stream column 2i + 1
    for i in (0, 5, 63):
        e = np.zeros((1, k // 2), np.float16)
        o = np.zeros((1, k // 2), np.float16)
        e[0, i] = 1.0
        y, _ = oracle.q4_gemv_half(W, e.view(np.uint16), o.view(np.uint16))
        assert np.array_equal(y[0], dense[:, 2 * i])
        y, _ = oracle.q4_gemv_half(W, o.view(np.uint16), e.view(np.uint16))
        assert np.array_equal(y[0], dense[:, 2 * i + 1])
    # and the HalfSet of f16 activations gives the plain GEMV of those values
    x16 = rng.standard_normal((3, k)).astype(np.float16)
    y1, S1 = oracle.q4_gemv_half(W, x16[:, 0::2].view(np.uint16), x16[:, 1::2].view(np.uint16))
    y2, S2 = oracle.q4_gemv(W, x16.astype(np.float64))
    assert np.array_equal(y1, y2) and np.array_equal(S1, S2)


def test_q8_0_decode_every_byte():
    # every signed byte value, against numpy's own int8 and float16 reading
    rng = np.random.default_rng(8)
    n, k = 8, 256
    q = np.arange(-128, 128, dtype=np.int16).reshape(8, 32)
    q = np.repeat(q[:, None, :], k // 32, axis=1).reshape(n, k)
    d = rng.uniform(0.0003, 0.0012, (n, k // 32)).astype(np.float16)
    H = wl.Q8_0Host(n, k, wl.pack_q8_0(q, d.view(np.uint16)))
    blk = H.blocks8
    ref = blk[:, :, 0:2].copy().view("<f2")[:, :, 0].astype(np.float64)[:, :, None] * \
        blk[:, :, 2:].view(np.int8).astype(np.float64)
    assert np.array_equal(oracle.dequant(oracle._hw(H)), ref.reshape(n, k))


def test_q8_0_upcast_of_q4_0_is_the_same_matrix():
    # crate inferencelayer, q4_0_to_q8_0n: the upcast keeps d and maps a
    # nibble q to q - 8, so both decoders must give the same weights
    rng = np.random.default_rng(9)
    H = wl.draw_q4_0(rng, 33, 160)
    H8 = wl.q4_0_to_q8_0(H)
    assert np.array_equal(oracle.dequant(oracle._hw(H)), oracle.dequant(oracle._hw(H8)))
    x = wl.draw_x(rng, 2, 160)
    assert np.array_equal(oracle.q4_gemv(oracle._hw(H), x)[0], oracle.q4_gemv(oracle._hw(H8), x)[0])


def test_q8_0_brute_force_fsum():
    rng = np.random.default_rng(10)
    H = wl.draw_q8_0(rng, 12, 96)
    x = wl.draw_x(rng, 2, 96)
    y, S = oracle.q4_gemv(oracle._hw(H), x)
    blk = H.blocks8
    dense = (blk[:, :, 0:2].copy().view("<f2")[:, :, 0].astype(np.float64)[:, :, None] *
             blk[:, :, 2:].view(np.int8).astype(np.float64)).reshape(12, 96)
    for r in range(2):
        for i in range(12):
            terms = dense[i] * x[r].astype(np.float64)
            assert abs(y[r, i] - math.fsum(terms)) <= 1e-12 * math.fsum(np.abs(terms))
            assert abs(S[r, i] - math.fsum(np.abs(terms))) <= 1e-12 * S[r, i]


# ---- Q4_K superblocks (crate inferencelayer, gemv_q5k_k_lcpp_src: f16 d and
# dmin, 12 bytes of 6-bit sub-scales and sub-mins, 128 nibble bytes;
# w = d*sc*q - dmin*mn).  The generator's bit-position table is written from
# the pack's description independently of the oracle's shift-and-mask decoder.

def test_q4_k_scale_table_is_a_bijection():
    # every one of the 96 bits of the 12 scale bytes holds exactly one bit of
    # one field
    pos = wl.Q4K_SCALE_BITS.reshape(-1, 2)
    flat = pos[:, 0] * 8 + pos[:, 1]
    assert sorted(flat.tolist()) == list(range(96))


@pytest.mark.parametrize("j", range(8))
def test_q4_k_scale_min_every_value(j):
    # every 6-bit value of both fields of sub-block j, the other fields random
    rng = np.random.default_rng(100 + j)
    for v in range(64):
        sc = rng.integers(0, 64, size=8)
        mn = rng.integers(0, 64, size=8)
        sc[j], mn[j] = v, 63 - v
        q = np.zeros((1, 256), dtype=np.uint8)
        blk = wl.pack_q4_k(q, sc[None], mn[None], np.zeros((1, 1), np.uint16), np.zeros((1, 1), np.uint16))
        for jj in range(8):
            assert oracle.q4_k_scale_min(blk[0, 0, 4:16], jj) == (sc[jj], mn[jj])


def test_q4_k_value_formula_exact():
    # each weight is d*sc*q - dmin*mn with one rounding (exact rationals)
    rng = np.random.default_rng(110)
    n, k = 6, 512
    q = rng.integers(0, 16, size=(n, k), dtype=np.uint8)
    sc = rng.integers(0, 64, size=(n, k // 32))
    mn = rng.integers(0, 64, size=(n, k // 32))
    d = rng.uniform(1e-4, 4e-4, (n, k // 256)).astype(np.float16)
    dm = rng.uniform(2e-4, 8e-4, (n, k // 256)).astype(np.float16)
    H = wl.Q4_KHost(n, k, wl.pack_q4_k(q, sc, mn, d.view(np.uint16), dm.view(np.uint16)))
    W = oracle.dequant(oracle._hw(H))
    for i in range(n):
        for e in range(0, k, 7):
            exact = (Fraction(float(d[i, e // 256])) * int(sc[i, e // 32]) * int(q[i, e])
                     - Fraction(float(dm[i, e // 256])) * int(mn[i, e // 32]))
            assert W[i, e] == float(exact)


def test_q4_k_nibble_order_one_hot():
    # row e of a 256 x 256 matrix has nibble 15 at element e and 0 elsewhere,
    # every scale 1, every min 0, d = 1: the decode is 15 * identity
    n = k = 256
    q = np.eye(n, k, dtype=np.uint8) * 15
    one = np.full((n, 1), np.float16(1.0)).view(np.uint16)
    H = wl.Q4_KHost(n, k, wl.pack_q4_k(q, np.ones((n, 8), int), np.zeros((n, 8), int), one,
                                       np.zeros((n, 1), np.uint16)))
    assert np.array_equal(oracle.dequant(oracle._hw(H)), 15.0 * np.eye(n))


def test_q4_k_equals_q4_0_with_shared_scale():
    # Q4_0 blocks whose eight scales in a superblock are equal are the Q4_K
    # superblock with d = dmin = that scale, every sc = 1 and every mn = 8:
    # d*q - 8d = d*(q - 8)
    rng = np.random.default_rng(111)
    n, k = 9, 512
    q = rng.integers(0, 16, size=(n, k), dtype=np.uint8)
    d = rng.uniform(0.005, 0.02, (n, k // 256)).astype(np.float16)
    H0 = wl.Q4_0Host(n, k, wl.pack_q4_0(q, np.repeat(d, 8, axis=1).view(np.uint16)))
    HK = wl.Q4_KHost(n, k, wl.pack_q4_k(q, np.ones((n, k // 32), int), np.full((n, k // 32), 8),
                                        d.view(np.uint16), d.view(np.uint16)))
    assert np.array_equal(oracle.dequant(oracle._hw(H0)), oracle.dequant(oracle._hw(HK)))


def test_q4_k_brute_force_fsum():
    rng = np.random.default_rng(112)
    n, k = 10, 256
    q = rng.integers(0, 16, size=(n, k), dtype=np.uint8)
    sc = rng.integers(0, 64, size=(n, k // 32))
    mn = rng.integers(0, 64, size=(n, k // 32))
    d = rng.uniform(1e-4, 4e-4, (n, 1)).astype(np.float16)
    dm = rng.uniform(2e-4, 8e-4, (n, 1)).astype(np.float16)
    H = wl.Q4_KHost(n, k, wl.pack_q4_k(q, sc, mn, d.view(np.uint16), dm.view(np.uint16)))
    x = wl.draw_x(rng, 2, k)
    y, S = oracle.q4_gemv(oracle._hw(H), x)
    dense = (d.astype(np.float64) * np.repeat(sc, 32, axis=1) * q
             - dm.astype(np.float64) * np.repeat(mn, 32, axis=1))
    for r in range(2):
        for i in range(n):
            terms = dense[i] * x[r].astype(np.float64)
            assert abs(y[r, i] - math.fsum(terms)) <= 1e-12 * math.fsum(np.abs(terms))
            assert abs(S[r, i] - math.fsum(np.abs(terms))) <= 1e-12 * S[r, i]


# ---- Q1 sign-bit superblocks (crate inferencelayer, gemv_q1_k_lcpp_src:
# bit i of a weight word is element i's sign, 1 -> +1, 0 -> -1; one f16 scale
# per 128 weights; 4.5 bytes per 32 weights)

def test_q1_every_byte_value():
    # every value of every sign byte, against numpy's own little-endian bit
    # reading and float16 decode
    rng = np.random.default_rng(120)
    n, k = 16, 2048
    blocks = np.empty((n, k // 128, 18), np.uint8)
    blocks[:, :, 2:] = np.arange(256, dtype=np.uint8).reshape(1, 16, 16).repeat(n, 0)
    d = rng.uniform(0.02, 0.06, (n, k // 128)).astype(np.float16)
    blocks[:, :, 0:2] = d.view(np.uint8).reshape(n, k // 128, 2)
    H = wl.Q1Host(n, k, blocks)
    bits = np.unpackbits(blocks[:, :, 2:], axis=2, bitorder="little").astype(np.float64)
    ref = (2.0 * bits - 1.0) * d.astype(np.float64)[:, :, None]
    assert np.array_equal(oracle.dequant(oracle._hw(H)), ref.reshape(n, k))
    # 16 bytes per superblock of 128, two of scale: 4.5 bytes per 32 weights
    assert blocks.size / (n * k / 32) == 4.5


def test_q1_sign_convention_and_positions():
    # all bits set is +d, none is -d; a single set bit lands on its element
    n, k = 130, 128
    bits = np.zeros((n, k), np.uint8)
    bits[0] = 1
    for e in range(k):
        bits[2 + e, e] = 1
    d = np.full((n, 1), np.float16(0.5)).view(np.uint16)
    W = oracle.dequant(oracle._hw(wl.Q1Host(n, k, wl.pack_q1(bits, d))))
    assert np.all(W[0] == 0.5) and np.all(W[1] == -0.5)
    assert np.array_equal(W[2:], np.where(np.eye(k, dtype=bool), 0.5, -0.5))


def test_q1_equals_q8_0_of_signs():
    # a Q1 superblock is the four Q8_0 blocks with the same d and q = +-1
    rng = np.random.default_rng(121)
    n, k = 21, 512
    bits = rng.integers(0, 2, (n, k), dtype=np.uint8)
    d = rng.uniform(0.02, 0.06, (n, k // 128)).astype(np.float16)
    H1 = wl.Q1Host(n, k, wl.pack_q1(bits, d.view(np.uint16)))
    H8 = wl.Q8_0Host(n, k, wl.pack_q8_0(2 * bits.astype(np.int16) - 1, np.repeat(d, 4, axis=1).view(np.uint16)))
    assert np.array_equal(oracle.dequant(oracle._hw(H1)), oracle.dequant(oracle._hw(H8)))


def test_q1_brute_force_fsum():
    rng = np.random.default_rng(122)
    H = wl.draw_q1(rng, 11, 384)
    x = wl.draw_x(rng, 3, 384)
    y, S = oracle.q4_gemv(oracle._hw(H), x)
    b = H.blocks1
    signs = 2.0 * np.unpackbits(b[:, :, 2:], axis=2, bitorder="little").astype(np.float64) - 1.0
    dense = (signs * b[:, :, 0:2].copy().view("<f2").astype(np.float64)).reshape(11, 384)
    for r in range(3):
        for i in range(11):
            terms = dense[i] * x[r].astype(np.float64)
            assert abs(y[r, i] - math.fsum(terms)) <= 1e-12 * math.fsum(np.abs(terms))
            assert abs(S[r, i] - math.fsum(np.abs(terms))) <= 1e-12 * S[r, i]


# ---- decode attention (honeycrisp/mod.rs: attn_state, gpu_attention and the
# fused RoPE + KV-append + SDPA dispatch)

def _attn_case(rng, H=8, Hkv=2, d=64, max_seq=48, position=29):
    q = rng.standard_normal((H, d))
    kn, vn = rng.standard_normal((Hkv, d)), rng.standard_normal((Hkv, d))
    kc = rng.standard_normal((Hkv, max_seq, d))
    vc = rng.standard_normal((Hkv, max_seq, d))
    kc[:, position + 1:] = np.nan       # never read: beyond the token
    vc[:, position + 1:] = np.nan
    return q, kn, vn, kc, vc


@pytest.mark.parametrize("window", [0, 1, 3, 30, 100])
def test_attn_brute_force_softmax(window):
    from scipy.special import softmax
    rng = np.random.default_rng(130 + window)
    H, Hkv, d, pos, scale = 8, 2, 64, 29, 0.125
    q, kn, vn, kc, vc = _attn_case(rng, H, Hkv, d, position=pos)
    out, bound, kc2, vc2 = oracle.attn_decode(q, kn, vn, kc, vc, pos, window, scale)
    # the append, and nothing else written
    assert np.array_equal(kc2[:, pos], kn) and np.array_equal(vc2[:, pos], vn)
    assert np.array_equal(kc2[:, :pos], kc[:, :pos]) and np.array_equal(vc2[:, :pos], vc[:, :pos])
    lo = max(0, pos + 1 - window) if window > 0 else 0
    G = H // Hkv
    for h in range(H):
        K, V = kc2[h // G, lo:pos + 1], vc2[h // G, lo:pos + 1]
        p = softmax(scale * (K @ q[h]))
        for e in range(0, d, 5):
            terms = p * V[:, e]
            assert abs(out[h, e] - math.fsum(terms)) <= 1e-12 * (1 + math.fsum(np.abs(terms)))
            assert abs(bound[h, e] - math.fsum(np.abs(terms))) <= 1e-12 * (1 + bound[h, e])


def test_attn_zero_query_is_the_window_mean():
    rng = np.random.default_rng(140)
    q, kn, vn, kc, vc = _attn_case(rng)
    out, _, _, vc2 = oracle.attn_decode(np.zeros_like(q), kn, vn, kc, vc, 29, 7, 0.3)
    for h in range(8):
        assert np.allclose(out[h], vc2[h // 4, 23:30].mean(axis=0), rtol=0, atol=1e-12)


def test_attn_gqa_grouping():
    # V of kv head j is the constant j + 1: consecutive query heads share one
    rng = np.random.default_rng(141)
    H, Hkv = 12, 3
    q, kn, vn, kc, vc = _attn_case(rng, H, Hkv)
    for j in range(Hkv):
        vc[j, :30] = j + 1.0
        vn[j] = j + 1.0
    out, _, _, _ = oracle.attn_decode(q, kn, vn, kc, vc, 29, 0, 0.2)
    for h in range(H):
        assert np.allclose(out[h], h // 4 + 1.0, rtol=0, atol=1e-12)


def test_attn_large_scale_is_the_argmax_row():
    rng = np.random.default_rng(142)
    q, kn, vn, kc, vc = _attn_case(rng)
    out, _, kc2, vc2 = oracle.attn_decode(q, kn, vn, kc, vc, 29, 0, 1e4)
    for h in range(8):
        t = int(np.argmax(kc2[h // 4, :30] @ q[h]))
        assert np.allclose(out[h], vc2[h // 4, t], rtol=0, atol=1e-9)


def test_rope_table_and_rotation():
    # the table against the pages' angle pos / theta^(2j/d), computed here
    # with numpy's vectorised functions
    c, s = oracle.rope_table(64, 16, 10000.0)
    ang = np.arange(64)[:, None] / 10000.0 ** (2.0 * np.arange(8)[None, :] / 16)
    assert np.allclose(c, np.cos(ang), rtol=0, atol=1e-15) and np.allclose(s, np.sin(ang), rtol=0, atol=1e-15)
    # a hand-worked rotation: d = 4, angles pi/2 and 0; element j pairs with j + 2
    x = oracle.rope_apply([1.0, 2.0, 3.0, 4.0], [0.0, 1.0], [1.0, 0.0])
    assert np.array_equal(x, [-3.0, 2.0, 1.0, 4.0])
    # rotations preserve each pair's norm, position 0 is the identity, and
    # dot products depend only on the position difference
    rng = np.random.default_rng(143)
    c, s = oracle.rope_table(512, 64, 10000.0)
    a, b = rng.standard_normal(64), rng.standard_normal(64)
    assert np.array_equal(oracle.rope_apply(a, c[0], s[0]), a)
    ra = oracle.rope_apply(a, c[77], s[77])
    assert np.allclose(ra[:32] ** 2 + ra[32:] ** 2, a[:32] ** 2 + a[32:] ** 2, rtol=1e-13)
    for p1, p2, dlt in [(5, 3, 100), (300, 17, 150), (40, 40, 471)]:
        d1 = oracle.rope_apply(a, c[p1], s[p1]) @ oracle.rope_apply(b, c[p2], s[p2])
        d2 = oracle.rope_apply(a, c[p1 + dlt], s[p1 + dlt]) @ oracle.rope_apply(b, c[p2 + dlt], s[p2 + dlt])
        assert abs(d1 - d2) <= 1e-11


def test_attn_rotates_q_and_appended_k():
    rng = np.random.default_rng(144)
    q, kn, vn, kc, vc = _attn_case(rng)
    c, s = oracle.rope_table(48, 64, 10000.0)
    out, bound, kc2, _ = oracle.attn_decode(q, kn, vn, kc, vc, 29, 0, 0.125, c, s)
    for j in range(2):
        assert np.allclose(kc2[j, 29], oracle.rope_apply(kn[j], c[29], s[29]), rtol=0, atol=0)
    # the same as attending with pre-rotated q and k and no tables
    qr = np.stack([oracle.rope_apply(q[h], c[29], s[29]) for h in range(8)])
    kr = np.stack([oracle.rope_apply(kn[j], c[29], s[29]) for j in range(2)])
    out2, bound2, _, _ = oracle.attn_decode(qr, kr, vn, kc, vc, 29, 0, 0.125)
    assert np.array_equal(out, out2) and np.array_equal(bound, bound2)
