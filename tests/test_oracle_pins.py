"""Pins for the CPU oracle: each test checks the oracle against something other
than itself -- the pages' E2M1 definition (golden fixtures), exact rational
arithmetic, brute force on tiny inputs, closed forms and invariants.  CPU only.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import fp4_linear as orc
from precision_gemm_row_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------- exact references

_GRID_F = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3),
           Fraction(4), Fraction(6)]


def _nearest_code_exact(y: float) -> int:
    """Nearest E2M1 magnitude by exact rational distance, ties to the even code,
    sign bit from y's sign.  Independent of the oracle's fp64 arithmetic."""
    mag = abs(Fraction(float(y)))
    best_d, best_c = None, None
    for c, g in enumerate(_GRID_F):
        d = abs(mag - g)
        if best_d is None or d < best_d or (d == best_d and c % 2 == 0):
            best_d, best_c = d, c
    return best_c | (8 if math.copysign(1.0, float(y)) < 0 else 0)


def _all_finite_bf16():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    exp = (bits >> 7) & 0xFF
    return bits[exp != 0xFF]


# ---------------------------------------------------------------- E2M1 format

def test_e2m1_decode_matches_golden_table():
    rows = _read_table("e2m1_codes.txt")
    assert len(rows) == 16
    for code, sign, exp, man, val in rows:
        code = int(code)
        assert (code >> 3) & 1 == int(sign)
        assert (code >> 1) & 3 == int(exp)
        assert code & 1 == int(man)
        assert orc.e2m1_decode(code) == float(val)
        assert math.copysign(1.0, orc.DECODE[code]) == math.copysign(1.0, float(val))


def test_e2m1_rounding_golden_cases():
    for y, code in _read_table("e2m1_rounding.txt"):
        got = int(orc.e2m1_round(np.array([np.float32(y)]))[0])
        assert got == int(code), (y, got, code)


def test_e2m1_round_exhaustive_bf16_exact_rational():
    # every finite BF16 value as the scaled input y (scale 1)
    bits = _all_finite_bf16()
    y = orc.bf16_to_f32(bits)
    got = orc.e2m1_round(y)
    want = np.array([_nearest_code_exact(v) for v in y.tolist()], dtype=np.uint8)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(y[i]), int(got[i]), int(want[i])) for i in bad[:10]]


@pytest.mark.parametrize("absmax", [1.0, 3.0, 0.7, 20.0, 2.0 ** -10, 1e-3, 65504.0, 7.123])
def test_e2m1_round_scaled_samples_exact_rational(absmax):
    rng = np.random.default_rng(123)
    bits = rng.choice(_all_finite_bf16(), size=3000)
    x = orc.bf16_to_f32(bits)
    s = orc.absmax_scale(np.array([absmax], dtype=np.float32))[0]
    with np.errstate(over="ignore"):
        y = x * s                               # fp32 products, as the quantizer forms them
    y = y[np.isfinite(y)]                       # |x| <= absmax keeps real inputs finite
    got = orc.e2m1_round(y)
    want = np.array([_nearest_code_exact(v) for v in y.tolist()], dtype=np.uint8)
    assert np.array_equal(got, want)


def test_scale_is_correctly_rounded_6_over_absmax():
    rng = np.random.default_rng(7)
    absmax = np.abs(orc.bf16_to_f32(rng.choice(_all_finite_bf16(), size=2000)))
    absmax = absmax[(absmax > 2.0 ** -120) & (absmax < 2.0 ** 120)]
    s = orc.absmax_scale(absmax)
    for a, sv in zip(absmax.tolist(), s.tolist()):
        exact = Fraction(6) / Fraction(a)
        half_ulp = Fraction(float(np.spacing(np.float32(sv)))) / 2
        assert abs(Fraction(sv) - exact) <= half_ulp
    # degenerate rows: zero and subnormal absmax give scale 1
    z = orc.absmax_scale(np.array([0.0, 1e-45], dtype=np.float32))
    assert z.tolist() == [1.0, 1.0]


# ---------------------------------------------------------------- row / column quantization

def _bf16_matrix(rng, shape, std=1.0):
    return wl.f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32) * np.float32(std))


def test_quantize_rows_bruteforce_small():
    rng = np.random.default_rng(0)
    A = orc.bf16_to_f32(_bf16_matrix(rng, (5, 12)))
    A[2] = 0.0
    A[3, 4] = -0.0
    codes, s = orc.quantize_rows(A)
    for i in range(A.shape[0]):
        row = A[i].tolist()
        amax = max(abs(v) for v in row)
        si = np.float32(1.0) if amax == 0 else np.float32(6.0) / np.float32(amax)
        assert s[i] == si
        for j, v in enumerate(row):
            c = int(codes[i, j // 2] >> (4 * (j % 2))) & 0xF
            assert c == _nearest_code_exact(float(np.float32(v) * si))


def test_quantize_cols_is_per_column_bruteforce():
    rng = np.random.default_rng(1)
    W = orc.bf16_to_f32(_bf16_matrix(rng, (8, 6), 0.02))
    W[:, 2] *= 50.0                         # one column with a distinct range
    codes_t, s = orc.quantize_cols(W)
    assert codes_t.shape == (6, 4) and s.shape == (6,)
    for j in range(6):
        amax = float(np.max(np.abs(W[:, j])))
        assert s[j] == np.float32(6.0) / np.float32(amax)
        for k in range(8):
            c = int(codes_t[j, k // 2] >> (4 * (k % 2))) & 0xF
            assert c == _nearest_code_exact(float(W[k, j] * s[j]))


def test_dequantized_values_on_grid_and_within_half_spacing():
    rng = np.random.default_rng(2)
    A = orc.bf16_to_f32(_bf16_matrix(rng, (64, 256)))
    codes, s = orc.quantize_rows(A)
    deq = orc.dequantize(codes, s)
    y = (A * s[:, None]).astype(np.float64)             # the quantizer's fp32 input
    q = orc.DECODE[orc.unpack_codes(codes)]
    assert np.all(np.isin(np.abs(q), orc.GRID))
    assert np.array_equal(deq, q / s[:, None].astype(np.float64))   # on the grid scaled by 1/s
    mag = np.abs(y)
    half = np.where(mag < 2, 0.25, np.where(mag < 4, 0.5, 1.0))
    assert np.all(np.abs(np.abs(q) - np.minimum(mag, 6.0)) <= half + 1e-6)
    # the largest element of every row lands on +-6 when 6/absmax * absmax rounds to 6
    idx = np.argmax(np.abs(A), axis=1)
    top = A[np.arange(64), idx] * s
    hit = np.abs(top) == np.float32(6.0)
    assert np.all(np.abs(q[np.arange(64), idx][hit]) == 6.0)


def test_lossless_grid_matrices_give_exact_product():
    # values on the E2M1 grid, every row / column reaching |6| times a power of two:
    # quantization is then lossless and the scaled FP4 GEMM equals A @ W exactly.
    rng = np.random.default_rng(3)
    M, K, N = 6, 16, 5
    A = rng.choice(orc.DECODE, size=(M, K))
    A[:, 0] = 6.0
    A *= 2.0 ** rng.integers(-3, 4, size=(M, 1))
    W = rng.choice(orc.DECODE, size=(K, N))
    W[1, :] = -6.0
    W *= 2.0 ** rng.integers(-5, 2, size=(1, N))
    a_codes, s_a = orc.quantize_rows(A.astype(np.float32))
    w_codes_t, s_w = orc.quantize_cols(W.astype(np.float32))
    Y = orc.linear_fwd(a_codes, s_a, w_codes_t, s_w)
    assert np.array_equal(Y, A @ W)


# ---------------------------------------------------------------- GEMM

def test_gemm_raw_bruteforce_fractions():
    rng = np.random.default_rng(4)
    M, K, N = 3, 10, 4
    a = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    w = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)

    def val(packed, r, k):
        c = int(packed[r, k // 2] >> (4 * (k % 2))) & 0xF
        return Fraction(orc.e2m1_decode(c))

    acc = orc.gemm_raw(a, w)
    for i in range(M):
        for j in range(N):
            ref = sum(val(a, i, k) * val(w, j, k) for k in range(K))
            assert Fraction(acc[i, j]) == ref


def test_gemm_raw_sampled_rows_cols_match_full():
    rng = np.random.default_rng(5)
    a = rng.integers(0, 256, size=(9, 32), dtype=np.uint8)
    w = rng.integers(0, 256, size=(7, 32), dtype=np.uint8)
    full = orc.gemm_raw(a, w)
    assert np.array_equal(orc.gemm_raw(a, w, rows=[8, 0, 3], cols=[6, 1]), full[np.ix_([8, 0, 3], [6, 1])])


def test_epilogue_unit_scales_is_raw_accumulator():
    rng = np.random.default_rng(6)
    a = rng.integers(0, 256, size=(4, 8), dtype=np.uint8)
    w = rng.integers(0, 256, size=(5, 8), dtype=np.uint8)
    Y = orc.linear_fwd(a, np.ones(4, np.float32), w, np.ones(5, np.float32))
    assert np.array_equal(Y, orc.gemm_raw(a, w))


def test_compensation_term_is_dA_times_W():
    rng = np.random.default_rng(8)
    M, K, N = 16, 32, 12
    A_bits = wl.f32_to_bf16_bits(rng.standard_t(3, size=(M, K)).astype(np.float32))
    W_bits = _bf16_matrix(rng, (K, N), 0.02)
    t, _, _ = orc.quantile_threshold(A_bits, 0.9)
    A_c, rp, ci, vals = orc.clamp_and_compensation(A_bits, t)
    a_codes, s_a = orc.quantize_rows(A_c)
    w_codes_t, s_w = orc.quantize_cols(orc.bf16_to_f32(W_bits))
    y0 = orc.linear_fwd(a_codes, s_a, w_codes_t, s_w)
    y1 = orc.linear_fwd(a_codes, s_a, w_codes_t, s_w, rp, ci, vals, W_bits)
    Wd = orc.bf16_to_f32(W_bits).astype(np.float64)
    dA = np.zeros((M, K))
    for i in range(M):
        for e in range(rp[i], rp[i + 1]):
            dA[i, ci[e]] += vals[e]
    assert rp[-1] > 0
    np.testing.assert_allclose(y1 - y0, dA @ Wd, rtol=0, atol=1e-12)
    # an empty dA changes nothing
    empty = np.zeros(M + 1, np.int32)
    y2 = orc.linear_fwd(a_codes, s_a, w_codes_t, s_w, empty, ci[:0], vals[:0], W_bits)
    assert np.array_equal(y2, y0)


def _magnitude_case(seed=21, M=5, K=32, N=6, q=0.8):
    """A tiny compensated layer with several dA entries per row (Student-t A)."""
    rng = np.random.default_rng(seed)
    A_bits = wl.f32_to_bf16_bits(rng.standard_t(3, size=(M, K)).astype(np.float32))
    W_bits = _bf16_matrix(rng, (K, N), 0.02)
    t, _, _ = orc.quantile_threshold(A_bits, q)
    A_c, rp, ci, cv = orc.clamp_and_compensation(A_bits, t)
    a_codes, s_a = orc.quantize_rows(A_c)
    w_codes_t, s_w = orc.quantize_cols(orc.bf16_to_f32(W_bits))
    return A_bits, W_bits, a_codes, s_a, w_codes_t, s_w, rp, ci, cv


def test_fwd_magnitude_bruteforce_fractions():
    """|acc/(s_A s_W)| + sum_k |dA[i,k]| |W[k,j]| with exact rationals: the size
    of the two terms the compensated output adds (the epilogue's fp32 rounding
    is relative to it), from the decoded codes, the exact fp32 scales and the
    exact BF16 weights."""
    A_bits, W_bits, a_codes, s_a, w_codes_t, s_w, rp, ci, cv = _magnitude_case()
    M, N, K = a_codes.shape[0], w_codes_t.shape[0], a_codes.shape[1] * 2
    assert rp[-1] >= M        # several entries
    mag = orc.linear_fwd_magnitude(a_codes, s_a, w_codes_t, s_w, rp, ci, cv, W_bits)
    Wf = orc.bf16_to_f32(W_bits)

    def dec(packed, r, k):
        return Fraction(orc.e2m1_decode(int(packed[r, k // 2] >> (4 * (k % 2))) & 0xF))

    for i in range(M):
        for j in range(N):
            acc = sum(dec(a_codes, i, k) * dec(w_codes_t, j, k) for k in range(K))
            ref = abs(acc) / (Fraction(float(s_a[i])) * Fraction(float(s_w[j])))
            for e in range(rp[i], rp[i + 1]):
                ref += abs(Fraction(float(cv[e]))) * abs(Fraction(float(Wf[ci[e], j])))
            assert abs(Fraction(float(mag[i, j])) - ref) <= Fraction(2.0 ** -50) * ref, (i, j)


def test_fwd_magnitude_invariants():
    """Triangle inequality (the magnitude bounds |Y|), independence of the signs
    of dA, no compensation = |uncompensated Y|, and a row subset = those rows."""
    A_bits, W_bits, a_codes, s_a, w_codes_t, s_w, rp, ci, cv = _magnitude_case(seed=22, M=8, K=64, N=10)
    mag = orc.linear_fwd_magnitude(a_codes, s_a, w_codes_t, s_w, rp, ci, cv, W_bits)
    Y = orc.linear_fwd(a_codes, s_a, w_codes_t, s_w, rp, ci, cv, W_bits)
    assert np.all(np.abs(Y) <= mag * (1 + 1e-12))
    flipped = orc.linear_fwd_magnitude(a_codes, s_a, w_codes_t, s_w, rp, ci, -cv, W_bits)
    assert np.array_equal(flipped, mag)
    empty = np.zeros(a_codes.shape[0] + 1, np.int32)
    y0 = orc.linear_fwd(a_codes, s_a, w_codes_t, s_w)
    assert np.array_equal(orc.linear_fwd_magnitude(a_codes, s_a, w_codes_t, s_w, empty, ci[:0], cv[:0], W_bits),
                          np.abs(y0))
    rows = [7, 2, 5]
    assert np.array_equal(orc.linear_fwd_magnitude(a_codes, s_a, w_codes_t, s_w, rp, ci, cv, W_bits, rows=rows),
                          mag[rows])
    # the compensation's magnitude adds: every entry moves it up by |dA| |W|
    assert np.all(mag >= np.abs(y0) - 1e-15)


def test_forward_approximates_dense_product():
    # with the compensation added back, the FP4 layer approximates A @ W; the
    # error is bounded by the E2M1 rounding error of A_clamped and W.
    rng = np.random.default_rng(9)
    M, K, N = 32, 128, 16
    A_bits = _bf16_matrix(rng, (M, K))
    W_bits = _bf16_matrix(rng, (K, N), 0.02)
    out = orc.linear_layer_forward(A_bits, W_bits, 0.99)
    A = orc.bf16_to_f32(A_bits).astype(np.float64)
    W = orc.bf16_to_f32(W_bits).astype(np.float64)
    ref = A @ W
    rel = np.linalg.norm(out["Y"] - ref) / np.linalg.norm(ref)
    assert rel < 0.2           # 4-bit operands: ~10 % relative error
    Aq = orc.dequantize(out["a_codes"], out["s_a"])
    Wq = orc.dequantize(out["w_codes_t"], out["s_w"]).T
    dA = orc.csr_to_dense(out["row_ptr"], out["col_idx"], out["vals"], (M, K))
    np.testing.assert_allclose(out["Y"], Aq @ Wq + dA @ W, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- quantile / clamp / CSR

def _brute_threshold(A_bits, q):
    mags = sorted(abs(float(v)) for v in orc.bf16_to_f32(A_bits).reshape(-1))
    n = len(mags)
    k = min(n, max(1, math.ceil(q * n)))
    return mags[k - 1], k


@pytest.mark.parametrize("q", [0.5, 0.9, 0.97, 0.99, 0.999, 1.0, 1e-9])
def test_quantile_bruteforce_and_invariants(q):
    rng = np.random.default_rng(10)
    A_bits = wl.f32_to_bf16_bits(rng.standard_t(3, size=(37, 29)).astype(np.float32))
    t, t_bits, k = orc.quantile_threshold(A_bits, q)
    bt, bk = _brute_threshold(A_bits, q)
    assert float(t) == bt and k == bk
    mags = np.abs(orc.bf16_to_f32(A_bits))
    assert np.count_nonzero(mags <= t) >= k
    assert np.count_nonzero(mags < t) <= k - 1


def test_quantile_heavy_ties():
    rng = np.random.default_rng(11)
    vals = np.array([0.5, -0.5, 1.0, 2.0, -2.0, 3.0], dtype=np.float32)
    A_bits = wl.f32_to_bf16_bits(rng.choice(vals, size=(50, 40)))
    for q in (0.3, 0.6, 0.9, 0.99):
        t, _, k = orc.quantile_threshold(A_bits, q)
        assert float(t) == _brute_threshold(A_bits, q)[0]


def test_clamp_identity_and_csr_structure():
    rng = np.random.default_rng(12)
    M, K = 40, 64
    A_bits = wl.f32_to_bf16_bits(rng.standard_t(3, size=(M, K)).astype(np.float32) * np.float32(3.0))
    for q in (0.9, 0.99, 1.0):
        t, _, k = orc.quantile_threshold(A_bits, q)
        A = orc.bf16_to_f32(A_bits)
        A_c, rp, ci, vals = orc.clamp_and_compensation(A_bits, t)
        D = orc.csr_to_dense(rp, ci, vals, (M, K)).astype(np.float32)
        assert np.array_equal((A_c + D).view(np.uint32), A.view(np.uint32)), "A_c + dA must equal A bitwise"
        clamped = np.abs(A) > t
        assert np.array_equal(D != 0, clamped)
        assert np.all(np.abs(A_c) <= t)
        assert rp[0] == 0 and np.all(np.diff(rp) >= 0) and rp[-1] == clamped.sum()
        assert rp[-1] <= A.size - k
        for i in range(M):
            cols = ci[rp[i]:rp[i + 1]]
            assert np.all(np.diff(cols) > 0)
            for c, v in zip(cols, vals[rp[i]:rp[i + 1]]):
                a = Fraction(float(A[i, c]))
                assert Fraction(float(v)) == a - (Fraction(float(t)) if a > 0 else -Fraction(float(t)))
        if q == 1.0:
            assert rp[-1] == 0


def test_clamp_rank_rule():
    assert orc.clamp_rank(1000, 0.999) == 999
    assert orc.clamp_rank(16777216, 0.999) == math.ceil(0.999 * 16777216)
    assert orc.clamp_rank(10, 1e-12) == 1
    assert orc.clamp_rank(10, 1.0) == 10


# ---------------------------------------------------------------- BF16 rounding helper

def test_f64_to_bf16_against_exact_rational():
    rng = np.random.default_rng(13)
    x = np.concatenate([rng.standard_normal(3000) * 10.0 ** rng.integers(-30, 30, 3000),
                        [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 0.0, -0.0]])
    bits = orc.f64_to_bf16(x)
    vals = orc.bf16_to_f32(bits)
    for xv, bv, b in zip(x.tolist(), vals.tolist(), bits.tolist()):
        # bv must be a nearest 8-significant-bit value, ties to an even last bit
        fx, fb = Fraction(xv), Fraction(bv)
        step = abs(Fraction(float(np.spacing(np.float32(bv))))) * 2 ** 16 if bv != 0 else Fraction(0)
        if bv == 0:
            assert abs(xv) < 1e-37
            continue
        assert abs(fx - fb) <= step / 2
        if abs(fx - fb) == step / 2:
            assert b & 1 == 0


# ---------------------------------------------------------------- DGE

@pytest.mark.parametrize("k,clip", [(5.0, 3.0), (3.0, 2.0), (8.0, 10.0)])
def test_dge_derivative_at_grid_points_and_midpoints(k, clip):
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0])
    assert np.allclose(orc.dge_derivative(grid, k, clip), 1.0 / k, rtol=1e-15)
    left = np.array([0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]) - 1e-12
    assert np.allclose(orc.dge_derivative(left, k, clip), 1.0 / k, rtol=1e-6)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    assert np.all(orc.dge_derivative(mids, k, clip) == clip)
    assert np.all(orc.dge_derivative(np.array([6.0, 6.5]), k, clip) == 1.0 / k)


def test_dge_k1_is_identity_with_unit_derivative_everywhere():
    # k = 1: f(x) = lo + delta/2 (1 + u) = x on every interval, so f' = 1,
    # including the interval midpoints (u = 0) and the grid points.
    x = np.concatenate([np.linspace(0, 5.999, 4001), [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]])
    assert np.allclose(orc.dge_surrogate(x, 1.0), x, rtol=0, atol=1e-12)
    assert np.all(orc.dge_derivative(x, 1.0, 3.0) == 1.0)


def test_dge_surrogate_continuous_monotone_and_hits_grid():
    k = 5.0
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0])
    assert np.allclose(orc.dge_surrogate(grid, k), grid, atol=0)
    ends = np.array([0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    assert np.allclose(orc.dge_surrogate(ends - 1e-13, k), ends, atol=1e-9)
    x = np.linspace(0, 6, 60001)
    f = orc.dge_surrogate(x, k)
    assert np.all(np.diff(f) >= -1e-15)


def test_dge_derivative_matches_finite_difference():
    k, clip = 5.0, 3.0
    rng = np.random.default_rng(14)
    x = rng.uniform(0, 6, 5000)
    lo, d = orc.dge_interval(x)
    u = np.abs(2 * (x - lo) / d - 1)
    keep = (u > 0.05) & (u < 0.95)
    x = x[keep]
    h = 1e-7
    fd = (orc.dge_surrogate(x + h, k) - orc.dge_surrogate(x - h, k)) / (2 * h)
    fp = orc.dge_derivative(x, k, clip)
    unclipped = fp < clip
    np.testing.assert_allclose(fd[unclipped], fp[unclipped], rtol=1e-5)


def test_wgrad_with_k1_is_plain_product_bruteforce():
    # k = 1: the surrogate is the identity, f' = 1, so dW = A^T dY.
    rng = np.random.default_rng(15)
    M, K, N = 7, 6, 4
    A = _bf16_matrix(rng, (M, K))
    dY = _bf16_matrix(rng, (M, N), 1e-3)
    W = _bf16_matrix(rng, (K, N), 0.02)
    _, s_w = orc.quantize_cols(orc.bf16_to_f32(W))
    dW = orc.wgrad_dge(A, dY, W, s_w, 1.0, 3.0)
    Af = orc.bf16_to_f32(A).tolist()
    Gf = orc.bf16_to_f32(dY).tolist()
    for r in range(K):
        for j in range(N):
            ref = sum(Fraction(Af[m][r]) * Fraction(Gf[m][j]) for m in range(M))
            assert dW[r, j] == np.float32(float(ref))


def test_wgrad_factor_symmetric_in_sign_and_uses_scaled_weight():
    rng = np.random.default_rng(16)
    M, K, N = 9, 6, 5
    A = _bf16_matrix(rng, (M, K))
    dY = _bf16_matrix(rng, (M, N), 1e-3)
    W = _bf16_matrix(rng, (K, N), 0.02)
    _, s_w = orc.quantize_cols(orc.bf16_to_f32(W))
    dW = orc.wgrad_dge(A, dY, W, s_w, 5.0, 3.0)
    dWn = orc.wgrad_dge(A, dY, W ^ np.uint16(0x8000), s_w, 5.0, 3.0)
    assert np.array_equal(dW, dWn)
    G = orc.bf16_to_f32(A).astype(np.float64).T @ orc.bf16_to_f32(dY).astype(np.float64)
    Wf = orc.bf16_to_f32(W)
    for r in range(K):
        for j in range(N):
            x = abs(float(Wf[r, j] * s_w[j]))
            assert dW[r, j] == np.float32(G[r, j] * float(orc.dge_derivative(np.array([x]), 5.0, 3.0)[0]))
    sub = orc.wgrad_dge(A, dY, W, s_w, 5.0, 3.0, rows=[4, 1], cols=[0, 3])
    assert np.array_equal(sub, dW[np.ix_([4, 1], [0, 3])])


# ---------------------------------------------------------------- input gradient (reading R16)

def test_dgrad_bruteforce_fractions():
    """Every entry against an exact rational sum of the BF16 products."""
    rng = np.random.default_rng(21)
    M, N, K = 3, 9, 4
    dY_bits = orc.f64_to_bf16(rng.standard_normal((M, N)) * 1e-3)
    W_bits = orc.f64_to_bf16(rng.standard_normal((K, N)) * 0.02)
    dY = orc.bf16_to_f32(dY_bits)
    W = orc.bf16_to_f32(W_bits)
    got = orc.linear_dgrad(dY_bits, W_bits)
    assert got.shape == (M, K)
    for m in range(M):
        for k in range(K):
            exact = sum(Fraction(float(dY[m, n])) * Fraction(float(W[k, n])) for n in range(N))
            assert got[m, k] == float(exact)


@pytest.mark.parametrize("K,N", [(24, 24), (16, 40), (40, 16)])
def test_dgrad_is_the_adjoint_of_the_forward_product(K, N):
    """The input gradient of L = <dY, X W> is the unique G with <G, X> = <dY, X W>
    for every X; a transposed or swapped operand breaks this (the square case
    K = N catches W in place of W^T)."""
    rng = np.random.default_rng(K * 100 + N)
    M = 7
    dY_bits = orc.f64_to_bf16(rng.standard_normal((M, N)))
    W_bits = orc.f64_to_bf16(rng.standard_normal((K, N)))
    G = orc.linear_dgrad(dY_bits, W_bits)
    dY = orc.bf16_to_f32(dY_bits).astype(np.float64)
    W = orc.bf16_to_f32(W_bits).astype(np.float64)
    for trial in range(3):
        X = rng.standard_normal((M, K))
        lhs = float(np.sum(G * X))
        rhs = float(np.sum(dY * (X @ W)))
        assert abs(lhs - rhs) <= 1e-12 * (np.sum(np.abs(G) * np.abs(X)) + 1.0)


def test_dgrad_sampled_rows_cols_match_full():
    rng = np.random.default_rng(5)
    dY_bits = orc.f64_to_bf16(rng.standard_normal((20, 48)))
    W_bits = orc.f64_to_bf16(rng.standard_normal((12, 48)))
    full = orc.linear_dgrad(dY_bits, W_bits)
    rows, cols = [0, 7, 19], [11, 2]
    assert np.array_equal(orc.linear_dgrad(dY_bits, W_bits, rows=rows, cols=cols), full[np.ix_(rows, cols)])


# ---------------------------------------------------------------- E4M3 (FP8 weight gradient)

def _e4m3_values_exact():
    """Finite non-negative E4M3 values as exact rationals, indexed by code 0..126:
    subnormals m/8 2^-6, normals (1 + m/8) 2^(e-7), e = 1..15 (code 127 is NaN)."""
    vals = []
    for c in range(127):
        e, m = c >> 3, c & 7
        vals.append(Fraction(m, 8) * Fraction(1, 64) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7))
    return vals


def _e4m3_nearest_exact(y: float) -> int:
    """Nearest finite E4M3 value by exact rational distance, ties to the even
    mantissa, magnitudes past 448 saturated, the sign bit from y."""
    vals = _e4m3_values_exact()
    mag = abs(Fraction(float(y)))
    if mag >= vals[-1]:
        c = 126
    else:
        hi = next(i for i, v in enumerate(vals) if v >= mag)
        lo = max(hi - 1, 0)
        dlo, dhi = mag - vals[lo], vals[hi] - mag
        c = lo if dlo < dhi else hi if dhi < dlo else (lo if lo % 2 == 0 else hi)
    return c | (0x80 if math.copysign(1.0, y) < 0 else 0)


def test_e4m3_decode_closed_form():
    vals = [orc.e4m3_decode(c) for c in range(256)]
    assert sum(math.isnan(v) for v in vals) == 2                      # S.1111.111 only
    assert max(v for v in vals if not math.isnan(v)) == 448.0
    assert orc.e4m3_decode(0x38) == 1.0 and orc.e4m3_decode(0x01) == 2.0 ** -9
    assert orc.e4m3_decode(0x08) == 2.0 ** -6 and orc.e4m3_decode(0x07) == 7 * 2.0 ** -9
    exact = _e4m3_values_exact()
    for c in range(127):
        assert Fraction(orc.e4m3_decode(c)) == exact[c]
        assert orc.e4m3_decode(c | 0x80) == -orc.e4m3_decode(c)


def test_e4m3_encode_exact_rational_on_values_midpoints_and_neighbours():
    exact = _e4m3_values_exact()
    pts = []
    for i in range(126):
        mid = (exact[i] + exact[i + 1]) / 2
        for v in (exact[i], mid):
            f = float(v)
            pts += [f, np.nextafter(f, 0.0), np.nextafter(f, np.inf)]
    pts += [448.0, 464.0, np.nextafter(464.0, 0.0), 465.0, 480.0, 1e4, 3.0e38, 0.0, 2.0 ** -11, 2.0 ** -10]
    x = np.array(pts + [-p for p in pts], dtype=np.float64)
    got = orc.e4m3_encode(x)
    want = np.array([_e4m3_nearest_exact(v) for v in x], dtype=np.uint8)
    np.testing.assert_array_equal(got, want)


def test_e4m3_golden_ties_and_saturation():
    # midpoints go to the even mantissa; everything at or past 448 stays at 448
    cases = {1 + 1 / 16: 0x38, 1 + 3 / 16: 0x3A, 2.0 ** -10: 0x00, 3 * 2.0 ** -10: 0x02,
             464.0: 0x7E, 1e9: 0x7E, -1e9: 0xFE, -0.0: 0x80, -2.0 ** -12: 0x80, 240.0: 0x77}
    got = orc.e4m3_encode(np.array(list(cases), dtype=np.float64))
    assert [int(c) for c in got] == list(cases.values())


def test_e4m3_encode_matches_torch_float8_in_range():
    """torch's float8_e4m3fn conversion rounds to nearest even but does not
    saturate, so the comparison stays below the saturation midpoint 464."""
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn in this torch")
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(200000) * np.exp2(rng.uniform(-14, 9, 200000))).astype(np.float32)
    x = x[np.abs(x) < 464.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(orc.e4m3_encode(x), ref)


def test_wgrad_fp8_is_scaled_encode_of_the_fp32_gradient():
    rng = np.random.default_rng(8)
    dW = (rng.standard_normal((7, 9)) * 1e-3).astype(np.float32)
    s = 448.0 / float(np.max(np.abs(dW)))
    codes, amax = orc.wgrad_dge_fp8(dW, s)
    assert amax == np.max(np.abs(dW))
    y = dW * np.float32(s)                                   # one fp32 multiply
    assert [int(c) for c in codes.ravel()] == [_e4m3_nearest_exact(float(v)) for v in y.ravel()]
    deq = np.array([orc.e4m3_decode(int(c)) for c in codes.ravel()]).reshape(dW.shape) / s
    # relative spacing of E4M3 is 2^-3, so the rounding error is at most 2^-4 relative
    # (normals) or 2^-10 / s absolute (subnormals)
    assert np.all(np.abs(deq - dW) <= np.maximum(np.abs(dW) * 2.0 ** -4, 2.0 ** -10 / s) * (1 + 1e-6))
    assert codes[np.unravel_index(np.argmax(np.abs(dW)), dW.shape)] & 0x7F == 0x7E
