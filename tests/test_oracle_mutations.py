"""Plant plausible mistakes in the oracle (on the CPU, by monkeypatching) and
check that at least one pin in test_oracle_pins fails for each.  This shows the
pins constrain every step: a dropped term, a wrong sign, an off-by-one index or
a swapped operand does not go unnoticed."""
import numpy as np
import pytest

from oracle import fp4_linear as orc
import tests.test_oracle_pins as pins


def _expect_failure(fn, *args):
    with pytest.raises(Exception):
        fn(*args)


def test_ties_away_from_zero_is_caught(monkeypatch):
    real = orc.e2m1_round

    def ties_away(y):
        y = np.asarray(y, dtype=np.float32)
        mag = np.minimum(np.abs(y).astype(np.float64), 6.0)
        d = np.abs(mag[..., None] - orc.GRID)
        nearest = d == d.min(axis=-1, keepdims=True)
        code = (7 - np.argmax(nearest[..., ::-1], axis=-1)).astype(np.uint8)   # larger on ties
        return code | (np.signbit(y).astype(np.uint8) << 3)

    monkeypatch.setattr(orc, "e2m1_round", ties_away)
    _expect_failure(pins.test_e2m1_rounding_golden_cases)
    _expect_failure(pins.test_e2m1_round_exhaustive_bf16_exact_rational)
    monkeypatch.setattr(orc, "e2m1_round", real)


def test_unsigned_zero_is_caught(monkeypatch):
    real = orc.e2m1_round

    def no_negative_zero(y):
        c = real(y)
        return np.where((c & 7) == 0, 0, c).astype(np.uint8)

    monkeypatch.setattr(orc, "e2m1_round", no_negative_zero)
    _expect_failure(pins.test_e2m1_rounding_golden_cases)


def test_inverted_scale_is_caught(monkeypatch):
    monkeypatch.setattr(orc, "absmax_scale", lambda a: (np.asarray(a, np.float32) / np.float32(6.0)))
    _expect_failure(pins.test_quantize_rows_bruteforce_small)
    _expect_failure(pins.test_scale_is_correctly_rounded_6_over_absmax)


def test_multiplied_instead_of_divided_scales_are_caught(monkeypatch):
    real_raw = orc.gemm_raw

    def bad_fwd(a_codes, s_a, w_codes_t, s_w, *args, **kw):
        acc = real_raw(a_codes, w_codes_t)
        return acc * (np.asarray(s_a, np.float64)[:, None] * np.asarray(s_w, np.float64)[None, :])

    monkeypatch.setattr(orc, "linear_fwd", bad_fwd)
    _expect_failure(pins.test_lossless_grid_matrices_give_exact_product)


def test_transposed_weight_operand_is_caught(monkeypatch):
    real_unpack = orc.unpack_codes

    def gemm_wrong_operand(a_codes, w_codes_t, rows=None, cols=None):
        a = 2.0 * orc.DECODE[real_unpack(a_codes)]
        w = 2.0 * orc.DECODE[real_unpack(w_codes_t)]
        w = w[::-1]                                # output columns permuted
        return (a @ w.T) / 4.0

    monkeypatch.setattr(orc, "gemm_raw", gemm_wrong_operand)
    _expect_failure(pins.test_gemm_raw_bruteforce_fractions)
    _expect_failure(pins.test_lossless_grid_matrices_give_exact_product)


def test_swapped_nibbles_in_unpack_are_caught(monkeypatch):
    def unpack_swapped(packed):
        packed = np.asarray(packed, dtype=np.uint8)
        out = np.empty((packed.shape[0], packed.shape[1] * 2), dtype=np.uint8)
        out[:, 0::2] = packed >> 4
        out[:, 1::2] = packed & 0xF
        return out

    monkeypatch.setattr(orc, "unpack_codes", unpack_swapped)
    # (a GEMM alone cannot see it: the same K permutation on both operands
    # leaves every dot product unchanged; the elementwise dequantization does)
    _expect_failure(pins.test_dequantized_values_on_grid_and_within_half_spacing)


def test_dropped_compensation_is_caught(monkeypatch):
    real = orc.linear_fwd

    def no_comp(a_codes, s_a, w_codes_t, s_w, row_ptr=None, col_idx=None, vals=None, W_bits=None, rows=None, cols=None):
        return real(a_codes, s_a, w_codes_t, s_w, rows=rows, cols=cols)

    monkeypatch.setattr(orc, "linear_fwd", no_comp)
    _expect_failure(pins.test_compensation_term_is_dA_times_W)
    _expect_failure(pins.test_forward_approximates_dense_product)


def test_quantile_off_by_one_is_caught(monkeypatch):
    def off_by_one(A_bits, q):
        mags = (np.asarray(A_bits, dtype=np.uint16) & np.uint16(0x7FFF)).reshape(-1)
        k = orc.clamp_rank(mags.size, q)
        t_bits = int(np.sort(mags)[min(k, mags.size - 1)])
        return orc.bf16_to_f32(np.array([t_bits], dtype=np.uint16))[0], t_bits, k

    monkeypatch.setattr(orc, "quantile_threshold", off_by_one)
    _expect_failure(pins.test_quantile_bruteforce_and_invariants, 0.9)


def test_non_strict_clamp_is_caught(monkeypatch):
    def clamp_ge(A_bits, t):
        A = orc.bf16_to_f32(A_bits)
        t = np.float32(t)
        mask = np.abs(A) >= t
        A_c = np.where(mask, np.copysign(t, A), A).astype(np.float32)
        dA = (A - A_c).astype(np.float32)
        row_ptr = np.zeros(A.shape[0] + 1, dtype=np.int64)
        row_ptr[1:] = np.cumsum(mask.sum(axis=1))
        rows, cols = np.nonzero(mask)
        return A_c, row_ptr.astype(np.int32), cols.astype(np.int32), dA[rows, cols]

    monkeypatch.setattr(orc, "clamp_and_compensation", clamp_ge)
    _expect_failure(pins.test_clamp_identity_and_csr_structure)


def test_wrong_sign_in_compensation_value_is_caught(monkeypatch):
    real = orc.clamp_and_compensation

    def flipped(A_bits, t):
        A_c, rp, ci, vals = real(A_bits, t)
        return A_c, rp, ci, -vals

    monkeypatch.setattr(orc, "clamp_and_compensation", flipped)
    _expect_failure(pins.test_clamp_identity_and_csr_structure)


def test_wrong_dge_exponent_is_caught(monkeypatch):
    real = orc.dge_derivative
    monkeypatch.setattr(orc, "dge_derivative", lambda x, k, clip: real(x, 1.0 / k, clip))
    _expect_failure(pins.test_dge_derivative_at_grid_points_and_midpoints, 5.0, 3.0)
    _expect_failure(pins.test_dge_derivative_matches_finite_difference)


def test_unscaled_weight_in_dge_is_caught(monkeypatch):
    real = orc.wgrad_dge

    def unscaled(A_bits, dY_bits, W_bits, s_w, k, clip, rows=None, cols=None):
        return real(A_bits, dY_bits, W_bits, np.ones_like(np.asarray(s_w)), k, clip, rows, cols)

    monkeypatch.setattr(orc, "wgrad_dge", unscaled)
    _expect_failure(pins.test_wgrad_factor_symmetric_in_sign_and_uses_scaled_weight)


def test_untransposed_weight_in_dgrad_is_caught(monkeypatch):
    def no_transpose(dY_bits, W_bits, rows=None, cols=None):
        dY = orc.bf16_to_f32(dY_bits).astype(np.float64)
        W = orc.bf16_to_f32(W_bits).astype(np.float64)
        return dY @ W        # dY W instead of dY W^T (same shape when K = N)

    monkeypatch.setattr(orc, "linear_dgrad", no_transpose)
    _expect_failure(pins.test_dgrad_is_the_adjoint_of_the_forward_product, 24, 24)


def _magnitude_with(body):
    """linear_fwd_magnitude rebuilt with one planted change in its compensation sum."""
    def mag(a_codes, s_a, w_codes_t, s_w, row_ptr, col_idx, vals, W_bits, rows=None):
        t1 = np.abs(orc.linear_fwd(a_codes, s_a, w_codes_t, s_w, rows=rows))
        rows_ = np.arange(np.asarray(a_codes).shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
        W = orc.bf16_to_f32(W_bits).astype(np.float64)
        rp = np.asarray(row_ptr, dtype=np.int64)
        return body(t1, rows_, W, rp, np.asarray(col_idx, np.int64), np.asarray(vals, np.float64))
    return mag


def test_magnitude_with_signed_compensation_is_caught(monkeypatch):
    def body(t1, rows, W, rp, ci, v):
        for r, i in enumerate(rows):
            t1[r] += v[rp[i]:rp[i + 1]] @ np.abs(W[ci[rp[i]:rp[i + 1]]])     # signed dA
        return t1
    monkeypatch.setattr(orc, "linear_fwd_magnitude", _magnitude_with(body))
    _expect_failure(pins.test_fwd_magnitude_bruteforce_fractions)
    _expect_failure(pins.test_fwd_magnitude_invariants)


def test_magnitude_with_signed_weights_is_caught(monkeypatch):
    def body(t1, rows, W, rp, ci, v):
        for r, i in enumerate(rows):
            t1[r] += np.abs(v[rp[i]:rp[i + 1]]) @ W[ci[rp[i]:rp[i + 1]]]     # signed W
        return t1
    monkeypatch.setattr(orc, "linear_fwd_magnitude", _magnitude_with(body))
    _expect_failure(pins.test_fwd_magnitude_bruteforce_fractions)


def test_magnitude_with_gemm_term_twice_is_caught(monkeypatch):
    def body(t1, rows, W, rp, ci, v):
        t1 = 2.0 * t1                                                       # GEMM term counted twice
        for r, i in enumerate(rows):
            t1[r] += np.abs(v[rp[i]:rp[i + 1]]) @ np.abs(W[ci[rp[i]:rp[i + 1]]])
        return t1
    monkeypatch.setattr(orc, "linear_fwd_magnitude", _magnitude_with(body))
    _expect_failure(pins.test_fwd_magnitude_bruteforce_fractions)


def test_magnitude_with_wrong_row_under_subset_is_caught(monkeypatch):
    def body(t1, rows, W, rp, ci, v):
        for r, i in enumerate(rows):
            a, b = rp[r], rp[r + 1]                                          # position, not the row index
            t1[r] += np.abs(v[a:b]) @ np.abs(W[ci[a:b]])
        return t1
    monkeypatch.setattr(orc, "linear_fwd_magnitude", _magnitude_with(body))
    _expect_failure(pins.test_fwd_magnitude_invariants)


def test_e4m3_ties_away_and_missing_saturation_are_caught(monkeypatch):
    real = orc.e4m3_encode

    def ties_away(y):
        y = np.asarray(y, dtype=np.float64)
        c = real(y)
        # where y sits exactly halfway between two codes, take the larger magnitude
        lo = np.array([abs(orc.e4m3_decode(int(v))) for v in c.ravel()]).reshape(c.shape)
        nxt = np.array([abs(orc.e4m3_decode(int(v & 0x7F) + 1)) if (v & 0x7F) < 0x7E else np.inf
                        for v in c.ravel()]).reshape(c.shape)
        tie = np.abs(y) == (lo + nxt) / 2
        return np.where(tie, c + 1, c).astype(np.uint8)

    monkeypatch.setattr(orc, "e4m3_encode", ties_away)
    _expect_failure(pins.test_e4m3_golden_ties_and_saturation)
    _expect_failure(pins.test_e4m3_encode_exact_rational_on_values_midpoints_and_neighbours)

    def no_saturation(y):
        c = real(y)
        big = np.abs(np.asarray(y, dtype=np.float64)) > 464.0
        return np.where(big, c | 0x7F, c).astype(np.uint8)

    monkeypatch.setattr(orc, "e4m3_encode", no_saturation)
    _expect_failure(pins.test_e4m3_golden_ties_and_saturation)
    _expect_failure(pins.test_e4m3_encode_exact_rational_on_values_midpoints_and_neighbours)
    monkeypatch.setattr(orc, "e4m3_encode", real)


def test_e4m3_wrong_exponent_bias_is_caught(monkeypatch):
    real = orc.e4m3_decode
    monkeypatch.setattr(orc, "e4m3_decode", lambda c: real(c) * 2.0)       # bias 6 instead of 7
    _expect_failure(pins.test_e4m3_decode_closed_form)
    monkeypatch.setattr(orc, "e4m3_decode", real)
    real_enc = orc.e4m3_encode
    monkeypatch.setattr(orc, "e4m3_encode", lambda y: real_enc(np.asarray(y, dtype=np.float64) / 2.0))
    _expect_failure(pins.test_e4m3_encode_exact_rational_on_values_midpoints_and_neighbours)
    _expect_failure(pins.test_e4m3_encode_matches_torch_float8_in_range)
    monkeypatch.setattr(orc, "e4m3_encode", real_enc)
