"""CPU oracle for the FP4 quantized linear layer.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this module: it is used by tests/, by __graft_entry__.smoke() and by
bench.py's cpu_baseline / reference arm, nowhere else.  It shares no code,
table or constant generator with the CUDA library; the only module both sides
read is the seeded input generator, which holds no arithmetic of the method.

What it computes, and where the pages say so
---------------------------------------------
Page 1, "首个 FP4 精度的大模型训练框架来了，来自微软研究院" (czzqal.com, a
machine-reworded copy of a QbitAI article), and page 2, "Microsoft Research
bringt den ersten FP4-Genauigkeitsrahmen für das Training großer Modelle heraus"
(topaibox.com), describe:

* the E2M1 format: 1 sign bit, 2 exponent bits, 1 mantissa bit (page 1, format
  passage; page 2, section "Quantifizierungsstrategien und Hardware-Anpassung");
* token-wise (row) quantization of the activation A and channel-wise (column)
  quantization of the weight W (page 1, granularity passage);
* "scale + shift" calibration into the FP4 range, then rounding to the nearest
  FP4 value through a lookup table (page 1, calibration passage; page 2, section
  "Innovationen in der Vorwärts- und Rückwärtspropagation");
* a quantile search over A that clamps its largest-magnitude outliers to a
  threshold, giving A_clamped, plus a sparse compensation matrix
  dA = A - A_clamped that is nonzero only at clamped positions (page 1,
  outlier passage; page 2, "Peak-Dämpfung und -Kompensation");
* a differentiable gradient estimator (DGE): hard quantization forward, and in
  backward a continuous differentiable function fitted to the quantizer whose
  derivative corrects the weight gradient (page 1, DGE passage; page 4,
  "Optimizing Large Language Model Training Using FP4 Quantization", abstract).

Readings where the pages are silent (each is stated where it is used):
R1 scale = 6/absmax as ONE fp32 division, applied as ONE fp32 multiply, no
   additive zero point; R2 round half to the even code, saturate above 6;
R3 the sign of a value that rounds to zero is kept (code 0x8); R4 a zero or
   non-finite 6/absmax gives scale 1; R6 the threshold is the order statistic
   k = ceil(q n) of |A| (BF16 values, no interpolation) and clamping is strict
   (|A| > t); R7 clamping happens before the row quantization; R8 the
   compensation multiplies dA by the original BF16 W; R9 the DGE surrogate is a
   per-interval power function with exponent 1/k and a clipped derivative;
   R11 accumulation and outputs in fp32 / BF16 (the pages' FP16 output is the
   authors' emulation detail); R12 element 2c of a row goes in the low nibble;
   R16 the input gradient (absent from the pages) is dY W^T with the BF16 W.
R17 the FP8 weight gradient for communication is E4M3 with one per-tensor
   scale from the caller, round half to even, saturating at 448.

Precision: fp64 wherever the pages fix no precision.  The quantizer itself
works in fp32 because its definition (R1) is an fp32 division and multiply.
"""
from __future__ import annotations

import math
from typing import Iterable, Optional, Sequence, Tuple

import numpy as np

# --------------------------------------------------------------------------
# E2M1 number format
# --------------------------------------------------------------------------


def e2m1_decode(code: int) -> float:
    """Value of a 4-bit E2M1 code.

    Page 1 (format passage) / page 2 ("Quantifizierungsstrategien und
    Hardware-Anpassung"): 2 exponent bits, 1 mantissa bit, 1 sign bit.  With the
    usual exponent bias of 1 and no Inf/NaN, exponent field 0 is subnormal
    (0.5 * m) and field e > 0 is 2^(e-1) * (1 + m/2).
    """
    sign = (code >> 3) & 1
    exp = (code >> 1) & 3
    man = code & 1
    if exp == 0:
        mag = 0.5 * man
    else:
        mag = 2.0 ** (exp - 1) * (1.0 + 0.5 * man)
    return -mag if sign else mag


#: decoded value of every code 0..15 (code 8 is -0.0)
DECODE = np.array([e2m1_decode(c) for c in range(16)], dtype=np.float64)
#: the non-negative grid, indexed by the 3-bit magnitude code
GRID = DECODE[:8].copy()


def e2m1_round(y: np.ndarray) -> np.ndarray:
    """Round fp32 values to E2M1 codes (0..15): nearest grid point, ties to the
    even code (mantissa bit 0), saturating at 6, sign kept (R2, R3).

    Page 1: values are mapped into the FP4 range and then rounded to the nearest
    FP4 value via a lookup table.  The nearest point is found by comparing the
    distance to every grid point; |y| is first limited to 6, which is the same
    as saturating because 6 is the nearest grid point to every |y| > 5.  All
    distances are exact in fp64 for |y| <= 6 with an fp32 |y|.
    """
    y = np.asarray(y, dtype=np.float32)
    out = np.empty(y.shape, dtype=np.uint8)
    flat_y = y.reshape(-1)
    flat_o = out.reshape(-1)
    even = (np.arange(8) % 2) == 0
    step = 1 << 20
    for s in range(0, flat_y.size, step):
        yy = flat_y[s:s + step]
        mag = np.minimum(np.abs(yy).astype(np.float64), 6.0)
        dist = np.abs(mag[:, None] - GRID[None, :])
        nearest = dist == dist.min(axis=1, keepdims=True)
        tie_even = nearest & even[None, :]
        code = np.where(tie_even.any(axis=1), np.argmax(tie_even, axis=1), np.argmax(nearest, axis=1))
        code = code.astype(np.uint8) | (np.signbit(yy).astype(np.uint8) << 3)
        flat_o[s:s + step] = code
    return out


# --------------------------------------------------------------------------
# BF16 helpers (bit-level, no library rounding)
# --------------------------------------------------------------------------


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """BF16 bit patterns -> fp32 values (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f64_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values straight to BF16 (8 significant bits, ties to even),
    returning uint16 bit patterns.  Rounds once (no detour through fp32).
    Covers the normal and subnormal BF16 range; overflow gives +-inf.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                              # x = m 2^e, 0.5 <= |m| < 1
    normal = np.abs(x) >= 2.0 ** -126
    r_norm = np.rint(m * 256.0) * np.exp2(e.astype(np.float64) - 8.0)   # rint is ties-to-even
    r_sub = np.rint(x * 2.0 ** 133) * 2.0 ** -133
    r = np.where(normal, r_norm, r_sub)
    with np.errstate(over="ignore"):
        r32 = r.astype(np.float32)                 # exact: r has <= 8 significant bits
    return (r32.view(np.uint32) >> 16).astype(np.uint16)


# --------------------------------------------------------------------------
# Scales and row / column quantization
# --------------------------------------------------------------------------


def absmax_scale(absmax: np.ndarray) -> np.ndarray:
    """s = 6 / absmax as one IEEE fp32 division (R1); s = 1 when absmax is 0 or
    6/absmax is not finite (R4).

    Page 1 (calibration passage): a scale factor maps the range to [-1, 1] and
    a "shift" factor maps [-1, 1] onto the FP4 range; read here as the single
    factor 6/absmax, since an additive offset would break the sign symmetry of
    E2M1 and the factoring of the scales out of the GEMM's K-sum.
    """
    absmax = np.asarray(absmax, dtype=np.float32)
    with np.errstate(divide="ignore", over="ignore"):
        s = np.float32(6.0) / absmax
    bad = (absmax == 0) | ~np.isfinite(s)
    return np.where(bad, np.float32(1.0), s).astype(np.float32)


def quantize_rows(X: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Token-wise (row) absmax quantization of an fp32 matrix X (M x K).

    Page 1 (granularity passage): A is quantized per row (token).  Returns the
    packed codes (M x K/2 uint8, element 2c in the low nibble, R12) and the
    fp32 scales s (M,), with code = E2M1(fl32(x * s)).
    """
    X = np.asarray(X, dtype=np.float32)
    M, K = X.shape
    assert K % 2 == 0
    assert np.isfinite(X).all(), "inputs must be finite (R5)"
    s = absmax_scale(np.max(np.abs(X), axis=1) if K else np.zeros(M, np.float32))
    Y = X * s[:, None]                                        # one fp32 multiply
    codes = e2m1_round(Y)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, s


def quantize_cols(W: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Channel-wise (column) quantization of W (K x N): a column of W is a row of
    W^T, so this is quantize_rows(W^T).  Output codes are N x K/2 (K-major).

    Page 1 (granularity passage): W is quantized per column (channel).
    """
    return quantize_rows(np.ascontiguousarray(np.asarray(W, dtype=np.float32).T))


def unpack_codes(packed: np.ndarray) -> np.ndarray:
    """Packed codes (R x C/2) -> code per element (R x C)."""
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty((packed.shape[0], packed.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = packed & 0xF
    out[:, 1::2] = packed >> 4
    return out


def dequantize(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """decode(code) / s per row, in fp64."""
    return DECODE[unpack_codes(packed)] / np.asarray(scales, dtype=np.float64)[:, None]


# --------------------------------------------------------------------------
# Quantile threshold, clamp and the sparse compensation matrix
# --------------------------------------------------------------------------


def clamp_rank(n: int, q: float) -> int:
    """k = ceil(q n) computed in IEEE double, limited to [1, n] (R6)."""
    if n <= 0:
        return 0
    return min(n, max(1, math.ceil(float(q) * float(n))))


def quantile_threshold(A_bits: np.ndarray, q: float) -> Tuple[np.float32, int, int]:
    """Threshold t = the k-th smallest |A| (k = ceil(q n), 1-based) over ALL
    elements of A, no interpolation (R6).

    Page 1 (outlier passage): a quantile search finds the largest-magnitude
    outliers of A.  |A| of a BF16 value is its bit pattern with the sign bit
    cleared, so the sort is over those 15-bit magnitudes.
    Returns (t as fp32, t's 15-bit magnitude pattern, k).
    """
    mags = (np.asarray(A_bits, dtype=np.uint16) & np.uint16(0x7FFF)).reshape(-1)
    k = clamp_rank(mags.size, q)
    t_bits = int(np.sort(mags, kind="stable")[k - 1])
    return bf16_to_f32(np.array([t_bits], dtype=np.uint16))[0], t_bits, k


def clamp_and_compensation(A_bits: np.ndarray, t: float):
    """A_clamped = sign(A) min(|A|, t) and dA = A - A_clamped in CSR form.

    Page 1 (outlier passage): outliers are limited to the threshold, giving
    A_clamped, and a sparse compensation matrix dA is built from A and
    A_clamped that is nonzero only where clamping happened.  Clamping is strict
    (|A| > t).  Rows in order; column indices ascending within a row; values
    fp32 (R13: A - (+-t) is exact in fp32 for these data, checked by the pins).
    Returns (A_clamped fp32, row_ptr int32 (M+1), col_idx int32, vals fp32).
    """
    A = bf16_to_f32(A_bits)
    t = np.float32(t)
    mask = np.abs(A) > t
    A_c = np.where(mask, np.copysign(t, A), A).astype(np.float32)
    dA = (A - A_c).astype(np.float32)
    counts = mask.sum(axis=1)
    row_ptr = np.zeros(A.shape[0] + 1, dtype=np.int64)
    row_ptr[1:] = np.cumsum(counts)
    rows, cols = np.nonzero(mask)            # row-major order: rows ascending, cols ascending
    vals = dA[rows, cols]
    return A_c, row_ptr.astype(np.int32), cols.astype(np.int32), vals.astype(np.float32)


def csr_to_dense(row_ptr, col_idx, vals, shape) -> np.ndarray:
    """Expand CSR to a dense fp64 matrix (duplicates would add up)."""
    D = np.zeros(shape, dtype=np.float64)
    row_ptr = np.asarray(row_ptr, dtype=np.int64)
    for i in range(shape[0]):
        a, b = row_ptr[i], row_ptr[i + 1]
        if b > a:
            np.add.at(D[i], np.asarray(col_idx[a:b], dtype=np.int64), np.asarray(vals[a:b], dtype=np.float64))
    return D


# --------------------------------------------------------------------------
# FP4 GEMM and its epilogue
# --------------------------------------------------------------------------


def gemm_raw(a_codes: np.ndarray, w_codes_t: np.ndarray, rows: Optional[Sequence[int]] = None,
             cols: Optional[Sequence[int]] = None) -> np.ndarray:
    """acc[i,j] = sum_k decode(qA[i,k]) * decode(qW[k,j]) with both operands as
    K-major code matrices (a_codes M x K/2, w_codes_t N x K/2).

    Page 1 (GeMM passage): block matrix multiplication in FP4; the pages reduce
    in FP16, here the sum is exact (R11).  Twice an E2M1 value is an integer in
    {0, +-1, +-2, +-3, +-4, +-6, +-8, +-12}; the products of those integers and
    all their partial sums are integers below 2^53, so the fp64 matrix product
    below is exact in any summation order.  Returns fp64 values (multiples of
    1/4) for the selected rows / columns.
    """
    a = unpack_codes(a_codes if rows is None else np.asarray(a_codes)[np.asarray(rows)])
    w = unpack_codes(w_codes_t if cols is None else np.asarray(w_codes_t)[np.asarray(cols)])
    a2 = 2.0 * DECODE[a]
    w2 = 2.0 * DECODE[w]
    acc4 = a2 @ w2.T
    return acc4 / 4.0


def linear_fwd(a_codes, s_a, w_codes_t, s_w, row_ptr=None, col_idx=None, vals=None, W_bits=None,
               rows: Optional[Sequence[int]] = None, cols: Optional[Sequence[int]] = None) -> np.ndarray:
    """Y[i,j] = acc[i,j] / (s_A[i] s_W[j]) + sum_{k in row i of dA} dA[i,k] W[k,j], in fp64.

    The per-row and per-column scales factor out of the K-sum (page 1,
    granularity passage: the row/column granularity matches the GEMM and needs
    no transpose), so they are applied once per output element.  The second
    term restores the clamped outlier mass with the original BF16 W (page 1,
    outlier passage "compensation"; R8).  Pass no CSR for the uncompensated Y.
    """
    M = np.asarray(a_codes).shape[0]
    N = np.asarray(w_codes_t).shape[0]
    rows = np.arange(M) if rows is None else np.asarray(rows, dtype=np.int64)
    cols = np.arange(N) if cols is None else np.asarray(cols, dtype=np.int64)
    acc = gemm_raw(a_codes, w_codes_t, rows, cols)
    sa = np.asarray(s_a, dtype=np.float64)[rows]
    sw = np.asarray(s_w, dtype=np.float64)[cols]
    Y = acc / (sa[:, None] * sw[None, :])
    if row_ptr is not None:
        W = bf16_to_f32(W_bits).astype(np.float64)
        rp = np.asarray(row_ptr, dtype=np.int64)
        for r, i in enumerate(rows):
            a, b = rp[i], rp[i + 1]
            if b > a:
                ks = np.asarray(col_idx[a:b], dtype=np.int64)
                v = np.asarray(vals[a:b], dtype=np.float64)
                Y[r] += v @ W[np.ix_(ks, cols)]
    return Y


def linear_fwd_magnitude(a_codes, s_a, w_codes_t, s_w, row_ptr, col_idx, vals, W_bits,
                         rows: Optional[Sequence[int]] = None) -> np.ndarray:
    """|acc / (s_A s_W)| + sum_k |dA[i,k]| |W[k,j]| in fp64: the size of the two
    terms the compensated output adds.  An fp32 evaluation of Y carries an
    absolute rounding error of a few fp32 ulps of this magnitude, which can be
    many BF16 ulps of Y when the terms cancel."""
    t1 = np.abs(linear_fwd(a_codes, s_a, w_codes_t, s_w, rows=rows))
    rows = np.arange(np.asarray(a_codes).shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    W = np.abs(bf16_to_f32(W_bits).astype(np.float64))
    rp = np.asarray(row_ptr, dtype=np.int64)
    for r, i in enumerate(rows):
        a, b = rp[i], rp[i + 1]
        if b > a:
            t1[r] += np.abs(np.asarray(vals[a:b], dtype=np.float64)) @ W[np.asarray(col_idx[a:b], dtype=np.int64)]
    return t1


# --------------------------------------------------------------------------
# Differentiable gradient estimator (weight gradient)
# --------------------------------------------------------------------------


def dge_interval(x: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Lower end lo and width delta of the E2M1 interval holding x >= 0:
    width 0.5 on [0, 2), 1 on [2, 4), 2 on [4, 6); x >= 6 gets (6, 0)."""
    x = np.asarray(x, dtype=np.float64)
    lo = np.where(x < 2.0, np.floor(x / 0.5) * 0.5,
                  np.where(x < 4.0, np.floor(x), np.where(x < 6.0, 4.0, 6.0)))
    delta = np.where(x < 2.0, 0.5, np.where(x < 4.0, 1.0, np.where(x < 6.0, 2.0, 0.0)))
    return lo, delta


def dge_surrogate(x: np.ndarray, k: float) -> np.ndarray:
    """Smooth stand-in for the quantizer on x >= 0 (R9):
    f(x) = lo + delta/2 (1 + sign(u) |u|^(1/k)), u = 2 (x - lo)/delta - 1.

    Page 1 (DGE passage): forward keeps hard quantization; backward refits the
    quantization function with a continuous differentiable function.  The pages
    do not print the function; this power form is the reading used here.  For
    x >= 6 it returns 6 (the saturated value).
    """
    x = np.asarray(x, dtype=np.float64)
    lo, delta = dge_interval(x)
    inside = delta > 0
    d = np.where(inside, delta, 1.0)
    u = 2.0 * (x - lo) / d - 1.0
    f = lo + 0.5 * d * (1.0 + np.sign(u) * np.abs(u) ** (1.0 / k))
    return np.where(inside, f, 6.0)


def dge_derivative(x: np.ndarray, k: float, clip: float) -> np.ndarray:
    """f'(x) = min(clip, (1/k) |u|^(1/k - 1)) with u as in dge_surrogate; x >= 6
    gives 1/k, the value the formula takes at every grid point (R9)."""
    x = np.asarray(x, dtype=np.float64)
    lo, delta = dge_interval(x)
    inside = delta > 0
    d = np.where(inside, delta, 1.0)
    u = np.abs(2.0 * (x - lo) / d - 1.0)
    with np.errstate(divide="ignore"):
        # |u|^e at u = 0 is +inf for e < 0 (clipped), 1 for e = 0 (k = 1: f is
        # the identity) and 0 for e > 0
        fp = (1.0 / k) * u ** (1.0 / k - 1.0)
    fp = np.minimum(clip, fp)
    return np.where(inside, fp, 1.0 / k)


def wgrad_dge(A_bits, dY_bits, W_bits, s_w, k: float, clip: float,
              rows: Optional[Sequence[int]] = None, cols: Optional[Sequence[int]] = None) -> np.ndarray:
    """dW[r,j] = (A^T dY)[r,j] * f'(|fl32(W[r,j] s_W[j])|), returned as fp32.

    Page 1 (DGE passage) and page 4 abstract ("differentiable quantization
    estimator for precise weight updates"): the weight gradient is corrected by
    the derivative of the smooth surrogate.  The surrogate is evaluated at the
    same scaled value the column quantizer rounds (one fp32 multiply); the scale
    cancels in the chain rule.  A^T dY is formed in fp64.  rows/cols select a
    sub-block of dW (rows index K, cols index N).
    """
    A = bf16_to_f32(A_bits).astype(np.float64)
    dY = bf16_to_f32(dY_bits).astype(np.float64)
    Kdim = A.shape[1]
    Ndim = dY.shape[1]
    rows = np.arange(Kdim) if rows is None else np.asarray(rows, dtype=np.int64)
    cols = np.arange(Ndim) if cols is None else np.asarray(cols, dtype=np.int64)
    G = A[:, rows].T @ dY[:, cols]
    W = bf16_to_f32(np.asarray(W_bits)[np.ix_(rows, cols)])
    x = np.abs(W * np.asarray(s_w, dtype=np.float32)[cols][None, :]).astype(np.float64)
    return (G * dge_derivative(x, k, clip)).astype(np.float32)


# --------------------------------------------------------------------------
# FP8 (E4M3) weight gradient, for gradient communication
# --------------------------------------------------------------------------
# Page 1, mixed-precision passage: the framework communicates gradients in FP8.
# The pages name neither the FP8 variant nor its scaling.  Reading R17: E4M3
# (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no infinities, the
# all-ones pattern S.1111.111 is NaN, so the largest finite magnitude is
# 1.75 * 2^8 = 448), one per-tensor fp32 scale s supplied by the caller
# (code = E4M3(fl32(dW * s)), dW ~ decode(code) / s), round half to the even
# mantissa, magnitudes above 448 saturate to 448, and max |dW| is returned so
# the caller can form the next step's scale (delayed per-tensor scaling).

E4M3_MAX = 448.0


def e4m3_decode(code: int) -> float:
    """Value of one E4M3 byte from its bit fields (NaN for S.1111.111)."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6          # subnormal: 0.m x 2^(1 - 7)
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def e4m3_encode(y: np.ndarray) -> np.ndarray:
    """E4M3 byte of each finite y (fp32 or fp64): nearest value, ties to the
    even mantissa, |y| above 448 gives 448, the sign kept for values that round
    to zero.  Works on the binary exponent, so every step is exact in fp64."""
    y = np.asarray(y, dtype=np.float64)
    assert np.all(np.isfinite(y)), "finite inputs only"
    a = np.abs(y)
    _, ex = np.frexp(a)                             # a = f 2^ex, f in [0.5, 1)
    e = np.maximum(ex - 1, -6)                      # unbiased exponent, subnormals share -6
    q = np.rint(a * np.exp2(3 - e))                 # mantissa units of 2^(e-3), half to even
    # q in [8, 16] for normals (16: carried into the next binade), [0, 8] below 2^-6
    carry = q >= 16
    e = np.where(carry, e + 1, e)
    q = np.where(carry, 8, q)
    normal = q >= 8
    mag = np.where(normal, ((e + 7) << 3) + (q - 8), q).astype(np.int64)
    # the magnitude pattern grows with the value, so past 448 (0x7E) it is cut
    # to 448 (0x7F would be NaN)
    mag = np.minimum(mag, 0x7E)
    return (mag | np.where(np.signbit(y), 0x80, 0)).astype(np.uint8)


def wgrad_dge_fp8(dW32: np.ndarray, scale: float) -> Tuple[np.ndarray, np.float32]:
    """E4M3 codes of fl32(dW * scale) and max |dW| (fp32), per reading R17.

    dW32 is the fp32 weight gradient (wgrad_dge); the product with the
    per-tensor scale is one fp32 multiply, rounded to nearest."""
    dW32 = np.asarray(dW32, dtype=np.float32)
    y = dW32 * np.float32(scale)
    return e4m3_encode(y), np.float32(np.max(np.abs(dW32))) if dW32.size else np.float32(0)


# --------------------------------------------------------------------------
# Input gradient (not on the pages)
# --------------------------------------------------------------------------


def linear_dgrad(dY_bits, W_bits, rows: Optional[Sequence[int]] = None,
                 cols: Optional[Sequence[int]] = None) -> np.ndarray:
    """dX[m,k] = sum_n dY[m,n] W[k,n], i.e. dX = dY W^T, in fp64.

    The pages give the forward pass and the DGE-corrected weight gradient but
    not the input gradient.  Reading R16: the chain rule of the forward's
    product A W, taken with the BF16 weight the caller passes (the unquantized
    W, as the compensation term uses).  Products of BF16 values are exact in
    fp64, so the result is the exact sum up to fp64 rounding; the caller rounds
    it to the output type.  rows select dX rows (tokens), cols select dX
    columns (input features).
    """
    dY = bf16_to_f32(np.asarray(dY_bits)).astype(np.float64)
    W = bf16_to_f32(np.asarray(W_bits)).astype(np.float64)
    rows = np.arange(dY.shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    cols = np.arange(W.shape[0]) if cols is None else np.asarray(cols, dtype=np.int64)
    return dY[rows] @ W[cols].T


# --------------------------------------------------------------------------
# One whole forward pass, for smoke tests and the CPU baseline
# --------------------------------------------------------------------------


def linear_layer_forward(A_bits, W_bits, q: float, rows: Optional[Iterable[int]] = None):
    """Quantile -> clamp + dA -> row / column quantization -> scaled FP4 GEMM +
    compensation, in the order page 1 gives (quantize at the start of forward,
    outlier clamp on A, FP4 GEMM).  Returns a dict of every intermediate."""
    t, t_bits, kk = quantile_threshold(A_bits, q)
    A_c, row_ptr, col_idx, vals = clamp_and_compensation(A_bits, t)
    a_codes, s_a = quantize_rows(A_c)
    w_codes_t, s_w = quantize_cols(bf16_to_f32(W_bits))
    rows = None if rows is None else list(rows)
    Y = linear_fwd(a_codes, s_a, w_codes_t, s_w, row_ptr, col_idx, vals, W_bits, rows=rows)
    return dict(t=t, t_bits=t_bits, k=kk, A_c=A_c, row_ptr=row_ptr, col_idx=col_idx, vals=vals,
                a_codes=a_codes, s_a=s_a, w_codes_t=w_codes_t, s_w=s_w, Y=Y)
