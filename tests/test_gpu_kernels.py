"""GPU parity of every kernel against the CPU oracle, element by element, on
seeded inputs at sizes the oracle finishes in seconds: several tiles, ragged
tails in M, N and K, and the degenerate cases (zero rows, negative zeros, ties,
q = 1, all-equal magnitudes).  All calls go through the C ABI."""
import numpy as np
import pytest
import torch

from oracle import fp4_linear as orc
from precision_gemm_row_gb300 import workloads as wl
from tests.gpu_common import (BF16_ULP_TOL, FROB_TOL, TC_SUM_BOUND, assert_bf16_compensated_close,
                              assert_no_device_flags, bf16_ulp_distance, dev_bf16, host_bits, rel_frobenius)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp4():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from precision_gemm_row_gb300 import build
    build.build()
    from precision_gemm_row_gb300 import fp4lin
    return fp4lin


def _normal_bits(seed, shape, std=1.0):
    rng = np.random.default_rng(seed)
    return wl.f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32) * np.float32(std))


def _t3_bits(seed, shape, scale=1.0):
    rng = np.random.default_rng(seed)
    return wl.f32_to_bf16_bits(rng.standard_t(3, size=shape).astype(np.float32) * np.float32(scale))


# ---------------------------------------------------------------- bounded waits

def test_bounded_wait_times_out_and_context_survives(fp4):
    fp4.fp4_selftest_bounded_wait(2000)          # 2 ms wait on an mbarrier nobody completes
    name, flags = fp4.fp4_device_status()
    assert name == "FP4_ERR_TIMEOUT" and flags & fp4.FLAG_TIMEOUT
    assert fp4.fp4_device_status() == ("FP4_OK", 0)   # flags were cleared
    x = torch.ones(1024, device="cuda")
    assert float(x.sum()) == 1024.0                    # context still usable


# ---------------------------------------------------------------- row / column quantization

@pytest.mark.parametrize("M,K", [(256, 512), (37, 96), (5, 4096), (3, 13824), (130, 11008), (1, 32)])
def test_quantize_rows_bit_exact(fp4, M, K):
    A_bits = _normal_bits(M * 7 + K, (M, K))
    A_bits[0, :] = 0                      # zero row -> scale 1, all codes 0
    if M > 2:
        A_bits[2, ::3] = 0x8000           # negative zeros keep their sign
        A_bits[1, 5] = wl.f32_to_bf16_bits(np.array([60.0], np.float32))[0]
    codes, s = fp4.fp4_quantize_rows(dev_bf16(A_bits))
    ref_codes, ref_s = orc.quantize_rows(orc.bf16_to_f32(A_bits))
    assert np.array_equal(s.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))
    assert np.array_equal(codes.cpu().numpy(), ref_codes)
    assert_no_device_flags(fp4)


@pytest.mark.parametrize("absmax", [6.0, 3.0, 12.0, 0.375, 1.5 * 2.0 ** -100])
def test_quantize_rows_every_bf16_value_bit_exact(fp4, absmax):
    # every finite BF16 magnitude up to absmax, both signs, in rows that each hold
    # absmax once: the scale is 6/absmax for every row, so all scaled values
    # (grid points, ties, boundaries, subnormals, zeros) are exercised
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = orc.bf16_to_f32(bits)
    keep = np.isfinite(vals) & (np.abs(vals) <= np.float32(absmax))
    bits = bits[keep]
    per_row = 255
    n_rows = -(-bits.size // per_row)
    pad = np.zeros(n_rows * per_row, np.uint16)
    pad[:bits.size] = bits
    top = wl.f32_to_bf16_bits(np.array([absmax], np.float32))[0]
    A_bits = np.concatenate([pad.reshape(n_rows, per_row), np.full((n_rows, 1), top, np.uint16)], axis=1)
    codes, s = fp4.fp4_quantize_rows(dev_bf16(A_bits))
    ref_codes, ref_s = orc.quantize_rows(orc.bf16_to_f32(A_bits))
    assert np.array_equal(s.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))
    got = codes.cpu().numpy()
    bad = np.argwhere(got != ref_codes)
    assert bad.size == 0, [(int(A_bits[r, 2 * c]), int(A_bits[r, 2 * c + 1]), int(got[r, c]), int(ref_codes[r, c]))
                           for r, c in bad[:8]]


def test_quantize_rows_with_fused_clamp_bit_exact(fp4):
    A_bits = _t3_bits(1, (96, 640), 2.0)
    t, _, _ = orc.quantile_threshold(A_bits, 0.97)
    A_c, _, _, _ = orc.clamp_and_compensation(A_bits, t)
    ref_codes, ref_s = orc.quantize_rows(A_c)
    t_dev = torch.tensor([float(t)], dtype=torch.float32, device="cuda")
    codes, s = fp4.fp4_quantize_rows(dev_bf16(A_bits), clamp_t=t_dev)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))
    assert np.array_equal(codes.cpu().numpy(), ref_codes)


@pytest.mark.parametrize("t", [2.7182817, 0.3, 1e30])
def test_quantize_rows_with_arbitrary_fp32_clamp(fp4, t):
    # a clamp threshold that is not a BF16 value is applied in fp32: x' = sign(x) min(|x|, t)
    A_bits = _t3_bits(7, (64, 512), 2.0)
    A = orc.bf16_to_f32(A_bits)
    tf = np.float32(t)
    A_c = np.where(np.abs(A) > tf, np.copysign(tf, A), A).astype(np.float32)
    ref_codes, ref_s = orc.quantize_rows(A_c)
    codes, s = fp4.fp4_quantize_rows(dev_bf16(A_bits), clamp_t=torch.tensor([t], dtype=torch.float32, device="cuda"))
    assert np.array_equal(s.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))
    assert np.array_equal(codes.cpu().numpy(), ref_codes)


def test_quantize_rows_strided_input(fp4):
    A_bits = _normal_bits(3, (20, 200))
    big = dev_bf16(A_bits)
    view = big[:, :160]                   # lda = 200 > K = 160
    codes = torch.full((20, 96), 0xAB, dtype=torch.uint8, device="cuda")   # ldc 96 > K/2, padding kept
    fp4.fp4_quantize_rows(view, codes=codes)
    ref_codes, _ = orc.quantize_rows(orc.bf16_to_f32(A_bits[:, :160]))
    got = codes.cpu().numpy()
    assert np.array_equal(got[:, :80], ref_codes)
    assert np.all(got[:, 80:] == 0xAB)


@pytest.mark.parametrize("K,N", [(512, 512), (96, 40), (2048, 264), (64, 8)])
def test_quantize_cols_bit_exact(fp4, K, N):
    W_bits = _normal_bits(K + N, (K, N), 0.02)
    W_bits[:, 1] = 0                      # zero column
    codes_t, s = fp4.fp4_quantize_cols(dev_bf16(W_bits))
    ref_codes, ref_s = orc.quantize_cols(orc.bf16_to_f32(W_bits))
    assert np.array_equal(s.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))
    assert np.array_equal(codes_t.cpu().numpy(), ref_codes)


# ---------------------------------------------------------------- quantile, clamp, CSR

def _check_outlier(fp4, A_bits, q, want_clamped=True):
    o = fp4.outlier_clamp_quantile(dev_bf16(A_bits), q, want_clamped=want_clamped)
    torch.cuda.synchronize()
    t, t_bits, k = orc.quantile_threshold(A_bits, q)
    A_c, rp, ci, cv = orc.clamp_and_compensation(A_bits, t)
    assert o["t"].cpu().numpy().view(np.uint32)[0] == np.float32(t).view(np.uint32)
    nnz = int(o["nnz"].item())
    assert nnz == rp[-1]
    assert np.array_equal(o["row_ptr"].cpu().numpy(), rp)
    assert np.array_equal(o["col_idx"][:nnz].cpu().numpy(), ci)
    assert np.array_equal(o["vals"][:nnz].cpu().numpy().view(np.uint32), cv.view(np.uint32))
    if want_clamped:
        assert np.array_equal(host_bits(o["A_clamped"]), (A_c.view(np.uint32) >> 16).astype(np.uint16))
    assert_no_device_flags(fp4)
    return o


@pytest.mark.parametrize("q", [0.99, 0.9, 0.5, 0.999, 1.0, 1e-7])
def test_outlier_clamp_c1_shape(fp4, q):
    lin = wl.WORKLOADS["c1_single_linear_256x512x512"].linears[0]
    A_bits = wl.WORKLOADS["c1_single_linear_256x512x512"].activation(lin)
    _check_outlier(fp4, A_bits, q)


@pytest.mark.parametrize("shape,q", [((300, 136), 0.97), ((1, 8), 0.5), ((7, 1000), 0.999), ((2048, 64), 0.99)])
def test_outlier_clamp_ragged_and_heavy_tails(fp4, shape, q):
    _check_outlier(fp4, _t3_bits(shape[0] + shape[1], shape, 3.0), q)


def test_outlier_clamp_heavy_ties_and_zeros(fp4):
    rng = np.random.default_rng(5)
    vals = wl.f32_to_bf16_bits(np.array([0.5, -0.5, 1.0, -2.0, 2.0, 3.0], np.float32))
    A_bits = rng.choice(vals, size=(64, 96))
    for q in (0.3, 0.6, 0.95, 1.0):
        _check_outlier(fp4, A_bits, q)
    _check_outlier(fp4, np.zeros((16, 32), np.uint16), 0.9)          # t = 0, nothing clamped


def test_outlier_clamp_repeated_calls_reuse_workspace(fp4):
    A1 = _t3_bits(11, (128, 256))
    A2 = _t3_bits(12, (128, 256), 10.0)
    o = _check_outlier(fp4, A1, 0.99)
    o2 = fp4.outlier_clamp_quantile(dev_bf16(A2), 0.99, out={"workspace": o["workspace"]})
    t, _, _ = orc.quantile_threshold(A2, 0.99)
    assert float(o2["t"].item()) == float(t)


@pytest.mark.parametrize("shape,q", [((256, 512), 0.99), ((300, 1056), 0.97), ((37, 13824), 0.999), ((5, 4096), 0.5),
                                     ((129, 96), 1.0)])
def test_fused_rows_outliers_matches_oracle_and_separate_calls(fp4, shape, q):
    A_bits = _t3_bits(shape[0] * 3 + shape[1], shape, 2.0)
    A = dev_bf16(A_bits)
    o = fp4.fp4_quantize_rows_outliers(A, q)
    torch.cuda.synchronize()
    t, _, _ = orc.quantile_threshold(A_bits, q)
    A_c, rp, ci, cv = orc.clamp_and_compensation(A_bits, t)
    ref_codes, ref_s = orc.quantize_rows(A_c)
    nnz = int(o["nnz"].item())
    assert o["t"].cpu().numpy().view(np.uint32)[0] == np.float32(t).view(np.uint32)
    assert np.array_equal(o["row_ptr"].cpu().numpy(), rp)
    assert np.array_equal(o["col_idx"][:nnz].cpu().numpy(), ci)
    assert np.array_equal(o["vals"][:nnz].cpu().numpy().view(np.uint32), cv.view(np.uint32))
    assert np.array_equal(o["codes"].cpu().numpy(), ref_codes)
    assert np.array_equal(o["scales"].cpu().numpy().view(np.uint32), ref_s.view(np.uint32))
    # same bytes as the two separate entry points
    o2 = fp4.outlier_clamp_quantile(A, q)
    codes2, s2 = fp4.fp4_quantize_rows(A, clamp_t=o2["t"])
    assert torch.equal(codes2, o["codes"]) and torch.equal(s2.view(torch.int32), o["scales"].view(torch.int32))
    assert_no_device_flags(fp4)


@pytest.mark.parametrize("q", [0.005, 0.3, 0.9999])
def test_fused_rows_outliers_every_finite_bf16_pattern(fp4, q):
    """All 65536 BF16 patterns (non-finite ones replaced by +-0) as a 256 x 256
    matrix, shuffled by rows: the packed magnitude max, the outlier test and the
    clamp must treat zeros, subnormals (q = 0.005 puts t among them), ties with
    t and the largest finite values exactly as the oracle's integer order."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = (bits & np.uint16(0x7F80)) != np.uint16(0x7F80)
    bits = np.where(finite, bits, bits & np.uint16(0x8000)).astype(np.uint16)
    A_bits = bits[np.random.default_rng(7).permutation(65536)].reshape(256, 256)
    o = fp4.fp4_quantize_rows_outliers(dev_bf16(A_bits), q)
    torch.cuda.synchronize()
    t, _, _ = orc.quantile_threshold(A_bits, q)
    A_c, rp, ci, cv = orc.clamp_and_compensation(A_bits, t)
    ref_codes, ref_s = orc.quantize_rows(A_c)
    nnz = int(o["nnz"].item())
    assert o["t"].cpu().numpy().view(np.uint32)[0] == np.float32(t).view(np.uint32)
    assert np.array_equal(o["row_ptr"].cpu().numpy(), rp)
    assert np.array_equal(o["col_idx"][:nnz].cpu().numpy(), ci)
    assert np.array_equal(o["vals"][:nnz].cpu().numpy().view(np.uint32), cv.view(np.uint32))
    assert np.array_equal(o["codes"].cpu().numpy(), ref_codes)
    assert np.array_equal(o["scales"].cpu().numpy().view(np.uint32), ref_s.view(np.uint32))
    assert_no_device_flags(fp4)


# ---------------------------------------------------------------- DGE weight gradient

@pytest.mark.parametrize("M,K,N", [(1, 8, 8), (1, 200, 264), (64, 128, 256), (256, 512, 512), (200, 136, 264),
                                   (1000, 384, 520), (1500, 1032, 520), (2048, 200, 264), (2304, 520, 520),
                                   (4100, 384, 136)])
@pytest.mark.parametrize("k,clip", [(5.0, 3.0), (1.0, 3.0)])
@pytest.mark.parametrize("workspace", ["auto", None])
def test_wgrad_dge(fp4, M, K, N, k, clip, workspace):
    """A single token (M = 1) and the smallest K, N; M >= 2048 tokens runs the GEMM
    as CTA pairs (256-row dW tiles; K = 200, 520 and 384 leave partial pair
    tiles, N = 264 / 136 partial column tiles).  With a
    workspace, these few-tile shapes with 2 or more 1024-token chunks (M = 1500
    and up) compute every tile as two halves of the token range (in 2048- or
    1024-token chunks, whichever halves it more evenly)."""
    A_bits = _normal_bits(M + 1, (M, K))
    dY_bits = _normal_bits(N + 2, (M, N), 1e-3)
    W_bits = _normal_bits(K + 3, (K, N), 0.02)
    _, s_w = orc.quantize_cols(orc.bf16_to_f32(W_bits))
    dW = fp4.fp4_linear_wgrad_dge(dev_bf16(A_bits), dev_bf16(dY_bits), dev_bf16(W_bits),
                                  torch.from_numpy(s_w).cuda(), k, clip, workspace=workspace)
    ref = orc.wgrad_dge(A_bits, dY_bits, W_bits, s_w, k, clip)
    err = rel_frobenius(dW.cpu().numpy(), ref)
    assert err <= FROB_TOL, err
    assert_no_device_flags(fp4)


# ---------------------------------------------------------------- input gradient

def _dgrad_ref(dY_bits, W_bits):
    ref = orc.linear_dgrad(dY_bits, W_bits)
    mag = orc.linear_dgrad(dY_bits & np.uint16(0x7FFF), W_bits & np.uint16(0x7FFF))
    return ref, mag


@pytest.mark.parametrize("M,N,K", [(1, 8, 8), (1, 2056, 264), (64, 128, 256), (200, 264, 136), (1000, 520, 392),
                                   (5, 8, 8), (129, 72, 1032), (300, 1096, 264), (300, 2056, 264), (2304, 4104, 520),
                                   (513, 16384, 8)])
@pytest.mark.parametrize("out", ["bf16", "fp32"])
@pytest.mark.parametrize("workspace", ["auto", None])
def test_dgrad(fp4, M, N, K, out, workspace):
    """N >= 2048 (a long reduction) runs CTA pairs (256-row tiles); M = 200, 1000,
    300, 2304, 513 leave partial row tiles, K = 136, 392, 264, 520, 8 partial
    column tiles, N = 264, 72, 1096, 2056, 4104 a partial last stage of 64.
    With a workspace, shapes with 2 or more 1024-element chunks (N = 1096 and
    up) split their few tiles into two halves of the N range (N = 2056 in
    1024-element chunks, halves of 1 and 2; N = 4104 in 2048-element chunks,
    halves of 1 and 2)."""
    dY_bits = _normal_bits(M + 7, (M, N), 1e-3)
    W_bits = _normal_bits(K + 11, (K, N), 0.02)
    dX = fp4.fp4_linear_dgrad(dev_bf16(dY_bits), dev_bf16(W_bits),
                              out_dtype=torch.bfloat16 if out == "bf16" else torch.float32, workspace=workspace)
    assert dX.shape == (M, K)
    ref, mag = _dgrad_ref(dY_bits, W_bits)
    if out == "bf16":
        assert_bf16_compensated_close(host_bits(dX), ref, mag, bound=TC_SUM_BOUND)
        got = orc.bf16_to_f32(host_bits(dX)).astype(np.float64)
        # rounding to BF16 dominates: the fp32 sums are far inside half an ulp
        assert rel_frobenius(got, ref) <= 2.0 ** -8
    else:
        got = dX.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - ref) <= TC_SUM_BOUND * mag)
        assert rel_frobenius(got, ref) <= FROB_TOL
    assert_no_device_flags(fp4)


def test_split_tail_is_deterministic_and_matches_whole_tiles(fp4):
    """The split tail (1.3B MLP up shapes: 176 weight-gradient tiles on 76 SM
    pairs leave 24 tiles for a last wave, computed as two halves) gives the same
    bits on every run, whichever half finishes first, and agrees with whole
    tiles to fp32 rounding of the two partial sums."""
    M, K, N = 8192, 2048, 5504
    assert fp4.fp4_linear_wgrad_dge_workspace(M, N, K) > 0
    A = torch.randn(M, K, device="cuda").bfloat16()
    dY = (torch.randn(M, N, device="cuda") * 1e-3).bfloat16()
    W = (torch.randn(K, N, device="cuda") * 0.02).bfloat16()
    s_w = (6.0 / W.float().abs().amax(0)).contiguous()
    runs = [fp4.fp4_linear_wgrad_dge(A, dY, W, s_w) for _ in range(3)]
    whole = fp4.fp4_linear_wgrad_dge(A, dY, W, s_w, workspace=None)
    for r in runs[1:]:
        assert torch.equal(r.view(torch.int32), runs[0].view(torch.int32))
    assert rel_frobenius(runs[0].cpu().numpy(), whole.cpu().numpy()) < 1e-6
    dX = [fp4.fp4_linear_dgrad(dY, W, out_dtype=torch.float32) for _ in range(3)]
    dX_whole = fp4.fp4_linear_dgrad(dY, W, out_dtype=torch.float32, workspace=None)
    for r in dX[1:]:
        assert torch.equal(r.view(torch.int32), dX[0].view(torch.int32))
    assert rel_frobenius(dX[0].cpu().numpy(), dX_whole.cpu().numpy()) < 1e-6
    assert_no_device_flags(fp4)


def test_linear_forward_and_backward_conveniences(fp4):
    """linear_forward / linear_backward chain the entry points of one layer step:
    their results equal the individual calls' (bit for bit) and the oracle's."""
    M, K, N, q = 200, 256, 264, 0.99
    A_bits = _t3_bits(11, (M, K), 2.0)
    W_bits = _normal_bits(12, (K, N), 0.02)
    dY_bits = _normal_bits(13, (M, N), 1e-3)
    A, W, dY = dev_bf16(A_bits), dev_bf16(W_bits), dev_bf16(dY_bits)
    Y, inter = fp4.linear_forward(A, W, q)
    dX, dW = fp4.linear_backward(A, W, dY, inter["s_w"])
    assert dX.shape == (M, K) and dX.dtype == torch.bfloat16 and dW.shape == (K, N)
    dW1 = fp4.fp4_linear_wgrad_dge(A, dY, W, inter["s_w"])
    dX1 = fp4.fp4_linear_dgrad(dY, W)
    assert torch.equal(dW.view(torch.int32), dW1.view(torch.int32))
    assert torch.equal(dX.view(torch.int16), dX1.view(torch.int16))
    _, s_w = orc.quantize_cols(orc.bf16_to_f32(W_bits))
    assert rel_frobenius(dW.cpu().numpy(), orc.wgrad_dge(A_bits, dY_bits, W_bits, s_w, 5.0, 3.0)) <= FROB_TOL
    ref, mag = _dgrad_ref(dY_bits, W_bits)
    assert_bf16_compensated_close(host_bits(dX), ref, mag, bound=TC_SUM_BOUND)
    assert_no_device_flags(fp4)


def test_dgrad_exact_on_integer_products(fp4):
    """Small integers: every product and partial sum is exact in fp32, so dX is
    the exact integer matrix bit for bit (checks operand order and tile
    placement without rounding in the way)."""
    M, N, K = 384, 4096, 264
    rng = np.random.default_rng(3)
    dY = rng.integers(-3, 4, size=(M, N)).astype(np.float32)
    W = rng.integers(-3, 4, size=(K, N)).astype(np.float32)
    dY_bits, W_bits = wl.f32_to_bf16_bits(dY), wl.f32_to_bf16_bits(W)
    dX = fp4.fp4_linear_dgrad(dev_bf16(dY_bits), dev_bf16(W_bits), out_dtype=torch.float32)
    ref = orc.linear_dgrad(dY_bits, W_bits)
    assert np.array_equal(dX.cpu().numpy(), ref.astype(np.float32))
    assert_no_device_flags(fp4)


def test_dgrad_output_leading_dimension(fp4):
    """dX written into a wider buffer: the columns past K keep their canary."""
    M, N, K, ld = 300, 520, 264, 272
    dY_bits = _normal_bits(1, (M, N), 1e-3)
    W_bits = _normal_bits(2, (K, N), 0.02)
    buf = torch.full((M, ld), -7.0, dtype=torch.float32, device="cuda")
    fp4.fp4_linear_dgrad(dev_bf16(dY_bits), dev_bf16(W_bits), dX=buf[:, :K])
    ref, mag = _dgrad_ref(dY_bits, W_bits)
    host = buf.cpu().numpy()
    assert np.all(host[:, K:] == -7.0)
    assert np.all(np.abs(host[:, :K].astype(np.float64) - ref) <= TC_SUM_BOUND * mag)
    assert_no_device_flags(fp4)


# ---------------------------------------------------------------- FP4 GEMM

def _random_codes(seed, rows, K):
    return np.random.default_rng(seed).integers(0, 256, size=(rows, K // 2), dtype=np.uint8)


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (256, 512, 512), (300, 520, 1056), (1, 8, 32), (129, 264, 96),
                                   (640, 1024, 2048)])
def test_gemm_raw_accumulator_bit_exact(fp4, M, N, K):
    a = _random_codes(M + K, M, K)
    w = _random_codes(N + K, N, K)
    Y = fp4.fp4_linear_fwd(torch.from_numpy(a).cuda(), None, torch.from_numpy(w).cuda(), None, K, out_type="raw")
    ref = orc.gemm_raw(a, w).astype(np.float32)
    got = Y.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), np.argwhere(got != ref)[:5]
    assert_no_device_flags(fp4)


@pytest.mark.parametrize("sign_pattern", ["all_pos", "alternating"])
def test_gemm_raw_exact_at_maximum_K(fp4, sign_pattern):
    # every product 6*6 = 36: the largest sums the exactness bound allows (K = 16384)
    M, N, K = 128, 256, 16384
    a = np.full((M, K // 2), 0x77, np.uint8)
    w = np.full((N, K // 2), 0x77, np.uint8)
    if sign_pattern == "alternating":
        a[::2] = 0xFF                       # rows of -6
        w[:, ::3] = 0xF7                    # every 3rd byte: (+6, -6)
    Y = fp4.fp4_linear_fwd(torch.from_numpy(a).cuda(), None, torch.from_numpy(w).cuda(), None, K, out_type="raw")
    ref = orc.gemm_raw(a, w).astype(np.float32)
    assert np.array_equal(Y.cpu().numpy(), ref)
    if sign_pattern == "all_pos":
        assert float(Y[0, 0]) == 36.0 * K


@pytest.mark.parametrize("workspace", ["auto", None])
@pytest.mark.parametrize("M,N,K,q", [(256, 512, 512, 0.99), (300, 520, 1056, 0.97), (129, 264, 96, 0.9)])
def test_linear_fwd_scaled_and_compensated(fp4, M, N, K, q, workspace):
    A_bits = _t3_bits(M, (M, K), 2.0)
    W_bits = _normal_bits(N, (K, N), 0.02)
    t, _, _ = orc.quantile_threshold(A_bits, q)
    A_c, rp, ci, cv = orc.clamp_and_compensation(A_bits, t)
    a_codes, s_a = orc.quantize_rows(A_c)
    w_codes, s_w = orc.quantize_cols(orc.bf16_to_f32(W_bits))
    d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    csr = {"row_ptr": d(rp), "col_idx": d(ci if ci.size else np.zeros(1, np.int32)),
           "vals": d(cv if cv.size else np.zeros(1, np.float32))}
    W = dev_bf16(W_bits)
    args = (d(a_codes), d(s_a), d(w_codes), d(s_w), K)
    y_comp = orc.linear_fwd(a_codes, s_a, w_codes, s_w, rp, ci, cv, W_bits)
    y_plain = orc.linear_fwd(a_codes, s_a, w_codes, s_w)
    # BF16, compensated: 1 ulp plus the fp32 bound of the epilogue sum (cancellation)
    yb = fp4.fp4_linear_fwd(*args, csr=csr, W=W, out_type="bf16", workspace=workspace)
    mag = orc.linear_fwd_magnitude(a_codes, s_a, w_codes, s_w, rp, ci, cv, W_bits)
    n_over = assert_bf16_compensated_close(host_bits(yb), y_comp, mag)
    assert n_over <= max(2, y_comp.size // 10000)
    # BF16 without compensation: strictly within 1 ulp
    yb0 = fp4.fp4_linear_fwd(*args, out_type="bf16")
    assert bf16_ulp_distance(host_bits(yb0), orc.f64_to_bf16(y_plain)).max() <= BF16_ULP_TOL
    # fp32, compensated: relative Frobenius
    yf = fp4.fp4_linear_fwd(*args, csr=csr, W=W, out_type="fp32", workspace=workspace)
    assert rel_frobenius(yf.cpu().numpy(), y_comp) <= FROB_TOL
    assert_no_device_flags(fp4)


@pytest.mark.parametrize("workspace", ["auto", None])
@pytest.mark.parametrize("bad_col", [-1, 96])
def test_linear_fwd_skips_and_reports_out_of_range_columns(fp4, workspace, bad_col):
    """A dA entry whose column lies outside W (a corrupt caller CSR) is skipped by
    both compensation paths and reported as FP4_ERR_INTERNAL; every other entry
    still counts (Y equals the oracle's result without that entry)."""
    M, N, K, q = 129, 264, 96, 0.9
    A_bits = _t3_bits(M + 5, (M, K), 2.0)
    W_bits = _normal_bits(N + 5, (K, N), 0.02)
    t, _, _ = orc.quantile_threshold(A_bits, q)
    A_c, rp, ci, cv = orc.clamp_and_compensation(A_bits, t)
    a_codes, s_a = orc.quantize_rows(A_c)
    w_codes, s_w = orc.quantize_cols(orc.bf16_to_f32(W_bits))
    e = int(rp[M // 2])                       # first entry of a middle row
    row = int(np.searchsorted(rp, e, side="right") - 1)
    assert rp[row] <= e < rp[row + 1]
    ci_bad = ci.copy()
    ci_bad[e] = bad_col
    keep = np.ones(ci.size, bool)
    keep[e] = False
    rp_ref = rp.copy()
    rp_ref[row + 1:] -= 1
    y_ref = orc.linear_fwd(a_codes, s_a, w_codes, s_w, rp_ref, ci[keep], cv[keep], W_bits)
    mag = orc.linear_fwd_magnitude(a_codes, s_a, w_codes, s_w, rp_ref, ci[keep], cv[keep], W_bits)
    d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    csr = {"row_ptr": d(rp), "col_idx": d(ci_bad), "vals": d(cv)}
    assert_no_device_flags(fp4)
    yb = fp4.fp4_linear_fwd(d(a_codes), d(s_a), d(w_codes), d(s_w), K, csr=csr, W=dev_bf16(W_bits), out_type="bf16",
                            workspace=workspace)
    name, flags = fp4.fp4_device_status()
    assert name == "FP4_ERR_INTERNAL" and flags & fp4.FLAG_INTERNAL, (name, flags)
    assert_bf16_compensated_close(host_bits(yb), y_ref, mag)
    assert_no_device_flags(fp4)


def _hot_channel_bits(seed, M, K, n_hot, scale=20.0):
    """N(0,1) activations with n_hot seeded channels multiplied by `scale` (outliers gather there)."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K)).astype(np.float32)
    hot = rng.choice(K, size=n_hot, replace=False)
    x[:, hot] *= scale
    return wl.f32_to_bf16_bits(x), np.sort(hot)


@pytest.mark.parametrize("M,N,K,n_hot", [(256, 512, 512, 10), (300, 520, 1056, 100), (129, 264, 2048, 128),
                                         (200, 240, 512, 129), (64, 16, 64, 1), (300, 520, 4096, 100),
                                         (100, 248, 4096, 7)])
def test_linear_fwd_compensation_paths_agree(fp4, M, N, K, n_hot):
    """dA confined to n_hot channels: up to 128 distinct columns run on the tensor
    cores (TF32 parts, several 32-column chunks), 129 fall back to the epilogue;
    both paths meet the compensated bound against the oracle.  K >= 4096 runs the
    GEMM as CTA pairs (256-row tiles; M = 100 and 300 leave partial pair tiles)."""
    A_bits, hot = _hot_channel_bits(M + n_hot, M, K, n_hot)
    W_bits = _normal_bits(N + K, (K, N), 0.02)
    # every entry of a hot channel above the threshold, none elsewhere: keep 30% of the hot entries
    q = 1.0 - 0.3 * n_hot / K
    t, _, _ = orc.quantile_threshold(A_bits, q)
    A_c, rp, ci, cv = orc.clamp_and_compensation(A_bits, t)
    assert set(np.unique(ci)) <= set(hot.tolist())
    distinct = np.unique(ci).size
    a_codes, s_a = orc.quantize_rows(A_c)
    w_codes, s_w = orc.quantize_cols(orc.bf16_to_f32(W_bits))
    d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    csr = {"row_ptr": d(rp), "col_idx": d(ci), "vals": d(cv)}
    W = dev_bf16(W_bits)
    args = (d(a_codes), d(s_a), d(w_codes), d(s_w), K)
    y_comp = orc.linear_fwd(a_codes, s_a, w_codes, s_w, rp, ci, cv, W_bits)
    mag = orc.linear_fwd_magnitude(a_codes, s_a, w_codes, s_w, rp, ci, cv, W_bits)
    for ws in ("auto", None):
        yb = fp4.fp4_linear_fwd(*args, csr=csr, W=W, out_type="bf16", workspace=ws)
        n_over = assert_bf16_compensated_close(host_bits(yb), y_comp, mag)
        assert n_over <= max(2, y_comp.size // 10000)
        yf = fp4.fp4_linear_fwd(*args, csr=csr, W=W, out_type="fp32", workspace=ws)
        assert rel_frobenius(yf.cpu().numpy(), y_comp) <= FROB_TOL
    assert distinct == n_hot or n_hot == 1
    assert_no_device_flags(fp4)


def test_linear_fwd_output_leading_dimension(fp4):
    M, N, K = 130, 48, 64
    a = _random_codes(1, M, K)
    w = _random_codes(2, N, K)
    Y = torch.full((M, 64), -7.0, dtype=torch.float32, device="cuda")
    fp4.fp4_linear_fwd(torch.from_numpy(a).cuda(), None, torch.from_numpy(w).cuda(), None, K, out_type="raw",
                       Y=Y[:, :N])
    got = Y.cpu().numpy()
    assert np.array_equal(got[:, :N], orc.gemm_raw(a, w).astype(np.float32))
    assert np.all(got[:, N:] == -7.0)


# ---------------------------------------------------------------- whole forward pass

def test_linear_forward_pipeline_c1(fp4):
    wlc = wl.WORKLOADS["c1_single_linear_256x512x512"]
    lin = wlc.linears[0]
    A_bits, W_bits = wlc.activation(lin), wlc.weight(lin)
    Y, inter = fp4.linear_forward(dev_bf16(A_bits), dev_bf16(W_bits), lin.q)
    ref = orc.linear_layer_forward(A_bits, W_bits, lin.q)
    assert float(inter["outlier"]["t"].item()) == float(ref["t"])
    assert np.array_equal(inter["a_codes"].cpu().numpy(), ref["a_codes"])
    assert np.array_equal(inter["w_codes_t"].cpu().numpy(), ref["w_codes_t"])
    mag = orc.linear_fwd_magnitude(ref["a_codes"], ref["s_a"], ref["w_codes_t"], ref["s_w"], ref["row_ptr"],
                                   ref["col_idx"], ref["vals"], W_bits)
    assert_bf16_compensated_close(host_bits(Y), ref["Y"], mag)
    assert_no_device_flags(fp4)


# ---------------------------------------------------------------- binding checks

def test_binding_rejects_undersized_or_mistyped_buffers(fp4):
    """The C ABI cannot see buffer sizes, so the binding checks every tensor it
    passes: an output too small, of the wrong dtype or on the wrong device is
    refused before any launch (nothing is written)."""
    K, N, M = 256, 64, 32
    W = dev_bf16(_normal_bits(1, (K, N), 0.02))
    A = dev_bf16(_normal_bits(2, (M, K)))
    u8 = lambda *s: torch.zeros(s, dtype=torch.uint8, device="cuda")
    f32 = lambda *s: torch.zeros(s, dtype=torch.float32, device="cuda")
    bad_calls = [
        lambda: fp4.fp4_quantize_cols(W, codes_t=u8(N - 1, K // 2)),
        lambda: fp4.fp4_quantize_cols(W, codes_t=u8(N, K // 2 - 16)),
        lambda: fp4.fp4_quantize_cols(W, scales=f32(N - 1)),
        lambda: fp4.fp4_quantize_cols(W, scales=torch.zeros(N, dtype=torch.float16, device="cuda")),
        lambda: fp4.fp4_quantize_cols(W, workspace=u8(8)),
        lambda: fp4.fp4_quantize_cols_noalloc(W, u8(N, K // 2), f32(N - 8)),
        lambda: fp4.fp4_quantize_cols_noalloc(W, u8(N, K // 2), torch.zeros(N)),            # host memory
        lambda: fp4.fp4_quantize_rows(A, codes=u8(M - 1, K // 2)),
        lambda: fp4.fp4_quantize_rows(A, scales=f32(M - 1)),
        lambda: fp4.fp4_quantize_rows_outliers(A, 0.99, out={"codes": u8(M, K // 2 - 16)}),
        lambda: fp4.fp4_quantize_rows_outliers(A, 0.99, out={"row_ptr": torch.zeros(M, dtype=torch.int32,
                                                                                      device="cuda")}),
        lambda: fp4.fp4_linear_wgrad_dge(A, dev_bf16(_normal_bits(3, (M, N))), W, f32(N - 1)),
        lambda: fp4.fp4_linear_dgrad(dev_bf16(_normal_bits(3, (M, N))), W, dX=f32(M, K - 8)),
    ]
    for i, call in enumerate(bad_calls):
        with pytest.raises(ValueError):
            call()
    codes, s_w = fp4.fp4_quantize_cols(W)
    a_codes, s_a = fp4.fp4_quantize_rows(A)
    with pytest.raises(ValueError):
        fp4.fp4_linear_fwd(a_codes, s_a, codes, s_w, K, Y=torch.zeros((M, N - 8), dtype=torch.bfloat16,
                                                                         device="cuda"))
    with pytest.raises(ValueError):
        fp4.fp4_linear_fwd(a_codes, s_a[: M - 1], codes, s_w, K)
    torch.cuda.synchronize()
    assert_no_device_flags(fp4)


# ---------------------------------------------------------------- wide pair tiles (K >= 4096)

@pytest.mark.parametrize("M,N,K", [(37, 8, 4096), (300, 240, 4096), (256, 480, 5120), (129, 1000, 4096),
                                   (1000, 5120, 4096), (8192, 4800, 4096), (512, 13824, 4096)])
def test_wide_gemm_raw_and_scaled(fp4, M, N, K):
    """The 256 x 480 pair-tile kernel that runs K >= 4096: a half narrower than 240
    (N = 8, 1000, 13824), a single half (N = 240), odd numbers of halves, partial
    pair rows (M = 37, 129, 1000), and a schedule that splits the last round of
    double tiles into single halves (M = 8192, N = 4800: 320 doubles on 76 pairs).
    The raw accumulator is checked against the oracle on small shapes and in full
    against torch._int_mm; BF16 output without compensation within 1 ulp."""
    from tests.gpu_common import assert_raw_acc_equals_int_mm
    a = _random_codes(M * 3 + N, M, K)
    w = _random_codes(N * 5 + K, N, K)
    da, dw = torch.from_numpy(a).cuda(), torch.from_numpy(w).cuda()
    raw = fp4.fp4_linear_fwd(da, None, dw, None, K, out_type="raw")
    assert_raw_acc_equals_int_mm(raw, da, dw)
    rows = np.unique(np.concatenate([np.arange(min(M, 3)), np.random.default_rng(M).choice(M, min(M, 24), replace=False),
                                     [M - 1]]))
    ref = orc.gemm_raw(a, w, rows=rows).astype(np.float32)
    got = raw[torch.from_numpy(rows).cuda()].cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    rng = np.random.default_rng(K + N)
    s_a = (rng.uniform(0.05, 4.0, M)).astype(np.float32)
    s_w = (rng.uniform(0.05, 4.0, N)).astype(np.float32)
    yb = fp4.fp4_linear_fwd(da, torch.from_numpy(s_a).cuda(), dw, torch.from_numpy(s_w).cuda(), K, out_type="bf16")
    y_ref = orc.linear_fwd(a, s_a, w, s_w, rows=rows)
    assert bf16_ulp_distance(host_bits(yb[torch.from_numpy(rows).cuda()]), orc.f64_to_bf16(y_ref)).max() <= BF16_ULP_TOL
    yf = fp4.fp4_linear_fwd(da, torch.from_numpy(s_a).cuda(), dw, torch.from_numpy(s_w).cuda(), K, out_type="fp32")
    np.testing.assert_allclose(yf[torch.from_numpy(rows).cuda()].cpu().numpy(), y_ref, rtol=2.0 ** -21, atol=0)
    assert_no_device_flags(fp4)


def test_outlier_pilot_misled_by_its_sample(fp4):
    """The row call draws a floor under the threshold from every 64th row of each
    CTA's row block (a pilot).  Here exactly those rows hold values 100 times
    larger, so the floor lands above the true threshold and the call must count
    the magnitudes below it in a second pass; t, the CSR and the codes stay
    bit-exact."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    M, K, q = 32 * sms, 512, 0.999
    rng = np.random.default_rng(11)
    x = rng.standard_normal((M, K)).astype(np.float32)
    sampled = np.zeros(M, bool)
    for b in range(sms):
        r0, r1 = M * b // sms, M * (b + 1) // sms
        sampled[r0:r1:64] = True
    x[sampled] *= np.float32(100.0)
    A_bits = wl.f32_to_bf16_bits(x)
    o = fp4.fp4_quantize_rows_outliers(dev_bf16(A_bits), q)
    t, t_bits, k = orc.quantile_threshold(A_bits, q)
    A_c, rp, ci, cv = orc.clamp_and_compensation(A_bits, t)
    # the true threshold lies among the large rows, and with 4x the exceedance
    # the pilot's floor is above it (the second pass is needed)
    assert float(o["t"].item()) == float(t)
    assert np.array_equal(o["row_ptr"].cpu().numpy(), rp)
    nnz = int(o["nnz"].item())
    assert nnz == rp[-1]
    assert np.array_equal(o["col_idx"][:nnz].cpu().numpy(), ci)
    assert np.array_equal(o["vals"][:nnz].cpu().numpy().view(np.uint32), cv.view(np.uint32))
    ref_codes, ref_s = orc.quantize_rows(A_c)
    assert np.array_equal(o["codes"].cpu().numpy(), ref_codes)
    assert np.array_equal(o["scales"].cpu().numpy().view(np.uint32), ref_s.view(np.uint32))
    assert_no_device_flags(fp4)


# ---------------------------------------------------------------- FP8 (E4M3) weight gradient

def _small_int_bits(seed, shape, lim):
    """BF16 patterns of integers in [-lim, lim]: sums of their products are exact in fp32."""
    rng = np.random.default_rng(seed)
    return wl.f32_to_bf16_bits(rng.integers(-lim, lim + 1, size=shape).astype(np.float32))


@pytest.mark.parametrize("M,K,N", [(300, 136, 264), (2100, 264, 136)])
@pytest.mark.parametrize("headroom", [1.0, 4.0])
@pytest.mark.parametrize("workspace", ["auto", None])
def test_wgrad_fp8_bit_exact_when_the_gradient_is_exact(fp4, M, K, N, headroom, workspace):
    """With k = 1 the DGE factor is exactly 1, and integer-valued A and dY make
    every sum exact in fp32, so dW is exact on both sides and the E4M3 codes
    must match the oracle's bit for bit: round half to even, sign of zero, and
    (headroom 4: the scale is 4x 448 / amax) saturation at 448.  M = 2100 runs
    CTA pairs and, with a workspace, the split tail."""
    A_bits = _small_int_bits(M, (M, K), 3)
    dY_bits = _small_int_bits(N + 1, (M, N), 2)
    W_bits = _normal_bits(K + 3, (K, N), 0.02)
    _, s_w = orc.quantize_cols(orc.bf16_to_f32(W_bits))
    ref32 = orc.wgrad_dge(A_bits, dY_bits, W_bits, s_w, 1.0, 3.0)
    scale = np.float32(headroom * 448.0 / float(np.max(np.abs(ref32))))
    ref_codes, ref_amax = orc.wgrad_dge_fp8(ref32, float(scale))
    codes, amax = fp4.fp4_linear_wgrad_dge(dev_bf16(A_bits), dev_bf16(dY_bits), dev_bf16(W_bits),
                                           torch.from_numpy(s_w).cuda(), 1.0, 3.0, workspace=workspace,
                                           dw_type="e4m3", dw_scale=torch.tensor([float(scale)], dtype=torch.float32, device="cuda"))
    np.testing.assert_array_equal(codes.cpu().numpy(), ref_codes)
    assert float(amax.item()) == float(ref_amax)
    if headroom > 1:
        assert np.count_nonzero((ref_codes & 0x7F) == 0x7E) > 0
    assert_no_device_flags(fp4)


@pytest.mark.parametrize("M,K,N", [(1, 8, 8), (1000, 392, 520), (4100, 384, 136)])
def test_wgrad_fp8_within_one_code_of_the_oracle(fp4, M, K, N):
    """With the DGE factor (k = 5) the fp32 gradient differs from the oracle's
    fp64 one in the last bits, so a code may differ by one step where fl32(dW s)
    lies next to a rounding boundary; every code is within one step of the
    oracle's, nearly all are equal, and amax agrees to fp32 rounding."""
    A_bits = _normal_bits(M + 1, (M, K))
    dY_bits = _normal_bits(N + 2, (M, N), 1e-3)
    W_bits = _normal_bits(K + 3, (K, N), 0.02)
    _, s_w = orc.quantize_cols(orc.bf16_to_f32(W_bits))
    ref32 = orc.wgrad_dge(A_bits, dY_bits, W_bits, s_w, 5.0, 3.0)
    scale = np.float32(448.0 / float(np.max(np.abs(ref32))))
    ref_codes, ref_amax = orc.wgrad_dge_fp8(ref32, float(scale))
    codes, amax = fp4.fp4_linear_wgrad_dge(dev_bf16(A_bits), dev_bf16(dY_bits), dev_bf16(W_bits),
                                           torch.from_numpy(s_w).cuda(), 5.0, 3.0, dw_type="e4m3",
                                           dw_scale=torch.tensor([float(scale)], dtype=torch.float32, device="cuda"))
    got = codes.cpu().numpy()

    def signed_step(c):   # E4M3 codes as a monotone signed integer scale
        c = c.astype(np.int32)
        return np.where(c & 0x80, -(c & 0x7F), c & 0x7F)

    assert np.max(np.abs(signed_step(got) - signed_step(ref_codes))) <= 1
    assert np.mean(got == ref_codes) >= 0.99
    assert abs(float(amax.item()) - float(ref_amax)) <= 1e-5 * float(ref_amax)
    assert_no_device_flags(fp4)


def test_wgrad_fp8_rejects_bad_arguments(fp4):
    A = dev_bf16(_normal_bits(1, (64, 64)))
    dY = dev_bf16(_normal_bits(2, (64, 64)))
    W = dev_bf16(_normal_bits(3, (64, 64)))
    s_w = torch.ones(64, dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        fp4.fp4_linear_wgrad_dge(A, dY, W, s_w, dw_type="e4m3")                  # no scale
    with pytest.raises(ValueError):
        fp4.fp4_linear_wgrad_dge(A, dY, W, s_w, dw_type="e5m2")
    with pytest.raises(ValueError):
        fp4.fp4_linear_wgrad_dge(A, dY, W, s_w, dw_scale=torch.ones(1, device="cuda"))   # fp32 with a scale


# ---------------------------------------------------------------- dense compensation

@pytest.mark.parametrize("M,K,N,q", [(300, 512, 264, 0.97), (2100, 1024, 520, 0.97), (129, 4096, 136, 0.99),
                                     (64, 64, 8, 0.9)])
@pytest.mark.parametrize("out", ["bf16", "fp32"])
@pytest.mark.parametrize("with_t", [True, False])
def test_linear_fwd_dense_compensation(fp4, M, K, N, q, out, with_t):
    """Heavy-tailed A clamped at a low quantile (dA in every tile), from the
    oracle's CSR and codes: Y = FP4 product + dA W with dA split into three BF16
    parts on the tensor cores.  fp32 Y within 1e-5 relative Frobenius of the
    fp64 oracle; BF16 Y within 1 ulp plus the tensor-core sum bound of the
    terms' magnitude.  3K >= 2048 (K = 1024, 4096) runs CTA pairs; K = 4096
    makes the FP4 product the 256 x 480 pair-tile kernel.  With the threshold t
    each entry is the two BF16 parts A and -sign(A) t (reduction 2K), without
    it three rounded parts (3K)."""
    A_bits = _t3_bits(M + K, (M, K))
    W_bits = _normal_bits(N + 7, (K, N), 0.02)
    t, _, _ = orc.quantile_threshold(A_bits, q)
    A_c, rp, ci, cv = orc.clamp_and_compensation(A_bits, t)
    assert rp[-1] >= 8 * M or M * K <= 4096          # dense enough to matter
    a_codes, s_a = orc.quantize_rows(A_c)
    w_codes, s_w = orc.quantize_cols(orc.bf16_to_f32(W_bits))
    csr = dict(row_ptr=torch.from_numpy(rp.astype(np.int32)).cuda(),
               col_idx=torch.from_numpy(np.asarray(ci, np.int32)).cuda(),
               vals=torch.from_numpy(np.asarray(cv, np.float32)).cuda())
    if with_t:
        csr["t"] = torch.tensor([float(t)], dtype=torch.float32, device="cuda")
    Y = fp4.fp4_linear_fwd_dense(torch.from_numpy(a_codes).cuda(), torch.from_numpy(s_a).cuda(),
                                 torch.from_numpy(w_codes).cuda(), torch.from_numpy(s_w).cuda(), K, csr=csr,
                                 W=dev_bf16(W_bits), out_type=out)
    y_ref = orc.linear_fwd(a_codes, s_a, w_codes, s_w, rp, ci, cv, W_bits)
    if out == "fp32":
        err = rel_frobenius(Y.cpu().numpy(), y_ref)
        assert err <= FROB_TOL, err
    else:
        mag = orc.linear_fwd_magnitude(a_codes, s_a, w_codes, s_w, rp, ci, cv, W_bits)
        assert_bf16_compensated_close(host_bits(Y), y_ref, mag, bound=TC_SUM_BOUND)
    assert_no_device_flags(fp4)


def test_linear_fwd_dense_rejects_bad_arguments(fp4):
    codes = torch.zeros((64, 48), dtype=torch.uint8, device="cuda")
    s = torch.ones(64, dtype=torch.float32, device="cuda")
    csr = dict(row_ptr=torch.zeros(65, dtype=torch.int32, device="cuda"),
               col_idx=torch.zeros(1, dtype=torch.int32, device="cuda"),
               vals=torch.zeros(1, dtype=torch.float32, device="cuda"))
    W = torch.zeros((96, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fp4.FP4Error):             # K % 64 != 0
        fp4.fp4_linear_fwd_dense(codes, s, torch.zeros((64, 48), dtype=torch.uint8, device="cuda"), s, 96,
                                 csr=csr, W=W)
    with pytest.raises(ValueError):
        fp4.fp4_linear_fwd_dense(codes, s, codes, s, 96, csr=csr, W=W, out_type="raw")


def test_linear_fwd_dense_reports_a_wrong_threshold(fp4):
    """A threshold that did not produce dA breaks the two-part premise: the
    call still multiplies a two-part rounding of each entry and raises the
    device-side INTERNAL flag."""
    M, K, N = 128, 256, 64
    A_bits = _t3_bits(5, (M, K))
    W_bits = _normal_bits(6, (K, N), 0.02)
    t, _, _ = orc.quantile_threshold(A_bits, 0.9)
    A_c, rp, ci, cv = orc.clamp_and_compensation(A_bits, t)
    a_codes, s_a = orc.quantize_rows(A_c)
    w_codes, s_w = orc.quantize_cols(orc.bf16_to_f32(W_bits))
    wrong = float(np.nextafter(np.float32(t), np.float32(np.inf)))     # not the clamp's threshold
    csr = dict(row_ptr=torch.from_numpy(rp.astype(np.int32)).cuda(),
               col_idx=torch.from_numpy(np.asarray(ci, np.int32)).cuda(),
               vals=torch.from_numpy(np.asarray(cv, np.float32)).cuda(),
               t=torch.tensor([wrong], dtype=torch.float32, device="cuda"))
    assert_no_device_flags(fp4)
    Y = fp4.fp4_linear_fwd_dense(torch.from_numpy(a_codes).cuda(), torch.from_numpy(s_a).cuda(),
                                 torch.from_numpy(w_codes).cuda(), torch.from_numpy(s_w).cuda(), K, csr=csr,
                                 W=dev_bf16(W_bits), out_type="fp32")
    name, flags = fp4.fp4_device_status()
    assert flags & 0x4, (name, flags)                                  # FP4_FLAG_INTERNAL (then cleared)
    y_ref = orc.linear_fwd(a_codes, s_a, w_codes, s_w, rp, ci, cv, W_bits)
    assert rel_frobenius(Y.cpu().numpy(), y_ref) <= 1e-4
    assert_no_device_flags(fp4)
