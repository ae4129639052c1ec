"""The allocation-free column quantizer (fp4_quantize_cols_noalloc) against the
regular one (fp4_quantize_cols with a caller workspace), through the C ABI.

fp4_quantize_cols_noalloc serves callers that cannot give the library scratch
memory; its column maxima live in a device array built into the library.  Two
calls in a row on different inputs show that each call starts from a cleared
array: the first call leaves large column maxima behind (values of scale 3),
the second quantizes smaller values (scale 0.02) in the same columns, so a
maximum left over from the first call would change the second call's scales
and codes.  Both calls are also checked against the oracle.  The file is
collected last so that, under `-x`, every other test has already run if this
one fails.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp4():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from precision_gemm_row_gb300 import build
    build.build()
    from precision_gemm_row_gb300 import fp4lin
    return fp4lin


def _weights(seed, K, N, std):
    rng = np.random.default_rng(seed)
    w = torch.from_numpy(rng.standard_normal((K, N)).astype(np.float32) * np.float32(std))
    return w.to(torch.bfloat16).cuda()


def test_noalloc_matches_workspace_variant_on_two_calls(fp4):
    from oracle import fp4_linear as orc
    # first call: large values over 5504 columns; second: small values over the
    # first 264 of the same columns (stale maxima would be larger than the new ones)
    cases = [(2048, 5504, 3.0, 0), (512, 264, 0.02, 1)]
    for K, N, std, seed in cases:
        W = _weights(seed, K, N, std)
        ref_codes, ref_scales = fp4.fp4_quantize_cols(W)
        codes = torch.full((N, K // 2), 0x5A, dtype=torch.uint8, device="cuda")
        scales = torch.full((N,), -1.0, dtype=torch.float32, device="cuda")
        st = fp4._lib.fp4_quantize_cols_noalloc(
            ctypes.c_void_p(W.data_ptr()), K, N, W.stride(0), ctypes.c_void_p(codes.data_ptr()), codes.stride(0),
            ctypes.c_void_p(scales.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == 0, fp4.status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(codes, ref_codes)
        assert torch.equal(scales.view(torch.int32), ref_scales.view(torch.int32))
        o_codes, o_scales = orc.quantize_cols(W.float().cpu().numpy())
        assert np.array_equal(codes.cpu().numpy(), o_codes)
        assert np.array_equal(scales.cpu().numpy().view(np.uint32), o_scales.view(np.uint32))
    assert fp4.fp4_device_status() == ("FP4_OK", 0)


def test_noalloc_rejects_too_many_columns(fp4):
    fake = ctypes.c_void_p(0x1000)     # never touched: the size check fails first
    st = fp4._lib.fp4_quantize_cols_noalloc(fake, 64, 65536 + 8, 65536 + 8, fake, 32, fake, None)
    assert fp4.status_string(st) == "FP4_ERR_SHAPE"
