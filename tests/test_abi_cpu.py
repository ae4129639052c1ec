"""The C-ABI library loads and exports every entry point include/fp4lin.h
declares; host-side argument validation and host-only helpers work without a
GPU (no kernel is launched here)."""
import ctypes
import math
import os
import re

import pytest

from precision_gemm_row_gb300 import build as fp4build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    path = fp4build.build()
    return ctypes.CDLL(path)


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "fp4lin.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return [n for n in names if n not in ("if", "return")]


def test_header_declares_the_hot_path_entry_points():
    names = set(_declared_functions())
    for fn in ("fp4_quantize_rows", "fp4_quantize_cols", "outlier_clamp_quantile", "fp4_linear_fwd",
               "fp4_linear_wgrad_dge", "fp4_linear_dgrad"):
        assert fn in names


def test_library_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), f"missing export {n}"


def test_binding_names_match_header():
    from precision_gemm_row_gb300 import fp4lin
    assert set(fp4lin.EXPORTS) == set(_declared_functions())
    for n in fp4lin.EXPORTS:
        if n not in ("fp4_status_string", "fp4_abi_version", "fp4_last_cuda_error"):
            assert hasattr(fp4lin, n)


def test_status_strings(lib):
    lib.fp4_status_string.restype = ctypes.c_char_p
    assert lib.fp4_status_string(0) == b"FP4_OK"
    assert lib.fp4_status_string(6) == b"FP4_ERR_TIMEOUT"
    assert lib.fp4_status_string(123) == b"FP4_ERR_UNKNOWN"
    assert lib.fp4_abi_version() == 2


def test_outlier_max_nnz_is_n_minus_rank(lib):
    lib.outlier_max_nnz.restype = ctypes.c_int64
    lib.outlier_max_nnz.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_double]
    for M, K, q in [(256, 512, 0.99), (8192, 2048, 0.999), (16384, 5120, 0.97), (7, 9, 1.0), (3, 8, 1e-9)]:
        n = M * K
        k = min(n, max(1, math.ceil(q * n)))
        assert lib.outlier_max_nnz(M, K, q) == n - k
    assert lib.outlier_max_nnz(4, 8, 0.0) == 0
    assert lib.outlier_max_nnz(4, 8, 1.5) == 0


def test_workspace_sizes(lib):
    lib.fp4_quantize_cols_workspace.restype = ctypes.c_size_t
    lib.fp4_quantize_cols_workspace.argtypes = [ctypes.c_int64]
    assert lib.fp4_quantize_cols_workspace(5504) >= 5504 * 4
    lib.outlier_clamp_quantile_workspace.restype = ctypes.c_size_t
    lib.outlier_clamp_quantile_workspace.argtypes = [ctypes.c_int64] * 3
    ws = lib.outlier_clamp_quantile_workspace(8192, 2048, 16778)
    assert ws >= 32768 * 4 + 8192 * 12 + 16778 * 8


def test_fwd_workspace_size(lib):
    lib.fp4_linear_fwd_workspace.restype = ctypes.c_size_t
    lib.fp4_linear_fwd_workspace.argtypes = [ctypes.c_int64] * 3
    small = lib.fp4_linear_fwd_workspace(256, 512, 512)
    big = lib.fp4_linear_fwd_workspace(8192, 5504, 2048)
    # two 512-byte TF32 planes per row of M and per row of N, plus small tables
    assert big >= 2 * 512 * (8192 + 5504)
    assert 0 < small < big
    assert lib.fp4_linear_fwd_workspace(256, 512, 48) == 0      # K not a multiple of 32
    assert lib.fp4_linear_fwd_workspace(0, 512, 512) == 0


def test_host_validation_rejects_bad_arguments_without_launching(lib):
    from precision_gemm_row_gb300 import fp4lin  # noqa: F401  (declares argtypes)
    L = fp4lin._lib
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first
    # K not a multiple of 32
    assert L.fp4_quantize_rows(fake, 4, 40, 40, None, fake, 32, fake, None) == 2
    # misaligned leading dimension
    assert L.fp4_quantize_rows(fake, 4, 64, 65, None, fake, 32, fake, None) == 3
    # null pointers
    assert L.fp4_quantize_rows(None, 4, 64, 64, None, fake, 32, fake, None) == 1
    # q outside (0, 1]
    assert L.outlier_clamp_quantile(fake, 4, 64, 64, 0.0, fake, fake, fake, fake, 10, None, None, 0, fake, 1 << 20,
                                    None) == 1
    # capacity below the bound
    assert L.outlier_clamp_quantile(fake, 4, 64, 64, 0.5, fake, fake, fake, fake, 10, None, None, 0, fake, 1 << 20,
                                    None) == 5
    # workspace too small
    assert L.outlier_clamp_quantile(fake, 4, 64, 64, 0.5, fake, fake, fake, fake, 200, None, None, 0, fake, 16,
                                    None) == 4
    # bad output type / bad K for the GEMM
    assert L.fp4_linear_fwd(fake, 32, fake, fake, 32, fake, 4, 8, 64, None, None, None, None, 0, fake, 7, 8,
                            None, 0, None) == 1
    assert L.fp4_linear_fwd(fake, 32, fake, fake, 32, fake, 4, 8, 48, None, None, None, None, 0, fake, 0, 8,
                            None, 0, None) == 2
    # partial CSR
    assert L.fp4_linear_fwd(fake, 32, fake, fake, 32, fake, 4, 8, 64, fake, None, None, None, 0, fake, 0, 8,
                            None, 0, None) == 1
    # compensation workspace given but too small
    assert L.fp4_linear_fwd(fake, 32, fake, fake, 32, fake, 4, 8, 64, fake, fake, fake, fake, 8, fake, 0, 8,
                            fake, 16, None) == 4
    # DGE parameters
    assert L.fp4_linear_wgrad_dge(fake, 64, fake, 8, fake, 8, fake, 4, 8, 64, 0.0, 3.0, fake, 0, 8, None, None, None, 0,
                                  None) == 1
    # unknown dW type; E4M3 without its scale or running maximum
    assert L.fp4_linear_wgrad_dge(fake, 64, fake, 8, fake, 8, fake, 4, 8, 64, 5.0, 3.0, fake, 2, 8, None, None, None, 0,
                                  None) == 1
    assert L.fp4_linear_wgrad_dge(fake, 64, fake, 8, fake, 8, fake, 4, 8, 64, 5.0, 3.0, fake, 1, 8, None, fake, None, 0,
                                  None) == 1
    assert L.fp4_linear_wgrad_dge(fake, 64, fake, 8, fake, 8, fake, 4, 8, 64, 5.0, 3.0, fake, 1, 8, fake, None, None, 0,
                                  None) == 1
    # input gradient: raw accumulator is not an output type; ragged N; misaligned leading dimension
    assert L.fp4_linear_dgrad(fake, 64, fake, 64, 4, 64, 16, fake, 2, 16, None, 0, None) == 1
    assert L.fp4_linear_dgrad(None, 64, fake, 64, 4, 64, 16, fake, 0, 16, None, 0, None) == 1
    assert L.fp4_linear_dgrad(fake, 64, fake, 64, 4, 60, 16, fake, 0, 16, None, 0, None) == 2
    assert L.fp4_linear_dgrad(fake, 64, fake, 64, 4, 64, 16, fake, 0, 12, None, 0, None) == 2
    assert L.fp4_linear_dgrad(fake, 64, fake, 64, 4, 64, 16, fake, 1, 20, None, 0, None) == 3
    assert L.fp4_quantize_cols(fake, 64, 12, 16, fake, 32, fake, fake, 1 << 10, None) == 2
    assert L.fp4_selftest_bounded_wait(0, None) == 1


def _declared_arities():
    """Number of parameters of every function include/fp4lin.h declares."""
    text = open(os.path.join(ROOT, "include", "fp4lin.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    out = {}
    for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(([^;{]*?)\)\s*;",
                         text, flags=re.M | re.S):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_argument_counts_match_header():
    """Every ctypes prototype in the binding takes as many arguments as the C
    declaration (a stale prototype would pass wrong values through the ABI)."""
    fp4build.build()
    from precision_gemm_row_gb300 import fp4lin
    arities = _declared_arities()
    assert len(arities) >= 12
    for name, n in arities.items():
        argtypes = getattr(fp4lin._lib, name).argtypes
        assert argtypes is not None, name
        assert len(argtypes) == n, (name, len(argtypes), n)


def test_dense_compensation_is_chosen_from_the_entry_bound(lib):
    """linear_forward multiplies dA densely when the host bound n - ceil(q n)
    averages at least DENSE_MIN_ROW_ENTRIES entries per row (and K % 64 == 0):
    the Student-t stress case at q = 0.97 / 0.99 (153 / 51 per row), not the
    13B layer at q = 0.999 (5 / 14 per row)."""
    from precision_gemm_row_gb300 import fp4lin
    assert fp4lin.outlier_max_nnz(16384, 5120, 0.97) == 16384 * 5120 - math.ceil(0.97 * 16384 * 5120)
    assert fp4lin.use_dense_compensation(16384, 5120, 0.97)
    assert fp4lin.use_dense_compensation(16384, 5120, 0.99)
    assert not fp4lin.use_dense_compensation(16384, 5120, 0.999)
    assert not fp4lin.use_dense_compensation(16384, 13824, 0.999)
    assert not fp4lin.use_dense_compensation(16384, 5120 + 32, 0.9)      # K % 64 != 0
    # the boundary: exactly DENSE_MIN_ROW_ENTRIES entries per row on average
    M, K = 1000, 6400
    q_at = 1.0 - fp4lin.DENSE_MIN_ROW_ENTRIES / K
    assert fp4lin.outlier_max_nnz(M, K, q_at) >= fp4lin.DENSE_MIN_ROW_ENTRIES * M - 1
