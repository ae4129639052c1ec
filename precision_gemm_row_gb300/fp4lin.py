"""Python binding of libfp4lin.so (ctypes), argument marshalling only.

Every function has the name of the C entry point it calls and takes torch CUDA
tensors.  Outputs that are not passed in are allocated with torch (PyTorch is
used for device memory and streams only); every step of the computation runs
in the library's CUDA kernels.  There is no fallback: if the library is not
built, importing this module raises ImportError, and a non-zero status from the
library raises FP4Error.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfp4lin.so")

FP4_OUT_BF16, FP4_OUT_FP32, FP4_OUT_RAW_ACC_FP32 = 0, 1, 2
_OUT_TYPES = {"bf16": FP4_OUT_BF16, "fp32": FP4_OUT_FP32, "raw": FP4_OUT_RAW_ACC_FP32}
FLAG_TIMEOUT, FLAG_CAPACITY, FLAG_INTERNAL = 0x1, 0x2, 0x4

# exported symbols, in the order include/fp4lin.h declares them
EXPORTS = (
    "fp4_status_string", "fp4_abi_version", "fp4_last_cuda_error", "fp4_quantize_rows", "fp4_quantize_cols_workspace",
    "fp4_quantize_cols", "fp4_quantize_cols_noalloc", "outlier_max_nnz", "outlier_clamp_quantile_workspace", "outlier_clamp_quantile",
    "fp4_quantize_rows_outliers", "fp4_linear_fwd_workspace", "fp4_linear_fwd", "fp4_linear_fwd_dense_workspace",
    "fp4_linear_fwd_dense", "fp4_linear_wgrad_dge", "fp4_linear_wgrad_dge_workspace",
    "fp4_linear_dgrad", "fp4_linear_dgrad_workspace",
    "fp4_device_status", "fp4_selftest_bounded_wait",
)


class FP4Error(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: {msg} ({status})")
        self.status = status
        self.status_name = msg


_c_i64, _c_sz, _c_vp, _c_int, _c_f, _c_d, _c_u32 = (ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int,
                                                    ctypes.c_float, ctypes.c_double, ctypes.c_uint32)


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"{path} is not built: run precision_gemm_row_gb300.build.build() (needs nvcc, sm_103a)")
    lib = ctypes.CDLL(path)
    sig = {
        "fp4_status_string": (ctypes.c_char_p, [_c_int]),
        "fp4_abi_version": (_c_int, []),
        "fp4_last_cuda_error": (ctypes.c_char_p, []),
        "fp4_quantize_rows": (_c_int, [_c_vp, _c_i64, _c_i64, _c_i64, _c_vp, _c_vp, _c_i64, _c_vp, _c_vp]),
        "fp4_quantize_cols_workspace": (_c_sz, [_c_i64]),
        "fp4_quantize_cols": (_c_int, [_c_vp, _c_i64, _c_i64, _c_i64, _c_vp, _c_i64, _c_vp, _c_vp, _c_sz, _c_vp]),
        "fp4_quantize_cols_noalloc": (_c_int, [_c_vp, _c_i64, _c_i64, _c_i64, _c_vp, _c_i64, _c_vp, _c_vp]),
        "outlier_max_nnz": (_c_i64, [_c_i64, _c_i64, _c_d]),
        "outlier_clamp_quantile_workspace": (_c_sz, [_c_i64, _c_i64, _c_i64]),
        "outlier_clamp_quantile": (_c_int, [_c_vp, _c_i64, _c_i64, _c_i64, _c_d, _c_vp, _c_vp, _c_vp, _c_vp,
                                            _c_i64, _c_vp, _c_vp, _c_i64, _c_vp, _c_sz, _c_vp]),
        "fp4_quantize_rows_outliers": (_c_int, [_c_vp, _c_i64, _c_i64, _c_i64, _c_d, _c_vp, _c_i64, _c_vp, _c_vp,
                                                _c_vp, _c_vp, _c_vp, _c_i64, _c_vp, _c_vp, _c_sz, _c_vp]),
        "fp4_linear_fwd_workspace": (_c_sz, [_c_i64, _c_i64, _c_i64]),
        "fp4_linear_fwd": (_c_int, [_c_vp, _c_i64, _c_vp, _c_vp, _c_i64, _c_vp, _c_i64, _c_i64, _c_i64, _c_vp,
                                    _c_vp, _c_vp, _c_vp, _c_i64, _c_vp, _c_int, _c_i64, _c_vp, _c_sz, _c_vp]),
        "fp4_linear_fwd_dense_workspace": (_c_sz, [_c_i64, _c_i64, _c_i64]),
        "fp4_linear_fwd_dense": (_c_int, [_c_vp, _c_i64, _c_vp, _c_vp, _c_i64, _c_vp, _c_i64, _c_i64, _c_i64,
                                          _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_i64, _c_vp, _c_int, _c_i64, _c_vp,
                                          _c_sz, _c_vp]),
        "fp4_linear_wgrad_dge": (_c_int, [_c_vp, _c_i64, _c_vp, _c_i64, _c_vp, _c_i64, _c_vp, _c_i64, _c_i64,
                                          _c_i64, _c_f, _c_f, _c_vp, _c_int, _c_i64, _c_vp, _c_vp, _c_vp, _c_sz,
                                          _c_vp]),
        "fp4_linear_wgrad_dge_workspace": (_c_sz, [_c_i64, _c_i64, _c_i64]),
        "fp4_linear_dgrad": (_c_int, [_c_vp, _c_i64, _c_vp, _c_i64, _c_i64, _c_i64, _c_i64, _c_vp, _c_int, _c_i64,
                                      _c_vp, _c_sz, _c_vp]),
        "fp4_linear_dgrad_workspace": (_c_sz, [_c_i64, _c_i64, _c_i64]),
        "fp4_device_status": (_c_int, [_c_vp, ctypes.POINTER(_c_u32)]),
        "fp4_selftest_bounded_wait": (_c_int, [_c_u32, _c_vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_lib = load_library()


def status_string(status: int) -> str:
    return _lib.fp4_status_string(status).decode()


def _check(fn: str, status: int) -> None:
    if status != 0:
        msg = status_string(status)
        if msg == "FP4_ERR_CUDA":
            msg += ": " + _lib.fp4_last_cuda_error().decode()
        raise FP4Error(fn, status, msg)


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _s(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _rowmajor(t: torch.Tensor, name: str, dtype: torch.dtype) -> int:
    if not t.is_cuda or t.dtype != dtype or t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D row-major CUDA {dtype} tensor (got {t.dtype}, {tuple(t.shape)}, "
                         f"strides {t.stride()}, device {t.device})")
    return t.stride(0) if t.shape[0] > 1 else max(t.stride(0), t.shape[1])


def _vec(t: torch.Tensor, name: str, dtype: torch.dtype, n: int, device) -> None:
    """A 1-D (or any contiguous) CUDA tensor of `dtype` with at least n elements on `device`."""
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous() or t.numel() < n or t.device != device:
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor of at least {n} elements on {device} "
                         f"(got {t.dtype}, {tuple(t.shape)}, device {t.device})")


def _mat(t: torch.Tensor, name: str, dtype: torch.dtype, rows: int, cols: int, device) -> int:
    """A row-major CUDA matrix of `dtype`, at least rows x cols, on `device`; returns its leading dimension."""
    ld = _rowmajor(t, name, dtype)
    if t.shape[0] < rows or t.shape[1] < cols or t.device != device:
        raise ValueError(f"{name} must be at least {rows} x {cols} on {device} (got {tuple(t.shape)} on {t.device})")
    return ld


def abi_version() -> int:
    return _lib.fp4_abi_version()


# ---------------------------------------------------------------- quantizers

def fp4_quantize_rows(A: torch.Tensor, clamp_t: Optional[torch.Tensor] = None, codes: Optional[torch.Tensor] = None,
                      scales: Optional[torch.Tensor] = None, stream=None):
    """Row-wise E2M1 quantization of A (M x K, BF16); returns (codes M x K/2 uint8, scales M fp32)."""
    lda = _rowmajor(A, "A", torch.bfloat16)
    M, K = A.shape
    if codes is None:
        codes = torch.empty((M, K // 2), dtype=torch.uint8, device=A.device)
    if scales is None:
        scales = torch.empty((M,), dtype=torch.float32, device=A.device)
    ldc = _mat(codes, "codes", torch.uint8, M, K // 2, A.device)
    _vec(scales, "scales", torch.float32, M, A.device)
    if clamp_t is not None:
        _vec(clamp_t, "clamp_t", torch.float32, 1, A.device)
    _check("fp4_quantize_rows", _lib.fp4_quantize_rows(_p(A), M, K, lda, _p(clamp_t), _p(codes), ldc, _p(scales),
                                                       _s(stream)))
    return codes, scales


def fp4_quantize_cols_workspace(N: int) -> int:
    return int(_lib.fp4_quantize_cols_workspace(N))


def fp4_quantize_cols(W: torch.Tensor, codes_t: Optional[torch.Tensor] = None, scales: Optional[torch.Tensor] = None,
                      workspace: Optional[torch.Tensor] = None, stream=None):
    """Column-wise E2M1 quantization of W (K x N, BF16); returns (codes_t N x K/2 uint8, scales N fp32)."""
    ldw = _rowmajor(W, "W", torch.bfloat16)
    K, N = W.shape
    if codes_t is None:
        codes_t = torch.empty((N, K // 2), dtype=torch.uint8, device=W.device)
    if scales is None:
        scales = torch.empty((N,), dtype=torch.float32, device=W.device)
    ws_bytes = fp4_quantize_cols_workspace(N)
    if workspace is None:
        workspace = torch.empty((max(ws_bytes, 16),), dtype=torch.uint8, device=W.device)
    ldc = _mat(codes_t, "codes_t", torch.uint8, N, K // 2, W.device)
    _vec(scales, "scales", torch.float32, N, W.device)
    _vec(workspace, "workspace", torch.uint8, ws_bytes, W.device)
    _check("fp4_quantize_cols", _lib.fp4_quantize_cols(_p(W), K, N, ldw, _p(codes_t), ldc, _p(scales), _p(workspace),
                                                       workspace.numel() * workspace.element_size(), _s(stream)))
    return codes_t, scales


def fp4_quantize_cols_noalloc(W: torch.Tensor, codes_t: torch.Tensor, scales: torch.Tensor, stream=None):
    """fp4_quantize_cols without a workspace (the library's built-in scratch;
    N <= 65536; calls must not overlap on the GPU).  Outputs must be passed in:
    this path is for callers that allocate nothing per call."""
    ldw = _rowmajor(W, "W", torch.bfloat16)
    K, N = W.shape
    ldc = _mat(codes_t, "codes_t", torch.uint8, N, K // 2, W.device)
    _vec(scales, "scales", torch.float32, N, W.device)
    _check("fp4_quantize_cols_noalloc", _lib.fp4_quantize_cols_noalloc(_p(W), K, N, ldw, _p(codes_t), ldc,
                                                                       _p(scales), _s(stream)))
    return codes_t, scales


# ---------------------------------------------------------------- outlier clamp

def outlier_max_nnz(M: int, K: int, q: float) -> int:
    return int(_lib.outlier_max_nnz(M, K, float(q)))


def outlier_clamp_quantile_workspace(M: int, K: int, nnz_capacity: int) -> int:
    return int(_lib.outlier_clamp_quantile_workspace(M, K, nnz_capacity))


def outlier_clamp_quantile(A: torch.Tensor, q: float, want_clamped: bool = False,
                           out: Optional[Dict[str, torch.Tensor]] = None, stream=None) -> Dict[str, torch.Tensor]:
    """Quantile threshold t of |A|, CSR of dA = A - A_clamped (and A_clamped on request).

    Returns a dict with t (1 fp32), row_ptr (M+1 int32), col_idx / vals (capacity-sized;
    the first nnz entries are valid), nnz (1 int64) and, if asked, A_clamped."""
    lda = _rowmajor(A, "A", torch.bfloat16)
    M, K = A.shape
    cap = outlier_max_nnz(M, K, q)
    dev = A.device
    o = dict(out) if out is not None else {}
    o.setdefault("t", torch.empty((1,), dtype=torch.float32, device=dev))
    o.setdefault("row_ptr", torch.empty((M + 1,), dtype=torch.int32, device=dev))
    o.setdefault("col_idx", torch.empty((max(cap, 1),), dtype=torch.int32, device=dev))
    o.setdefault("vals", torch.empty((max(cap, 1),), dtype=torch.float32, device=dev))
    o.setdefault("nnz", torch.empty((1,), dtype=torch.int64, device=dev))
    ws_bytes = outlier_clamp_quantile_workspace(M, K, o["col_idx"].numel())
    o.setdefault("workspace", torch.empty((ws_bytes,), dtype=torch.uint8, device=dev))
    if want_clamped:
        o.setdefault("A_clamped", torch.empty_like(A))
    ac = o.get("A_clamped") if want_clamped else None
    ldac = _mat(ac, "A_clamped", torch.bfloat16, M, K, dev) if ac is not None else 0
    _check_outlier_outputs(o, M, cap, dev)
    _vec(o["workspace"], "workspace", torch.uint8, ws_bytes, dev)
    ws = o["workspace"]
    _check("outlier_clamp_quantile", _lib.outlier_clamp_quantile(
        _p(A), M, K, lda, float(q), _p(o["t"]), _p(o["row_ptr"]), _p(o["col_idx"]), _p(o["vals"]),
        o["col_idx"].numel(), _p(o["nnz"]), _p(ac), ldac, _p(ws), ws.numel(), _s(stream)))
    return o


def _check_outlier_outputs(o: Dict[str, torch.Tensor], M: int, cap: int, device) -> None:
    _vec(o["t"], "t", torch.float32, 1, device)
    _vec(o["row_ptr"], "row_ptr", torch.int32, M + 1, device)
    _vec(o["col_idx"], "col_idx", torch.int32, cap, device)
    _vec(o["vals"], "vals", torch.float32, cap, device)
    _vec(o["nnz"], "nnz", torch.int64, 1, device)
    if o["col_idx"].numel() != o["vals"].numel():
        raise ValueError("col_idx and vals must have the same capacity")


def fp4_quantize_rows_outliers(A: torch.Tensor, q: float, out: Optional[Dict[str, torch.Tensor]] = None,
                               stream=None) -> Dict[str, torch.Tensor]:
    """Threshold, clamp, CSR of dA and the row codes / scales of A_clamped in one call.
    Returns the outlier_clamp_quantile dict plus 'codes' (M x K/2) and 'scales' (M)."""
    lda = _rowmajor(A, "A", torch.bfloat16)
    M, K = A.shape
    cap = outlier_max_nnz(M, K, q)
    dev = A.device
    o = dict(out) if out is not None else {}
    o.setdefault("t", torch.empty((1,), dtype=torch.float32, device=dev))
    o.setdefault("row_ptr", torch.empty((M + 1,), dtype=torch.int32, device=dev))
    o.setdefault("col_idx", torch.empty((max(cap, 1),), dtype=torch.int32, device=dev))
    o.setdefault("vals", torch.empty((max(cap, 1),), dtype=torch.float32, device=dev))
    o.setdefault("nnz", torch.empty((1,), dtype=torch.int64, device=dev))
    o.setdefault("codes", torch.empty((M, K // 2), dtype=torch.uint8, device=dev))
    o.setdefault("scales", torch.empty((M,), dtype=torch.float32, device=dev))
    ws_bytes = outlier_clamp_quantile_workspace(M, K, o["col_idx"].numel())
    o.setdefault("workspace", torch.empty((ws_bytes,), dtype=torch.uint8, device=dev))
    ldc = _mat(o["codes"], "codes", torch.uint8, M, K // 2, dev)
    _vec(o["scales"], "scales", torch.float32, M, dev)
    _check_outlier_outputs(o, M, cap, dev)
    _vec(o["workspace"], "workspace", torch.uint8, ws_bytes, dev)
    ws = o["workspace"]
    _check("fp4_quantize_rows_outliers", _lib.fp4_quantize_rows_outliers(
        _p(A), M, K, lda, float(q), _p(o["codes"]), ldc, _p(o["scales"]), _p(o["t"]), _p(o["row_ptr"]),
        _p(o["col_idx"]), _p(o["vals"]), o["col_idx"].numel(), _p(o["nnz"]), _p(ws), ws.numel(), _s(stream)))
    return o


# ---------------------------------------------------------------- GEMMs

def fp4_linear_fwd_workspace(M: int, N: int, K: int) -> int:
    """Bytes of workspace fp4_linear_fwd uses to run the compensation on the tensor cores."""
    return int(_lib.fp4_linear_fwd_workspace(M, N, K))


def fp4_linear_fwd(a_codes: torch.Tensor, s_a: Optional[torch.Tensor], w_codes_t: torch.Tensor,
                   s_w: Optional[torch.Tensor], K: int, csr: Optional[Dict[str, torch.Tensor]] = None,
                   W: Optional[torch.Tensor] = None, out_type: str = "bf16", Y: Optional[torch.Tensor] = None,
                   workspace="auto", stream=None) -> torch.Tensor:
    """Y = (qA qW^T) / (s_A s_W^T) [+ dA W]; out_type 'bf16', 'fp32' or 'raw' (unscaled accumulator).

    workspace: "auto" allocates one when csr is given (compensation on the tensor
    cores when dA has few distinct columns); None forces the epilogue path; or a
    caller-owned CUDA uint8 tensor of at least fp4_linear_fwd_workspace(M, N, K) bytes.
    """
    dev = a_codes.device
    M, N = a_codes.shape[0], w_codes_t.shape[0]
    lda_c = _mat(a_codes, "a_codes", torch.uint8, M, K // 2, dev)
    ldw_c = _mat(w_codes_t, "w_codes_t", torch.uint8, N, K // 2, dev)
    yt = _OUT_TYPES[out_type]
    if yt != FP4_OUT_RAW_ACC_FP32:
        _vec(s_a, "s_a", torch.float32, M, dev)
        _vec(s_w, "s_w", torch.float32, N, dev)
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16 if yt == FP4_OUT_BF16 else torch.float32, device=dev)
    ldy = _mat(Y, "Y", torch.bfloat16 if yt == FP4_OUT_BF16 else torch.float32, M, N, dev)
    rp = ci = cv = None
    ldw = 0
    ws, ws_bytes = None, 0
    if csr is not None:
        rp, ci, cv = csr["row_ptr"], csr["col_idx"], csr["vals"]
        _vec(rp, "row_ptr", torch.int32, M + 1, dev)
        _vec(ci, "col_idx", torch.int32, 0, dev)
        _vec(cv, "vals", torch.float32, 0, dev)
        ldw = _mat(W, "W", torch.bfloat16, K, N, dev)
        if isinstance(workspace, str):
            if workspace != "auto":
                raise ValueError("workspace must be 'auto', None or a CUDA uint8 tensor")
            workspace = torch.empty(fp4_linear_fwd_workspace(M, N, K), dtype=torch.uint8, device=a_codes.device)
        if workspace is not None:
            _vec(workspace, "workspace", torch.uint8, fp4_linear_fwd_workspace(M, N, K), dev)
            ws, ws_bytes = workspace, workspace.numel() * workspace.element_size()
    _check("fp4_linear_fwd", _lib.fp4_linear_fwd(
        _p(a_codes), lda_c, _p(s_a), _p(w_codes_t), ldw_c, _p(s_w), M, N, K, _p(rp), _p(ci), _p(cv), _p(W), ldw,
        _p(Y), yt, ldy, _p(ws), ws_bytes, _s(stream)))
    return Y


def fp4_linear_fwd_dense_workspace(M: int, N: int, K: int) -> int:
    """Bytes of workspace fp4_linear_fwd_dense needs on the current device."""
    return int(_lib.fp4_linear_fwd_dense_workspace(M, N, K))


def fp4_linear_fwd_dense(a_codes: torch.Tensor, s_a: torch.Tensor, w_codes_t: torch.Tensor, s_w: torch.Tensor,
                         K: int, csr: Dict[str, torch.Tensor], W: torch.Tensor, out_type: str = "bf16",
                         Y: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                         stream=None) -> torch.Tensor:
    """Y = (qA qW^T) / (s_A s_W^T) + dA W with dA multiplied densely on the BF16
    tensor cores; for a dense dA.  csr may hold "t", the clamp threshold that
    produced dA (as fp4_quantize_rows_outliers returns it): then each entry is
    two exact BF16 parts instead of three."""
    dev = a_codes.device
    M, N = a_codes.shape[0], w_codes_t.shape[0]
    lda_c = _mat(a_codes, "a_codes", torch.uint8, M, K // 2, dev)
    ldw_c = _mat(w_codes_t, "w_codes_t", torch.uint8, N, K // 2, dev)
    if out_type not in ("bf16", "fp32"):
        raise ValueError("out_type must be 'bf16' or 'fp32'")
    yt = _OUT_TYPES[out_type]
    _vec(s_a, "s_a", torch.float32, M, dev)
    _vec(s_w, "s_w", torch.float32, N, dev)
    ydt = torch.bfloat16 if yt == FP4_OUT_BF16 else torch.float32
    if Y is None:
        Y = torch.empty((M, N), dtype=ydt, device=dev)
    ldy = _mat(Y, "Y", ydt, M, N, dev)
    rp, ci, cv = csr["row_ptr"], csr["col_idx"], csr["vals"]
    _vec(rp, "row_ptr", torch.int32, M + 1, dev)
    _vec(ci, "col_idx", torch.int32, 0, dev)
    _vec(cv, "vals", torch.float32, 0, dev)
    ldw = _mat(W, "W", torch.bfloat16, K, N, dev)
    t = csr.get("t")
    if t is not None:
        _vec(t, "t", torch.float32, 1, dev)
    need = fp4_linear_fwd_dense_workspace(M, N, K)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    _vec(workspace, "workspace", torch.uint8, need, dev)
    _check("fp4_linear_fwd_dense", _lib.fp4_linear_fwd_dense(
        _p(a_codes), lda_c, _p(s_a), _p(w_codes_t), ldw_c, _p(s_w), M, N, K, _p(rp), _p(ci), _p(cv), _p(t), _p(W),
        ldw, _p(Y), yt, ldy, _p(workspace), workspace.numel(), _s(stream)))
    return Y


def _bwd_workspace(workspace, nbytes: int, device):
    """(pointer, bytes) for the backward GEMMs' split-tail workspace: "auto"
    allocates what the call needs (nothing when it never splits), None runs
    without, or a caller-owned CUDA uint8 tensor."""
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError("workspace must be 'auto', None or a CUDA uint8 tensor")
        if nbytes == 0:
            return None, 0
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
    if workspace is None:
        return None, 0
    _vec(workspace, "workspace", torch.uint8, nbytes, device)
    return workspace, workspace.numel() * workspace.element_size()


def fp4_linear_wgrad_dge_workspace(M: int, N: int, K: int) -> int:
    """Bytes of split-tail workspace fp4_linear_wgrad_dge uses on the current device."""
    return int(_lib.fp4_linear_wgrad_dge_workspace(M, N, K))


def fp4_linear_dgrad_workspace(M: int, N: int, K: int) -> int:
    """Bytes of split-tail workspace fp4_linear_dgrad uses on the current device."""
    return int(_lib.fp4_linear_dgrad_workspace(M, N, K))


DW_TYPES = {"fp32": 0, "e4m3": 1}


def fp4_linear_wgrad_dge(A: torch.Tensor, dY: torch.Tensor, W: torch.Tensor, s_w: torch.Tensor,
                         dge_k: float = 5.0, dge_clip: float = 3.0, dW: Optional[torch.Tensor] = None,
                         workspace="auto", stream=None, dw_type: str = "fp32",
                         dw_scale: Optional[torch.Tensor] = None, dw_amax: Optional[torch.Tensor] = None):
    """dW = (A^T dY) * f'(|W s_W|) (K x N).  workspace: see _bwd_workspace.

    dw_type "fp32" returns dW in fp32.  dw_type "e4m3" returns (codes, amax):
    codes K x N uint8 = E4M3(fl32(dW * scale)) with dw_scale a 1-element fp32
    device tensor, and amax the 1-element fp32 tensor max |dW|."""
    if dw_type not in DW_TYPES:
        raise ValueError(f"dw_type must be one of {sorted(DW_TYPES)}")
    fp8 = dw_type == "e4m3"
    lda = _rowmajor(A, "A", torch.bfloat16)
    M, K = A.shape
    N = dY.shape[1]
    lddy = _mat(dY, "dY", torch.bfloat16, M, N, A.device)
    ldw = _mat(W, "W", torch.bfloat16, K, N, A.device)
    _vec(s_w, "s_w", torch.float32, N, A.device)
    out_dtype = torch.uint8 if fp8 else torch.float32
    if dW is None:
        dW = torch.empty((K, N), dtype=out_dtype, device=A.device)
    lddw = _mat(dW, "dW", out_dtype, K, N, A.device)
    if fp8:
        if dw_scale is None:
            raise ValueError("dw_type 'e4m3' needs dw_scale (a 1-element fp32 device tensor)")
        _vec(dw_scale, "dw_scale", torch.float32, 1, A.device)
        if dw_amax is None:
            dw_amax = torch.empty(1, dtype=torch.float32, device=A.device)
        _vec(dw_amax, "dw_amax", torch.float32, 1, A.device)
    elif dw_scale is not None or dw_amax is not None:
        raise ValueError("dw_scale / dw_amax apply to dw_type 'e4m3' only")
    ws, ws_bytes = _bwd_workspace(workspace, fp4_linear_wgrad_dge_workspace(M, N, K), A.device)
    _check("fp4_linear_wgrad_dge", _lib.fp4_linear_wgrad_dge(
        _p(A), lda, _p(dY), lddy, _p(W), ldw, _p(s_w), M, N, K, float(dge_k), float(dge_clip), _p(dW),
        DW_TYPES[dw_type], lddw, _p(dw_scale) if fp8 else None, _p(dw_amax) if fp8 else None,
        _p(ws), ws_bytes, _s(stream)))
    return (dW, dw_amax) if fp8 else dW


def fp4_linear_dgrad(dY: torch.Tensor, W: torch.Tensor, out_dtype: torch.dtype = torch.bfloat16,
                     dX: Optional[torch.Tensor] = None, workspace="auto", stream=None) -> torch.Tensor:
    """dX = dY W^T (M x K), BF16 or fp32; fp32 accumulation.  workspace: see _bwd_workspace."""
    lddy = _rowmajor(dY, "dY", torch.bfloat16)
    M, N = dY.shape
    K = W.shape[0]
    if W.shape[1] != N:
        raise ValueError(f"W must be K x {N} (got {tuple(W.shape)})")
    ldw = _mat(W, "W", torch.bfloat16, K, N, dY.device)
    if dX is None:
        dX = torch.empty((M, K), dtype=out_dtype, device=dY.device)
    if dX.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError(f"dX must be bfloat16 or float32 (got {dX.dtype})")
    lddx = _mat(dX, "dX", dX.dtype, M, K, dY.device)
    dx_type = FP4_OUT_BF16 if dX.dtype == torch.bfloat16 else FP4_OUT_FP32
    ws, ws_bytes = _bwd_workspace(workspace, fp4_linear_dgrad_workspace(M, N, K), dY.device)
    _check("fp4_linear_dgrad", _lib.fp4_linear_dgrad(
        _p(dY), lddy, _p(W), ldw, M, N, K, _p(dX), dx_type, lddx, _p(ws), ws_bytes, _s(stream)))
    return dX


# ---------------------------------------------------------------- status

def fp4_device_status(stream=None):
    """Synchronizes the stream; returns (status name, flags) and clears the device flags."""
    flags = ctypes.c_uint32(0)
    st = _lib.fp4_device_status(_s(stream), ctypes.byref(flags))
    return status_string(st), int(flags.value)


def fp4_selftest_bounded_wait(timeout_us: int, stream=None) -> None:
    _check("fp4_selftest_bounded_wait", _lib.fp4_selftest_bounded_wait(int(timeout_us), _s(stream)))


# ---------------------------------------------------------------- one layer

# dA averaging at least this many entries per row is multiplied densely
# (fp4_linear_fwd_dense); the bound is n - ceil(q n), known on the host.
DENSE_MIN_ROW_ENTRIES = 28


def use_dense_compensation(M: int, K: int, q: float) -> bool:
    """Whether linear_forward multiplies dA densely for this shape and quantile."""
    return K % 64 == 0 and outlier_max_nnz(M, K, q) >= DENSE_MIN_ROW_ENTRIES * M


def linear_forward(A: torch.Tensor, W: torch.Tensor, q: float, out_type: str = "bf16", stream=None,
                   dense: Optional[bool] = None):
    """The whole forward of the quantized linear layer: quantile threshold,
    clamp + CSR of dA + row quantization of A_clamped (one fused pass), column
    quantization of W, FP4 GEMM with scales and compensation.  dense: multiply
    dA on the BF16 tensor cores as a dense matrix (None: when
    use_dense_compensation says so).  Returns (Y, intermediates)."""
    o = fp4_quantize_rows_outliers(A, q, stream=stream)
    w_codes_t, s_w = fp4_quantize_cols(W, stream=stream)
    M, K = A.shape
    if dense is None:
        dense = use_dense_compensation(M, K, q) and out_type in ("bf16", "fp32")
    if dense:
        Y = fp4_linear_fwd_dense(o["codes"], o["scales"], w_codes_t, s_w, K, csr=o, W=W, out_type=out_type,
                                 stream=stream)
    else:
        Y = fp4_linear_fwd(o["codes"], o["scales"], w_codes_t, s_w, K, csr=o, W=W, out_type=out_type,
                           stream=stream)
    return Y, dict(outlier=o, a_codes=o["codes"], s_a=o["scales"], w_codes_t=w_codes_t, s_w=s_w)


def linear_backward(A: torch.Tensor, W: torch.Tensor, dY: torch.Tensor, s_w: torch.Tensor, dge_k: float = 5.0,
                    dge_clip: float = 3.0, dx_dtype: torch.dtype = torch.bfloat16, stream=None):
    """The backward of the quantized linear layer: the DGE-corrected weight
    gradient dW (K x N, fp32) and the input gradient dX = dY W^T (M x K).
    s_w: the column scales of W from the forward (linear_forward's "s_w").
    Returns (dX, dW)."""
    dW = fp4_linear_wgrad_dge(A, dY, W, s_w, dge_k, dge_clip, stream=stream)
    dX = fp4_linear_dgrad(dY, W, out_dtype=dx_dtype, stream=stream)
    return dX, dW
