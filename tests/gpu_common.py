"""Helpers shared by the GPU parity tests: host <-> device transfer of BF16 bit
patterns and the comparison rules (bit-exact, BF16 ulp distance, relative
Frobenius error)."""
import os

import numpy as np
import torch

BF16_ULP_TOL = 1          # final BF16 outputs: within 1 BF16 ulp
FROB_TOL = 1e-5           # compensated fp32 outputs and DGE weight gradients
FP32_SUM_BOUND = 2.0 ** -20   # fp32 epilogue rounding, relative to the terms' magnitude
# BF16 products summed on the tensor core (backward GEMMs): each 2048-term chunk
# is 128 MMA steps into an fp32 accumulator, each add within 2^-23 (truncation)
# of a partial sum bounded by the chunk's sum of |terms|; the chunks are added
# in fp32 (at most 8 adds, 2^-24 each).  Allowing 2^-23 more per step for the
# 16-term sum inside an MMA gives |error| <= ((128 + 128) 2^-23 + 8 2^-24) sum
# |terms| for the longest reduction (16384 terms: 8 chunks), below 2^-14 sum |terms|
# (tests/test_tolerance_model.py derives and models it).
TC_SUM_BOUND = 2.0 ** -14


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_ulp_distance(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in BF16 ulps between two BF16 bit patterns (+0 and -0 coincide)."""
    def key(b):
        b = np.asarray(b, dtype=np.uint16).astype(np.int64)
        mag = b & 0x7FFF
        return np.where(b & 0x8000, -mag, mag)
    return np.abs(key(a_bits) - key(b_bits))


def rel_frobenius(got: np.ndarray, ref: np.ndarray) -> float:
    ref = np.asarray(ref, dtype=np.float64)
    num = np.linalg.norm(np.asarray(got, dtype=np.float64) - ref)
    den = np.linalg.norm(ref)
    return float(num / den) if den > 0 else float(num)


def assert_no_device_flags(fp4lin):
    name, flags = fp4lin.fp4_device_status()
    assert flags == 0 and name == "FP4_OK", (name, flags)


def bf16_ulp_of(y: np.ndarray) -> np.ndarray:
    """Spacing of BF16 values at |y| (8 significant bits)."""
    y = np.abs(np.asarray(y, dtype=np.float64))
    _, e = np.frexp(np.where(y > 0, y, 2.0 ** -126))
    return np.exp2(e.astype(np.float64) - 8.0)


def assert_bf16_compensated_close(got_bits: np.ndarray, y_ref: np.ndarray, magnitude: np.ndarray,
                                  bound: float = FP32_SUM_BOUND):
    """Compensated BF16 output: within 1 BF16 ulp of the fp64 result plus the
    fp32 rounding bound of the epilogue's sum (FP32_SUM_BOUND x the magnitude of
    the two added terms), which is what any fp32 epilogue can guarantee when
    the GEMM term and the compensation cancel."""
    from oracle import fp4_linear as orc
    got = orc.bf16_to_f32(got_bits).astype(np.float64)
    allowed = bf16_ulp_of(y_ref) + bound * magnitude
    bad = np.abs(got - y_ref) > allowed
    assert not bad.any(), (np.argwhere(bad)[:5], got[bad][:5], y_ref[bad][:5])
    return int(np.count_nonzero(bf16_ulp_distance(got_bits, orc.f64_to_bf16(y_ref)) > BF16_ULP_TOL))


def _golden_e2m1_x2() -> list:
    """Twice the value of every E2M1 code (an integer), read from the golden
    format table tests/golden/e2m1_codes.txt (written from the pages' bit layout)."""
    vals = {}
    with open(os.path.join(os.path.dirname(__file__), "golden", "e2m1_codes.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            if line:
                vals[int(line[0])] = int(round(2 * float(line[4])))
    return [vals[c] for c in range(16)]


def codes_to_int8_x2(packed: torch.Tensor) -> torch.Tensor:
    """Packed E2M1 codes (R x C/2 uint8, element 2c in the low nibble) -> R x C int8
    holding twice each value, on the tensors' device (test-side decode by table)."""
    lut = torch.tensor(_golden_e2m1_x2(), dtype=torch.int8, device=packed.device)
    lo = lut[(packed & 15).long()]
    hi = lut[(packed >> 4).long()]
    return torch.stack((lo, hi), dim=-1).reshape(packed.shape[0], 2 * packed.shape[1])


def assert_raw_acc_equals_int_mm(raw: torch.Tensor, a_codes: torch.Tensor, w_codes_t: torch.Tensor):
    """The whole M x N raw FP4 accumulator against torch._int_mm (cuBLASLt int8,
    an independent library) on the x2 integer codes: 4 acc == (2 qA)(2 qW)^T
    exactly (every value is an integer below 2^24, so fp32 holds it exactly)."""
    a8 = codes_to_int8_x2(a_codes)
    w8 = codes_to_int8_x2(w_codes_t)
    ref = torch._int_mm(a8, w8.t())
    got = raw.mul(4.0)
    assert torch.equal(got, got.round()), "raw accumulator is not a multiple of 1/4"
    bad = (got.to(torch.int32) != ref)
    assert not bool(bad.any()), (int(bad.sum()), torch.nonzero(bad)[:5].tolist())
