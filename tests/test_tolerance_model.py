"""Where the backward GEMMs' tolerance comes from, checked on the CPU.

The input gradient dX = dY W^T is a BF16 product summed on the tensor core.  Its
parity tests allow 1 BF16 ulp plus TC_SUM_BOUND x sum |terms| per output
(tests/gpu_common.py).  The bound follows from an accumulation model:
  * the reduction is split into chunks of 2048 terms (128 MMA steps of 16),
    each accumulated in fp32 in tensor memory;
  * every MMA step forms its 16-term sum and adds it to the fp32 accumulator,
    and both the step's sum and the add may truncate (round toward zero):
    each error is below 2^-23 of a partial sum whose size is at most the
    chunk's sum of |terms|;
  * the chunk sums are added in fp32 registers with round to nearest (2^-24
    of at most the whole sum of |terms| per add).
So |error| <= (2 * 128 * 2^-23 + n_chunks * 2^-24) sum |terms|, which for the
longest reduction here (16384 terms, 8 chunks) is 260 * 2^-23 < 2^-14.

The tests below run that model in numpy (exact products in fp64, truncating
fp32 adds) on data shaped like the 13B layer's input gradient and on
all-positive terms (where truncation errors never cancel), and check that the
observed error stays inside TC_SUM_BOUND while the bound is not vacuous.
"""
import numpy as np
import pytest

from precision_gemm_row_gb300 import workloads as wl
from tests.gpu_common import TC_SUM_BOUND

CHUNK, STEP = 2048, 16


def _rz_f32(x: np.ndarray) -> np.ndarray:
    """fp64 -> fp32 rounded toward zero."""
    r = x.astype(np.float32)
    over = np.abs(r.astype(np.float64)) > np.abs(x)
    r[over] = np.nextafter(r[over], np.float32(0.0))
    return r


def _tensor_core_sum_model(terms: np.ndarray) -> np.ndarray:
    """Row sums of `terms` (rows x L, exact fp64 products) as the model above
    forms them: truncating fp32 accumulation of 16-term steps per 2048-term
    chunk, chunks added in fp32 with round to nearest."""
    rows, L = terms.shape
    total = np.zeros(rows, np.float32)
    for c0 in range(0, L, CHUNK):
        acc = np.zeros(rows, np.float32)
        for s0 in range(c0, min(L, c0 + CHUNK), STEP):
            step = _rz_f32(terms[:, s0:s0 + STEP].sum(axis=1))
            acc = _rz_f32(acc.astype(np.float64) + step.astype(np.float64))
        total = total + acc                                 # fp32, round to nearest
    return total


def _analytic_bound(L: int) -> float:
    n_chunks = -(-L // CHUNK)
    return 2 * (CHUNK // STEP) * 2.0 ** -23 + n_chunks * 2.0 ** -24


def test_bound_covers_the_longest_reduction():
    assert _analytic_bound(16384) <= TC_SUM_BOUND
    assert _analytic_bound(16384) > TC_SUM_BOUND / 2      # and is not far from it


@pytest.mark.parametrize("L", [5120, 13824])
def test_model_error_inside_bound_on_layer_shaped_data(L):
    rng = np.random.default_rng(L)
    dY = wl.bf16_bits_to_f32_view(wl.f32_to_bf16_bits(
        rng.standard_normal((32, L)).astype(np.float32) * np.float32(1e-3))).astype(np.float64)
    W = wl.bf16_bits_to_f32_view(wl.f32_to_bf16_bits(
        rng.standard_normal((8, L)).astype(np.float32) * np.float32(0.02))).astype(np.float64)
    terms = (dY[:, None, :] * W[None, :, :]).reshape(-1, L)       # exact: BF16 x BF16 fits fp64
    err = np.abs(_tensor_core_sum_model(terms).astype(np.float64) - terms.sum(axis=1))
    scale = np.abs(terms).sum(axis=1)
    assert np.all(err <= _analytic_bound(L) * scale)
    assert np.all(err <= TC_SUM_BOUND * scale)


def test_model_error_inside_bound_when_truncations_never_cancel():
    rng = np.random.default_rng(1)
    L = 16384
    terms = rng.uniform(0.5, 1.0, size=(16, L)) * 2.0 ** rng.integers(-8, 0, size=(16, L))
    err = np.abs(_tensor_core_sum_model(terms).astype(np.float64) - terms.sum(axis=1))
    scale = terms.sum(axis=1)
    worst = float(np.max(err / scale))
    assert worst <= _analytic_bound(L) <= TC_SUM_BOUND
    # truncation here always loses in the same direction, so the error is a
    # visible part of the bound (the bound is not vacuous for this model)
    assert worst > 2.0 ** -23
