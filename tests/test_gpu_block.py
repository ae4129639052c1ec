"""NEXT-4: a LLaMA decoder block stepped on synthetic tokens with its seven
linear layers on the FP4 library (forward with outlier clamp + compensation,
DGE weight gradient and input gradient in backward, SGD on fp32 masters)."""
import math

import numpy as np
import pytest
import torch

from oracle import fp4_linear as orc
from tests.gpu_common import FROB_TOL, assert_no_device_flags, rel_frobenius

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def blk():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from precision_gemm_row_gb300 import build
    build.build()
    from precision_gemm_row_gb300 import block, fp4lin
    return block, fp4lin


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def test_block_loss_decreases_over_sgd_steps(blk):
    block, fp4lin = blk
    losses = block.train(block.BlockConfig(), steps=5)
    assert all(math.isfinite(l) for l in losses), losses
    assert all(b < a for a, b in zip(losses, losses[1:])), losses
    assert losses[-1] < 0.95 * losses[0], losses
    assert_no_device_flags(fp4lin)


@pytest.mark.parametrize("name", ["q_proj", "down_proj"])
def test_block_step_weight_gradient_matches_oracle(blk, name):
    """One step's DGE weight gradient of a linear inside the block, on sampled
    rows of dW, against the oracle fed the same BF16 A, dY and W."""
    block, fp4lin = blk
    cfg = block.BlockConfig(batch=1, seq=1024)
    b = block.LlamaBlock(cfg)
    rec = {}
    loss = b.step(record=rec)
    assert math.isfinite(loss)
    r = rec[name]
    assert r["nnz"] > 0                      # the clamp found outliers to compensate
    K = r["A"].shape[1]
    rows = np.sort(np.random.default_rng(3).choice(K, size=48, replace=False))
    ref = orc.wgrad_dge(_bits(r["A"]), _bits(r["dY"]), _bits(r["W"]), r["s_w"].cpu().numpy(),
                        cfg.dge_k, cfg.dge_clip, rows=rows)
    got = r["dW"][torch.from_numpy(rows).cuda()].cpu().numpy()
    err = rel_frobenius(got, ref)
    assert err <= FROB_TOL, err
    assert_no_device_flags(fp4lin)


def test_block_trains_with_fp8_weight_gradients(blk):
    """The same steps with the weight gradients carried as E4M3 codes under
    delayed per-tensor scaling: the loss still falls every step and stays
    close to the fp32-gradient run's."""
    block, fp4lin = blk
    ref = block.train(block.BlockConfig(), steps=4)
    fp8 = block.train(block.BlockConfig(fp8_grads=True), steps=4)
    assert all(math.isfinite(l) for l in fp8), fp8
    assert all(b < a for a, b in zip(fp8, fp8[1:])), fp8
    assert fp8[0] == pytest.approx(ref[0], rel=1e-6)          # the same first forward
    assert all(abs(a - b) <= 0.02 * b for a, b in zip(fp8, ref)), (fp8, ref)
    assert_no_device_flags(fp4lin)
