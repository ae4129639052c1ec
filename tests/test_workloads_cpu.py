"""Host-side input layouts: the shared-input fusion of linears (one GEMM over
the members' weights side by side) and bench.py's linear selection.  Checked on
small slices of the seeded inputs; no GPU."""
import os
import sys
import types

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from oracle import fp4_linear as orc  # noqa: E402
from precision_gemm_row_gb300 import workloads as wl  # noqa: E402


def _small_decoder():
    """The 7B decoder-layer structure at a size the oracle handles in milliseconds."""
    return wl._decoder("tiny_layer", 7, "tiny decoder layer", 64, 96, 160)


def test_fusion_groups_linears_by_activation_and_keeps_the_flops():
    base = _small_decoder()
    fused = wl.fuse_shared_inputs(base)
    assert [l.name for l in fused.linears] == ["q_proj+k_proj+v_proj", "o_proj", "gate_proj+up_proj", "down_proj"]
    assert [l.N for l in fused.linears] == [3 * 96, 96, 2 * 160, 96]
    assert sum(l.M * l.K * l.N for l in fused.linears) == sum(l.M * l.K * l.N for l in base.linears)


def test_fused_inputs_are_the_members_side_by_side():
    base = _small_decoder()
    fused = wl.fuse_shared_inputs(base)
    qkv = fused.linears[0]
    members = fused.members[qkv.name]
    assert np.array_equal(fused.activation(qkv), base.activation(members[0]))
    W, dY = fused.weight(qkv), fused.grad(qkv)
    c0 = 0
    for m in members:
        assert np.array_equal(W[:, c0:c0 + m.N], base.weight(m))
        assert np.array_equal(dY[:, c0:c0 + m.N], base.grad(m))
        c0 += m.N


def test_fused_products_split_into_the_members_and_dgrad_sums():
    """Y_cat = A W_cat is the members' Y side by side, and dY_cat W_cat^T is the
    sum of the members' input gradients: the identities the fused GEMM relies on."""
    base = _small_decoder()
    fused = wl.fuse_shared_inputs(base)
    lin = fused.linears[2]            # gate + up
    A = orc.bf16_to_f32(fused.activation(lin)).astype(np.float64)
    W = orc.bf16_to_f32(fused.weight(lin)).astype(np.float64)
    Y = A @ W
    dX = orc.linear_dgrad(fused.grad(lin), fused.weight(lin))
    c0, dX_sum = 0, 0.0
    for m in fused.members[lin.name]:
        Wm = orc.bf16_to_f32(base.weight(m)).astype(np.float64)
        assert np.allclose(Y[:, c0:c0 + m.N], A @ Wm, rtol=1e-13, atol=1e-15)
        dX_sum = dX_sum + orc.linear_dgrad(base.grad(m), base.weight(m))
        c0 += m.N
    assert np.allclose(dX, dX_sum, rtol=1e-12, atol=1e-15)


def test_bench_linear_selection():
    import bench
    args = types.SimpleNamespace(workload="c4_llama13b_layer_16384tok", fuse_shared_input=False, linear=["down_proj"])
    work = bench.select_linears(wl, args)
    assert [(l.name, l.K, l.N) for l in work.linears] == [("down_proj", 13824, 5120)]
    args = types.SimpleNamespace(workload="c3_llama7b_layer_8192tok", fuse_shared_input=True,
                                 linear=["gate_proj+up_proj"])
    assert [l.N for l in bench.select_linears(wl, args).linears] == [2 * 11008]
    args = types.SimpleNamespace(workload="c2_llama1.3b_mlp_up_8192x2048x5504", fuse_shared_input=False,
                                 linear=["q_proj"])
    with pytest.raises(SystemExit):
        bench.select_linears(wl, args)


def test_reference_arm_line_on_the_small_workload():
    """bench.py --impl reference times the oracle on the host; its JSON line
    carries the contract's keys (checked on the 256 x 512 x 512 workload, which
    it times in full)."""
    import bench
    args = types.SimpleNamespace(workload="c1_single_linear_256x512x512", steps=1, warmup=3, cpu_sample=16,
                                 fuse_shared_input=False, linear=[])
    line = bench.run_reference(args)
    assert line["impl"] == "reference" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["unit"] == "TFLOP/s" and line["metric"].startswith("FP4 linear fwd+bwd TFLOPS")
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["steps"] == 1 and line["warmup"] == 3
    # measured, not extrapolated: the step time is what the sub-problem took, and
    # the value is the sub-problem's work over that time
    assert line["extrapolated"] is False
    cb = line["cpu_baseline"]
    assert line["ms_per_step"] == pytest.approx(cb["step_s"] * 1e3, abs=1e-3)
    assert line["value"] == pytest.approx(cb["sample_flops_per_step"] / cb["step_s"] / 1e12, rel=2e-3)
    # the small workload is timed in full (every token and output column), whatever the sample
    assert cb["sample_flops_per_step"] == 6 * 256 * 512 * 512
    assert cb["sample"].startswith("the whole problem")
    assert line["config"]["workload"] == "c1_single_linear_256x512x512"
    assert line["config"]["linears"] == [["linear", 256, 512, 512, 0.99]]


def test_row_prefix_draws_equal_the_whole_draw():
    """The oracle's sub-problem draws only the first rows of A and dY; every
    activation kind gives the same values as the first rows of the full draw."""
    for kind in ("normal", "normal_x20", "normal_redraw15", "normal_4x20", "student_t3"):
        full = wl.draw_activation(7, "a", 96, 64, kind)
        assert np.array_equal(wl.draw_activation(7, "a", 96, 64, kind, rows=10), full[:10]), kind
    assert np.array_equal(wl.draw_grad(7, "g", 96, 40, rows=5), wl.draw_grad(7, "g", 96, 40)[:5])
