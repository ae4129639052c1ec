"""Full-size parity on every workload (the 1.3B / 7B / 13B LLaMA shapes and the
Student-t stress case), run through the same launches bench.py times
(bench.StepPlan).  The oracle recomputes sampled outputs one by one:

* threshold t: exact order statistic over ALL of |A| (full sort);
* CSR: every row's count against a full count of |A| > t; column indices and
  values bit-exact on sampled rows;
* row codes / scales bit-exact on sampled rows; column codes / scales bit-exact
  on every column;
* the whole M x N raw FP4 accumulator against torch._int_mm (cuBLASLt int8) on
  the x2 integer codes; raw accumulators bit-exact and BF16 Y (1 ulp + fp32 sum
  bound) against the oracle, from the oracle's own codes, on sampled rows;
* DGE weight gradient within 1e-5 relative Frobenius on sampled feature rows, and its E4M3
  form within one code of the oracle's encoding there;
* BF16 input gradient dY W^T within 1 ulp + the tensor-core sum bound on sampled rows.
"""
import types

import numpy as np
import pytest
import torch

from oracle import fp4_linear as orc
from precision_gemm_row_gb300 import workloads as wl
from tests.gpu_common import (FROB_TOL, TC_SUM_BOUND, assert_bf16_compensated_close, assert_no_device_flags,
                              assert_raw_acc_equals_int_mm, dev_bf16, host_bits, rel_frobenius)

pytestmark = pytest.mark.gpu

N_SAMPLE = 40


@pytest.fixture(scope="module")
def fp4():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from precision_gemm_row_gb300 import build
    build.build()
    from precision_gemm_row_gb300 import fp4lin
    return fp4lin


def _sample(n, seed):
    rng = np.random.default_rng(seed)
    s = rng.choice(n, size=min(N_SAMPLE, n), replace=False)
    return np.unique(np.concatenate([s, [0, n - 1]]))


def _distinct_cases(work):
    """One linear per distinct (activation, weight) shape so every kernel sees every shape."""
    seen, out = set(), []
    for lin in work.linears:
        key = (lin.act, lin.K, lin.N, lin.q, lin.weight_name or lin.name)
        shape_key = (lin.act, lin.K, lin.N, lin.q)
        if shape_key in seen:
            continue
        seen.add(shape_key)
        out.append(lin)
    return out


CASES = [(k, lin.name) for k in wl.WORKLOAD_ORDER for lin in _distinct_cases(wl.WORKLOADS[k])]


@pytest.mark.parametrize("workload,linear", CASES)
def test_full_size_linear(fp4, workload, linear):
    import bench
    work = wl.WORKLOADS[workload]
    lin = next(l for l in work.linears if l.name == linear)
    A_bits, W_bits, dY_bits = work.activation(lin), work.weight(lin), work.grad(lin)
    plan = bench.StepPlan(fp4, types.SimpleNamespace(linears=[lin]),
                          [(dev_bf16(A_bits), dev_bf16(W_bits), dev_bf16(dY_bits))])
    plan.run()
    plan.run()                       # second pass over the same buffers (workspace reuse)
    torch.cuda.synchronize()
    act, step = next(iter(plan.acts.values())), plan.lins[0]
    assert_no_device_flags(fp4)
    M, K, N = lin.M, lin.K, lin.N
    rows = _sample(M, 1)
    frows = _sample(K, 3)

    # threshold over all of |A|
    t, t_bits, k = orc.quantile_threshold(A_bits, lin.q)
    assert act.out["t"].cpu().numpy().view(np.uint32)[0] == np.float32(t).view(np.uint32)
    # CSR row counts for every row, entries for sampled rows
    rp = act.out["row_ptr"].cpu().numpy().astype(np.int64)
    counts = np.count_nonzero((A_bits & np.uint16(0x7FFF)) > np.uint16(t_bits), axis=1)
    assert np.array_equal(np.diff(rp), counts) and rp[0] == 0
    assert int(act.out["nnz"].item()) == rp[-1] <= orc.clamp_rank(M * K, 1.0) - k
    A_c_s, rp_s, ci_s, cv_s = orc.clamp_and_compensation(A_bits[rows], t)
    ci_g = act.out["col_idx"].cpu().numpy()
    cv_g = act.out["vals"].cpu().numpy()
    for r, i in enumerate(rows):
        seg = slice(rp[i], rp[i + 1])
        assert np.array_equal(ci_g[seg], ci_s[rp_s[r]:rp_s[r + 1]])
        assert np.array_equal(cv_g[seg].view(np.uint32), cv_s[rp_s[r]:rp_s[r + 1]].view(np.uint32))
    # row quantization of A_clamped on sampled rows
    ref_a, ref_sa = orc.quantize_rows(A_c_s)
    assert np.array_equal(act.out["codes"][torch.from_numpy(rows).cuda()].cpu().numpy(), ref_a)
    assert np.array_equal(act.out["scales"].cpu().numpy()[rows].view(np.uint32), ref_sa.view(np.uint32))
    # column quantization of W: every column against the oracle
    Wf = orc.bf16_to_f32(W_bits)
    ref_w, ref_sw = orc.quantize_cols(Wf)
    assert np.array_equal(step.w_codes.cpu().numpy(), ref_w)
    assert np.array_equal(step.s_w.cpu().numpy().view(np.uint32), ref_sw.view(np.uint32))
    # GEMM: the whole M x N raw accumulator against cuBLASLt int8 on the codes,
    # and the sampled rows (raw and compensated BF16 Y) against the oracle, built
    # from the oracle's own codes and scales
    raw = fp4.fp4_linear_fwd(act.out["codes"], None, step.w_codes, None, K, out_type="raw")
    assert_raw_acc_equals_int_mm(raw, act.out["codes"], step.w_codes)
    ref_raw = orc.gemm_raw(ref_a, ref_w).astype(np.float32)
    assert np.array_equal(raw[torch.from_numpy(rows).cuda()].cpu().numpy().view(np.uint32), ref_raw.view(np.uint32))
    del raw
    y_ref = orc.linear_fwd(ref_a, ref_sa, ref_w, ref_sw, rp_s, ci_s, cv_s, W_bits)
    mag = orc.linear_fwd_magnitude(ref_a, ref_sa, ref_w, ref_sw, rp_s, ci_s, cv_s, W_bits)
    y_gpu = host_bits(step.Y[torch.from_numpy(rows).cuda()])
    # a dense dA is summed on the tensor cores (the backward engine's bound)
    assert_bf16_compensated_close(y_gpu, y_ref, mag, **({"bound": TC_SUM_BOUND} if step.dense else {}))
    # DGE weight gradient on sampled feature rows
    dw_ref = orc.wgrad_dge(A_bits, dY_bits, W_bits, ref_sw, 5.0, 3.0, rows=frows)
    dw_gpu = step.dW[torch.from_numpy(frows).cuda()].cpu().numpy()
    assert rel_frobenius(dw_gpu, dw_ref) <= FROB_TOL
    # the FP8 (E4M3) weight gradient of the same launch shape, with a scale set
    # from the oracle's sampled gradient: codes within one step of the oracle's
    # encoding of its own gradient, almost all equal; the returned max |dW|
    # covers the sampled rows and agrees with the fp32 gradient's
    scale = np.float32(448.0 / float(np.max(np.abs(dw_ref))))
    codes8, amax = fp4.fp4_linear_wgrad_dge(act.A, step.dY, step.W, step.s_w, 5.0, 3.0, dw_type="e4m3",
                                            dw_scale=torch.tensor([float(scale)], dtype=torch.float32,
                                                                  device="cuda"))
    ref8, _ = orc.wgrad_dge_fp8(dw_ref, float(scale))
    got8 = codes8[torch.from_numpy(frows).cuda()].cpu().numpy().astype(np.int32)
    step_of = lambda c: np.where(c & 0x80, -(c & 0x7F), c & 0x7F)
    assert np.max(np.abs(step_of(got8) - step_of(ref8.astype(np.int32)))) <= 1
    assert np.mean(got8 == ref8) >= 0.99
    amax = float(amax.item())
    assert amax >= float(np.max(np.abs(dw_ref))) * (1 - 1e-5)
    assert amax == float(step.dW.abs().max().item())
    del codes8
    # input gradient on sampled token rows
    dx_ref = orc.linear_dgrad(dY_bits, W_bits, rows=rows)
    dx_mag = orc.linear_dgrad(dY_bits & np.uint16(0x7FFF), W_bits & np.uint16(0x7FFF), rows=rows)
    assert_bf16_compensated_close(host_bits(step.dX[torch.from_numpy(rows).cuda()]), dx_ref, dx_mag,
                                  bound=TC_SUM_BOUND)
    assert_no_device_flags(fp4)


def test_fused_shared_input_linears_7b_layer(fp4):
    """Linears reading the same activation as one GEMM over their weights side
    by side (q/k/v: N = 12288, gate/up: N = 22016): every member's Y, column
    codes and dW are its column block, and dX is the sum of the members' input
    gradients; checked against the oracle member by member on sampled rows."""
    import bench
    base = wl.WORKLOADS["c3_llama7b_layer_8192tok"]
    work = wl.fuse_shared_inputs(base)
    fused = [l for l in work.linears if len(work.members[l.name]) > 1]
    assert [l.N for l in fused] == [3 * 4096, 2 * 11008]
    for lin in fused:
        A_bits = work.activation(lin)
        W_bits, dY_bits = work.weight(lin), work.grad(lin)
        plan = bench.StepPlan(fp4, types.SimpleNamespace(linears=[lin]),
                              [(dev_bf16(A_bits), dev_bf16(W_bits), dev_bf16(dY_bits))])
        plan.run()
        torch.cuda.synchronize()
        assert_no_device_flags(fp4)
        act, step = next(iter(plan.acts.values())), plan.lins[0]
        rows, frows = _sample(lin.M, 5), _sample(lin.K, 6)
        # the oracle's threshold, CSR and row codes of the sampled rows
        t, _, _ = orc.quantile_threshold(A_bits, lin.q)
        A_c_s, rp_s, ci_s, cv_s = orc.clamp_and_compensation(A_bits[rows], t)
        ref_a, ref_sa = orc.quantize_rows(A_c_s)
        assert np.array_equal(act.out["codes"][torch.from_numpy(rows).cuda()].cpu().numpy(), ref_a)
        w_codes, s_w = step.w_codes.cpu().numpy(), step.s_w.cpu().numpy()
        raw = fp4.fp4_linear_fwd(act.out["codes"], None, step.w_codes, None, lin.K, out_type="raw")
        assert_raw_acc_equals_int_mm(raw, act.out["codes"], step.w_codes)
        del raw
        Y = host_bits(step.Y[torch.from_numpy(rows).cuda()])
        dW = step.dW[torch.from_numpy(frows).cuda()].cpu().numpy()
        dx_ref = np.zeros((rows.size, lin.K))
        dx_mag = np.zeros((rows.size, lin.K))
        c0 = 0
        for m in work.members[lin.name]:
            blk = slice(c0, c0 + m.N)
            Wm, dYm = base.weight(m), base.grad(m)
            ref_w, ref_sw = orc.quantize_cols(orc.bf16_to_f32(Wm))      # every column of the member
            assert np.array_equal(w_codes[blk], ref_w)
            assert np.array_equal(s_w[blk].view(np.uint32), ref_sw.view(np.uint32))
            y_ref = orc.linear_fwd(ref_a, ref_sa, ref_w, ref_sw, rp_s, ci_s, cv_s, Wm)
            mag = orc.linear_fwd_magnitude(ref_a, ref_sa, ref_w, ref_sw, rp_s, ci_s, cv_s, Wm)
            assert_bf16_compensated_close(Y[:, blk], y_ref, mag)
            dw_ref = orc.wgrad_dge(A_bits, dYm, Wm, ref_sw, 5.0, 3.0, rows=frows)
            assert rel_frobenius(dW[:, blk], dw_ref) <= FROB_TOL
            dx_ref += orc.linear_dgrad(dYm, Wm, rows=rows)
            dx_mag += orc.linear_dgrad(dYm & np.uint16(0x7FFF), Wm & np.uint16(0x7FFF), rows=rows)
            c0 += m.N
        assert_bf16_compensated_close(host_bits(step.dX[torch.from_numpy(rows).cuda()]), dx_ref, dx_mag,
                                      bound=TC_SUM_BOUND)
        assert_no_device_flags(fp4)
