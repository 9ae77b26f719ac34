"""GPU parity of fused_add_rmsnorm and fused_swiglu (through the C-ABI)
against the fp64 oracle.

Tolerances.  The new residual is the bf16 rounding of a sum of two bf16
values, computed exactly in fp32 for these inputs: it must equal the
oracle's bit for bit.  The outputs are bf16 roundings of fp32 results whose
own error (a sum of squares over the row, rsqrtf, __expf, a division) is far
below a bf16 unit, so each output is within one bf16 unit in the last place
of the exact value: |out - ref| <= 2^-8 |ref|, with a 1/64 margin for the
fp32 error when the exact value sits just above a power of two (the fp32
sum of squares over 8960 values can be off by about 2^-16 relative).
"""

import numpy as np
import pytest
import torch

import exact_attention_47_gb300 as attn
import oracle
import workloads
from parity import to64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
ULP = 2.0 ** -8


def _assert_ulp(got, ref, what):
    got = to64(got) if isinstance(got, torch.Tensor) else np.asarray(got, dtype=np.float64)
    assert np.isfinite(got).all(), what + ": non-finite output"
    err = np.abs(got - ref)
    bound = ULP * (1.0 + 2.0 ** -6) * np.abs(ref)
    worst = float((err - bound).max())
    assert worst <= 0.0, "%s: %d values beyond one bf16 ulp (worst excess %.3g)" % (
        what, int((err > bound).sum()), worst)


@pytest.mark.parametrize("rows,hidden", [(1, 8), (3, 1536), (17, 4096), (257, 264), (1000, 1536), (5, 8960)])
def test_add_rmsnorm_matches_oracle(rows, hidden):
    x, res, w = workloads.add_rmsnorm_inputs(rows, hidden, seed=rows + hidden)
    ref_out, ref_r = oracle.add_rmsnorm(x.double().numpy(), res.double().numpy(), w.double().numpy(), 1e-6)
    dres = res.to(DEV)
    out, dres = attn.fused_add_rmsnorm(x.to(DEV), dres, w.to(DEV), eps=1e-6)
    torch.cuda.synchronize()
    assert np.array_equal(to64(dres), ref_r), "residual differs from bf16(x + residual)"
    _assert_ulp(out, ref_out, "rmsnorm %dx%d" % (rows, hidden))


def test_add_rmsnorm_full_workload():
    c = workloads.FUSION_CONFIGS["qwen_add_rmsnorm"]
    x, res, w = workloads.add_rmsnorm_inputs(c["rows"], c["hidden"], c["seed"])
    ref_out, ref_r = oracle.add_rmsnorm(x.double().numpy(), res.double().numpy(), w.double().numpy(), 1e-6)
    out, dres = attn.fused_add_rmsnorm(x.to(DEV), res.to(DEV), w.to(DEV), eps=1e-6)
    torch.cuda.synchronize()
    assert np.array_equal(to64(dres), ref_r)
    _assert_ulp(out, ref_out, "qwen_add_rmsnorm")


def test_add_rmsnorm_large_eps_and_zero_rows():
    """eps dominating the mean square, and rows that sum to exactly zero."""
    x, res, w = workloads.add_rmsnorm_inputs(6, 64, seed=5)
    res[:2] = -x[:2]                                      # x + residual = 0 exactly
    ref_out, ref_r = oracle.add_rmsnorm(x.double().numpy(), res.double().numpy(), w.double().numpy(), 10.0)
    out, dres = attn.fused_add_rmsnorm(x.to(DEV), res.to(DEV), w.to(DEV), eps=10.0)
    torch.cuda.synchronize()
    assert np.array_equal(to64(dres), ref_r)
    assert np.all(to64(out)[:2] == 0.0)
    _assert_ulp(out, ref_out, "eps 10")


@pytest.mark.parametrize("rows,F", [(1, 8), (7, 200), (33, 8960), (1000, 2048), (3, 8)])
def test_swiglu_matches_oracle(rows, F):
    gu = workloads.swiglu_inputs(rows, F, seed=rows * 7 + F)
    out = attn.fused_swiglu(gu.to(DEV))
    torch.cuda.synchronize()
    _assert_ulp(out, oracle.swiglu(gu.double().numpy()), "swiglu %dx%d" % (rows, F))


def test_swiglu_full_workload_sampled_rows():
    c = workloads.FUSION_CONFIGS["qwen_swiglu"]
    gu = workloads.swiglu_inputs(c["rows"], c["F"], c["seed"])
    out = attn.fused_swiglu(gu.to(DEV))
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.arange(0, c["rows"], 61), [c["rows"] - 1]]))
    _assert_ulp(to64(out)[rows], oracle.swiglu(gu[rows].double().numpy()), "qwen_swiglu")


def test_fusions_empty_and_rejected():
    x = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    out, _ = attn.fused_add_rmsnorm(x, x.clone(), torch.ones(64, dtype=torch.bfloat16, device=DEV))
    assert out.numel() == 0
    assert attn.fused_swiglu(torch.empty((0, 16), dtype=torch.bfloat16, device=DEV)).numel() == 0
    with pytest.raises(attn.AttnError) as e:
        attn.fused_swiglu(torch.zeros((4, 24), dtype=torch.bfloat16, device=DEV))   # F = 12
    assert e.value.status == 2                            # ATTN_ERR_UNSUPPORTED: F not a multiple of 8
