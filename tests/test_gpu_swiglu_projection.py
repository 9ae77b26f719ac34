"""GPU parity of swiglu_projection (the gate/up GEMM with SiLU * up in its
epilogue, through the C-ABI) against the fp64 oracle.

Tolerance.  The products x_k W_fk of bf16 values are exact in fp32; the
tensor cores add them in fp32, in an order the test does not fix, so the
projected g and u carry at most (hidden - 1) 2^-23 sum_k |x_k W_fk| of
summation error (the standard bound for fp32 summation in any order, with
truncating additions allowed).  That error passes through
out = silu(g) u as |silu'(g) u| dg + |silu(g)| du; silu itself (__expf, one
division) is exact to about 2^-21 relative; the result is rounded once to
bf16.  So each element must satisfy
    |out - ref| <= 2^-8 (1 + 2^-6) |ref| + 1.01 (|silu'(g) u| A_g + |silu(g)| A_u),
A = (hidden - 1) 2^-23 (|x| |W|^T), computed in fp64 from the same inputs.
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


def _bound(x, w):
    x = np.asarray(x, np.float64)
    w = np.asarray(w, np.float64)
    F = w.shape[0] // 2
    g, u = x @ w[:F].T, x @ w[F:].T
    ref = oracle.swiglu_projection(x, w)
    scale = (x.shape[1] - 1) * 2.0 ** -23
    a_g = scale * (np.abs(x) @ np.abs(w[:F]).T)
    a_u = scale * (np.abs(x) @ np.abs(w[F:]).T)
    sig = 1.0 / (1.0 + np.exp(-g))
    dsilu = sig * (1.0 + g * (1.0 - sig))
    silu = g * sig
    return ref, 2.0 ** -8 * (1.0 + 2.0 ** -6) * np.abs(ref) + 1.01 * (np.abs(dsilu * u) * a_g + np.abs(silu) * a_u)


def _check(out, x, w, what):
    got = to64(out) if isinstance(out, torch.Tensor) else np.asarray(out, np.float64)
    ref, bound = _bound(x, w)
    assert np.isfinite(got).all(), what + ": non-finite output"
    err = np.abs(got - ref)
    frac = float((err / bound).max())
    assert frac <= 1.0, "%s: %d values beyond the bound (worst %.3f of it)" % (what, int((err > bound).sum()), frac)
    print("%s: worst error %.3f of the bound, max |err| %.3g" % (what, frac, float(err.max())))


SHAPES = [  # rows, hidden, F: ragged row tiles, several K steps and feature tiles
    (1, 64, 128), (200, 128, 256), (513, 1536, 384), (130, 320, 1024), (128, 64, 128), (1000, 768, 640),
]


@pytest.mark.parametrize("rows,hidden,F", SHAPES)
def test_swiglu_projection_matches_oracle(rows, hidden, F):
    x, w = workloads.swiglu_projection_inputs(rows, hidden, F, seed=rows + hidden + F)
    out = attn.swiglu_projection(x.to(DEV), w.to(DEV))
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    _check(out, x.double().numpy(), w.double().numpy(), "proj %dx%dx%d" % (rows, hidden, F))


def test_swiglu_projection_full_workload_sampled_rows():
    c = workloads.FUSION_CONFIGS["qwen_swiglu_projection"]
    x, w = workloads.swiglu_projection_inputs(c["rows"], c["hidden"], c["F"], c["seed"])
    out = attn.swiglu_projection(x.to(DEV), w.to(DEV))
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    rows = np.unique(np.concatenate([np.arange(0, c["rows"], 379), [127, 128, c["rows"] - 1]]))
    _check(to64(out)[rows], x[rows].double().numpy(), w.double().numpy(), "qwen_swiglu_projection")


def test_swiglu_projection_matches_unfused_path_shape_and_rejects():
    # Empty problem, and sizes the kernel does not tile.
    x = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    w = torch.zeros((256, 64), dtype=torch.bfloat16, device=DEV)
    assert attn.swiglu_projection(x, w).shape == (0, 128)
    with pytest.raises(attn.AttnError) as e:
        attn.swiglu_projection(torch.zeros((4, 96), dtype=torch.bfloat16, device=DEV),
                               torch.zeros((256, 96), dtype=torch.bfloat16, device=DEV))   # hidden 96
    assert e.value.status == 2
    with pytest.raises(attn.AttnError) as e:
        attn.swiglu_projection(torch.zeros((4, 64), dtype=torch.bfloat16, device=DEV),
                               torch.zeros((192, 64), dtype=torch.bfloat16, device=DEV))   # F = 96
    assert e.value.status == 2
