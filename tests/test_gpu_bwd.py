"""GPU parity of attn_bwd (through the C-ABI) against the fp64 oracle.

The GPU forward gives O and the LSE, attn_bwd the gradients; the oracle
computes the exact gradients from the same bf16 inputs.  A gradient tensor g
is compared relative to its largest reference magnitude:
    max |g - ref| <= 2e-2 * max |ref|,   mean |g - ref| <= 2e-3 * max |ref|
(the forward's bounds on O, whose entries are of unit scale, carried over to
the scale of each gradient: P and dS are rounded to bf16 before their MMAs,
D uses the bf16 O, and the results are rounded to bf16).  The scale is
floored at 1e-3, so a gradient that vanishes identically (one allowed key:
P = 1 whatever the scores, so dQ = dK = 0) is held to 2e-5 absolute.
"""

import ctypes

import numpy as np
import pytest
import torch

import exact_attention_47_gb300 as attn
import oracle
import workloads
from parity import assert_rel_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _case(B, Hq, Hkv, N, d, seed):
    q, k, v = workloads.prefill_inputs(B, Hq, Hkv, N, d, seed)
    g = torch.Generator().manual_seed(seed + 1)
    do = torch.randn((B, Hq, N, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    return q, k, v, do


def _gpu(q, k, v, do, causal, scale):
    q, k, v, do = (t.to(DEV) for t in (q, k, v, do))
    o, lse = attn.attn_fwd(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = attn.attn_bwd(q, k, v, o, lse, do, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    return dq, dk, dv


def _assert_grad_close(got, ref, what):
    assert_rel_close(got, ref, what)


SHAPES = [  # B, Hq, Hkv, N, d — ragged tails, several tiles, GQA / MQA
    (1, 2, 2, 128, 64), (1, 2, 1, 200, 128), (2, 4, 2, 256, 128), (1, 6, 2, 333, 64),
    (1, 4, 4, 512, 128), (1, 3, 1, 1, 64), (1, 12, 2, 1024, 128),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%dHq%dHkv%dN%dd%d" % s)
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_matches_oracle(shape, causal):
    B, Hq, Hkv, N, d = shape
    q, k, v, do = _case(B, Hq, Hkv, N, d, seed=500 + N + d)
    scale = workloads.default_scale(d)
    dq, dk, dv = _gpu(q, k, v, do, causal, scale)
    rq, rk, rv = oracle.attention_backward(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                           do.double().numpy(), scale, causal)
    _assert_grad_close(dq, rq, "dq %s" % (shape,))
    _assert_grad_close(dk, rk, "dk %s" % (shape,))
    _assert_grad_close(dv, rv, "dv %s" % (shape,))


def test_bwd_deterministic():
    q, k, v, do = _case(1, 4, 2, 384, 128, seed=42)
    a = _gpu(q, k, v, do, True, 0.1)
    b = _gpu(q, k, v, do, True, 0.1)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_bwd_workspace_too_small_is_rejected():
    q, k, v, do = (t.to(DEV) for t in _case(1, 2, 2, 256, 64, seed=43))
    o, lse = attn.attn_fwd(q, k, v)
    small = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(ValueError, match="workspace has 16 bytes"):      # the binding's check
        attn.attn_bwd(q, k, v, o, lse, do, workspace=small)
    p = [ctypes.c_void_p(t.data_ptr()) for t in (q, k, v, o, lse, do)]
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    st = attn.load_library().attn_bwd(*p, *(ctypes.c_void_p(t.data_ptr()) for t in (dq, dk, dv)),
                                      1, 2, 2, 256, 64, 1, 0.125, ctypes.c_void_p(small.data_ptr()), 16,
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 5                                                       # the C-ABI's: ATTN_ERR_WORKSPACE
