"""GPU check of the FMA-pipe exp2 (attn_selftest_exp2_poly, through the
C-ABI) against exp2 in fp64 and against the special-function unit's exp2
as torch computes it: relative error below 2^-18 over [-125, 127]; below
2^-125 and not negative under -126 (-inf included)."""

import numpy as np
import pytest
import torch

import exact_attention_47_gb300 as attn

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
BOUND = 2.0 ** -18


def test_exp2_poly_within_bound():
    rng = np.random.default_rng(11)
    x = np.concatenate([np.linspace(-125.0, 127.0, 1000001), rng.uniform(-125.0, 127.0, 200001),
                        np.arange(-125, 127, dtype=np.float64) + 0.5]).astype(np.float32)
    y = attn.selftest_exp2_poly(torch.from_numpy(x).to(DEV))
    torch.cuda.synchronize()
    got = y.cpu().double().numpy()
    rel = np.abs(got / np.exp2(x.astype(np.float64)) - 1.0)
    assert rel.max() < BOUND, float(rel.max())
    # Beside the special-function unit's exp2 (torch.exp2 on the GPU).
    ref_sfu = torch.exp2(torch.from_numpy(x).to(DEV)).cpu().double().numpy()
    assert np.abs(got / ref_sfu - 1.0).max() < 2 * BOUND


def test_exp2_poly_underflow_odd_length_and_in_place():
    x = torch.tensor([-126.5, -150.0, -1e30, float("-inf"), 0.0, 1.0, -1.0], dtype=torch.float32, device=DEV)
    y = attn.selftest_exp2_poly(x)                     # odd length: the last pair is half used
    torch.cuda.synchronize()
    got = y.cpu().double().numpy()
    assert np.all(got[:4] >= 0.0) and np.all(got[:4] < 2.0 ** -125)
    assert np.all(np.abs(got[4:] / np.array([1.0, 2.0, 0.5]) - 1.0) < BOUND)
    z = x.clone()
    attn.selftest_exp2_poly(z, y=z)                    # in place
    torch.cuda.synchronize()
    assert torch.equal(z, y)
    assert attn.selftest_exp2_poly(torch.empty(0, device=DEV)).numel() == 0
