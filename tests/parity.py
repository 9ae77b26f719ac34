"""Helpers of the GPU parity tests: tolerances and seeded-input plumbing.

Tolerances (bf16 inputs, fp32 accumulation, bf16 output) against the fp64
oracle on the same bf16 values: O max-abs <= 2e-2 and mean-abs <= 2e-3,
LSE max-abs <= 1e-3.
"""

import numpy as np
import torch

O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_MAX_ABS = 1e-3


def to64(t):
    return t.detach().float().cpu().double().numpy()


def assert_attn_close(o, lse, o_ref, lse_ref, what=""):
    o = to64(o) if isinstance(o, torch.Tensor) else o
    err = np.abs(o - o_ref)
    assert np.all(np.isfinite(o)), "%s: non-finite output" % what
    assert err.max() <= O_MAX_ABS, "%s: O max-abs %.4g" % (what, err.max())
    assert err.mean() <= O_MEAN_ABS, "%s: O mean-abs %.4g" % (what, err.mean())
    if lse is not None:
        lse = to64(lse) if isinstance(lse, torch.Tensor) else lse
        fin = np.isfinite(lse_ref)
        assert np.array_equal(np.isfinite(lse), fin), "%s: LSE finiteness differs" % what
        if fin.any():
            lerr = np.abs(lse[fin] - lse_ref[fin])
            assert lerr.max() <= LSE_MAX_ABS, "%s: LSE max-abs %.4g" % (what, lerr.max())
        assert np.array_equal(lse[~fin], lse_ref[~fin]), "%s: -inf LSE mismatch" % what
    return err.max(), err.mean()


def sample_rows(N, every, extra=()):
    """Rows the oracle evaluates at full size: every `every`-th row, both
    ends, both sides of every 128-row tile boundary near the ends."""
    rows = set(range(0, N, every))
    for r in (0, 1, 2, 126, 127, 128, 129, 255, 256, N // 2, N - 129, N - 128, N - 2, N - 1):
        if 0 <= r < N:
            rows.add(r)
    rows.update(r for r in extra if 0 <= r < N)
    return np.array(sorted(rows))
