"""Helpers of the GPU parity tests: tolerances, comparisons that record their
margins, and seeded-input plumbing.

Tolerances (bf16 inputs, fp32 accumulation, bf16 output) against the fp64
oracle on the same bf16 values: O max-abs <= 2e-2 and mean-abs <= 2e-3,
LSE max-abs <= 1e-3.  Tensors of other scales (gradients, SSD outputs and
states) are held to the same two bounds relative to their largest reference
magnitude.

Every comparison appends its errors to MARGINS; the test session prints them
at the end (tests/conftest.py), so a run shows how close each case came to
its bound, not only that it passed.
"""

import numpy as np
import torch

O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_MAX_ABS = 1e-3

MARGINS = []        # (test id, what, {name: (error, bound)})
CURRENT = ""        # id of the running test (set by tests/conftest.py)


def to64(t):
    return t.detach().float().cpu().double().numpy()


def _record(what, **pairs):
    MARGINS.append((CURRENT, what, pairs))


def assert_attn_close(o, lse, o_ref, lse_ref, what=""):
    o = to64(o) if isinstance(o, torch.Tensor) else o
    err = np.abs(o - o_ref)
    assert np.all(np.isfinite(o)), "%s: non-finite output" % what
    pairs = {"O max": (float(err.max()), O_MAX_ABS), "O mean": (float(err.mean()), O_MEAN_ABS)}
    if lse is not None:
        lse = to64(lse) if isinstance(lse, torch.Tensor) else lse
        fin = np.isfinite(lse_ref)
        assert np.array_equal(np.isfinite(lse), fin), "%s: LSE finiteness differs" % what
        if fin.any():
            pairs["LSE max"] = (float(np.abs(lse[fin] - lse_ref[fin]).max()), LSE_MAX_ABS)
        assert np.array_equal(lse[~fin], lse_ref[~fin]), "%s: -inf LSE mismatch" % what
    _record(what, **pairs)
    assert err.max() <= O_MAX_ABS, "%s: O max-abs %.4g" % (what, err.max())
    assert err.mean() <= O_MEAN_ABS, "%s: O mean-abs %.4g" % (what, err.mean())
    if "LSE max" in pairs:
        assert pairs["LSE max"][0] <= LSE_MAX_ABS, "%s: LSE max-abs %.4g" % (what, pairs["LSE max"][0])
    return err.max(), err.mean()


def assert_rel_close(got, ref, what, floor=1e-3):
    """max |got - ref| <= 2e-2 s and mean |got - ref| <= 2e-3 s with
    s = max(max |ref|, floor): the attention bounds at the tensor's own scale."""
    got = to64(got) if isinstance(got, torch.Tensor) else np.asarray(got, dtype=np.float64)
    scale = max(float(np.abs(ref).max()), floor)
    err = np.abs(got - ref)
    assert np.isfinite(got).all(), what + ": non-finite values"
    _record(what, **{"max/s": (float(err.max()) / scale, O_MAX_ABS),
                     "mean/s": (float(err.mean()) / scale, O_MEAN_ABS)})
    assert err.max() <= O_MAX_ABS * scale, "%s: max-abs %.4g vs %.4g x 2e-2" % (what, err.max(), scale)
    assert err.mean() <= O_MEAN_ABS * scale, "%s: mean-abs %.4g vs %.4g x 2e-3" % (what, err.mean(), scale)


def margin_lines():
    """One line per recorded comparison: each error and its fraction of the
    bound (1.00 = at the bound)."""
    lines = []
    for test, what, pairs in MARGINS:
        cols = "  ".join("%s %.3g (%.2f)" % (k, e, e / b) for k, (e, b) in pairs.items())
        worst = max(e / b for e, b in pairs.values()) if pairs else 0.0
        lines.append("%.2f  %s  | %s %s" % (worst, cols, test, what))
    return lines


def sample_rows(N, every, extra=()):
    """Rows the oracle evaluates at full size: every `every`-th row, both
    ends, both sides of every 128-row tile boundary near the ends."""
    rows = set(range(0, N, every))
    for r in (0, 1, 2, 126, 127, 128, 129, 255, 256, N // 2, N - 129, N - 128, N - 2, N - 1):
        if 0 <= r < N:
            rows.add(r)
    rows.update(r for r in extra if 0 <= r < N)
    return np.array(sorted(rows))
