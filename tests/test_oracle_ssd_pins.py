"""Pins of the fp64 oracle's Mamba-2 SSD forward (``oracle.ssd_*``).

The recurrence (the definition) is pinned to its unrolled form — every
output written as an explicit sum over earlier tokens with the products of
the decays between them (brute-force loops) — and to closed forms (no
decay: a running sum of outer products; total forgetting: only the current
token).  The chunked algorithm is pinned to the recurrence for chunk sizes
from 1 to the whole sequence, ragged last chunks, an initial state and
grouped B/C; its pieces to what the page states they compute (the
log2-scaled cumulative sum restarting at every chunk; the states at chunk
checkpoints).  Plausible mistakes are written out as mutants, and each must
fail a pin.
"""

import numpy as np
import pytest

import oracle
import workloads


def _case(batch, L, H, P, N, G, seed, h0=False, decay_scale=1.0):
    d = workloads.ssd_inputs(batch, L, H, P, N, G, seed)
    x, B, C = (d[k].double().numpy() for k in ("x", "B", "C"))
    dt, A = d["dt"].double().numpy() * decay_scale, d["A"].double().numpy()
    init = np.random.default_rng(seed).standard_normal((batch, H, P, N)) if h0 else None
    return x, dt, A, B, C, init


def _diff(a, b):
    a, b = np.asarray(a), np.asarray(b)
    if a.shape != b.shape or not np.isfinite(a).all():
        return np.inf
    return float(np.abs(a - b).max())


# ------------------------------------------------- pins of the recurrence

def test_recurrence_equals_unrolled_sum():
    """y_t = sum_{s<=t} (c_t . b_s) prod_{s<r<=t} e^{a_r} x_s + prod_{r<=t} e^{a_r} h0 c_t."""
    x, dt, A, B, C, h0 = _case(1, 9, 2, 3, 4, 1, seed=1, h0=True, decay_scale=10.0)
    y, hf = oracle.ssd_recurrence(x, dt, A, B, C, h0)
    L = x.shape[1]
    for h in range(2):
        a = A[h] * dt[0, :, h]
        for t in range(L):
            acc = np.exp(a[:t + 1].sum()) * (h0[0, h] @ C[0, t, 0])
            for s in range(t + 1):
                acc = acc + (C[0, t, 0] @ B[0, s, 0]) * np.exp(a[s + 1:t + 1].sum()) * x[0, s, h]
            assert _diff(y[0, t, h], acc) <= 1e-12
        state = np.exp(a.sum()) * h0[0, h]
        for s in range(L):
            state = state + np.exp(a[s + 1:].sum()) * np.outer(x[0, s, h], B[0, s, 0])
        assert _diff(hf[0, h], state) <= 1e-12


def test_recurrence_without_decay_is_running_sum():
    """A = 0: h_t = sum_{s<=t} x_s b_s^T (a cumulative sum), y_t = h_t c_t."""
    x, dt, A, B, C, _ = _case(2, 11, 3, 4, 5, 1, seed=2)
    y, hf = oracle.ssd_recurrence(x, dt, np.zeros_like(A), B, C)
    outer = np.einsum("btp,btn->btpn", x[:, :, 1], B[:, :, 0])
    run = np.cumsum(outer, axis=1)
    assert _diff(y[:, :, 1], np.einsum("btpn,btn->btp", run, C[:, :, 0])) <= 1e-12
    assert _diff(hf[:, 1], run[:, -1]) <= 1e-12


def test_recurrence_with_total_forgetting_keeps_current_token():
    """exp(a_t) = 0 (underflow): h_t = x_t b_t^T, so y_t = (c_t . b_t) x_t."""
    x, dt, A, B, C, _ = _case(1, 7, 2, 3, 4, 1, seed=3)
    y, hf = oracle.ssd_recurrence(x, np.full_like(dt, 1e4), A, B, C)
    cb = np.einsum("btn,btn->bt", C[:, :, 0], B[:, :, 0])
    assert _diff(y, cb[:, :, None, None] * x) <= 1e-12
    assert _diff(hf[0, 0], np.outer(x[0, -1, 0], B[0, -1, 0])) <= 1e-12


# ------------------------------------------ pins of the chunked algorithm

CHUNK_CASES = [  # batch, L, H, P, N, G, chunk, h0
    (2, 37, 4, 8, 16, 2, 1, False), (1, 37, 4, 8, 16, 2, 8, True), (2, 64, 2, 16, 8, 1, 16, True),
    (1, 50, 3, 4, 4, 3, 50, False), (1, 50, 3, 4, 4, 1, 64, True), (2, 33, 2, 8, 8, 1, 7, True),
]


def pin_chunked_equals_recurrence(fn):
    worst = 0.0
    for batch, L, H, P, N, G, chunk, h0 in CHUNK_CASES:
        x, dt, A, B, C, init = _case(batch, L, H, P, N, G, seed=L + chunk, h0=h0, decay_scale=5.0)
        y, hf = oracle.ssd_recurrence(x, dt, A, B, C, init)
        yc, hfc = fn(x, dt, A, B, C, chunk, init)
        worst = max(worst, _diff(yc, y) / max(1.0, np.abs(y).max()), _diff(hfc, hf) / max(1.0, np.abs(hf).max()))
    return worst


def test_chunked_equals_recurrence():
    assert pin_chunked_equals_recurrence(oracle.ssd_chunked) <= 1e-12


def test_chunk_cumsum_is_log2_scaled_and_restarts():
    x, dt, A, B, C, _ = _case(2, 21, 3, 2, 2, 1, seed=5)
    g = oracle.ssd_chunk_cumsum(dt, A, 8)                        # chunks of 8, 8, 5
    for c, (t0, t1) in enumerate(((0, 8), (8, 16), (16, 21))):
        nat = np.cumsum(dt[:, t0:t1, :] * A, axis=1).transpose(0, 2, 1)
        assert _diff(np.exp2(g[:, :, c, :t1 - t0]), np.exp(nat)) <= 1e-12
        assert _diff(g[:, :, c, 0], oracle.ssd.LOG2E * (dt[:, t0, :] * A)) <= 1e-12   # restarts
    assert np.all(g <= 0)                                         # a_t < 0: exponents never positive


def test_fwd_pass_state_gives_states_at_chunk_checkpoints():
    """Each chunk's initial state is the recurrence's state just before the
    chunk; the final state is the recurrence's final state."""
    batch, L, H, P, N, G, chunk = 1, 30, 2, 4, 6, 1, 8
    x, dt, A, B, C, init = _case(batch, L, H, P, N, G, seed=6, h0=True, decay_scale=3.0)
    g = oracle.ssd_chunk_cumsum(dt, A, chunk)
    S_init, hf = oracle.ssd_fwd_pass_state(x, B, g, chunk, init)
    for c in range(g.shape[2]):
        t = c * chunk
        _, h_before = oracle.ssd_recurrence(x[:, :t], dt[:, :t], A, B[:, :t], C[:, :t], init)
        assert _diff(S_init[:, c], h_before) <= 1e-12
    _, h_all = oracle.ssd_recurrence(x, dt, A, B, C, init)
    assert _diff(hf, h_all) <= 1e-12


# ---------------------------------------------------------------- mutants

def _chunked_mutant(kind):
    """The oracle's chunked pipeline with one plausible mistake."""
    def fn(x, dt, A, B, C, chunk, h0=None):
        bs, L, H, P = x.shape
        N = B.shape[3]
        hpg = H // B.shape[2]
        nc = (L + chunk - 1) // chunk
        a = dt * A[None, None, :]
        y = np.zeros((bs, L, H, P))
        S = np.zeros((bs, H, P, N)) if h0 is None else np.array(h0, dtype=np.float64)
        run = np.zeros((bs, H))
        for c in range(nc):
            t0, t1 = c * chunk, min(L, (c + 1) * chunk)
            n = t1 - t0
            gl = np.cumsum(a[:, t0:t1], axis=1).transpose(0, 2, 1) * oracle.ssd.LOG2E
            if kind == "global_cumsum":
                gl = gl + run[:, :, None]
                run = gl[:, :, -1]
            ex = np.exp if kind == "natural_exp" else np.exp2
            mask = np.triu(np.ones((n, n), bool)) if kind == "upper_mask" else np.tril(np.ones((n, n), bool))
            for b in range(bs):
                for h in range(H):
                    gc, Bc, Cc = gl[b, h], B[b, t0:t1, h // hpg], C[b, t0:t1, h // hpg]
                    diff = gc[None, :] - gc[:, None] if kind == "sign_flip" else gc[:, None] - gc[None, :]
                    M = (Cc @ Bc.T) * ex(np.where(mask, diff, -np.inf))
                    carry = (Cc @ S[b, h].T) * (1.0 if kind == "no_h0_decay" else ex(gc)[:, None])
                    y[b, t0:t1, h] = M @ x[b, t0:t1, h] + carry
                    w = ex(gc[-1] - gc)
                    inc = (x[b, t0:t1, h] * w[:, None]).T @ Bc
                    S[b, h] = (1.0 if kind == "no_state_decay" else ex(gc[-1])) * S[b, h] + inc
        return y, S
    return fn


MUTANTS = ["global_cumsum", "natural_exp", "upper_mask", "sign_flip", "no_h0_decay", "no_state_decay"]


@pytest.mark.parametrize("kind", MUTANTS)
def test_chunked_mutant_is_caught(kind):
    with np.errstate(all="ignore"):
        assert not (pin_chunked_equals_recurrence(_chunked_mutant(kind)) <= 1e-12), kind


def test_mutant_template_reproduces_oracle():
    assert pin_chunked_equals_recurrence(_chunked_mutant("none")) <= 1e-12
