"""fp64 reference of the Mamba-2 SSD forward (state-space duality, chunked) —
TEST INFRASTRUCTURE ONLY.

"Accelerating Mamba-2 with high-performance forward kernels in NVIDIA CUDA
Tile": a linear recurrence with a fixed-size hidden state per head,
    h_t = exp(a_t) h_{t-1} + x_t b_t^T,    y_t = h_t c_t,    a_t = A[h] dt[t, h] < 0,
is evaluated chunk by chunk with matrix products (the "jump formula" gives
the state at chunk checkpoints; inside a chunk the outputs are
(C B^T o exp(G - G^T) o causal mask) X, as in softmax attention's masked
matrix), in three kernels: a per-chunk cumulative sum of a_t scaled by
log2(e) (so later exponentials are exp2), ``fwd_pass_state`` (a sequential
loop over chunks giving each chunk's initial state and the final state),
and the output of each chunk from its inputs and its initial state.

Notation and layouts (the page fixes no layout; these are the readings):
  x  [batch, L, H, P]   inputs of the recurrence (P = head dim)
  dt [batch, L, H]      time steps (> 0);  A [H] (< 0) per-head decay rate
  B, C [batch, L, G, N] (N = state size; head h uses group h // (H // G))
  h  [batch, H, P, N]   hidden state (h0 optional, zero by default)
  y  [batch, L, H, P]
The page's a_t is used as printed: the recurrence takes x_t as it is (a
caller wanting Mamba-2's discretised input passes x_t * dt_t).
"""

import numpy as np

LOG2E = 1.4426950408889634


def _group(H, G):
    if H % G != 0:
        raise ValueError("H must be a multiple of G")
    return H // G


def ssd_recurrence(x, dt, A, B, C, h0=None):
    """The plain definition: the recurrence, one time step at a time, in fp64.
    Returns (y [batch, L, H, P], h_final [batch, H, P, N])."""
    x, dt, A, B, C = (np.asarray(t, dtype=np.float64) for t in (x, dt, A, B, C))
    bs, L, H, P = x.shape
    N = B.shape[3]
    hpg = _group(H, B.shape[2])
    y = np.zeros((bs, L, H, P))
    hf = np.zeros((bs, H, P, N))
    for b in range(bs):
        for h in range(H):
            g = h // hpg
            st = np.zeros((P, N)) if h0 is None else np.array(h0[b, h], dtype=np.float64)
            for t in range(L):
                st = np.exp(A[h] * dt[b, t, h]) * st + np.outer(x[b, t, h], B[b, t, g])
                y[b, t, h] = st @ C[b, t, g]
            hf[b, h] = st
    return y, hf


def ssd_chunk_cumsum(dt, A, chunk):
    """Kernel 1: within each chunk, the running sum of a_t = A[h] dt[t, h],
    scaled by log2(e) (exp2 of it is exp of the natural sum).  It restarts at
    every chunk (not a global cumulative sum).  Returns g [batch, H, n_chunks,
    chunk]; positions past the end of a ragged last chunk hold the chunk's
    last value."""
    dt, A = np.asarray(dt, dtype=np.float64), np.asarray(A, dtype=np.float64)
    bs, L, H = dt.shape
    nc = (L + chunk - 1) // chunk
    g = np.zeros((bs, H, nc, chunk))
    for c in range(nc):
        t0, t1 = c * chunk, min(L, (c + 1) * chunk)
        a = (dt[:, t0:t1, :] * A[None, None, :]).transpose(0, 2, 1)      # [batch, H, len]
        cs = np.cumsum(a, axis=-1) * LOG2E
        g[:, :, c, :t1 - t0] = cs
        g[:, :, c, t1 - t0:] = cs[:, :, -1:]
    return g


def ssd_fwd_pass_state(x, B, g, chunk, h0=None):
    """fwd_pass_state: the sequential loop over chunks.  With s the chunk's
    first position, n its length and g its log2-scaled running sums, the jump
    formula carries the state across the chunk:
        S_next = 2^(g_last) S + sum_j 2^(g_last - g_j) x_j b_j^T.
    Returns (S_init [batch, n_chunks, H, P, N] — each chunk's initial state —
    and the final state [batch, H, P, N])."""
    x, B, g = (np.asarray(t, dtype=np.float64) for t in (x, B, g))
    bs, L, H, P = x.shape
    N = B.shape[3]
    hpg = _group(H, B.shape[2])
    nc = g.shape[2]
    S_init = np.zeros((bs, nc, H, P, N))
    S = np.zeros((bs, H, P, N)) if h0 is None else np.array(h0, dtype=np.float64)
    for c in range(nc):
        S_init[:, c] = S
        t0, t1 = c * chunk, min(L, (c + 1) * chunk)
        n = t1 - t0
        for b in range(bs):
            for h in range(H):
                gc = g[b, h, c, :n]
                w = np.exp2(gc[-1] - gc)                                     # decay to the chunk end
                inc = (x[b, t0:t1, h] * w[:, None]).T @ B[b, t0:t1, h // hpg]
                S[b, h] = np.exp2(gc[-1]) * S[b, h] + inc
    return S_init, S


def ssd_chunk_output(x, B, C, g, S_init, chunk):
    """The output of every chunk from its own inputs and its initial state:
        y_i = sum_{j <= i} (c_i . b_j) 2^(g_i - g_j) x_j  +  2^(g_i) S c_i,
    i, j positions in the chunk (the causal mask keeps j <= i, so every
    exponent is <= 0).  Returns y [batch, L, H, P]."""
    x, B, C, g, S_init = (np.asarray(t, dtype=np.float64) for t in (x, B, C, g, S_init))
    bs, L, H, P = x.shape
    hpg = _group(H, B.shape[2])
    y = np.zeros((bs, L, H, P))
    for c in range(g.shape[2]):
        t0, t1 = c * chunk, min(L, (c + 1) * chunk)
        n = t1 - t0
        causal = np.tril(np.ones((n, n), dtype=bool))
        for b in range(bs):
            for h in range(H):
                gc = g[b, h, c, :n]
                Cc, Bc = C[b, t0:t1, h // hpg], B[b, t0:t1, h // hpg]
                diff = np.where(causal, gc[:, None] - gc[None, :], -np.inf)
                M = (Cc @ Bc.T) * np.exp2(diff)
                y[b, t0:t1, h] = M @ x[b, t0:t1, h] + np.exp2(gc)[:, None] * (Cc @ S_init[b, c, h].T)
    return y


def ssd_chunked(x, dt, A, B, C, chunk, h0=None):
    """The chunked SSD forward: kernel 1, fwd_pass_state, then the chunk
    outputs.  Returns (y, h_final), equal to ``ssd_recurrence`` up to
    rounding."""
    g = ssd_chunk_cumsum(dt, A, chunk)
    S_init, hf = ssd_fwd_pass_state(x, B, g, chunk, h0)
    return ssd_chunk_output(x, B, C, g, S_init, chunk), hf
