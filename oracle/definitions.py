"""fp64 reference definitions of exact attention (prefill, paged decode,
chunked prefill over a paged cache, and the backward pass).

TEST INFRASTRUCTURE ONLY — see the package docstring.  Nothing on the GPU
product path imports this module.

Notation follows the pages: Q, K, V tensors; logits ``s``; the softmax
stabiliser ``m`` (row maximum); the running denominator ``l``; output O.

Layouts (the pages fix none; these are the readings used everywhere):
  prefill  q [B, Hq, N, d], k/v [B, Hkv, N, d]; o [B, Hq, N, d]; lse [B, Hq, N]
  decode   q [S, Hq, d]; k_cache/v_cache [num_blocks, Hkv, block_size, d];
           block_table [S, max_blocks] int; seq_lens [S] int;
           o [S, Hq, d]; lse [S, Hq]
  chunked  q [S, Hq, N, d] new queries, k_new/v_new [S, Hkv, N, d];
  prefill  paged caches and block_table as for decode; ctx_lens [S] int
           (tokens already cached); o [S, Hq, N, d]; lse [S, Hq, N]
Query head h reads KV head g = h // (Hq // Hkv) (contiguous GQA groups).
LSE is the natural log of the sum of exp of the *scaled* logits.
"""

import numpy as np

_NEG_INF = -np.inf


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def score_matrix(q_rows, k_rows, scale):
    """Scaled dot-product logits s_ij = scale * <q_i, k_j>.

    "Advanced attention mechanisms – II", section "Tiling", step 2 (Q x K^T
    for a pair of tiles gives the t x t score matrix); here the whole
    sequence is one tile.  The product is a library matmul in fp64.
    """
    return float(scale) * (_f64(q_rows) @ _f64(k_rows).T)


def softmax_probs(s, allowed):
    """Row softmax of logits ``s`` over the ``allowed`` entries (mask).

    "Advanced attention mechanisms – II", section "Softmax stabiliser":
    p_i = exp(l_i - m) / sum_j exp(l_j - m) with m the row maximum, so every
    numerator lies in [0, 1].  Disallowed entries get probability 0 (the mask
    step of section "Why?", A -> A').  Returns (p, m, l) where m is the row
    maximum over allowed entries and l the stabilised denominator.  A row with
    no allowed entry returns p = 0, m = -inf, l = 0.
    """
    s = _f64(s)
    allowed = np.asarray(allowed, dtype=bool)
    masked = np.where(allowed, s, _NEG_INF)
    m = masked.max(axis=-1)
    safe_m = np.where(np.isfinite(m), m, 0.0)
    e = np.where(allowed, np.exp(masked - safe_m[..., None]), 0.0)
    l = e.sum(axis=-1)
    p = np.divide(e, l[..., None], out=np.zeros_like(e), where=l[..., None] > 0)
    return p, m, l


def _causal_allowed(rows, n_keys):
    """Causal mask for prefill (Nq == Nk): query i sees keys j <= i."""
    rows = np.asarray(rows)
    return np.arange(n_keys)[None, :] <= rows[:, None]


def attention(q, k, v, scale, causal, rows=None):
    """Exact attention, the plain definition (the naive path the method replaces).

    "Advanced attention mechanisms – II", section "Why?": A = Q K^T, mask A to
    A', softmax A' to A'', then A'' V; with the stabiliser of section "Softmax
    stabiliser".  "Fast attention kernels and operator fusion accelerate AI
    models", section "FlashAttention-style attention and Paged Attention":
    the fused kernel computes the same function.

    q [B, Hq, N, d], k/v [B, Hkv, N, d].  ``rows`` optionally selects query
    rows (rows are independent by definition, so a subset is exact for those
    rows).  Returns (o [B, Hq, R, d], lse [B, Hq, R]) in fp64, R = len(rows).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    group = Hq // Hkv
    n_keys = k.shape[2]
    rows = np.arange(N) if rows is None else np.asarray(rows, dtype=np.int64)
    o = np.zeros((B, Hq, rows.size, v.shape[3]))
    lse = np.zeros((B, Hq, rows.size))
    # Row chunks only bound memory: each row's arithmetic is unchanged.
    chunk = 1024
    for b in range(B):
        for h in range(Hq):
            g = h // group
            for r0 in range(0, rows.size, chunk):
                rr = rows[r0:r0 + chunk]
                s = score_matrix(q[b, h, rr], k[b, g], scale)
                if causal:
                    allowed = _causal_allowed(rr, n_keys)
                else:
                    allowed = np.ones_like(s, dtype=bool)
                p, m, l = softmax_probs(s, allowed)
                o[b, h, r0:r0 + rr.size] = p @ v[b, g]
                with np.errstate(divide="ignore"):
                    lse[b, h, r0:r0 + rr.size] = m + np.log(l)
    return o, lse


def attention_backward(q, k, v, do, scale, causal):
    """Gradients of exact attention with respect to q, k and v.

    The forward is the plain definition of ``attention`` ("Advanced attention
    mechanisms – II", section "Why?"); section "Flash Attention" keeps the
    softmax statistics so that the backward pass can recompute the attention
    matrix instead of storing it.  This is the chain rule of that definition
    written out, with upstream gradient ``do`` = dL/dO:

        P    = softmax(s) over the allowed keys,  s = scale * Q K^T
        dV   = P^T dO                      (O = P V)
        dP   = dO V^T
        dS_ij = P_ij * (dP_ij - sum_k P_ik dP_ik)   (Jacobian of the row softmax)
        dQ   = scale * dS K,   dK = scale * dS^T Q

    Disallowed (masked) entries have P = 0 and so no gradient.  With GQA the
    K/V gradients of a KV head are summed over the query heads that read it.
    Returns (dq [B,Hq,N,d], dk [B,Hkv,N,d], dv [B,Hkv,N,d]) in fp64.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    group = Hq // Hkv
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            g = h // group
            s = score_matrix(q[b, h], k[b, g], scale)
            allowed = _causal_allowed(np.arange(N), k.shape[2]) if causal else np.ones_like(s, dtype=bool)
            p, _, _ = softmax_probs(s, allowed)
            dv[b, g] += p.T @ do[b, h]
            dp = do[b, h] @ v[b, g].T
            ds = p * (dp - (p * dp).sum(axis=-1, keepdims=True))
            dq[b, h] = float(scale) * (ds @ k[b, g])
            dk[b, g] += float(scale) * (ds.T @ q[b, h])
    return dq, dk, dv


def attention_online(q, k, v, scale, causal, tile):
    """Tile-by-tile attention with the running-max / running-sum softmax.

    "Advanced attention mechanisms – II", section "Tiling": step 1 splits
    K and V into tiles of ``tile`` rows; step 2 computes the tile's scores
    Q K_t^T; step 3 accumulates tile by tile.  Section "Incremental / online
    softmax": the value after every tile but the last is incomplete and the
    last tile reaches the exact result.  The page's own formula image is
    missing; the reading used is the standard one: keep per row the running
    maximum m, the running denominator l and the running unnormalised output
    acc; for each tile with logits s,
        m_new = max(m, max_j s_j)
        acc   = acc * exp(m - m_new) + sum_j exp(s_j - m_new) v_j
        l     = l   * exp(m - m_new) + sum_j exp(s_j - m_new)
    and finally o = acc / l, lse = m + log l.  fp64 throughout.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    group = Hq // Hkv
    n_keys = k.shape[2]
    dv = v.shape[3]
    o = np.zeros((B, Hq, N, dv))
    lse = np.zeros((B, Hq, N))
    rows = np.arange(N)
    for b in range(B):
        for h in range(Hq):
            g = h // group
            m = np.full(N, _NEG_INF)
            l = np.zeros(N)
            acc = np.zeros((N, dv))
            for j0 in range(0, n_keys, tile):
                kt = k[b, g, j0:j0 + tile]
                vt = v[b, g, j0:j0 + tile]
                s = score_matrix(q[b, h], kt, scale)
                keys = np.arange(j0, j0 + kt.shape[0])
                if causal:
                    allowed = keys[None, :] <= rows[:, None]
                else:
                    allowed = np.ones_like(s, dtype=bool)
                s = np.where(allowed, s, _NEG_INF)
                m_new = np.maximum(m, s.max(axis=1))
                # Rows that have seen no allowed key yet keep m = -inf.
                shift = np.where(np.isfinite(m_new), m_new, 0.0)
                alpha = np.where(np.isfinite(m), np.exp(m - shift), 0.0)
                e = np.where(allowed, np.exp(s - shift[:, None]), 0.0)
                acc = acc * alpha[:, None] + e @ vt
                l = l * alpha + e.sum(axis=1)
                m = m_new
            o[b, h] = acc / l[:, None]
            lse[b, h] = m + np.log(l)
    return o, lse


def split_partials(q_rows, k_rows, v_rows, scale, allowed, bounds):
    """Per-split partial softmax state over disjoint key ranges.

    For each key range [a, b) in ``bounds`` return (m_s, l_s, acc_s): the
    range's row maximum, stabilised denominator and unnormalised output
    sum_j exp(s_j - m_s) v_j.  The pages say nothing about splitting keys
    across workers; this is the same running-state algebra as the online
    softmax ("Advanced attention mechanisms – II", "Incremental / online
    softmax") applied to ranges that are processed independently.
    """
    s = score_matrix(q_rows, k_rows, scale)
    v_rows = _f64(v_rows)
    parts = []
    for a, b in bounds:
        ss = s[:, a:b]
        al = np.asarray(allowed)[:, a:b]
        masked = np.where(al, ss, _NEG_INF)
        m = masked.max(axis=1) if b > a else np.full(s.shape[0], _NEG_INF)
        shift = np.where(np.isfinite(m), m, 0.0)
        e = np.where(al, np.exp(masked - shift[:, None]), 0.0)
        parts.append((m, e.sum(axis=1), e @ v_rows[a:b]))
    return parts


def combine_partials(parts):
    """Merge independent partial states into the exact softmax result.

    With M = max_s m_s and w_s = exp(m_s - M): l = sum_s w_s l_s,
    o = sum_s w_s acc_s / l, lse = M + log l.  Splits with m_s = -inf
    (no allowed key) carry weight 0.  Rows with no allowed key at all
    return o = 0, lse = -inf.
    """
    ms = np.stack([p[0] for p in parts])
    M = ms.max(axis=0)
    shift = np.where(np.isfinite(M), M, 0.0)
    w = np.where(np.isfinite(ms), np.exp(ms - shift[None, :]), 0.0)
    l = sum(w[i] * parts[i][1] for i in range(len(parts)))
    acc = sum(w[i][:, None] * parts[i][2] for i in range(len(parts)))
    o = np.divide(acc, l[:, None], out=np.zeros_like(acc), where=l[:, None] > 0)
    with np.errstate(divide="ignore"):
        lse = np.where(l > 0, M + np.log(np.where(l > 0, l, 1.0)), _NEG_INF)
    return o, lse


def gather_paged_keys(cache, block_table_row, seq_len, kv_head, block_size):
    """Translate logical positions to physical cache slots, one by one.

    "Fast attention kernels and operator fusion accelerate AI models",
    section "FlashAttention-style attention and Paged Attention": the paged
    cache stores fixed-size blocks and a block table maps logical positions
    to physical blocks; the kernel translates every position through it.
    Position p lives at cache[block_table[p // block_size], kv_head,
    p % block_size].  Returns a [seq_len, d] fp64 array.
    """
    d = cache.shape[3]
    out = np.zeros((int(seq_len), d))
    for p in range(int(seq_len)):
        phys = int(block_table_row[p // block_size])
        out[p] = cache[phys, kv_head, p % block_size]
    return out


def decode_paged(q, k_cache, v_cache, block_table, seq_lens, scale,
                 block_size=16):
    """Single-token decode over a paged KV cache (plain definition).

    The query of sequence b is its last token and attends to all
    seq_lens[b] cached keys (no mask within them).  Keys and values are
    fetched through the block table (``gather_paged_keys``) and the
    definition of ``attention`` is applied to the one query row.  A sequence
    with no cached key returns o = 0 and lse = -inf.

    q [S, Hq, d]; caches [num_blocks, Hkv, block_size, d];
    returns (o [S, Hq, d], lse [S, Hq]) in fp64.
    """
    q = _f64(q)
    k_cache = np.asarray(k_cache)
    v_cache = np.asarray(v_cache)
    S, Hq, d = q.shape
    Hkv = k_cache.shape[1]
    group = Hq // Hkv
    o = np.zeros((S, Hq, v_cache.shape[3]))
    lse = np.full((S, Hq), _NEG_INF)
    for b in range(S):
        L = int(seq_lens[b])
        if L == 0:
            continue
        for g in range(Hkv):
            kk = gather_paged_keys(k_cache, block_table[b], L, g, block_size)
            vv = gather_paged_keys(v_cache, block_table[b], L, g, block_size)
            heads = slice(g * group, (g + 1) * group)
            s = score_matrix(q[b, heads], kk, scale)
            p, m, l = softmax_probs(s, np.ones_like(s, dtype=bool))
            o[b, heads] = p @ vv
            lse[b, heads] = m + np.log(l)
    return o, lse


def prefill_paged(q, k_new, v_new, k_cache, v_cache, block_table, ctx_lens, scale,
                  block_size=16, rows=None):
    """Chunked prefill over a paged KV cache (plain definition).

    "Fast attention kernels and operator fusion accelerate AI models",
    section "FlashAttention-style attention and Paged Attention": the KV cache
    grows as tokens arrive and lives in fixed-size blocks that a block table
    maps from logical positions; every position goes through that table.
    The step that fills the cache for a chunk of new tokens is read as:

      1. append: new token i of sequence b takes logical position
         ctx_lens[b] + i; its key and value rows are stored at
         cache[block_table[b][pos // block_size], g, pos % block_size];
      2. the slots past the sequence's new length in its last block are set
         to zero (they hold no token; clearing them keeps stale values out of
         the block);
      3. attend: new query i (position ctx_lens[b] + i) sees logical keys
         0 .. ctx_lens[b] + i — the whole cached prefix plus the new tokens up
         to itself (the causal mask at an offset) — gathered through the
         table (``gather_paged_keys``), with the definition of ``attention``.

    q [S, Hq, N, d]; k_new / v_new [S, Hkv, N, d]; caches
    [num_blocks, Hkv, block_size, d] (not modified: updated copies are
    returned); block_table [S, max_blocks] int; ctx_lens [S] int.
    ``rows`` optionally selects the new-query rows of step 3 (rows are
    independent by definition, so a subset is exact for those rows).
    Returns (o [S, Hq, R, d], lse [S, Hq, R], k_cache_out, v_cache_out) in
    fp64, R = len(rows) (N by default).
    """
    q, k_new, v_new = _f64(q), _f64(k_new), _f64(v_new)
    kc = np.array(k_cache, dtype=np.float64, copy=True)
    vc = np.array(v_cache, dtype=np.float64, copy=True)
    S, Hq, N, d = q.shape
    Hkv = k_new.shape[1]
    group = Hq // Hkv
    # Steps 1 and 2: the cache update.
    for b in range(S):
        ctx = int(ctx_lens[b])
        for g in range(Hkv):
            for i in range(N):
                pos = ctx + i
                phys = int(block_table[b][pos // block_size])
                kc[phys, g, pos % block_size] = k_new[b, g, i]
                vc[phys, g, pos % block_size] = v_new[b, g, i]
            end = ctx + N
            if N > 0 and end % block_size != 0:
                phys = int(block_table[b][end // block_size])
                kc[phys, g, end % block_size:] = 0.0
                vc[phys, g, end % block_size:] = 0.0
    # Step 3: attention of the new queries over the updated cache.
    rows = np.arange(N) if rows is None else np.asarray(rows, dtype=np.int64)
    o = np.zeros((S, Hq, rows.size, v_new.shape[3]))
    lse = np.zeros((S, Hq, rows.size))
    for b in range(S):
        ctx = int(ctx_lens[b])
        n_keys = ctx + N
        allowed = np.arange(n_keys)[None, :] <= (ctx + rows)[:, None]
        for g in range(Hkv):
            kk = gather_paged_keys(kc, block_table[b], n_keys, g, block_size)
            vv = gather_paged_keys(vc, block_table[b], n_keys, g, block_size)
            for h in range(g * group, (g + 1) * group):
                s = score_matrix(q[b, h, rows], kk, scale)
                p, m, l = softmax_probs(s, allowed)
                o[b, h] = p @ vv
                lse[b, h] = m + np.log(l)
    return o, lse, kc, vc
