"""Pins of the fp64 oracle's chunked prefill over a paged cache
(``oracle.prefill_paged``).

Each pin checks the oracle against something other than its own code:
torch's ``scaled_dot_product_attention`` and ``logsumexp`` in fp64 over the
logical (unpaged) key sequence that the input generator drew before storing
it through the table (a library routine), a brute-force walk over every slot
of the updated cache, closed forms, and invariants of the method (splitting a
chunk in two changes nothing; relabelling the physical blocks changes
nothing; the last new token is a decode step over the updated cache).
Plausible mistakes are written out as mutants, and each must fail a pin.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads


def _case(seed, ctx_lens, N, Hq=4, Hkv=2, d=8, spare=2, nan_unused=True):
    return workloads.paged_prefill_inputs(len(ctx_lens), Hq, Hkv, N, d, seed, ctx_lens=ctx_lens,
                                          spare_blocks=spare, nan_unused=nan_unused)


def _np(t):
    return t.double().numpy()


def _run(fn, x, scale, q=None, k_new=None, v_new=None, k_cache=None, v_cache=None,
         table=None, ctx=None):
    return fn(_np(x["q"]) if q is None else q,
              _np(x["k_new"]) if k_new is None else k_new,
              _np(x["v_new"]) if v_new is None else v_new,
              _np(x["k_cache"]) if k_cache is None else k_cache,
              _np(x["v_cache"]) if v_cache is None else v_cache,
              x["block_table"].numpy() if table is None else table,
              x["ctx_lens"].numpy() if ctx is None else ctx, scale, x["block_size"])


def _diff(a, b):
    """max |a - b|, or inf when a value is not finite where the other is."""
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    if a.shape != b.shape:
        return np.inf
    fa, fb = np.isfinite(a), np.isfinite(b)
    if (fa != fb).any() or (a[~fa] != b[~fb]).any():
        return np.inf
    return float(np.abs(a[fa] - b[fb]).max()) if fa.any() else 0.0


def _cache_equal(a, b):
    return np.array_equal(a, b, equal_nan=True) and np.array_equal(np.signbit(a), np.signbit(b))


# ---------------------------------------------------------------- the pins

def pin_sdpa(fn):
    """O and LSE equal torch SDPA / logsumexp over [prefix ; new keys], with
    query i allowed keys j <= ctx + i (fp64, K/V repeated per query head)."""
    N, Hq, Hkv = 19, 6, 2
    x = _case(21, [0, 5, 16, 37], N, Hq=Hq, Hkv=Hkv, d=16)
    scale = 0.35
    o, lse, _, _ = _run(fn, x, scale)
    worst = 0.0
    for b, ctx in enumerate(x["ctx_lens"].tolist()):
        K = torch.cat([x["k_prefix"][b].double(), x["k_new"][b].double()], dim=1)
        V = torch.cat([x["v_prefix"][b].double(), x["v_new"][b].double()], dim=1)
        K = K.repeat_interleave(Hq // Hkv, dim=0)
        V = V.repeat_interleave(Hq // Hkv, dim=0)
        Q = x["q"][b].double()
        mask = torch.arange(ctx + N)[None, :] <= (ctx + torch.arange(N))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=scale)
        logits = (scale * Q @ K.transpose(-1, -2)).masked_fill(~mask, float("-inf"))
        worst = max(worst, _diff(o[b], ref.numpy()), _diff(lse[b], torch.logsumexp(logits, -1).numpy()))
    return worst


def pin_cache_slots(fn):
    """Every slot of every block a sequence owns holds, after the call, its
    logical token (prefix, then the new rows) or zero past the new length;
    every other slot of the pool is unchanged (NaN included).  A walk over
    all slots, brute force."""
    N, Hkv = 21, 2
    x = _case(22, [3, 16, 30, 0], N, Hkv=Hkv, spare=3)
    _, _, kc, vc = _run(fn, x, 0.5)
    table = x["block_table"].numpy()
    bs = x["block_size"]
    bad = 0
    for out, cin, new, pref in ((kc, x["k_cache"], x["k_new"], x["k_prefix"]),
                                (vc, x["v_cache"], x["v_new"], x["v_prefix"])):
        cin = _np(cin)
        owned = np.zeros((cin.shape[0], bs), dtype=bool)
        for b, ctx in enumerate(x["ctx_lens"].tolist()):
            L = ctx + N
            logical = np.concatenate([_np(pref[b]), _np(new[b])], axis=1)   # [Hkv, L, d]
            for lb in range((L + bs - 1) // bs):
                phys = int(table[b, lb])
                for s in range(bs):
                    p = lb * bs + s
                    want = logical[:, p] if p < L else np.zeros_like(logical[:, 0])
                    bad += not _cache_equal(out[phys, :, s], want)
                    owned[phys, s] = True
        rest_out = out.transpose(0, 2, 1, 3)[~owned]
        rest_in = cin.transpose(0, 2, 1, 3)[~owned]
        bad += not _cache_equal(rest_out, rest_in)
    return float(bad)


def pin_closed_forms(fn):
    """(a) A sequence whose only token is the new one returns its value row
    and LSE = scale * |q . k| of that one key; (b) when every value row of a
    sequence (prefix and new) is the same vector, every output row is it."""
    x = _case(23, [0, 7], 1, Hq=2, Hkv=1, d=8)
    scale = 0.6
    o, lse, _, _ = _run(fn, x, scale)
    q, kn, vn = _np(x["q"]), _np(x["k_new"]), _np(x["v_new"])
    worst = max(_diff(o[0, :, 0], np.repeat(vn[0, :, 0], 2, axis=0)),
                _diff(lse[0, :, 0], scale * (q[0, :, 0] * kn[0, 0, 0]).sum(-1)))
    # (b): overwrite every value row with one vector, in the cache and in the new rows.
    y = _case(24, [5, 33], 12, Hq=4, Hkv=2, d=8, nan_unused=False)
    row = np.linspace(-1.0, 1.0, 8)
    vc = np.empty(tuple(y["v_cache"].shape))
    vc[:] = row
    vn = np.empty(tuple(y["v_new"].shape))
    vn[:] = row
    o, _, _, _ = _run(fn, y, 0.4, v_new=vn, v_cache=vc)
    return max(worst, _diff(o, np.broadcast_to(row, o.shape)))


def pin_chunk_split(fn):
    """Prefilling N1 then N2 new tokens (the second call on the first call's
    cache, its prefix N1 longer) gives the same outputs and the same final
    cache as prefilling all N1 + N2 at once."""
    N1, N2 = 13, 22
    x = _case(25, [4, 16, 29], N1 + N2, Hq=4, Hkv=2, d=8)
    scale = 0.45
    q, kn, vn = _np(x["q"]), _np(x["k_new"]), _np(x["v_new"])
    ctx = x["ctx_lens"].numpy()
    o, lse, kc, vc = _run(fn, x, scale)
    o1, l1, kc1, vc1 = _run(fn, x, scale, q=q[:, :, :N1], k_new=kn[:, :, :N1], v_new=vn[:, :, :N1])
    o2, l2, kc2, vc2 = _run(fn, x, scale, q=q[:, :, N1:], k_new=kn[:, :, N1:], v_new=vn[:, :, N1:],
                            k_cache=kc1, v_cache=vc1, ctx=ctx + N1)
    worst = max(_diff(o[:, :, :N1], o1), _diff(o[:, :, N1:], o2),
                _diff(lse[:, :, :N1], l1), _diff(lse[:, :, N1:], l2))
    if not (_cache_equal(kc, kc2) and _cache_equal(vc, vc2)):
        worst = np.inf
    return worst


def pin_block_relabel(fn):
    """Moving every physical block to another index (and the table with it)
    leaves O and LSE unchanged and moves the updated cache the same way."""
    x = _case(26, [9, 40, 0], 17, Hq=4, Hkv=1, d=8, spare=4)
    scale = 0.3
    o, lse, kc, vc = _run(fn, x, scale)
    nb = x["k_cache"].shape[0]
    perm = np.random.default_rng(7).permutation(nb)          # block i moves to perm[i]
    table = x["block_table"].numpy()
    table2 = np.where(table >= 0, perm[np.maximum(table, 0)], -1)
    kcin, vcin = _np(x["k_cache"]), _np(x["v_cache"])
    kc_in2, vc_in2 = np.empty_like(kcin), np.empty_like(vcin)
    kc_in2[perm], vc_in2[perm] = kcin, vcin
    o2, lse2, kc2, vc2 = _run(fn, x, scale, k_cache=kc_in2, v_cache=vc_in2, table=table2)
    worst = max(_diff(o, o2), _diff(lse, lse2))
    if not (_cache_equal(kc2[perm], kc) and _cache_equal(vc2[perm], vc)):
        worst = np.inf
    return worst


def pin_last_token_is_decode(fn):
    """The last new token of each sequence attends to every cached key, so
    its row equals a decode step (``oracle.decode_paged``, pinned on its own)
    over the updated cache with seq_lens = ctx + N."""
    N = 11
    x = _case(27, [0, 20, 47], N, Hq=6, Hkv=2, d=16)
    scale = 0.25
    o, lse, kc, vc = _run(fn, x, scale)
    od, ld = oracle.decode_paged(_np(x["q"])[:, :, N - 1], kc, vc, x["block_table"].numpy(),
                                 x["ctx_lens"].numpy() + N, scale, x["block_size"])
    return max(_diff(o[:, :, N - 1], od), _diff(lse[:, :, N - 1], ld))


PINS = [(pin_sdpa, 1e-12), (pin_cache_slots, 0.0), (pin_closed_forms, 1e-12),
        (pin_chunk_split, 1e-12), (pin_block_relabel, 0.0), (pin_last_token_is_decode, 1e-12)]


@pytest.mark.parametrize("pin,tol", PINS, ids=lambda x: getattr(x, "__name__", str(x)))
def test_paged_prefill_oracle_passes_pin(pin, tol):
    assert pin(oracle.prefill_paged) <= tol


# ---------------------------------------------------------------- mutants

def _mutant(kind):
    """The oracle's chunked prefill with one plausible mistake."""
    def fn(q, k_new, v_new, k_cache, v_cache, table, ctx_lens, scale, bs=16):
        S, Hq, N, d = q.shape
        Hkv = k_new.shape[1]
        G = Hq // Hkv
        kc, vc = np.array(k_cache, copy=True), np.array(v_cache, copy=True)
        for b in range(S):
            ctx = int(ctx_lens[b])
            for g in range(Hkv):
                for i in range(N):
                    pos = i if kind == "write_from_zero" else ctx + i
                    kc[int(table[b][pos // bs]), g, pos % bs] = k_new[b, g, i]
                    vc[int(table[b][pos // bs]), g, pos % bs] = v_new[b, g, i]
                end = ctx + N
                if N > 0 and end % bs and kind != "no_tail_clear":
                    kc[int(table[b][end // bs]), g, end % bs:] = 0.0
                    vc[int(table[b][end // bs]), g, end % bs:] = 0.0
        src_k, src_v = (k_cache, v_cache) if kind == "attend_stale_cache" else (kc, vc)
        o = np.zeros((S, Hq, N, d))
        lse = np.zeros((S, Hq, N))
        for b in range(S):
            ctx = int(ctx_lens[b])
            keys, rows = np.arange(ctx + N)[None, :], np.arange(N)[:, None]
            if kind == "mask_ignores_prefix":
                allowed = keys <= rows
            elif kind == "mask_strict":
                allowed = keys < ctx + rows
            else:
                allowed = keys <= ctx + rows
            for h in range(Hq):
                g = h % Hkv if kind == "wrong_kv_head" else h // G
                kk = oracle.gather_paged_keys(src_k, table[b], ctx + N, g, bs)
                vv = oracle.gather_paged_keys(src_v, table[b], ctx + N, g, bs)
                p, m, l = oracle.softmax_probs(oracle.score_matrix(q[b, h], kk, scale), allowed)
                o[b, h] = p @ vv
                with np.errstate(divide="ignore", invalid="ignore"):
                    lse[b, h] = m + np.log(l)
        return o, lse, kc, vc
    return fn


MUTANTS = ["write_from_zero", "no_tail_clear", "attend_stale_cache", "mask_ignores_prefix",
           "mask_strict", "wrong_kv_head"]


@pytest.mark.parametrize("kind", MUTANTS)
def test_paged_prefill_mutant_is_caught(kind):
    bad = _mutant(kind)
    with np.errstate(all="ignore"):
        caught = any(not (pin(bad) <= tol) for pin, tol in PINS)
    assert caught, kind


def test_mutant_framework_reproduces_oracle():
    """The mutant template without a mistake passes every pin, so a caught
    mutant is caught for its mistake."""
    good = _mutant("none")
    for pin, tol in PINS:
        assert pin(good) <= tol, pin.__name__
