"""Pins for the fp64 oracle, against things other than the oracle itself.

Each test pins the oracle to brute force with the textbook (unstabilised)
softmax, hand-worked closed forms, a library routine, or an invariant that
the mathematics fixes.  The mutation tests at the end plant plausible
mistakes in the oracle (on the CPU) and check that some pin catches each.

Sources: "Advanced attention mechanisms – II" (Aryan Das), sections "Why?",
"Tiling", "Softmax stabiliser", "Incremental / online softmax";
"Fast attention kernels and operator fusion accelerate AI models", section
"FlashAttention-style attention and Paged Attention".
"""

import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import oracle.definitions as oa
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * std


def brute_force(q, k, v, scale, causal):
    """Scalar loops with the unstabilised textbook softmax
    p_j = exp(s_j) / sum exp(s_j) (section "Softmax stabiliser", first
    formula), lse = log(sum exp(s_j)).  Inputs are kept small so exp does
    not overflow; this shares no code or formula shape with the oracle."""
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    o = np.zeros(q.shape[:3] + (v.shape[3],))
    lse = np.zeros(q.shape[:3])
    for b in range(B):
        for h in range(Hq):
            g = h // G
            for i in range(N):
                keys = range(i + 1) if causal else range(k.shape[2])
                ex = {}
                for j in keys:
                    dot = 0.0
                    for c in range(d):
                        dot += float(q[b, h, i, c]) * float(k[b, g, j, c])
                    ex[j] = math.exp(scale * dot)
                z = sum(ex.values())
                for c in range(v.shape[3]):
                    o[b, h, i, c] = sum(ex[j] * float(v[b, g, j, c]) for j in ex) / z
                lse[b, h, i] = math.log(z)
    return o, lse


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("N", [1, 2, 3, 17])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (4, 2), (3, 1)])
def test_brute_force_small(N, causal, Hq, Hkv):
    d = 8
    q = _rand((1, Hq, N, d), 1 + N, 0.7)
    k = _rand((1, Hkv, N, d), 2 + N, 0.7)
    v = _rand((1, Hkv, N, 5), 3 + N)
    scale = 0.35
    o, lse = oracle.attention(q, k, v, scale, causal)
    ob, lb = brute_force(q, k, v, scale, causal)
    assert np.max(np.abs(o - ob)) <= 1e-12
    assert np.max(np.abs(lse - lb)) <= 1e-12


def test_brute_force_tiny_config_rows():
    """The tiny workload (B1 H2 N256 d64) itself, on a handful of rows."""
    cfg = workloads.PREFILL_CONFIGS["tiny"]
    q, k, v = workloads.prefill_inputs(cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["N"], cfg["d"], cfg["seed"])
    q, k, v = (t.double().numpy() for t in (q, k, v))
    scale = workloads.default_scale(cfg["d"])
    rows = np.array([0, 1, 77, 255])
    for causal in (False, True):
        o, lse = oracle.attention(q, k, v, scale, causal, rows=rows)
        ob, lb = brute_force(q[:, :, rows], k, v, scale, False) if not causal else (None, None)
        if causal:
            # brute force over the causal prefix of each sampled row
            for idx, r in enumerate(rows):
                obr, lbr = brute_force(q[:, :, r:r + 1], k[:, :, :r + 1], v[:, :, :r + 1], scale, False)
                assert np.max(np.abs(o[:, :, idx] - obr[:, :, 0])) <= 1e-12
                assert np.max(np.abs(lse[:, :, idx] - lbr[:, :, 0])) <= 1e-12
        else:
            assert np.max(np.abs(o - ob)) <= 1e-12
            assert np.max(np.abs(lse - lb)) <= 1e-12


# ------------------------------------------------------------- closed forms

def _golden():
    with open(os.path.join(GOLDEN, "three_keys_closed_form.json")) as f:
        return json.load(f)


def _arr(x):
    return np.array(x, dtype=np.float64)


def test_golden_three_keys_prefill():
    g = _golden()["prefill"]
    q, k, v = _arr(g["q"]), _arr(g["k"]), _arr(g["v"])
    o, lse = oracle.attention(q, k, v, g["scale"], False)
    assert np.allclose(o, _arr(g["expected_noncausal_o"]), atol=1e-12, rtol=0)
    assert np.allclose(lse, _arr(g["expected_noncausal_lse"]), atol=1e-12, rtol=0)
    o, lse = oracle.attention(q, k, v, g["scale"], True)
    assert np.allclose(o, _arr(g["expected_causal_o"]), atol=1e-12, rtol=0)
    assert np.allclose(lse, _arr(g["expected_causal_lse"]), atol=1e-12, rtol=0)


def test_golden_three_keys_paged():
    g = _golden()["paged"]
    conv = lambda x: np.array(x, dtype=object).astype(np.float64)  # "nan" strings
    o, lse = oracle.decode_paged(_arr(g["q"]), conv(g["k_cache"]), conv(g["v_cache"]),
                                 np.array(g["block_table"]), np.array(g["seq_lens"]),
                                 g["scale"], block_size=g["block_size"])
    assert np.allclose(o, _arr(g["expected_o"]), atol=1e-12, rtol=0)
    assert np.allclose(lse, _arr(g["expected_lse"]), atol=1e-12, rtol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_equal_scores_give_mean_of_v(causal):
    """q = 0 makes every logit 0: o_i is the mean of the allowed V rows and
    lse_i = ln(#allowed) (i+1 causal, N otherwise)."""
    N, d = 37, 16
    q = np.zeros((1, 2, N, d))
    k = _rand((1, 1, N, d), 5)
    v = _rand((1, 1, N, 9), 6)
    o, lse = oracle.attention(q, k, v, 0.125, causal)
    for i in range(N):
        n = i + 1 if causal else N
        assert np.allclose(o[0, :, i], v[0, 0, :n].mean(axis=0), atol=1e-13, rtol=0)
        assert np.allclose(lse[0, :, i], math.log(n), atol=1e-13, rtol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_v_gives_constant_output(causal):
    N, d = 50, 8
    q = _rand((2, 2, N, d), 7, 2.0)
    k = _rand((2, 2, N, d), 8, 2.0)
    c = _rand((5,), 9)
    v = np.broadcast_to(c, (2, 2, N, 5)).copy()
    o, _ = oracle.attention(q, k, v, 0.5, causal)
    assert np.max(np.abs(o - c)) <= 1e-13


def test_causal_row_zero_is_v0():
    N, d = 20, 8
    q = _rand((1, 3, N, d), 10, 3.0)
    k = _rand((1, 3, N, d), 11, 3.0)
    v = _rand((1, 3, N, d), 12)
    o, lse = oracle.attention(q, k, v, 0.3, True)
    assert np.array_equal(o[:, :, 0], v[:, :, 0])
    assert np.allclose(lse[:, :, 0], 0.3 * np.einsum("bhc,bhc->bh", q[:, :, 0], k[:, :, 0]),
                       atol=1e-13, rtol=0)


def test_one_dominant_key_selects_its_value():
    """A key whose logit exceeds every other by 200 gets weight 1 - O(e^-200)."""
    N, d = 9, 4
    q = np.zeros((1, 1, 1, d)); q[..., 0] = 1.0
    k = _rand((1, 1, N, d), 13) * 0.01
    k[0, 0, 4, 0] = 200.0
    v = _rand((1, 1, N, 3), 14)
    o, lse = oracle.attention(q, k, v, 1.0, False)
    assert np.allclose(o[0, 0, 0], v[0, 0, 4], atol=1e-12, rtol=0)


# --------------------------------------------------------------- invariants

@pytest.mark.parametrize("causal", [False, True])
def test_probabilities_are_a_distribution(causal):
    """Section "Softmax stabiliser": stabilised numerators lie in [0, 1];
    every row of P sums to 1."""
    N = 64
    s = _rand((N, N), 15, 8.0)
    allowed = oa._causal_allowed(np.arange(N), N) if causal else np.ones((N, N), bool)
    p, m, l = oracle.softmax_probs(s, allowed)
    assert np.all(p >= 0) and np.all(p <= 1)
    assert np.max(np.abs(p.sum(axis=1) - 1)) <= 1e-12
    assert np.all(p[~allowed] == 0)
    assert np.all((l >= 1) & (l <= N))  # the max entry contributes exp(0) = 1


def test_shift_invariance():
    """Adding a constant c to every logit of a row leaves o unchanged and
    shifts lse by c.  Realised by k_j -> k_j + u with <q_i, u> = c/scale for
    one query row: q = e0 * a, u = e0 * c/(scale a)."""
    N, d, scale = 30, 6, 0.4
    q = _rand((1, 1, 1, d), 16); q[..., 0] = 1.5
    k = _rand((1, 1, N, d), 17)
    v = _rand((1, 1, N, d), 18)
    c = 7.25
    u = np.zeros(d); u[0] = c / (scale * 1.5)
    q[..., 1:] = 0.0
    o1, l1 = oracle.attention(q, k, v, scale, False)
    o2, l2 = oracle.attention(q, k + u, v, scale, False)
    assert np.max(np.abs(o1 - o2)) <= 1e-12
    assert np.max(np.abs((l2 - l1) - c)) <= 1e-12


@pytest.mark.parametrize("tile", [1, 7, 64, 100])
@pytest.mark.parametrize("causal", [False, True])
def test_online_blocked_equals_one_shot(tile, causal):
    """Section "Incremental / online softmax": partial values are
    incomplete, the last step reaches the exact result."""
    N, d = 100, 16
    q = _rand((2, 4, N, d), 19, 1.5)
    k = _rand((2, 2, N, d), 20, 1.5)
    v = _rand((2, 2, N, d), 21)
    o1, l1 = oracle.attention(q, k, v, 0.25, causal)
    o2, l2 = oracle.attention_online(q, k, v, 0.25, causal, tile)
    assert np.max(np.abs(o1 - o2)) <= 1e-12
    assert np.max(np.abs(l1 - l2)) <= 1e-12


def test_online_partial_is_incomplete():
    """Stopping the online loop before the last tile is not the answer."""
    N, d = 40, 8
    q = _rand((1, 1, N, d), 22, 2.0)
    k = _rand((1, 1, N, d), 23, 2.0)
    v = _rand((1, 1, N, d), 24)
    o_full, _ = oracle.attention(q, k, v, 0.5, False)
    o_part, _ = oracle.attention(q, k[:, :, :30], v[:, :, :30], 0.5, False)
    assert np.max(np.abs(o_full - o_part)) > 1e-3


@pytest.mark.parametrize("bounds", [[(0, 13), (13, 40), (40, 64)],
                                    [(0, 64)],
                                    [(0, 0), (0, 32), (32, 64), (64, 64)]])
def test_split_combine_equals_one_shot(bounds):
    N, d = 64, 8
    q = _rand((5, d), 25, 2.0)
    k = _rand((N, d), 26, 2.0)
    v = _rand((N, d), 27)
    allowed = np.ones((5, N), bool)
    allowed[0, 10:] = False  # one row that only some splits can see
    parts = oracle.split_partials(q, k, v, 0.5, allowed, bounds)
    o, lse = oracle.combine_partials(parts)
    p, m, l = oracle.softmax_probs(oracle.score_matrix(q, k, 0.5), allowed)
    assert np.max(np.abs(o - p @ v)) <= 1e-12
    assert np.max(np.abs(lse - (m + np.log(l)))) <= 1e-12


def test_combine_with_no_allowed_key():
    parts = [(np.array([-np.inf]), np.array([0.0]), np.zeros((1, 3)))]
    o, lse = oracle.combine_partials(parts)
    assert np.all(o == 0) and lse[0] == -np.inf


# ------------------------------------------------------------ library cross-check

@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_sdpa_fp64_tiny(causal):
    """torch scaled_dot_product_attention (named on the page "Fast attention
    kernels ...", section "FlashAttention-style attention ..."), CPU, fp64."""
    cfg = workloads.PREFILL_CONFIGS["tiny"]
    q, k, v = workloads.prefill_inputs(cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["N"], cfg["d"], cfg["seed"])
    q, k, v = (t.double() for t in (q, k, v))
    scale = workloads.default_scale(cfg["d"])
    ref = F.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=scale)
    o, _ = oracle.attention(q.numpy(), k.numpy(), v.numpy(), scale, causal)
    assert np.max(np.abs(o - ref.numpy())) <= 1e-10


@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_sdpa_fp64_gqa(causal):
    q, k, v = workloads.prefill_inputs(1, 12, 2, 96, 32, seed=31)
    q, k, v = (t.double() for t in (q, k, v))
    ref = F.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=0.2, enable_gqa=True)
    o, _ = oracle.attention(q.numpy(), k.numpy(), v.numpy(), 0.2, causal)
    assert np.max(np.abs(o - ref.numpy())) <= 1e-10


def test_gqa_equals_repeated_kv_heads():
    """Contiguous groups: head h reads KV head h // (Hq/Hkv)."""
    q = _rand((1, 6, 20, 8), 32)
    k = _rand((1, 2, 20, 8), 33)
    v = _rand((1, 2, 20, 8), 34)
    o1, l1 = oracle.attention(q, k, v, 0.3, True)
    o2, l2 = oracle.attention(q, np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1), 0.3, True)
    assert np.max(np.abs(o1 - o2)) == 0 and np.max(np.abs(l1 - l2)) == 0


# -------------------------------------------------------------------- paged

def _small_decode(seed=40, **kw):
    args = dict(num_seqs=5, Hq=6, Hkv=2, d=16, seed=seed, len_lo=1, len_hi=70)
    args.update(kw)
    return workloads.decode_inputs(**args)


def test_paged_equals_contiguous_last_row():
    """Decode of a paged sequence equals the last row of causal prefill over
    the same keys laid out contiguously (the query is the last token)."""
    inp = _small_decode()
    kc = inp["k_cache"].double().numpy(); vc = inp["v_cache"].double().numpy()
    q = inp["q"].double().numpy()
    o, lse = oracle.decode_paged(q, kc, vc, inp["block_table"].numpy(),
                                 inp["seq_lens"].numpy(), 0.25)
    for b, L in enumerate(inp["seq_lens"].tolist()):
        for g in range(2):
            kk = oracle.gather_paged_keys(kc, inp["block_table"][b].numpy(), L, g, 16)
            vv = oracle.gather_paged_keys(vc, inp["block_table"][b].numpy(), L, g, 16)
            qq = np.zeros((1, 3, L, 16))
            qq[0, :, L - 1] = q[b, 3 * g:3 * g + 3]
            op, lp = oracle.attention(qq, kk[None, None], vv[None, None], 0.25, True, rows=[L - 1])
            assert np.max(np.abs(op[0, :, 0] - o[b, 3 * g:3 * g + 3])) <= 1e-12
            assert np.max(np.abs(lp[0, :, 0] - lse[b, 3 * g:3 * g + 3])) <= 1e-12


def test_paged_translation_by_hand():
    """gather_paged_keys against a direct, hand-indexed construction."""
    kc = np.arange(4 * 1 * 4 * 2, dtype=np.float64).reshape(4, 1, 4, 2)
    table = np.array([3, 1, 0])
    got = oracle.gather_paged_keys(kc, table, 10, 0, 4)
    want = np.concatenate([kc[3, 0], kc[1, 0], kc[0, 0, :2]])
    assert np.array_equal(got, want)


def test_paged_permutation_invariance():
    """Moving blocks to other physical slots and rewriting the table gives
    the identical result (paging does not change the logical elements)."""
    inp = _small_decode(seed=41)
    kc = inp["k_cache"].double().numpy(); vc = inp["v_cache"].double().numpy()
    table = inp["block_table"].numpy()
    perm = np.random.default_rng(3).permutation(kc.shape[0])  # new slot of old block
    kc2 = np.empty_like(kc); vc2 = np.empty_like(vc)
    kc2[perm] = kc; vc2[perm] = vc
    table2 = np.where(table >= 0, perm[np.maximum(table, 0)], -1)
    args = (inp["q"].double().numpy(),)
    o1, l1 = oracle.decode_paged(*args, kc, vc, table, inp["seq_lens"].numpy(), 0.3)
    o2, l2 = oracle.decode_paged(*args, kc2, vc2, table2, inp["seq_lens"].numpy(), 0.3)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_paged_unused_slots_do_not_leak():
    inp = _small_decode(seed=42, nan_unused=True)
    o, lse = oracle.decode_paged(inp["q"].double().numpy(), inp["k_cache"].double().numpy(),
                                 inp["v_cache"].double().numpy(), inp["block_table"].numpy(),
                                 inp["seq_lens"].numpy(), 0.3)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))


def test_paged_empty_sequence():
    inp = _small_decode(seed=43, seq_lens=[0, 5, 16, 17, 1])
    o, lse = oracle.decode_paged(inp["q"].double().numpy(), inp["k_cache"].double().numpy(),
                                 inp["v_cache"].double().numpy(), inp["block_table"].numpy(),
                                 inp["seq_lens"].numpy(), 0.3)
    assert np.all(o[0] == 0) and np.all(lse[0] == -np.inf)
    assert np.all(np.isfinite(o[1:])) and np.all(np.isfinite(lse[1:]))


def test_paged_single_key_returns_its_value():
    inp = _small_decode(seed=44, seq_lens=[1, 1, 1, 1, 1])
    o, lse = oracle.decode_paged(inp["q"].double().numpy(), inp["k_cache"].double().numpy(),
                                 inp["v_cache"].double().numpy(), inp["block_table"].numpy(),
                                 inp["seq_lens"].numpy(), 0.3)
    vc = inp["v_cache"].double().numpy()
    for b in range(5):
        phys = int(inp["block_table"][b, 0])
        for h in range(6):
            assert np.array_equal(o[b, h], vc[phys, h // 3, 0])


# ---------------------------------------------------------------- mutations

def _pins_pass():
    """A compact subset of the pins above, used against planted mistakes."""
    try:
        test_brute_force_small(3, True, 4, 2)
        test_brute_force_small(17, False, 4, 2)
        test_golden_three_keys_prefill()
        test_causal_row_zero_is_v0()
        test_gqa_equals_repeated_kv_heads()
        test_matches_torch_sdpa_fp64_gqa(True)
        return True
    except AssertionError:
        return False


def test_pins_pass_unmodified():
    assert _pins_pass()


def test_mutation_strict_causal_mask_is_caught(monkeypatch):
    # off by one: query i no longer sees its own key
    monkeypatch.setattr(oa, "_causal_allowed",
                        lambda rows, n: np.arange(n)[None, :] < np.asarray(rows)[:, None])
    assert not _pins_pass()


def test_mutation_dropped_scale_is_caught(monkeypatch):
    monkeypatch.setattr(oa, "score_matrix", lambda q, k, scale: np.asarray(q, float) @ np.asarray(k, float).T)
    assert not _pins_pass()


def test_mutation_wrong_gqa_head_map_is_caught(monkeypatch):
    real = oa.attention

    def wrong(q, k, v, scale, causal, rows=None):
        # head h reads KV head h % Hkv instead of h // G
        q = np.asarray(q, float); Hq, Hkv = q.shape[1], np.asarray(k).shape[1]
        idx = np.arange(Hq) % Hkv
        return real(q, np.asarray(k, float)[:, idx], np.asarray(v, float)[:, idx], scale, causal, rows)

    monkeypatch.setattr(oracle, "attention", wrong)
    assert not _pins_pass()


def test_mutation_unnormalised_output_is_caught(monkeypatch):
    real = oa.softmax_probs

    def wrong(s, allowed):
        p, m, l = real(s, allowed)
        return p * l[..., None] / (l[..., None] + 1.0), m, l

    monkeypatch.setattr(oa, "softmax_probs", wrong)
    assert not _pins_pass()
