"""GPU parity of attn_prefill_paged (through the C-ABI) against the fp64 oracle.

The chunked prefill appends new K/V rows to the paged cache and attends each
new query causally over the cached prefix and the new tokens up to itself.
Checked: O and LSE within the forward's tolerances; the updated cache equal
to the oracle's bit for bit (every slot of the pool, including the NaN that
the generator leaves in unused slots); prefixes that end inside a block, on
a block edge and on a 128-key tile edge; new-token counts of 1, ragged
tails and several query blocks; GQA / MQA / MHA and d = 64 / 128; the full
chunked-prefill workload on sampled rows; and how it composes with
attn_fwd, with a second chunk and with attn_decode_paged.
"""

import numpy as np
import pytest
import torch

import exact_attention_47_gb300 as attn
import oracle
import workloads
from parity import assert_attn_close, sample_rows, to64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _dev(x):
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def _gpu(x, scale, d=None):
    d = d or _dev(x)
    o, lse = attn.attn_prefill_paged(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"],
                                     d["block_table"], d["ctx_lens"], scale=scale)
    torch.cuda.synchronize()
    return o, lse, d


def _ref(x, scale, rows=None):
    return oracle.prefill_paged(x["q"].double().numpy(), x["k_new"].double().numpy(),
                                x["v_new"].double().numpy(), x["k_cache"].double().numpy(),
                                x["v_cache"].double().numpy(), x["block_table"].numpy(),
                                x["ctx_lens"].numpy(), scale, x["block_size"], rows=rows)


def _assert_cache_equal(got, want, what):
    got = to64(got)
    ok = np.array_equal(got, want, equal_nan=True) and np.array_equal(np.signbit(got), np.signbit(want))
    assert ok, "%s: cache differs in %d values" % (what, int((~((got == want) | (np.isnan(got) & np.isnan(want)))).sum()))


CASES = [  # S, Hq, Hkv, N, d, ctx_lens
    (2, 2, 2, 128, 64, [0, 0]),
    (3, 4, 2, 200, 128, [1, 15, 16]),
    (2, 6, 2, 333, 64, [127, 129]),
    (1, 12, 2, 513, 128, [1000]),
    (4, 4, 1, 1, 128, [0, 5, 31, 250]),
    (2, 8, 8, 256, 128, [300, 17]),
    (3, 12, 2, 700, 128, [128, 2000, 77]),
    (2, 16, 1, 37, 64, [255, 256]),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "S%dHq%dHkv%dN%dd%d-ctx%s" % (c[:5] + ("_".join(map(str, c[5])),)))
def test_prefill_paged_matches_oracle(case):
    S, Hq, Hkv, N, d, ctx = case
    x = workloads.paged_prefill_inputs(S, Hq, Hkv, N, d, seed=600 + N + d, ctx_lens=ctx, spare_blocks=3)
    scale = workloads.default_scale(d)
    o, lse, dx = _gpu(x, scale)
    assert attn.device_status() == 0
    ro, rl, rk, rv = _ref(x, scale)
    assert_attn_close(o, lse, ro, rl, what=str(case))
    _assert_cache_equal(dx["k_cache"], rk, "k_cache")
    _assert_cache_equal(dx["v_cache"], rv, "v_cache")


def test_chunked_prefill_workload_sampled_rows():
    c = workloads.PAGED_PREFILL_CONFIGS["qwen_chunked_prefill"]
    x = workloads.paged_prefill_inputs(c["num_seqs"], c["Hq"], c["Hkv"], c["N_new"], c["d"], c["seed"],
                                       ctx_lo=c["ctx_lo"], ctx_hi=c["ctx_hi"])
    scale = workloads.default_scale(c["d"])
    o, lse, dx = _gpu(x, scale)
    assert attn.device_status() == 0
    rows = sample_rows(c["N_new"], 97)
    ro, rl, rk, rv = _ref(x, scale, rows=rows)
    assert_attn_close(to64(o)[:, :, rows], to64(lse)[:, :, rows], ro, rl, what="qwen_chunked_prefill")
    _assert_cache_equal(dx["k_cache"], rk, "k_cache")
    _assert_cache_equal(dx["v_cache"], rv, "v_cache")


def test_zero_prefix_equals_attn_fwd():
    """With nothing cached the chunk is an ordinary causal prefill: the same
    kernel arithmetic on the same values, so the outputs agree bit for bit."""
    S, Hq, Hkv, N, d = 2, 6, 2, 300, 128
    x = workloads.paged_prefill_inputs(S, Hq, Hkv, N, d, seed=71, ctx_lens=[0, 0])
    scale = workloads.default_scale(d)
    o, lse, dx = _gpu(x, scale)
    of, lf = attn.attn_fwd(dx["q"], dx["k_new"], dx["v_new"], causal=True, scale=scale)
    torch.cuda.synchronize()
    assert torch.equal(o, of) and torch.equal(lse, lf)


def test_two_chunks_then_decode():
    """Prefill in two chunks, then decode one more token: each step on the
    GPU over the cache the previous GPU step left, each checked against the
    oracle run the same way on its own cache."""
    S, Hq, Hkv, d = 3, 12, 2, 128
    N1, N2 = 150, 260
    x = workloads.paged_prefill_inputs(S, Hq, Hkv, N1 + N2 + 1, d, seed=72, ctx_lens=[0, 33, 512])
    scale = workloads.default_scale(d)
    dx = _dev(x)
    ctx = x["ctx_lens"].numpy()
    rk, rv = x["k_cache"].double().numpy(), x["v_cache"].double().numpy()
    table = x["block_table"].numpy()
    q, kn, vn = (x[n].double().numpy() for n in ("q", "k_new", "v_new"))
    for lo, hi in ((0, N1), (N1, N1 + N2)):
        o, lse = attn.attn_prefill_paged(dx["q"][:, :, lo:hi].contiguous(),
                                         dx["k_new"][:, :, lo:hi].contiguous(),
                                         dx["v_new"][:, :, lo:hi].contiguous(), dx["k_cache"],
                                         dx["v_cache"], dx["block_table"],
                                         (dx["ctx_lens"] + lo).to(torch.int32), scale=scale)
        torch.cuda.synchronize()
        assert attn.device_status() == 0
        ro, rl, rk, rv = oracle.prefill_paged(q[:, :, lo:hi], kn[:, :, lo:hi], vn[:, :, lo:hi], rk, rv,
                                              table, ctx + lo, scale)
        assert_attn_close(o, lse, ro, rl, what="chunk %d:%d" % (lo, hi))
    _assert_cache_equal(dx["k_cache"], rk, "k_cache after two chunks")
    # The last token: a one-token chunk appends its K/V (and attends, which
    # is itself a decode step), then attn_decode_paged decodes it.
    lo = N1 + N2
    o1, l1 = attn.attn_prefill_paged(dx["q"][:, :, lo:].contiguous(), dx["k_new"][:, :, lo:].contiguous(),
                            dx["v_new"][:, :, lo:].contiguous(), dx["k_cache"], dx["v_cache"],
                            dx["block_table"], (dx["ctx_lens"] + lo).to(torch.int32), scale=scale)
    ro1, rl1, rk, rv = oracle.prefill_paged(q[:, :, lo:], kn[:, :, lo:], vn[:, :, lo:], rk, rv, table,
                                            ctx + lo, scale)
    seq_lens = (dx["ctx_lens"] + lo + 1).to(torch.int32)
    od, ld = attn.attn_decode_paged(dx["q"][:, :, lo].contiguous(), dx["k_cache"], dx["v_cache"],
                                    dx["block_table"], seq_lens, scale=scale)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    rod, rld = oracle.decode_paged(q[:, :, lo], rk, rv, table, ctx + lo + 1, scale)
    assert_attn_close(o1, l1, ro1, rl1, what="one-token chunk")
    assert_attn_close(od, ld, rod, rld, what="decode after prefill")


def test_bad_ctx_len_is_reported():
    """A ctx_lens entry beyond the table is reported; that sequence is not
    written and every loop stays bounded (the other sequence is unaffected)."""
    S, Hq, Hkv, N, d = 2, 4, 2, 64, 64
    x = workloads.paged_prefill_inputs(S, Hq, Hkv, N, d, seed=73, ctx_lens=[10, 20])
    scale = workloads.default_scale(d)
    dx = _dev(x)
    dx["ctx_lens"] = torch.tensor([10, 10 ** 6], dtype=torch.int32, device=DEV)
    o, lse, dx = _gpu(x, scale, d=dx)
    assert attn.device_status() & attn.ATTN_DEV_BAD_SEQLEN
    ro, rl, _, _ = _ref(x, scale)
    assert_attn_close(o[:1], lse[:1], ro[:1], rl[:1], what="good sequence")


def test_bad_block_entry_is_reported():
    S, Hq, Hkv, N, d = 1, 2, 1, 40, 64
    x = workloads.paged_prefill_inputs(S, Hq, Hkv, N, d, seed=74, ctx_lens=[30])
    dx = _dev(x)
    dx["block_table"][0, 1] = x["num_blocks"] + 5          # a prefix block outside the pool
    _gpu(x, workloads.default_scale(d), d=dx)
    assert attn.device_status() & attn.ATTN_DEV_BAD_BLOCK


def test_empty_chunk_launches_nothing():
    x = workloads.paged_prefill_inputs(2, 2, 2, 0, 64, seed=75, ctx_lens=[3, 4])
    before = x["k_cache"].clone()
    o, lse, dx = _gpu(x, 0.125)
    assert o.numel() == 0 and lse.numel() == 0
    assert torch.equal(dx["k_cache"].cpu().view(torch.int16), before.view(torch.int16))


def test_many_sequences_keep_query_block_order():
    """More sequences than the start-up cost ranking holds (257 > 256): the
    kernel walks the units in query-block order instead; same results."""
    S, Hq, Hkv, N, d = 257, 2, 1, 3, 64
    ctx = [(7 * b) % 41 for b in range(S)]
    x = workloads.paged_prefill_inputs(S, Hq, Hkv, N, d, seed=76, ctx_lens=ctx)
    scale = workloads.default_scale(d)
    o, lse, dx = _gpu(x, scale)
    assert attn.device_status() == 0
    ro, rl, rk, _ = _ref(x, scale)
    assert_attn_close(o, lse, ro, rl, what="257 sequences")
    _assert_cache_equal(dx["k_cache"], rk, "k_cache")
