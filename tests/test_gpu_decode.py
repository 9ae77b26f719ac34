"""GPU parity of attn_decode_paged (through the C-ABI) against the fp64 oracle.

Covers the full paged-decode workload (64 sequences, Hq 12, Hkv 2, d 128,
lengths U[128, 4096], block_size 16, permuted block table) on every output,
the ragged lengths around block edges, empty sequences, NaN in unused slots,
paging invariances, and the device-side checks of bad table entries.
"""

import ctypes

import numpy as np
import pytest
import torch

import exact_attention_47_gb300 as attn
import oracle
import workloads
from parity import assert_attn_close, to64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def to_dev(inp):
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def run(inp, scale, **kw):
    d = to_dev(inp)
    o, lse = attn.attn_decode_paged(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                    d["seq_lens"], scale=scale, **kw)
    torch.cuda.synchronize()
    return o, lse


def ref(inp, scale):
    return oracle.decode_paged(inp["q"].double().numpy(), inp["k_cache"].double().numpy(),
                               inp["v_cache"].double().numpy(), inp["block_table"].numpy(),
                               inp["seq_lens"].numpy(), scale)


def test_paged_decode_config_all_outputs():
    c = workloads.DECODE_CONFIGS["paged_decode"]
    inp = workloads.decode_inputs(c["num_seqs"], c["Hq"], c["Hkv"], c["d"], c["seed"],
                                  c["len_lo"], c["len_hi"])
    scale = workloads.default_scale(c["d"])
    o, lse = run(inp, scale)
    assert attn.device_status() == 0
    assert_attn_close(o, lse, *ref(inp, scale), what="paged_decode")


@pytest.mark.parametrize("Hq,Hkv,d", [(12, 2, 128), (8, 8, 64), (16, 1, 128), (6, 3, 64)])
def test_ragged_lengths(Hq, Hkv, d):
    lens = [1, 15, 16, 17, 31, 32, 33, 100, 255, 256, 257, 700, 4096]
    inp = workloads.decode_inputs(len(lens), Hq, Hkv, d, seed=20 + Hq + d, seq_lens=lens,
                                  len_hi=4096)
    scale = workloads.default_scale(d)
    o, lse = run(inp, scale)
    assert attn.device_status() == 0
    assert_attn_close(o, lse, *ref(inp, scale), what="ragged")


def test_empty_sequence_gives_zero_and_minus_inf():
    inp = workloads.decode_inputs(4, 12, 2, 128, seed=21, seq_lens=[0, 5, 0, 40], len_hi=64)
    o, lse = run(inp, 0.1)
    o_ref, lse_ref = ref(inp, 0.1)
    assert_attn_close(o, lse, o_ref, lse_ref, what="empty")
    assert torch.all(o[0] == 0) and torch.all(torch.isneginf(lse[0]))


def test_nan_in_unused_slots_does_not_leak():
    inp = workloads.decode_inputs(6, 12, 2, 128, seed=22, seq_lens=[1, 7, 17, 30, 49, 63],
                                  len_hi=64, nan_unused=True)
    o, lse = run(inp, 0.1)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    assert_attn_close(o, lse, *ref(inp, 0.1), what="nan slots")


def test_permuted_pool_gives_identical_bits():
    inp = workloads.decode_inputs(8, 12, 2, 128, seed=23, len_lo=1, len_hi=600)
    o1, l1 = run(inp, 0.1)
    nb = inp["k_cache"].shape[0]
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(5))
    k2 = torch.empty_like(inp["k_cache"]); v2 = torch.empty_like(inp["v_cache"])
    k2[perm] = inp["k_cache"]; v2[perm] = inp["v_cache"]
    t = inp["block_table"].long()
    t2 = torch.where(t >= 0, perm[t.clamp(min=0)], t).to(torch.int32)
    inp2 = dict(inp, k_cache=k2, v_cache=v2, block_table=t2)
    o2, l2 = run(inp2, 0.1)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_decode_equals_prefill_last_row():
    """Paging changes only where keys live: decode == last row of the causal
    forward over the same keys laid out contiguously (both on the GPU)."""
    L, Hq, Hkv, d = 333, 12, 2, 128
    inp = workloads.decode_inputs(1, Hq, Hkv, d, seed=24, seq_lens=[L], len_hi=512)
    o_dec, l_dec = run(inp, 0.088)
    kc, vc, table = inp["k_cache"], inp["v_cache"], inp["block_table"][0]
    pos = torch.arange(L)
    phys = table[pos // 16].long()
    k = kc[phys, :, pos % 16].permute(1, 0, 2).unsqueeze(0).contiguous()   # [1,Hkv,L,d]
    v = vc[phys, :, pos % 16].permute(1, 0, 2).unsqueeze(0).contiguous()
    q = torch.zeros(1, Hq, L, d, dtype=torch.bfloat16)
    q[0, :, L - 1] = inp["q"][0]
    o_fwd, l_fwd = attn.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, scale=0.088)
    torch.cuda.synchronize()
    assert (o_fwd[0, :, L - 1].float() - o_dec[0].float()).abs().max().item() <= 2e-2
    assert (l_fwd[0, :, L - 1] - l_dec[0]).abs().max().item() <= 1e-3


@pytest.mark.parametrize("ctas", [1, 3, 7, 64, 0])
def test_work_split_does_not_change_the_result(ctas):
    """One CTA walks every sequence; a few CTAs split sequences into many
    parts; a full wave gives the minimum chunk.  All agree with the oracle."""
    inp = workloads.decode_inputs(9, 12, 2, 128, seed=25, len_lo=1, len_hi=2000,
                                  seq_lens=[1, 700, 0, 17, 2000, 256, 1999, 33, 1024])
    try:
        attn.set_decode_max_ctas(ctas)
        o, lse = run(inp, 0.1)
    finally:
        attn.set_decode_max_ctas(0)
    assert attn.device_status() == 0
    assert_attn_close(o, lse, *ref(inp, 0.1), what="ctas %d" % ctas)


def test_deterministic():
    inp = workloads.decode_inputs(9, 12, 2, 128, seed=26, len_lo=1, len_hi=3000)
    o1, l1 = run(inp, 0.1)
    o2, l2 = run(inp, 0.1)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_bad_block_entry_is_reported_not_faulted():
    inp = workloads.decode_inputs(3, 12, 2, 128, seed=27, seq_lens=[40, 40, 40], len_hi=64)
    attn.device_status()  # clear
    bad = inp["block_table"].clone()
    bad[1, 1] = inp["k_cache"].shape[0] + 100        # outside the pool
    o, lse = run(dict(inp, block_table=bad), 0.1)
    assert attn.device_status() & attn.ATTN_DEV_BAD_BLOCK
    # the other sequences are untouched
    o_ref, lse_ref = ref(inp, 0.1)
    assert_attn_close(to64(o)[[0, 2]], to64(lse)[[0, 2]], o_ref[[0, 2]], lse_ref[[0, 2]])


def test_bad_seq_len_is_clamped_and_reported():
    inp = workloads.decode_inputs(2, 12, 2, 128, seed=28, seq_lens=[32, 20], len_hi=32,
                                  max_blocks_per_seq=2)
    attn.device_status()
    sl = inp["seq_lens"].clone()
    sl[1] = 1000                                     # more than 2 blocks of 16
    run(dict(inp, seq_lens=sl), 0.1)
    assert attn.device_status() & attn.ATTN_DEV_BAD_SEQLEN


def test_small_workspace_is_rejected():
    inp = workloads.decode_inputs(2, 12, 2, 128, seed=29, len_lo=1, len_hi=64)
    ws = torch.empty(64, dtype=torch.uint8, device=DEV)
    with pytest.raises(ValueError, match="workspace has 64 bytes"):      # the binding's check
        run(inp, 0.1, workspace=ws)
    d = to_dev(inp)
    o = torch.empty_like(d["q"])
    S, Hq, dh = d["q"].shape
    nb, Hkv = d["k_cache"].shape[:2]
    p = [ctypes.c_void_p(d[n].data_ptr()) for n in ("q", "k_cache", "v_cache", "block_table", "seq_lens")]
    st = attn.load_library().attn_decode_paged(*p, S, Hq, Hkv, dh, 16, d["block_table"].shape[1], nb, 0.1,
                                               ctypes.c_void_p(o.data_ptr()), None,
                                               ctypes.c_void_p(ws.data_ptr()), 64,
                                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 5                                                       # the C-ABI's: ATTN_ERR_WORKSPACE


def test_bounded_wait_times_out_and_reports():
    """A barrier nothing completes: the kernel gives up after 20 ms, sets
    the timeout bit and returns; the context stays usable."""
    flags = attn.selftest_wait_timeout(20_000_000)
    assert flags & attn.ATTN_DEV_TIMEOUT
    x = torch.ones(4, device=DEV)
    assert float(x.sum()) == 4.0
    assert attn.device_status() == 0


def _call(d, scale, o, lse, ws):
    attn.attn_decode_paged(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"],
                           scale=scale, o=o, lse=lse, workspace=ws)


def _outs(inp):
    S, Hq, d = inp["q"].shape
    return (torch.empty(S, Hq, d, dtype=torch.bfloat16, device=DEV),
            torch.empty(S, Hq, dtype=torch.float32, device=DEV))


def test_workspace_garbage_and_reuse():
    """The per-run arrival counters live in the caller's workspace: random
    bytes on entry, or the state another call left, must not change a
    result.  Several CTAs per sequence, so most runs are split."""
    a = workloads.decode_inputs(9, 12, 2, 128, seed=28, len_lo=1, len_hi=3000)
    b = workloads.decode_inputs(5, 12, 2, 128, seed=29, seq_lens=[2990, 1, 600, 2048, 77], len_hi=3000)
    mb = max(a["block_table"].shape[1], b["block_table"].shape[1])
    need = attn.attn_decode_paged_workspace_size(9, 12, 128, mb)
    ws = torch.randint(0, 256, (need,), dtype=torch.uint8, generator=torch.Generator().manual_seed(3)).to(DEV)
    da, db = to_dev(a), to_dev(b)
    oa, la = _outs(a)
    ob, lb = _outs(b)
    try:
        attn.set_decode_max_ctas(13)
        _call(da, 0.1, oa, la, ws)
        torch.cuda.synchronize()
        first = (oa.clone(), la.clone())
        _call(db, 0.1, ob, lb, ws)
        _call(da, 0.1, oa, la, ws)
        torch.cuda.synchronize()
    finally:
        attn.set_decode_max_ctas(0)
    assert attn.device_status() == 0
    assert_attn_close(first[0], first[1], *ref(a, 0.1), what="garbage workspace")
    assert_attn_close(ob, lb, *ref(b, 0.1), what="reused workspace")
    assert torch.equal(first[0], oa) and torch.equal(first[1], la)


@pytest.mark.parametrize("early", [0, 1, 2])
def test_graph_replay_reuses_counters(early):
    """A captured decode replays with the same counter tag every time; each
    call must leave the counters as it found them.  Two decodes back to back
    in one graph also exercise the programmatic dependency between them."""
    a = workloads.decode_inputs(9, 12, 2, 128, seed=30, len_lo=1, len_hi=2500)
    b = workloads.decode_inputs(9, 12, 2, 128, seed=31, len_lo=1, len_hi=2500)
    da, db = to_dev(a), to_dev(b)
    mb = max(a["block_table"].shape[1], b["block_table"].shape[1])
    ws = torch.zeros(attn.attn_decode_paged_workspace_size(9, 12, 128, mb), dtype=torch.uint8, device=DEV)
    oa, la = _outs(a)
    ob, lb = _outs(b)
    try:
        attn.set_decode_early_plan(early)
        _call(da, 0.1, oa, la, ws)
        _call(db, 0.1, ob, lb, ws)
        torch.cuda.synchronize()
        eager = [t.clone() for t in (oa, la, ob, lb)]
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(g):
                _call(da, 0.1, oa, la, ws)
                _call(db, 0.1, ob, lb, ws)
        torch.cuda.current_stream().wait_stream(side)
        for _ in range(3):
            for t in (oa, la, ob, lb):
                t.fill_(7.0)
            g.replay()
            torch.cuda.synchronize()
            assert all(torch.equal(x, y) for x, y in zip(eager, (oa, la, ob, lb)))
    finally:
        attn.set_decode_early_plan(0)
    assert attn.device_status() == 0
    assert_attn_close(oa, la, *ref(a, 0.1), what="graph replay a")
    assert_attn_close(ob, lb, *ref(b, 0.1), what="graph replay b")


def test_early_plan_gives_identical_bits():
    """The early plan only moves the split plan (level 1), and the first
    cache copies (level 2), before the wait for the preceding kernel: same
    split, same bits.  Chained calls with different lengths check that no
    call plans with another's lengths."""
    c = workloads.DECODE_CONFIGS["paged_decode"]
    inps = [workloads.decode_inputs(c["num_seqs"], c["Hq"], c["Hkv"], c["d"], c["seed"] + 50 * i,
                                    c["len_lo"], c["len_hi"]) for i in range(3)]
    devs = [to_dev(x) for x in inps]
    scale = workloads.default_scale(c["d"])
    res = {}
    for early in (0, 1, 2):
        try:
            attn.set_decode_early_plan(early)
            outs = []
            for d in devs:
                S = d["q"].shape[0]
                mb = d["block_table"].shape[1]
                ws = torch.empty(attn.attn_decode_paged_workspace_size(S, c["Hq"], c["d"], mb),
                                 dtype=torch.uint8, device=DEV)
                o, lse = _outs(d)
                _call(d, scale, o, lse, ws)
                outs.append((o, lse))
            torch.cuda.synchronize()
            res[early] = outs
        finally:
            attn.set_decode_early_plan(0)
    assert attn.device_status() == 0
    for level in (1, 2):
        for (o0, l0), (o1, l1) in zip(res[0], res[level]):
            assert torch.equal(o0, o1) and torch.equal(l0, l1)
    assert_attn_close(*res[2][2], *ref(inps[2], scale), what="early plan, third call")


@pytest.mark.parametrize("S,Hq,Hkv,d,lo,hi", [
    (48, 16, 1, 128, 1, 400),     # 16 query heads per KV head: the 14-stage ring
    (40, 8, 8, 64, 1, 300),       # d = 64, one query head per KV head
    (6, 12, 2, 128, 3000, 9000),  # few long sequences: every CTA inside one run
], ids=["G16", "d64", "long"])
def test_early_stream_levels_give_identical_bits(S, Hq, Hkv, d, lo, hi):
    """Every level of the early plan gives the same bits on the other kernel
    instances too: short sequences put last blocks of sequences among the
    first blocks of most CTAs (which the early stream leaves for after the
    wait), long ones give CTAs whose first blocks are all early."""
    inp = workloads.decode_inputs(S, Hq, Hkv, d, seed=60 + Hq + d, len_lo=lo, len_hi=hi)
    dv = to_dev(inp)
    scale = workloads.default_scale(d)
    ws = torch.empty(attn.attn_decode_paged_workspace_size(S, Hq, d, dv["block_table"].shape[1]),
                     dtype=torch.uint8, device=DEV)
    res = {}
    try:
        for early in (0, 1, 2):
            attn.set_decode_early_plan(early)
            o, lse = _outs(dv)
            for _ in range(2):                         # back to back: the second overlaps the first
                _call(dv, scale, o, lse, ws)
            torch.cuda.synchronize()
            res[early] = (o, lse)
    finally:
        attn.set_decode_early_plan(0)
    assert attn.device_status() == 0
    for level in (1, 2):
        assert torch.equal(res[0][0], res[level][0]) and torch.equal(res[0][1], res[level][1])
    assert_attn_close(*res[2], *ref(inp, scale), what="early stream, S %d Hq %d Hkv %d d %d" % (S, Hq, Hkv, d))


def test_long_sequences_split_into_many_parts():
    """Eight 16384-token sequences over one wave: every (sequence, KV head)
    run is split over about ten CTAs, so the part that arrives last merges
    ten or more published parts (several passes of the merge)."""
    inp = workloads.decode_inputs(8, 12, 2, 128, seed=32, len_lo=16384, len_hi=16384)
    o, lse = run(inp, 0.088)
    assert attn.device_status() == 0
    assert_attn_close(o, lse, *ref(inp, 0.088), what="8 x 16384 tokens")
