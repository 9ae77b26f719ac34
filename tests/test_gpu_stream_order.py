"""Stream order across launches (GPU).

Every kernel of the library is launched as a programmatic dependent of the
work before it in the stream: its CTAs may start while that kernel drains,
and they wait for it before touching global memory.  These tests put a
kernel that writes a call's inputs (or reads its outputs) immediately before
(or after) the call, on one stream, and check that every call sees the new
data: results equal those of the same call on freshly made tensors, and the
oracle where it is cheap.
"""

import pytest
import torch

import exact_attention_47_gb300 as attn
import oracle
import workloads
from parity import assert_attn_close, to64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def test_forward_sees_inputs_written_just_before():
    """q, k, v are overwritten by device copies right before each forward;
    back to back, with no synchronisation in between."""
    B, Hq, Hkv, N, d = 2, 4, 2, 384, 128
    inputs = [workloads.prefill_inputs(B, Hq, Hkv, N, d, seed=70 + i) for i in range(3)]
    dev_inputs = [tuple(t.to(DEV) for t in x) for x in inputs]
    q, k, v = (torch.empty_like(t) for t in dev_inputs[0])
    outs = []
    for qi, ki, vi in dev_inputs:
        q.copy_(qi)
        k.copy_(ki)
        v.copy_(vi)
        o, lse = attn.attn_fwd(q, k, v, causal=True, scale=0.09)
        outs.append((o, lse))
    torch.cuda.synchronize()
    for (qi, ki, vi), (o, lse) in zip(dev_inputs, outs):
        o_ref, lse_ref = attn.attn_fwd(qi, ki, vi, causal=True, scale=0.09)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    assert attn.device_status() == 0


def test_forward_output_read_just_after():
    """A torch kernel that reads the forward's output right after it sees the
    finished result (and the next forward, which overwrites the output
    buffer, waits for that reader)."""
    B, Hq, Hkv, N, d = 1, 4, 4, 256, 64
    x = [workloads.prefill_inputs(B, Hq, Hkv, N, d, seed=80 + i) for i in range(2)]
    a = tuple(t.to(DEV) for t in x[0])
    b = tuple(t.to(DEV) for t in x[1])
    o = torch.empty_like(a[0])
    attn.attn_fwd(*a, causal=False, scale=0.1, o=o)
    first = o.float().sum(dim=-1)          # reads o right after the first forward
    attn.attn_fwd(*b, causal=False, scale=0.1, o=o)
    torch.cuda.synchronize()
    o_a, _ = attn.attn_fwd(*a, causal=False, scale=0.1)
    torch.cuda.synchronize()
    assert torch.equal(first, o_a.float().sum(dim=-1))


@pytest.mark.parametrize("early", [0, 1, 2])
def test_decode_sees_lengths_and_queries_written_just_before(early):
    """Without the early plan, seq_lens may be written by the kernel right
    before the decode (a fill); the queries may always be.  With the early
    plan (either level) the lengths come from a host copy and only q is
    rewritten."""
    S, Hq, Hkv, d = 6, 12, 2, 128
    inp = workloads.decode_inputs(S, Hq, Hkv, d, seed=90, len_lo=700, len_hi=700)
    dv = {k: (t.to(DEV) if isinstance(t, torch.Tensor) else t) for k, t in inp.items()}
    qs = [torch.randn(S, Hq, d, generator=torch.Generator().manual_seed(91 + i)).to(torch.bfloat16).to(DEV)
          for i in range(3)]
    lens = [700, 333, 17]
    q = torch.empty_like(qs[0])
    seq_lens = dv["seq_lens"].clone()
    outs = []
    try:
        attn.set_decode_early_plan(early)
        for i in range(3):
            q.copy_(qs[i])
            if not early:
                seq_lens.fill_(lens[i])
            o, lse = attn.attn_decode_paged(q, dv["k_cache"], dv["v_cache"], dv["block_table"], seq_lens,
                                            scale=0.1)
            outs.append((o, lse))
        torch.cuda.synchronize()
    finally:
        attn.set_decode_early_plan(0)
    assert attn.device_status() == 0
    for i, (o, lse) in enumerate(outs):
        L = 700 if early else lens[i]
        ref_inp = dict(inp, q=qs[i].cpu(), seq_lens=torch.full((S,), L, dtype=torch.int32))
        o_ref, lse_ref = oracle.decode_paged(to64(ref_inp["q"]), to64(inp["k_cache"]), to64(inp["v_cache"]),
                                             inp["block_table"].numpy(), ref_inp["seq_lens"].numpy(), 0.1)
        assert_attn_close(o, lse, o_ref, lse_ref, what="decode after a write, call %d" % i)


def test_chained_fusions_consume_the_previous_output():
    """add + RMSNorm writes the residual in place and its output; SwiGLU then
    reads a tensor built from that output by a torch kernel: every step sees
    its predecessor's result."""
    rows, hidden = 512, 1536
    x, res, w = workloads.add_rmsnorm_inputs(rows, hidden, seed=95)
    x, res, w = x.to(DEV), res.to(DEV), w.to(DEV)
    res0 = res.clone()
    out1, _ = attn.fused_add_rmsnorm(x, res, w)
    out2, _ = attn.fused_add_rmsnorm(out1, res, w)   # reads out1 and the updated residual
    gu = torch.cat([out2, out1], dim=1).contiguous()  # [rows, 2 * hidden]: gate = out2, up = out1
    y = attn.fused_swiglu(gu)
    torch.cuda.synchronize()
    # The same chain with a synchronisation after every call.
    r = res0.clone()
    a1, _ = attn.fused_add_rmsnorm(x, r, w)
    torch.cuda.synchronize()
    a2, _ = attn.fused_add_rmsnorm(a1, r, w)
    torch.cuda.synchronize()
    y_ref = attn.fused_swiglu(torch.cat([a2, a1], dim=1).contiguous())
    torch.cuda.synchronize()
    assert torch.equal(out1, a1) and torch.equal(out2, a2) and torch.equal(res, r) and torch.equal(y, y_ref)


def _last_blocks_first(inp):
    """The same decode inputs with the physical blocks relabelled so that
    block b is the last block of sequence b: the last blocks of all the
    sequences form one contiguous slice of each cache."""
    table = inp["block_table"].clone()
    lens = inp["seq_lens"].tolist()
    nb = inp["k_cache"].shape[0]
    last = [int(table[b, (L + 15) // 16 - 1]) for b, L in enumerate(lens)]
    rest = [i for i in range(nb) if i not in set(last)]
    order = last + rest                                # new id -> old id
    new_id = torch.empty(nb, dtype=torch.int64)
    new_id[torch.tensor(order)] = torch.arange(nb)
    valid = table >= 0
    table[valid] = new_id[table[valid].long()].to(torch.int32)
    return dict(inp, block_table=table, k_cache=inp["k_cache"][order].contiguous(),
                v_cache=inp["v_cache"][order].contiguous())


@pytest.mark.parametrize("early", [0, 1, 2])
def test_decode_sees_last_blocks_written_just_before(early):
    """The newest token's block of every sequence (its last block) may be
    written by the kernel right before the decode at every early-plan
    level.  Here two residual-add kernels, launched as programmatic
    dependents that let their own dependents start early, rewrite the last
    K and V blocks of all 40 sequences in place just before the call; with
    lengths of 1 to 300 tokens every CTA's first blocks include last blocks,
    which the early stream of level 2 must leave for after the wait."""
    S, Hq, Hkv, d = 40, 12, 2, 128
    inp = _last_blocks_first(workloads.decode_inputs(S, Hq, Hkv, d, seed=97, len_lo=1, len_hi=300))
    g = torch.Generator().manual_seed(98)
    rows = S * Hkv * 16
    # Large changes to the keys move the scores; V changes by half its own
    # scale, so |O| stays in the range of the other decode cases (a bf16 ulp
    # of 8 is 0.0625 by itself, beyond the absolute bound).
    xk = (4 * torch.randn(rows, d, generator=g)).to(torch.bfloat16).to(DEV)
    xv = (0.5 * torch.randn(rows, d, generator=g)).to(torch.bfloat16).to(DEV)
    w = torch.ones(d, dtype=torch.bfloat16, device=DEV)
    dv = {k: (t.to(DEV) if isinstance(t, torch.Tensor) else t) for k, t in inp.items()}
    try:
        attn.set_decode_early_plan(early)
        for _ in range(2):                            # a warm call, then the checked one
            kc, vc = dv["k_cache"].clone(), dv["v_cache"].clone()
            torch.cuda.synchronize()
            attn.fused_add_rmsnorm(xk, kc[:S].view(rows, d), w)
            attn.fused_add_rmsnorm(xv, vc[:S].view(rows, d), w)
            o, lse = attn.attn_decode_paged(dv["q"], kc, vc, dv["block_table"], dv["seq_lens"], scale=0.1)
            torch.cuda.synchronize()
    finally:
        attn.set_decode_early_plan(0)
    assert attn.device_status() == 0
    kc64, vc64 = to64(kc.cpu()), to64(vc.cpu())
    args = (to64(inp["q"]),)
    tail = (inp["block_table"].numpy(), inp["seq_lens"].numpy(), 0.1)
    o_new, lse_new = oracle.decode_paged(*args, kc64, vc64, *tail)
    o_old, _ = oracle.decode_paged(*args, to64(inp["k_cache"]), to64(inp["v_cache"]), *tail)
    # The rewrite moves the outputs far beyond the tolerance, so a stale read would show.
    assert abs(o_new - o_old).max() > 0.5
    assert_attn_close(o, lse, o_new, lse_new, what="decode after last blocks rewritten, early %d" % early)
