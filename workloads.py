"""Seeded synthetic inputs shared by the tests, ``bench.py`` and the oracle checks.

This module only draws random numbers and lays them out: it holds none of
the attention arithmetic, so both the CUDA path and the fp64 oracle can be
fed from it without sharing any code with each other.

Every tensor is drawn in fp32 from ``torch.Generator().manual_seed(seed)``
on the CPU and rounded to bf16 (round-to-nearest-even); the oracle consumes
the exact bf16 values (upcast to fp64) and the GPU gets the same bits.

The shapes mirror the pages' workloads: GPT-2-sized heads ("Advanced
attention mechanisms – II", section "Flash Attention"), a Qwen2.5-1.5B-style
GQA layer and block_size = 16 paged decode ("Fast attention kernels and
operator fusion accelerate AI models", section "FlashAttention-style
attention and Paged Attention").  No model weights or datasets are used.
"""

import math

import torch

BLOCK_SIZE = 16

# name -> parameters of the five workloads
PREFILL_CONFIGS = {
    "tiny": dict(B=1, Hq=2, Hkv=2, N=256, d=64, std=1.0, key_offset=False, seed=0),
    "gpt2_small": dict(B=8, Hq=12, Hkv=12, N=1024, d=64, std=1.0, key_offset=False, seed=1),
    "qwen_gqa_prefill": dict(B=4, Hq=12, Hkv=2, N=4096, d=128, std=1.0, key_offset=False, seed=2),
    "long_context": dict(B=1, Hq=16, Hkv=16, N=16384, d=128, std=0.5, key_offset=True, seed=3),
}
DECODE_CONFIGS = {
    "paged_decode": dict(num_seqs=64, Hq=12, Hkv=2, d=128, len_lo=128, len_hi=4096, seed=4),
}


def _randn(gen, shape, std=1.0):
    x = torch.randn(*shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x


def prefill_inputs(B, Hq, Hkv, N, d, seed, std=1.0, key_offset=False):
    """q [B,Hq,N,d], k/v [B,Hkv,N,d] bf16 (CPU), entries ~ N(0, std^2).

    With ``key_offset`` every key row j of every head gets one extra
    N(0, 1) draw added to all of its d components (a per-row offset that
    widens the range of the logits, as in the long-context workload).
    """
    gen = torch.Generator().manual_seed(int(seed))
    q = _randn(gen, (B, Hq, N, d), std)
    k = _randn(gen, (B, Hkv, N, d), std)
    v = _randn(gen, (B, Hkv, N, d), std)
    if key_offset:
        k = k + _randn(gen, (B, Hkv, N, 1))
    return (q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16))


def default_scale(d):
    """1/sqrt(d) rounded to fp32 — the value handed to both sides."""
    return float(torch.tensor(1.0 / math.sqrt(d), dtype=torch.float32))


def decode_inputs(num_seqs, Hq, Hkv, d, seed, len_lo=128, len_hi=4096,
                  seq_lens=None, block_size=BLOCK_SIZE, permute=True,
                  nan_unused=True, max_blocks_per_seq=None, spare_blocks=0):
    """Paged-cache decode inputs.

    seq_lens ~ U{len_lo..len_hi} (inclusive) unless given.  The physical
    pool holds exactly sum ceil(L/16) blocks (+ ``spare_blocks`` unused
    ones); each sequence's table row is a consecutive slice of one random
    permutation of the pool (identity when ``permute`` is False), padded
    with -1.  Cache slots past a sequence's length in its last block are
    filled with NaN (``nan_unused``) so that reading them would show.

    Returns a dict of CPU tensors: q [S,Hq,d] bf16, k_cache / v_cache
    [num_blocks,Hkv,block_size,d] bf16, block_table [S,max_blocks] int32,
    seq_lens [S] int32.
    """
    gen = torch.Generator().manual_seed(int(seed))
    if seq_lens is None:
        seq_lens = torch.randint(len_lo, len_hi + 1, (num_seqs,), generator=gen)
    seq_lens = torch.as_tensor(seq_lens, dtype=torch.int64)
    nblk = [(int(L) + block_size - 1) // block_size for L in seq_lens]
    if max_blocks_per_seq is None:
        max_blocks_per_seq = max(1, (len_hi + block_size - 1) // block_size, max(nblk + [1]))
    num_blocks = sum(nblk) + int(spare_blocks)
    num_blocks = max(num_blocks, 1)
    if permute:
        perm = torch.randperm(num_blocks, generator=gen)
    else:
        perm = torch.arange(num_blocks)
    table = torch.full((num_seqs, max_blocks_per_seq), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(nblk):
        table[b, :n] = perm[off:off + n].to(torch.int32)
        off += n
    q = _randn(gen, (num_seqs, Hq, d)).to(torch.bfloat16)
    k_cache = _randn(gen, (num_blocks, Hkv, block_size, d)).to(torch.bfloat16)
    v_cache = _randn(gen, (num_blocks, Hkv, block_size, d)).to(torch.bfloat16)
    if nan_unused:
        for b, L in enumerate(seq_lens.tolist()):
            if L % block_size:
                phys = int(table[b, L // block_size])
                k_cache[phys, :, L % block_size:] = float("nan")
                v_cache[phys, :, L % block_size:] = float("nan")
    return dict(q=q, k_cache=k_cache, v_cache=v_cache, block_table=table,
                seq_lens=seq_lens.to(torch.int32), block_size=block_size,
                max_blocks_per_seq=max_blocks_per_seq, num_blocks=num_blocks)


PAGED_PREFILL_CONFIGS = {
    # A chunk of 2048 new tokens per sequence on top of a cached prefix, with
    # the Qwen2.5-1.5B-style GQA geometry and block_size = 16.
    "qwen_chunked_prefill": dict(num_seqs=4, Hq=12, Hkv=2, N_new=2048, d=128,
                                 ctx_lo=0, ctx_hi=6144, seed=5),
}


def paged_prefill_inputs(num_seqs, Hq, Hkv, N_new, d, seed, ctx_lo=0, ctx_hi=4096,
                         ctx_lens=None, block_size=BLOCK_SIZE, permute=True,
                         nan_unused=True, max_blocks_per_seq=None, spare_blocks=0):
    """Chunked-prefill inputs over a paged cache.

    Sequence b already holds ctx_lens[b] ~ U{ctx_lo..ctx_hi} cached tokens
    (unless given) and brings N_new new ones.  Its table row gets
    ceil((ctx + N_new) / 16) blocks: a consecutive slice of one random
    permutation of the pool (identity when ``permute`` is False), padded
    with -1.  The prefix keys/values are drawn in logical order and stored
    through the table; every other slot of the pool (the slots the new
    tokens will take, the tail of each last block, ``spare_blocks``) holds
    NaN when ``nan_unused``, else N(0, 1) draws.

    Returns a dict of CPU tensors: q [S,Hq,N_new,d], k_new / v_new
    [S,Hkv,N_new,d], k_cache / v_cache [num_blocks,Hkv,block_size,d] bf16,
    block_table [S,max_blocks] int32, ctx_lens [S] int32, and k_prefix /
    v_prefix (lists of [Hkv, ctx_lens[b], d] bf16: the same prefix values in
    logical order), plus block_size, max_blocks_per_seq, num_blocks.
    """
    gen = torch.Generator().manual_seed(int(seed))
    if ctx_lens is None:
        ctx_lens = torch.randint(ctx_lo, ctx_hi + 1, (num_seqs,), generator=gen)
    ctx_lens = torch.as_tensor(ctx_lens, dtype=torch.int64)
    total = [int(c) + int(N_new) for c in ctx_lens]
    nblk = [(t + block_size - 1) // block_size for t in total]
    if max_blocks_per_seq is None:
        max_blocks_per_seq = max(nblk + [1])
    num_blocks = max(sum(nblk) + int(spare_blocks), 1)
    perm = torch.randperm(num_blocks, generator=gen) if permute else torch.arange(num_blocks)
    table = torch.full((num_seqs, max_blocks_per_seq), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(nblk):
        table[b, :n] = perm[off:off + n].to(torch.int32)
        off += n
    q = _randn(gen, (num_seqs, Hq, N_new, d)).to(torch.bfloat16)
    k_new = _randn(gen, (num_seqs, Hkv, N_new, d)).to(torch.bfloat16)
    v_new = _randn(gen, (num_seqs, Hkv, N_new, d)).to(torch.bfloat16)
    shape = (num_blocks, Hkv, block_size, d)
    if nan_unused:
        k_cache = torch.full(shape, float("nan"), dtype=torch.bfloat16)
        v_cache = torch.full(shape, float("nan"), dtype=torch.bfloat16)
    else:
        k_cache = _randn(gen, shape).to(torch.bfloat16)
        v_cache = _randn(gen, shape).to(torch.bfloat16)
    k_prefix, v_prefix = [], []
    for b, c in enumerate(ctx_lens.tolist()):
        kp = _randn(gen, (Hkv, c, d)).to(torch.bfloat16)
        vp = _randn(gen, (Hkv, c, d)).to(torch.bfloat16)
        pos = torch.arange(c)
        phys = table[b, pos // block_size].long()
        slot = pos % block_size
        k_cache[phys, :, slot] = kp.permute(1, 0, 2)
        v_cache[phys, :, slot] = vp.permute(1, 0, 2)
        k_prefix.append(kp)
        v_prefix.append(vp)
    return dict(q=q, k_new=k_new, v_new=v_new, k_cache=k_cache, v_cache=v_cache,
                block_table=table, ctx_lens=ctx_lens.to(torch.int32), k_prefix=k_prefix,
                v_prefix=v_prefix, block_size=block_size,
                max_blocks_per_seq=max_blocks_per_seq, num_blocks=num_blocks)


FUSION_CONFIGS = {
    # One Qwen2.5-1.5B-sized layer over the 4 x 4096 tokens of the prefill
    # workload: hidden size 1536, MLP intermediate size 8960.
    "qwen_add_rmsnorm": dict(rows=16384, hidden=1536, seed=6),
    "qwen_swiglu": dict(rows=16384, F=8960, seed=7),
    # The same layer's gate/up projection with the activation fused in.
    "qwen_swiglu_projection": dict(rows=16384, hidden=1536, F=8960, seed=9),
}


def add_rmsnorm_inputs(rows, hidden, seed):
    """x, residual [rows, hidden] ~ N(0, 1) and weight [hidden] ~ N(1, 0.1^2), bf16 (CPU)."""
    gen = torch.Generator().manual_seed(int(seed))
    x = _randn(gen, (rows, hidden)).to(torch.bfloat16)
    residual = _randn(gen, (rows, hidden)).to(torch.bfloat16)
    weight = (1.0 + 0.1 * _randn(gen, (hidden,))).to(torch.bfloat16)
    return x, residual, weight


def swiglu_inputs(rows, F, seed):
    """Merged gate/up projection output [rows, 2F] bf16 (CPU): gate columns
    ~ N(0, 2^2) (so SiLU sees both its linear and its vanishing side), up
    columns ~ N(0, 1)."""
    gen = torch.Generator().manual_seed(int(seed))
    g = _randn(gen, (rows, F), 2.0)
    u = _randn(gen, (rows, F))
    return torch.cat([g, u], dim=1).to(torch.bfloat16)


def swiglu_projection_inputs(rows, hidden, F, seed):
    """Activations x [rows, hidden] ~ N(0, 1) and a merged gate/up weight
    [2F, hidden] (gate rows first), bf16 (CPU).  Gate weights have std
    2 / sqrt(hidden), so the projected gate is about N(0, 2^2) and SiLU sees
    both its linear and its vanishing side; up weights 1 / sqrt(hidden)."""
    gen = torch.Generator().manual_seed(int(seed))
    x = _randn(gen, (rows, hidden)).to(torch.bfloat16)
    wg = _randn(gen, (F, hidden), 2.0 / hidden ** 0.5)
    wu = _randn(gen, (F, hidden), 1.0 / hidden ** 0.5)
    return x, torch.cat([wg, wu], dim=0).to(torch.bfloat16)


SSD_CONFIGS = {
    # A Mamba-2-2.7B-sized layer (d_model 2560, expand 2: 80 heads of 64,
    # state 128, one group, chunk 256) over 4 sequences of 4096 tokens.
    "mamba2_ssd": dict(batch=4, L=4096, H=80, P=64, N=128, G=1, chunk=256, seed=8),
}


def ssd_inputs(batch, L, H, P, N, G, seed):
    """Mamba-2 SSD inputs (CPU): x [batch, L, H, P], B, C [batch, L, G, N] bf16
    ~ N(0, 1); dt [batch, L, H] fp32 log-uniform in [1e-3, 1e-1]; A [H] fp32
    = -exp(U[0, ln 16]) (decay rates in [1, 16], negative)."""
    gen = torch.Generator().manual_seed(int(seed))
    x = _randn(gen, (batch, L, H, P)).to(torch.bfloat16)
    B = _randn(gen, (batch, L, G, N)).to(torch.bfloat16)
    C = _randn(gen, (batch, L, G, N)).to(torch.bfloat16)
    lo, hi = math.log(1e-3), math.log(1e-1)
    dt = torch.exp(lo + (hi - lo) * torch.rand((batch, L, H), generator=gen, dtype=torch.float32))
    A = -torch.exp(math.log(16.0) * torch.rand((H,), generator=gen, dtype=torch.float32))
    return dict(x=x, dt=dt, A=A, B=B, C=C)
