"""attn_decode_paged_noalloc: the decode for callers that cannot allocate.

Some callers of this library may not allocate device memory when they run
the decode (a plugin inside a host framework that owns all device memory,
or a serving loop that must not call cudaMalloc because it can synchronize
the device).  attn_decode_paged_noalloc serves them from a fixed device
array built into the library.  This file checks, through the C-ABI:
  - two calls in a row give bit for bit the results of the workspace entry
    point (the same kernels over the same split; only where the partial
    results are kept differs), and the first also matches the fp64 oracle;
  - with the outputs passed in, a call allocates no device memory (neither
    torch's counters nor the device's free memory move);
  - sizes beyond the array are refused before anything is launched.
It is named to run after every other test file and also passes when run
alone.
"""

import gc

import pytest
import torch

import exact_attention_47_gb300 as attn
import oracle
import workloads
from parity import assert_attn_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
SCALE = 0.0883883


def _inputs(seq_lens, seed):
    inp = workloads.decode_inputs(len(seq_lens), 12, 2, 128, seed=seed, seq_lens=seq_lens,
                                  len_hi=4096)
    return inp, {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def _args(d):
    return d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"]


def test_noalloc_matches_workspace_entry_point_twice():
    # Two calls in a row with different length mixes: the second call reuses
    # the array the first one left behind.
    first = _inputs([1, 700, 0, 17, 4096, 256, 1999, 33, 1024, 3000, 15, 16], seed=71)
    second = _inputs([4096, 5, 2048, 129, 0, 3500], seed=72)
    for i, (host, d) in enumerate((first, second)):
        o_ref, lse_ref = attn.attn_decode_paged(*_args(d), scale=SCALE)
        o_na, lse_na = attn.attn_decode_paged_noalloc(*_args(d), scale=SCALE)
        torch.cuda.synchronize()
        assert attn.device_status() == 0
        assert torch.equal(o_na, o_ref), "call %d: o differs from the workspace entry point" % i
        assert torch.equal(lse_na, lse_ref), "call %d: lse differs from the workspace entry point" % i
        if i == 0:
            ro, rl = oracle.decode_paged(host["q"].double().numpy(), host["k_cache"].double().numpy(),
                                         host["v_cache"].double().numpy(), host["block_table"].numpy(),
                                         host["seq_lens"].numpy(), SCALE)
            assert_attn_close(o_na, lse_na, ro, rl, what="noalloc vs oracle")


def test_noalloc_call_allocates_no_device_memory():
    _, d = _inputs([3000, 1, 4096, 64, 777, 2048, 0, 1500], seed=73)
    o = torch.empty_like(d["q"])
    lse = torch.empty(d["q"].shape[:2], dtype=torch.float32, device=DEV)
    attn.attn_decode_paged_noalloc(*_args(d), scale=SCALE, o=o, lse=lse)   # first call: set-up
    torch.cuda.synchronize()
    o_first = o.clone()
    # No garbage collection during the measured call: objects of earlier
    # tests freed in the middle of it would move the counters.
    gc.collect()
    gc.disable()
    try:
        before = torch.cuda.memory_stats()
        free = torch.cuda.mem_get_info()[0]
        attn.attn_decode_paged_noalloc(*_args(d), scale=SCALE, o=o, lse=lse)
        torch.cuda.synchronize()
        after = torch.cuda.memory_stats()
        free_after = torch.cuda.mem_get_info()[0]
    finally:
        gc.enable()
    # torch's cumulative counts of allocation requests and of segments it
    # took from the device, and the device's own free memory.
    for key in ("allocation.all.allocated", "segment.all.allocated", "allocated_bytes.all.allocated"):
        assert after[key] == before[key], key
    assert free_after == free
    assert attn.device_status() == 0
    assert torch.equal(o, o_first)


def test_noalloc_refuses_sizes_beyond_its_array():
    # 64 sequences x 12 heads with up to 1024 blocks each need far more than
    # the 8 MiB array: refused before anything is launched.
    q = torch.zeros(64, 12, 128, dtype=torch.bfloat16, device=DEV)
    kc = torch.zeros(4, 2, 16, 128, dtype=torch.bfloat16, device=DEV)
    table = torch.zeros(64, 1024, dtype=torch.int32, device=DEV)
    lens = torch.ones(64, dtype=torch.int32, device=DEV)
    with pytest.raises(attn.AttnError, match="WORKSPACE"):
        attn.attn_decode_paged_noalloc(q, kc, kc, table, lens)
