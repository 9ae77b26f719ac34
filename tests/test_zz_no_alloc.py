"""attn_decode_paged_noalloc: the decode for callers that cannot allocate.

Some callers of this library may not allocate device memory when they run
the decode (a plugin inside a host framework that owns all device memory,
or a serving loop that must not call cudaMalloc because it can synchronize
the device).  attn_decode_paged_noalloc serves them from a fixed device
array built into the library.  This file checks, through the C-ABI, that two
calls in a row give the same results as the workspace entry point, and that
sizes beyond the array are refused.  It is named to run after every other
test file and also passes when run alone.
"""

import pytest
import torch

import exact_attention_47_gb300 as attn
import workloads
from parity import assert_attn_close, to64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _inputs(seq_lens, seed):
    inp = workloads.decode_inputs(len(seq_lens), 12, 2, 128, seed=seed, seq_lens=seq_lens,
                                  len_hi=4096)
    return {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def _both(d, scale):
    args = (d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"])
    o_ref, lse_ref = attn.attn_decode_paged(*args, scale=scale)
    o_na, lse_na = attn.attn_decode_paged_noalloc(*args, scale=scale)
    torch.cuda.synchronize()
    return o_na, lse_na, o_ref, lse_ref


def test_noalloc_matches_workspace_entry_point_twice():
    # Two calls in a row with different length mixes: the second call reuses
    # the array the first one left behind.
    first = _inputs([1, 700, 0, 17, 4096, 256, 1999, 33, 1024, 3000, 15, 16], seed=71)
    second = _inputs([4096, 5, 2048, 129, 0, 3500], seed=72)
    for d in (first, second):
        o_na, lse_na, o_ref, lse_ref = _both(d, 0.0883883)
        assert attn.device_status() == 0
        assert_attn_close(o_na, lse_na, to64(o_ref), to64(lse_ref), what="noalloc vs workspace")


def test_noalloc_refuses_sizes_beyond_its_array():
    # 64 sequences x 12 heads with up to 1024 blocks each need far more than
    # the 8 MiB array: refused before anything is launched.
    q = torch.zeros(64, 12, 128, dtype=torch.bfloat16, device=DEV)
    kc = torch.zeros(4, 2, 16, 128, dtype=torch.bfloat16, device=DEV)
    table = torch.zeros(64, 1024, dtype=torch.int32, device=DEV)
    lens = torch.ones(64, dtype=torch.int32, device=DEV)
    with pytest.raises(attn.AttnError, match="WORKSPACE"):
        attn.attn_decode_paged_noalloc(q, kc, kc, table, lens)
