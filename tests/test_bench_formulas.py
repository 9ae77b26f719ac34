"""The work counts ``bench.py`` divides by, checked against brute force.

Every rate in the bench line is (work per call) / (CUDA-event time); these
tests count the work independently on small cases: allowed (query, key)
pairs by enumerating the mask, and bytes by listing every tensor a call
reads or writes.  CPU only.
"""

import numpy as np

import bench
import workloads


def test_fwd_flops_is_four_d_per_half_square():
    # The causal convention is N^2 / 2 pairs per (batch, head): 4 d flops per pair.
    c = dict(B=2, Hq=3, N=10, d=8)
    assert bench.fwd_flops(c) == 4 * 8 * 2 * 3 * (10 * 10 / 2)


def test_paged_prefill_flops_counts_allowed_pairs():
    Hq, N, d = 3, 7, 16
    ctx = [0, 5, 16, 33]
    pairs = 0
    for P in ctx:
        keys = np.arange(P + N)
        for i in range(N):
            pairs += int((keys <= P + i).sum())          # the chunk's causal mask at offset P
    assert bench.paged_prefill_flops(ctx, Hq, N, d) == 4.0 * d * Hq * pairs


def test_decode_bytes_lists_every_tensor():
    inp = workloads.decode_inputs(5, 4, 2, 64, seed=3, len_lo=1, len_hi=100)
    S, Hq, Hkv, d = 5, 4, 2, 64
    L = inp["seq_lens"].numpy().astype(np.int64)
    expect = 0
    expect += int(L.sum()) * Hkv * d * 2 * 2            # every addressed K and V row, bf16
    expect += S * Hq * d * 2                            # q
    expect += S * Hq * d * 2                            # o
    expect += S * Hq * 4                                # lse
    expect += inp["block_table"].numel() * 4 + S * 4    # table, lengths
    assert bench.decode_bytes(inp, Hq, Hkv, d) == expect


def test_fusion_byte_counts():
    rows, hidden, F = 37, 264, 200
    bf16 = 2
    x = residual_in = residual_out = out = rows * hidden * bf16
    weight = hidden * bf16
    gate_up, act = rows * 2 * F * bf16, rows * F * bf16
    got = bench.fusion_bytes(rows, hidden, F)
    assert got["add_rmsnorm"] == x + residual_in + residual_out + out + weight
    assert got["swiglu"] == gate_up + act


def test_ssd_flops_counts_the_matrix_form():
    # Per chunk of n positions: the masked C B^T once per B/C group (n^2/2
    # pairs of N multiply-adds), and per head its product with X over the
    # same pairs (P multiply-adds each), the state update and the carried
    # state's output (P N multiply-adds per position each).
    batch, L, H, G, P, N, chunk = 2, 300, 6, 2, 8, 16, 128
    total = 0
    for c0 in range(0, L, chunk):
        n = min(chunk, L - c0)
        pairs = n * n / 2
        total += G * pairs * 2 * N                       # C B^T per group
        total += H * pairs * 2 * P                       # (.) X per head
        total += H * (n * 2 * P * N + n * 2 * P * N)     # (x w)^T B, C S^T per head
    assert bench.ssd_flops(batch, L, H, G, P, N, chunk) == batch * total


def test_ssd_bytes_lists_every_tensor():
    batch, L, H, G, P, N = 2, 300, 4, 2, 64, 128
    d = workloads.ssd_inputs(batch, L, H, P, N, G, seed=1)
    reads = sum(t.numel() * t.element_size() for t in d.values())      # x, dt, A, B, C
    writes = batch * L * H * P * 2 + batch * H * P * N * 4             # y (bf16), final state (fp32)
    assert bench.ssd_bytes(batch, L, H, G, P, N) == reads + writes


def test_swiglu_projection_flops_is_the_gemm():
    # [rows, hidden] x [hidden, 2F]: one multiply-add per (row, output column, k).
    rows, hidden, F = 5, 64, 128
    assert bench.swiglu_projection_flops(rows, hidden, F) == 2 * rows * (2 * F) * hidden
