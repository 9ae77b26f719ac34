"""GPU parity of ssd_chunked_fwd (through the C-ABI) against the fp64 oracle.

Tolerance (the pages state none).  The kernels round x * 2^(g_last - g_j),
the decay-weighted C B^T entries and each chunk's initial state to bf16
before their matrix products (for the second half of a 256-token chunk also
x * 2^(g_m - g_j) and the state times 2^(g_m), m = 127), accumulate in fp32
and round y to bf16: the same kind of rounding steps as the attention
forward's P, so its bounds are carried over relative to the output's scale:
max |y - ref| <= 2e-2 * max |ref|, mean |y - ref| <= 2e-3 * max |ref|; the
same for the final state.
"""

import numpy as np
import pytest
import torch

import exact_attention_47_gb300 as attn
import oracle
import workloads
from parity import assert_rel_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _close(got, ref, what):
    assert_rel_close(got, ref, what)


def _run(d, chunk, h0=None):
    dev = {k: v.to(DEV) for k, v in d.items()}
    y, hf = attn.ssd_chunked_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], chunk=chunk,
                                 h0=None if h0 is None else torch.as_tensor(h0, dtype=torch.float32).to(DEV))
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    return y, hf


CASES = [  # batch, L, H, G, N, chunk, with h0
    (1, 64, 2, 1, 64, 64, False), (2, 200, 4, 2, 128, 64, False), (1, 300, 3, 1, 128, 128, True),
    (1, 512, 2, 1, 64, 256, True), (1, 1, 2, 1, 64, 64, False), (2, 777, 2, 1, 128, 256, True),
    # more than 16 heads per group (two output blocks, the second partial),
    # an odd number of heads per group, several groups
    (1, 300, 20, 1, 128, 256, False), (1, 129, 5, 1, 64, 128, False), (2, 130, 8, 2, 64, 128, True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b%dL%dH%dG%dN%dQ%d%s" % (c[:6] + ("h0" if c[6] else "",)))
def test_ssd_matches_oracle(case):
    batch, L, H, G, N, chunk, with_h0 = case
    d = workloads.ssd_inputs(batch, L, H, 64, N, G, seed=900 + L + N)
    h0 = np.random.default_rng(L).standard_normal((batch, H, 64, N)) if with_h0 else None
    y, hf = _run(d, chunk, h0)
    ry, rh = oracle.ssd_recurrence(*(d[k].double().numpy() for k in ("x", "dt", "A", "B", "C")),
                                   None if h0 is None else np.asarray(h0, np.float32).astype(np.float64))
    _close(y, ry, "y %s" % (case,))
    _close(hf, rh, "h_final %s" % (case,))


def test_ssd_full_workload_sampled_heads():
    c = workloads.SSD_CONFIGS["mamba2_ssd"]
    d = workloads.ssd_inputs(c["batch"], c["L"], c["H"], c["P"], c["N"], c["G"], c["seed"])
    y, hf = _run(d, c["chunk"])
    for b, h in ((0, 0), (1, 17), (3, 79)):
        sel = {k: d[k].double().numpy() for k in ("x", "dt", "A", "B", "C")}
        ry, rh = oracle.ssd_chunked(sel["x"][b:b + 1, :, h:h + 1], sel["dt"][b:b + 1, :, h:h + 1],
                                    sel["A"][h:h + 1], sel["B"][b:b + 1], sel["C"][b:b + 1], c["chunk"])
        _close(y[b:b + 1, :, h:h + 1], ry, "y b%d h%d" % (b, h))
        _close(hf[b:b + 1, h:h + 1], rh, "h_final b%d h%d" % (b, h))


def test_ssd_rejects_unsupported_shapes():
    d = workloads.ssd_inputs(1, 64, 2, 64, 64, 1, seed=1)
    dev = {k: v.to(DEV) for k, v in d.items()}
    with pytest.raises(attn.AttnError) as e:
        attn.ssd_chunked_fwd(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], chunk=100)
    assert e.value.status == 2
