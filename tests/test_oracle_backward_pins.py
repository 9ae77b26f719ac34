"""Pins of the fp64 oracle's attention backward (``oracle.attention_backward``).

Each pin checks the oracle against something other than its own formula:
central finite differences of the forward definition (brute force), torch
autograd through ``scaled_dot_product_attention`` in fp64 (a library
routine), and closed forms the mathematics fixes.  Plausible mistakes in the
gradient formulas are written out as mutants, and each must fail a pin.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads


def _inputs(B, Hq, Hkv, N, d, seed):
    q, k, v = workloads.prefill_inputs(B, Hq, Hkv, N, d, seed)
    g = torch.Generator().manual_seed(seed + 7)
    do = torch.randn((B, Hq, N, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    return q.double().numpy(), k.double().numpy(), v.double().numpy(), do.double().numpy()


def _loss(q, k, v, do, scale, causal):
    o, _ = oracle.attention(q, k, v, scale, causal)
    return float((o * do).sum())


# ---------------------------------------------------------------- the pins

def pin_finite_differences(bwd, causal):
    """Central differences of L = sum(O * dO) for every input element."""
    q, k, v, do = _inputs(1, 2, 1, 5, 3, seed=11)
    scale = 0.7
    dq, dk, dv = bwd(q, k, v, do, scale, causal)
    h = 1e-6
    worst = 0.0
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = dict(q=q, k=k, v=v)
            args_m = dict(q=q, k=k, v=v)
            args_p[name] = xp
            args_m[name] = xm
            num = (_loss(args_p["q"], args_p["k"], args_p["v"], do, scale, causal) -
                   _loss(args_m["q"], args_m["k"], args_m["v"], do, scale, causal)) / (2 * h)
            worst = max(worst, abs(num - g[idx]))
    return worst


def pin_torch_autograd(bwd, causal):
    """torch autograd of SDPA in fp64 (K/V repeated per query head, their
    gradients summed back over each group)."""
    B, Hq, Hkv, N, d = 1, 4, 2, 33, 16
    q, k, v, do = _inputs(B, Hq, Hkv, N, d, seed=12)
    scale = d ** -0.5
    dq, dk, dv = bwd(q, k, v, do, scale, causal)
    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(k, requires_grad=True)
    tv = torch.tensor(v, requires_grad=True)
    G = Hq // Hkv
    o = torch.nn.functional.scaled_dot_product_attention(
        tq, tk.repeat_interleave(G, dim=1), tv.repeat_interleave(G, dim=1),
        is_causal=causal, scale=scale)
    (o * torch.tensor(do)).sum().backward()
    return max(np.abs(dq - tq.grad.numpy()).max(), np.abs(dk - tk.grad.numpy()).max(),
               np.abs(dv - tv.grad.numpy()).max())


def pin_constant_v(bwd, causal):
    """Equal V rows make O independent of the scores: dQ = dK = 0."""
    q, k, v, do = _inputs(1, 2, 2, 40, 8, seed=13)
    v[:] = v[:, :, :1, :]
    dq, dk, _ = bwd(q, k, v, do, 0.5, causal)
    return max(np.abs(dq).max(), np.abs(dk).max())


def pin_sums(bwd, causal):
    """Every row of P sums to 1, so sum_j dV_j = sum_i dO_i; and adding one
    vector to every key leaves O unchanged, so sum_j dK_j = 0."""
    q, k, v, do = _inputs(1, 3, 3, 50, 8, seed=14)
    _, dk, dv = bwd(q, k, v, do, 0.4, causal)
    return max(np.abs(dv.sum(axis=2) - do.sum(axis=2)).max(), np.abs(dk.sum(axis=2)).max())


def pin_gqa(bwd, causal):
    """A KV head shared by G query heads gets the sum of the gradients it
    would get as G separate (repeated) KV heads."""
    B, Hq, Hkv, N, d = 1, 6, 2, 30, 8
    q, k, v, do = _inputs(B, Hq, Hkv, N, d, seed=15)
    G = Hq // Hkv
    dq, dk, dv = bwd(q, k, v, do, 0.3, causal)
    rq, rk, rv = bwd(q, np.repeat(k, G, axis=1), np.repeat(v, G, axis=1), do, 0.3, causal)
    rk = rk.reshape(B, Hkv, G, N, d).sum(axis=2)
    rv = rv.reshape(B, Hkv, G, N, d).sum(axis=2)
    return max(np.abs(dq - rq).max(), np.abs(dk - rk).max(), np.abs(dv - rv).max())


PINS = [(pin_finite_differences, 1e-6), (pin_torch_autograd, 1e-10), (pin_constant_v, 1e-12),
        (pin_sums, 1e-10), (pin_gqa, 1e-12)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("pin,tol", PINS, ids=lambda x: getattr(x, "__name__", str(x)))
def test_backward_oracle_passes_pin(pin, tol, causal):
    assert pin(oracle.attention_backward, causal) <= tol


# ---------------------------------------------------------------- mutants

def _mutant(kind):
    """The oracle's backward with one plausible mistake."""
    def bwd(q, k, v, do, scale, causal):
        B, Hq, N, d = q.shape
        Hkv = k.shape[1]
        G = Hq // Hkv
        dq = np.zeros_like(q)
        dk = np.zeros_like(k)
        dv = np.zeros_like(v)
        for b in range(B):
            for h in range(Hq):
                g = h // G
                s = scale * (q[b, h] @ k[b, g].T)
                allowed = np.tril(np.ones((N, N), bool)) if (causal and kind != "no_mask") else np.ones((N, N), bool)
                p, _, _ = oracle.softmax_probs(s, allowed)
                dv[b, g] += (p if kind == "p_not_transposed" else p.T) @ do[b, h]
                dp = do[b, h] @ v[b, g].T
                ds = p * dp if kind == "no_rowsum_term" else p * (dp - (p * dp).sum(axis=-1, keepdims=True))
                sc = 1.0 if kind == "no_scale" else scale
                dq[b, h] = sc * (ds @ k[b, g])
                dk[b, g] += sc * (ds.T @ q[b, h])
        return dq, dk, dv
    return bwd


@pytest.mark.parametrize("kind", ["no_rowsum_term", "no_scale", "p_not_transposed", "no_mask"])
def test_backward_mutant_is_caught(kind):
    bad = _mutant(kind)
    caught = any(pin(bad, causal) > tol for pin, tol in PINS for causal in (False, True))
    assert caught, kind


def test_mutant_framework_reproduces_oracle():
    """The mutant template without a mistake is the oracle (so a caught mutant
    is caught for its mistake, not for a difference in the template)."""
    q, k, v, do = _inputs(1, 4, 2, 20, 8, seed=16)
    for causal in (False, True):
        ref = oracle.attention_backward(q, k, v, do, 0.6, causal)
        same = _mutant("none")(q, k, v, do, 0.6, causal)
        for a, b in zip(ref, same):
            assert np.abs(a - b).max() <= 1e-12
