"""Pins of the fp64 oracle's operator fusions (``oracle.add_rmsnorm``,
``oracle.swiglu``, ``oracle.swiglu_projection``, ``oracle.round_bf16``).

Each pin checks the oracle against something other than its own code:
torch's own bf16 conversion and bf16 addition, ``torch.nn.functional.rms_norm``
and ``silu`` in fp64 (library routines), and closed forms (unit RMS of the
normalised row, scale invariance, a constant row, silu(0) = 0 and
silu(g) - silu(-g) = g).  Plausible mistakes are written out as mutants,
and each must fail a pin.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads


def _np(t):
    return t.double().numpy()


# ---------------------------------------------------------------- round_bf16

def test_round_bf16_matches_torch_conversion():
    g = torch.Generator().manual_seed(3)
    x = torch.randn(200000, generator=g, dtype=torch.float32) * torch.exp2(torch.randint(-20, 20, (200000,), generator=g).float())
    assert np.array_equal(oracle.round_bf16(x.double().numpy()), x.to(torch.bfloat16).double().numpy())


def test_round_bf16_ties_to_even():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: the even neighbour is 1;
    # 1 + 3 * 2^-8 lies halfway between 1 + 2^-7 and 1 + 2^-6: the even one is 1 + 2^-6.
    got = oracle.round_bf16([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 3.0])
    assert got.tolist() == [1.0, 1 + 2.0 ** -6, -1.0, 3.0]


# ---------------------------------------------------------------- the pins

def pin_rmsnorm_vs_torch(fn):
    """out = torch rms_norm (fp64) of the stored residual row."""
    x, res, w = workloads.add_rmsnorm_inputs(37, 264, seed=11)
    out, r = fn(_np(x), _np(res), _np(w), 1e-6)
    ref = torch.nn.functional.rms_norm(torch.tensor(r), (264,), torch.tensor(_np(w)), 1e-6)
    return float(np.abs(out - ref.numpy()).max())


def pin_residual_is_bf16_add(fn):
    """The new residual equals torch's bf16 addition of the two inputs."""
    x, res, w = workloads.add_rmsnorm_inputs(64, 512, seed=12)
    _, r = fn(_np(x), _np(res), _np(w), 1e-6)
    return float(np.abs(r - (x + res).double().numpy()).max())


def pin_unit_rms(fn):
    """With weight 1 and eps 0 every output row has mean square 1."""
    x, res, _ = workloads.add_rmsnorm_inputs(20, 300, seed=13)
    out, _ = fn(_np(x), _np(res), np.ones(300), 0.0)
    return float(np.abs((out * out).mean(axis=1) - 1.0).max())


def pin_scale_invariance(fn):
    """With eps 0, scaling both inputs by 4 (exact in bf16) leaves the output unchanged."""
    x, res, w = workloads.add_rmsnorm_inputs(9, 128, seed=14)
    a, _ = fn(_np(x), _np(res), _np(w), 0.0)
    b, _ = fn(4 * _np(x), 4 * _np(res), _np(w), 0.0)
    return float(np.abs(a - b).max())


def pin_constant_row(fn):
    """A row of constant c (x = c, residual = 0) gives out = w * c / sqrt(c^2 + eps)."""
    w = np.linspace(0.5, 1.5, 16)
    c, eps = 0.75, 0.25
    out, _ = fn(np.full((1, 16), c), np.zeros((1, 16)), w, eps)
    return float(np.abs(out[0] - w * c / np.sqrt(c * c + eps)).max())


RMS_PINS = [(pin_rmsnorm_vs_torch, 1e-12), (pin_residual_is_bf16_add, 0.0), (pin_unit_rms, 1e-12),
            (pin_scale_invariance, 1e-12), (pin_constant_row, 1e-15)]


def pin_swiglu_vs_torch(fn):
    gu = workloads.swiglu_inputs(33, 200, seed=15)
    g, u = _np(gu[:, :200]), _np(gu[:, 200:])
    ref = torch.nn.functional.silu(torch.tensor(g)) * torch.tensor(u)
    return float(np.abs(fn(_np(gu)) - ref.numpy()).max())


def pin_swiglu_closed_forms(fn):
    """silu(0) * u = 0; with u = 1, silu(g) - silu(-g) = g."""
    g = np.linspace(-6.0, 6.0, 25)
    zero = fn(np.concatenate([np.zeros((1, 25)), np.ones((1, 25))], axis=1))
    plus = fn(np.concatenate([g[None], np.ones((1, 25))], axis=1))
    minus = fn(np.concatenate([-g[None], np.ones((1, 25))], axis=1))
    return float(max(np.abs(zero).max(), np.abs(plus - minus - g).max()))


SWIGLU_PINS = [(pin_swiglu_vs_torch, 1e-12), (pin_swiglu_closed_forms, 1e-12)]


def pin_projection_vs_torch(fn):
    """torch's fp64 matmuls of the two weight halves and its silu."""
    x, w = workloads.swiglu_projection_inputs(29, 64, 48, seed=16)
    xt, wt = torch.tensor(_np(x)), torch.tensor(_np(w))
    ref = torch.nn.functional.silu(xt @ wt[:48].T) * (xt @ wt[48:].T)
    return float(np.abs(fn(_np(x), _np(w)) - ref.numpy()).max())


def pin_projection_identity_weights(fn):
    """W_gate = 2 I and W_up = I (hidden = F) give silu(2 x) * x elementwise."""
    x = np.linspace(-4.0, 4.0, 40).reshape(5, 8)
    w = np.concatenate([2.0 * np.eye(8), np.eye(8)], axis=0)
    return float(np.abs(fn(x, w) - 2.0 * x / (1.0 + np.exp(-2.0 * x)) * x).max())


def pin_projection_single_feature(fn):
    """One feature with gate weight row a and up weight row b: the gate and
    up inputs are the dot products x.a and x.b, worked by hand."""
    x = np.array([[1.0, 2.0, -1.0]])
    w = np.array([[0.5, 0.0, 1.0],      # g = 0.5 - 1 = -0.5
                  [1.0, 1.0, 1.0]])     # u = 1 + 2 - 1 = 2
    return float(abs(fn(x, w)[0, 0] - (-0.5 / (1.0 + np.exp(0.5)) * 2.0)))


PROJ_PINS = [(pin_projection_vs_torch, 1e-12), (pin_projection_identity_weights, 1e-12),
             (pin_projection_single_feature, 1e-15)]


@pytest.mark.parametrize("pin,tol", RMS_PINS, ids=lambda x: getattr(x, "__name__", str(x)))
def test_add_rmsnorm_oracle_passes_pin(pin, tol):
    assert pin(oracle.add_rmsnorm) <= tol


@pytest.mark.parametrize("pin,tol", SWIGLU_PINS, ids=lambda x: getattr(x, "__name__", str(x)))
def test_swiglu_oracle_passes_pin(pin, tol):
    assert pin(oracle.swiglu) <= tol


@pytest.mark.parametrize("pin,tol", PROJ_PINS, ids=lambda x: getattr(x, "__name__", str(x)))
def test_swiglu_projection_oracle_passes_pin(pin, tol):
    assert pin(oracle.swiglu_projection) <= tol


# ---------------------------------------------------------------- mutants

def _rms_mutant(kind):
    def fn(x, residual, weight, eps):
        s = np.asarray(x, np.float64) + np.asarray(residual, np.float64)
        r = s if kind == "unrounded_residual" else oracle.round_bf16(s)
        ms = (r * r).sum(-1, keepdims=True) if kind == "sum_not_mean" else (r * r).mean(-1, keepdims=True)
        den = np.sqrt(ms) + eps if kind == "eps_outside_sqrt" else np.sqrt(ms + eps)
        w = 1.0 if kind == "no_weight" else np.asarray(weight, np.float64)
        return r / den * w, r
    return fn


def _swiglu_mutant(kind):
    def fn(gate_up):
        gate_up = np.asarray(gate_up, np.float64)
        F = gate_up.shape[-1] // 2
        g, u = gate_up[..., :F], gate_up[..., F:]
        if kind == "gate_up_swapped":
            g, u = u, g
        act = 1.0 / (1.0 + np.exp(-g)) if kind == "sigmoid_not_silu" else g / (1.0 + np.exp(-g))
        return act * u
    return fn


def _projection_mutant(kind):
    def fn(x, w_gate_up):
        x = np.asarray(x, np.float64)
        w = np.asarray(w_gate_up, np.float64)
        F = w.shape[0] // 2
        wg, wu = (w[0::2], w[1::2]) if kind == "interleaved_halves" else (w[:F], w[F:])
        if kind == "gate_up_swapped":
            wg, wu = wu, wg
        g, u = x @ wg.T, x @ wu.T
        if kind == "no_activation":
            return g * u
        if kind == "exp_sign":
            return g / (1.0 + np.exp(g)) * u
        return g / (1.0 + np.exp(-g)) * u
    return fn


@pytest.mark.parametrize("kind", ["unrounded_residual", "sum_not_mean", "eps_outside_sqrt", "no_weight"])
def test_add_rmsnorm_mutant_is_caught(kind):
    assert any(not (pin(_rms_mutant(kind)) <= tol) for pin, tol in RMS_PINS), kind


@pytest.mark.parametrize("kind", ["gate_up_swapped", "sigmoid_not_silu"])
def test_swiglu_mutant_is_caught(kind):
    assert any(not (pin(_swiglu_mutant(kind)) <= tol) for pin, tol in SWIGLU_PINS), kind


@pytest.mark.parametrize("kind", ["gate_up_swapped", "interleaved_halves", "no_activation", "exp_sign"])
def test_swiglu_projection_mutant_is_caught(kind):
    assert any(not (pin(_projection_mutant(kind)) <= tol) for pin, tol in PROJ_PINS), kind


def test_mutant_templates_reproduce_oracle():
    for pin, tol in RMS_PINS:
        assert pin(_rms_mutant("none")) <= tol, pin.__name__
    for pin, tol in SWIGLU_PINS:
        assert pin(_swiglu_mutant("none")) <= tol, pin.__name__
    for pin, tol in PROJ_PINS:
        assert pin(_projection_mutant("none")) <= tol, pin.__name__
