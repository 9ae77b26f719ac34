"""fp64 reference of the operator fusions beside attention — TEST INFRASTRUCTURE ONLY.

"Fast attention kernels and operator fusion accelerate AI models", section
"Operator fusion": a transformer layer's residual add followed by RMSNorm,
and the SwiGLU block's SiLU and elementwise product, are separate kernels in
a naive implementation, each writing its intermediate tensor to HBM; fusing
them into one kernel removes those round trips and leaves the mathematical
function unchanged (only rounding order may differ).  These are the plain
definitions of what the fused kernels compute.

Layouts (the page fixes none): rows of a [rows, hidden] activation matrix;
the SwiGLU input is the merged gate/up projection output [rows, 2F] with
the gate in columns 0..F-1 and the up projection in columns F..2F-1; the
merged gate/up weight is [2F, hidden] (rows = output features, gate rows
first), as a linear layer stores it.
"""

import numpy as np


def round_bf16(x):
    """Round-to-nearest, ties-to-even, to bfloat16 (8 significant bits,
    fp32's exponent range), written out from its definition: the significand
    in [0.5, 1) is scaled by 2^8 and rounded half-to-even.  Returns the
    rounded values as fp64.  (Subnormal and overflowing inputs are outside
    what the tests feed it.)"""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)


def add_rmsnorm(x, residual, weight, eps):
    """Residual add followed by RMSNorm, one row at a time.

    The residual stream is stored in bf16, so its new value is the sum
    rounded to bf16 (what an unfused add kernel would store); RMSNorm then
    normalises that stored row:
        r   = bf16(x + residual)
        out = r / sqrt(mean_j(r_j^2) + eps) * weight
    x, residual [rows, hidden]; weight [hidden].  Returns (out, r) in fp64
    (out before its own rounding to the output type).
    """
    x = np.asarray(x, dtype=np.float64)
    residual = np.asarray(residual, dtype=np.float64)
    weight = np.asarray(weight, dtype=np.float64)
    r = round_bf16(x + residual)
    ms = np.mean(r * r, axis=-1, keepdims=True)
    return r / np.sqrt(ms + float(eps)) * weight, r


def swiglu(gate_up):
    """SwiGLU activation of a merged gate/up projection output:
        out = silu(g) * u,  silu(g) = g / (1 + exp(-g)),
    g = gate_up[..., :F], u = gate_up[..., F:].  Returns fp64 [..., F]."""
    gate_up = np.asarray(gate_up, dtype=np.float64)
    F = gate_up.shape[-1] // 2
    g, u = gate_up[..., :F], gate_up[..., F:]
    return g / (1.0 + np.exp(-g)) * u


def swiglu_projection(x, w_gate_up):
    """The SwiGLU block's gate/up projection followed by its activation, the
    steps the page fuses into one kernel ("Operator fusion"):
        g = x W_gate^T,  u = x W_up^T,  out = silu(g) * u,
    x [rows, hidden], w_gate_up [2F, hidden] with W_gate = rows 0..F-1 and
    W_up = rows F..2F-1.  Returns fp64 [rows, F]."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w_gate_up, dtype=np.float64)
    F = w.shape[0] // 2
    g = x @ w[:F].T
    u = x @ w[F:].T
    return g / (1.0 + np.exp(-g)) * u
