"""SwiGLU backward, float64 (the operand it feeds to the weight gradient).

Test infrastructure only (see the package docstring).

The weight-gradient pages say the utility kernels around the FP8 weight
gradient include a cast fused with SwiGLU ("Is DeepGEMM directly applicable
to backward in training?", LyricZhao, 26 Feb 2025).  The pages give no
formula; this is the standard SwiGLU of a MoE expert's up/gate projection:

    h = [g | u]              forward pre-activations, [T, 2I] (gate half first)
    a = silu(g) * u          silu(g) = g * sigma(g),  sigma(g) = 1 / (1 + e^-g)

and its backward for the upstream gradient da = dL/da [T, I]:

    du = da * silu(g)
    dg = da * u * silu'(g),  silu'(g) = sigma(g) * (1 + g * (1 - sigma(g)))

``dh = [dg | du]`` is the A operand of the up/gate weight gradient
(dW = dh^T x); ``a`` recomputed is the B operand of the down-projection's
(dW_down = dy^T a).  Each is then cast by columns (``quant_colblock``).
"""
import numpy as np


def sigmoid(g):
    g = np.asarray(g, dtype=np.float64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-g))


def swiglu_backward(h, da):
    """Returns ``(dh [T, 2I], a [T, I])`` in float64 from ``h [T, 2I]`` and
    ``da [T, I]`` (any float dtype, converted exactly)."""
    h = np.asarray(h, dtype=np.float64)
    da = np.asarray(da, dtype=np.float64)
    T, I2 = h.shape
    if I2 % 2 or da.shape != (T, I2 // 2):
        raise ValueError("h must be [T, 2I] and da [T, I]")
    I = I2 // 2
    g, u = h[:, :I], h[:, I:]
    s = sigmoid(g)
    silu = g * s
    dsilu = s * (1.0 + g * (1.0 - s))
    dh = np.concatenate([da * u * dsilu, da * silu], axis=1)
    return dh, silu * u


def swiglu_backward_cast(h, da, gran_k: int = 128, with_a: bool = True):
    """Column-block casts of ``dh`` (and of ``a`` if ``with_a``): the float64
    values, then ``quant_colblock``.  Returns ``(dh, a, (q_dh, sf_dh),
    (q_a, sf_a) or None)``."""
    from .quant import quant_colblock
    dh, a = swiglu_backward(h, da)
    return dh, a, quant_colblock(dh, gran_k), (quant_colblock(a, gran_k) if with_a else None)
