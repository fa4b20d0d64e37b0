"""LayerNorm over the hidden dimension, forward and hand-derived backward.

Follows "LLM Lab 06: build a Megatron-style Transformer Block from scratch",
section 2: `F.layer_norm(x, (hidden,))`, i.e. per token, normalise over the
hidden features with the biased variance and eps = 1e-5; "02 - How a whole
Transformer block is split", section 2: LayerNorm is a local per-token op.

Test infrastructure only (see the package docstring).
"""
import numpy as np


def ln_fwd(x, gamma=None, beta=None, eps=1e-5):
    """y = gamma * (x - mean) / sqrt(var + eps) + beta per row of x [T, H].

    var is the biased variance (divide by H). gamma/beta None = no affine.
    Returns (y, mean [T], rstd [T]) with rstd = 1/sqrt(var + eps).
    """
    x = np.asarray(x, dtype=np.float64)
    mean = x.mean(axis=-1)
    var = ((x - mean[:, None]) ** 2).mean(axis=-1)
    rstd = 1.0 / np.sqrt(var + eps)
    xhat = (x - mean[:, None]) * rstd[:, None]
    y = xhat
    if gamma is not None:
        y = y * gamma[None, :]
    if beta is not None:
        y = y + beta[None, :]
    return y, mean, rstd


def ln_bwd(dy, x, mean, rstd, gamma=None):
    """Backward of ln_fwd for one row-normalised input.

    With xhat = (x - mean) * rstd and g = dy * gamma:
        dx = rstd * (g - mean_H(g) - xhat * mean_H(g * xhat))
        dgamma = sum_T dy * xhat,   dbeta = sum_T dy.
    Derived from d xhat_j / d x_i = rstd * (delta_ij - 1/H - xhat_i xhat_j / H).
    Returns (dx, dgamma, dbeta); dgamma/dbeta are None without affine.
    """
    dy = np.asarray(dy, dtype=np.float64)
    xhat = (x - mean[:, None]) * rstd[:, None]
    g = dy * gamma[None, :] if gamma is not None else dy
    dx = rstd[:, None] * (g - g.mean(axis=-1, keepdims=True)
                          - xhat * (g * xhat).mean(axis=-1, keepdims=True))
    if gamma is None:
        return dx, None, None
    return dx, (dy * xhat).sum(axis=0), dy.sum(axis=0)
