"""erf-GELU and interleaved SwiGLU, forward and derivative.

* GELU: "LLM Lab 06: build a Megatron-style Transformer Block from scratch",
  section 2 uses `F.gelu`, whose default is the exact (erf) form
  gelu(u) = u * Phi(u), Phi the standard normal CDF.
* SwiGLU: "02 - How a whole Transformer block is split", section 1: fc1
  emits 2*ffn columns (gate and up); the activation is silu(gate) * up, and
  the gate and up halves of the same segment are kept together by an
  interleaved layout. The pages give no block size; the reading used here:
  fc1 output columns are blocks of `gb` columns alternating gate, up:
  [gate_0 (gb) | up_0 (gb) | gate_1 | up_1 | ...], so activation column
  i*gb + c = silu(gate block i, col c) * (up block i, col c).

Test infrastructure only.
"""
import numpy as np
from scipy.special import erf

_SQRT2 = np.sqrt(2.0)
_INV_SQRT_2PI = 1.0 / np.sqrt(2.0 * np.pi)


def gelu(u):
    return 0.5 * u * (1.0 + erf(u / _SQRT2))


def gelu_grad(u):
    """d/du [u Phi(u)] = Phi(u) + u phi(u)."""
    return 0.5 * (1.0 + erf(u / _SQRT2)) + u * _INV_SQRT_2PI * np.exp(-0.5 * u * u)


def silu(g):
    return g / (1.0 + np.exp(-g))


def silu_grad(g):
    """d/dg [g sigma(g)] = sigma(g) (1 + g (1 - sigma(g)))."""
    s = 1.0 / (1.0 + np.exp(-g))
    return s * (1.0 + g * (1.0 - s))


def glu_split(u, gb):
    """Split interleaved fc1 output u [T, 2F] into (gate [T, F], up [T, F])."""
    T, two_f = u.shape
    assert two_f % (2 * gb) == 0
    v = u.reshape(T, two_f // (2 * gb), 2, gb)
    return v[:, :, 0, :].reshape(T, two_f // 2), v[:, :, 1, :].reshape(T, two_f // 2)


def glu_merge(dgate, dup, gb):
    """Inverse of glu_split: interleave [T, F] gate/up halves back to [T, 2F]."""
    T, F = dgate.shape
    out = np.empty((T, F // gb, 2, gb))
    out[:, :, 0, :] = dgate.reshape(T, F // gb, gb)
    out[:, :, 1, :] = dup.reshape(T, F // gb, gb)
    return out.reshape(T, 2 * F)


def swiglu_fwd(u, gb):
    gate, up = glu_split(u, gb)
    return silu(gate) * up


def swiglu_bwd(da, u, gb):
    """Gradient wrt the interleaved pre-activation u given da = dL/d(silu(g)*up)."""
    gate, up = glu_split(u, gb)
    return glu_merge(da * up * silu_grad(gate), da * silu(gate), gb)
