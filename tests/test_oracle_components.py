"""Pins for the oracle's building blocks (CPU only).

Each check ties an oracle function to something other than itself: a closed
form, an invariant, central finite differences in float64, or a library
routine that computes the same definition (torch CPU float64, scipy).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import logsumexp

import oracle
from megatron_transformer_layer_fwd_gb300.inputs import round_to_bf16

RNG = np.random.default_rng(1234)


def fd_grad(f, x, idx_list, h=1e-6):
    """Central differences of scalar f at x for the given flat indices."""
    out = []
    flat = x.reshape(-1)
    for i in idx_list:
        old = flat[i]
        flat[i] = old + h
        fp = f()
        flat[i] = old - h
        fm = f()
        flat[i] = old
        out.append((fp - fm) / (2 * h))
    return np.array(out)


# ------------------------------------------------------------------ LayerNorm

def test_ln_closed_form_mean_and_variance():
    x = RNG.standard_normal((16, 64)) * 3.0 + 1.5
    eps = 1e-5
    y, mean, rstd = oracle.ln_fwd(x, eps=eps)
    assert np.abs(y.mean(axis=1)).max() <= 1e-12
    var_x = np.var(x, axis=1)                      # biased variance, library
    np.testing.assert_allclose((y ** 2).mean(axis=1), var_x / (var_x + eps), rtol=1e-12)
    np.testing.assert_allclose(mean, x.mean(axis=1), rtol=1e-13)


def test_ln_matches_torch_layer_norm_with_affine():
    x = RNG.standard_normal((7, 40))
    g = 1 + 0.1 * RNG.standard_normal(40)
    b = 0.1 * RNG.standard_normal(40)
    y, _, _ = oracle.ln_fwd(x, g, b, 1e-5)
    ref = F.layer_norm(torch.tensor(x), (40,), torch.tensor(g), torch.tensor(b), 1e-5).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_ln_affine_invariance_without_eps():
    x = RNG.standard_normal((5, 32))
    y1, _, _ = oracle.ln_fwd(x, eps=0.0)
    y2, _, _ = oracle.ln_fwd(3.7 * x - 2.0, eps=0.0)
    np.testing.assert_allclose(y1, y2, atol=1e-12)


@pytest.mark.parametrize("affine", [False, True])
def test_ln_backward_finite_differences(affine):
    x = RNG.standard_normal((4, 8))
    g = 1 + 0.3 * RNG.standard_normal(8) if affine else None
    b = 0.2 * RNG.standard_normal(8) if affine else None
    dy = RNG.standard_normal((4, 8))
    loss = lambda: float((dy * oracle.ln_fwd(x, g, b, 1e-5)[0]).sum())
    _, mean, rstd = oracle.ln_fwd(x, g, b, 1e-5)
    dx, dg, db = oracle.ln_bwd(dy, x, mean, rstd, g)
    idx = list(range(x.size))
    np.testing.assert_allclose(dx.reshape(-1), fd_grad(loss, x, idx), rtol=1e-6, atol=1e-8)
    if affine:
        np.testing.assert_allclose(dg, fd_grad(loss, g, range(8)), rtol=1e-6, atol=1e-8)
        np.testing.assert_allclose(db, fd_grad(loss, b, range(8)), rtol=1e-6, atol=1e-8)


def test_ln_backward_constant_dy_is_zero():
    x = RNG.standard_normal((6, 16))
    _, mean, rstd = oracle.ln_fwd(x)
    dx, _, _ = oracle.ln_bwd(np.full((6, 16), 0.25), x, mean, rstd)
    assert np.abs(dx).max() <= 1e-12


def test_ln_backward_adjoint_identity():
    """<dy, J dx> = <J^T dy, dx> with J dx from a directional finite difference."""
    x = RNG.standard_normal((3, 12))
    dxv = RNG.standard_normal((3, 12))
    dy = RNG.standard_normal((3, 12))
    h = 1e-6
    jdx = (oracle.ln_fwd(x + h * dxv)[0] - oracle.ln_fwd(x - h * dxv)[0]) / (2 * h)
    _, mean, rstd = oracle.ln_fwd(x)
    jt_dy, _, _ = oracle.ln_bwd(dy, x, mean, rstd)
    assert abs((dy * jdx).sum() - (jt_dy * dxv).sum()) < 1e-7


# ---------------------------------------------------------------- activations

def test_gelu_matches_torch_erf_gelu_and_odd_identity():
    u = np.linspace(-6, 6, 1001)
    np.testing.assert_allclose(oracle.gelu(u), F.gelu(torch.tensor(u)).numpy(), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(oracle.gelu(u) - oracle.gelu(-u), u, atol=1e-13)
    assert oracle.gelu(np.array([0.0]))[0] == 0.0


def test_gelu_and_silu_derivatives_by_finite_differences():
    u = np.linspace(-5, 5, 41)
    h = 1e-6
    np.testing.assert_allclose(oracle.gelu_grad(u), (oracle.gelu(u + h) - oracle.gelu(u - h)) / (2 * h),
                               rtol=1e-7, atol=1e-9)
    np.testing.assert_allclose(oracle.silu_grad(u), (oracle.silu(u + h) - oracle.silu(u - h)) / (2 * h),
                               rtol=1e-7, atol=1e-9)
    np.testing.assert_allclose(oracle.silu(u), F.silu(torch.tensor(u)).numpy(), rtol=1e-12)


def test_swiglu_interleave_equals_deinterleaved_standard_swiglu():
    T, F_, gb = 3, 8, 2
    u = RNG.standard_normal((T, 2 * F_))
    # independent de-interleave by explicit index lists
    gate_cols = [blk * 2 * gb + c for blk in range(F_ // gb) for c in range(gb)]
    up_cols = [blk * 2 * gb + gb + c for blk in range(F_ // gb) for c in range(gb)]
    ref = F.silu(torch.tensor(u[:, gate_cols])).numpy() * u[:, up_cols]
    np.testing.assert_allclose(oracle.swiglu_fwd(u, gb), ref, rtol=1e-13)


def test_swiglu_backward_finite_differences():
    T, F_, gb = 2, 4, 2
    u = RNG.standard_normal((T, 2 * F_))
    da = RNG.standard_normal((T, F_))
    loss = lambda: float((da * oracle.swiglu_fwd(u, gb)).sum())
    du = oracle.swiglu_bwd(da, u, gb)
    np.testing.assert_allclose(du.reshape(-1), fd_grad(loss, u, range(u.size)), rtol=1e-6, atol=1e-9)


def test_round_to_bf16_matches_torch():
    a = np.concatenate([RNG.standard_normal(10000) * 10.0 ** RNG.integers(-30, 30, 10000),
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8])])
    ref = torch.tensor(a, dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(round_to_bf16(a), ref)


# ------------------------------------------------------------------ attention

def _qkv(B, nq, nkv, S, d, scale=1.0):
    return (RNG.standard_normal((B, nq, S, d)) * scale, RNG.standard_normal((B, nkv, S, d)) * scale,
            RNG.standard_normal((B, nkv, S, d)))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq,nkv", [(4, 4), (4, 2), (4, 1)])
def test_attention_matches_torch_sdpa(causal, nq, nkv):
    q, k, v = _qkv(2, nq, nkv, 9, 5)
    o, lse = oracle.attention_fwd(q, k, v, causal)
    ref = F.scaled_dot_product_attention(torch.tensor(q), torch.tensor(k), torch.tensor(v),
                                         is_causal=causal, enable_gqa=True).numpy()
    np.testing.assert_allclose(o, ref, rtol=1e-11, atol=1e-12)
    # lse by scipy's logsumexp of the explicitly masked scores
    rep = nq // nkv
    for h in range(nq):
        s = q[0, h] @ k[0, h // rep].T / math.sqrt(5)
        if causal:
            s[np.triu_indices(9, 1)] = -np.inf
        np.testing.assert_allclose(lse[0, h], logsumexp(s, axis=1), rtol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_attention_probabilities_rows_sum_to_one_and_causal_zero(causal):
    S = 6
    q, k, _ = _qkv(1, 2, 2, S, S)
    v = np.broadcast_to(np.eye(S), (1, 2, S, S)).copy()      # V = I  =>  O = P
    p, _ = oracle.attention_fwd(q, k, v, causal)
    np.testing.assert_allclose(p.sum(axis=-1), 1.0, rtol=1e-13)
    assert (p >= 0).all()
    if causal:
        assert np.abs(p[..., np.triu_indices(S, 1)[0], np.triu_indices(S, 1)[1]]).max() == 0.0
        np.testing.assert_allclose(p[..., 0, 0], 1.0)


def test_attention_zero_queries_give_uniform_and_prefix_means():
    q, k, v = _qkv(1, 2, 1, 7, 4)
    q[:] = 0.0
    o, _ = oracle.attention_fwd(q, k, v, False)
    np.testing.assert_allclose(o[0, 1], np.broadcast_to(v[0, 0].mean(0), (7, 4)), rtol=1e-13)
    oc, _ = oracle.attention_fwd(q, k, v, True)
    prefix = np.cumsum(v[0, 0], axis=0) / np.arange(1, 8)[:, None]
    np.testing.assert_allclose(oc[0, 0], prefix, rtol=1e-12)
    np.testing.assert_allclose(oc[0, :, 0], v[0, 0, 0][None, :].repeat(2, 0), rtol=1e-13)


def test_gqa_equals_mha_with_repeated_kv():
    q, k, v = _qkv(2, 6, 2, 5, 3)
    o, _ = oracle.attention_fwd(q, k, v, True)
    o2, _ = oracle.attention_fwd(q, np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1), True)
    np.testing.assert_allclose(o, o2, rtol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nkv", [2, 1])
def test_attention_backward_finite_differences(causal, nkv):
    q, k, v = _qkv(1, 2, nkv, 4, 4)
    do = RNG.standard_normal(q.shape)
    loss = lambda: float((do * oracle.attention_fwd(q, k, v, causal)[0]).sum())
    dq, dk, dv = oracle.attention_bwd(do, q, k, v, causal)
    for arr, grad in ((q, dq), (k, dk), (v, dv)):
        np.testing.assert_allclose(grad.reshape(-1), fd_grad(loss, arr, range(arr.size)),
                                   rtol=1e-6, atol=1e-8)


def test_attention_backward_matches_torch_autograd():
    q, k, v = _qkv(2, 4, 2, 6, 3)
    do = RNG.standard_normal(q.shape)
    tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    F.scaled_dot_product_attention(tq, tk, tv, is_causal=True, enable_gqa=True).backward(torch.tensor(do))
    dq, dk, dv = oracle.attention_bwd(do, q, k, v, True)
    for a, t in ((dq, tq), (dk, tk), (dv, tv)):
        np.testing.assert_allclose(a, t.grad.numpy(), rtol=1e-10, atol=1e-12)
