"""Pins for the oracle's cross-entropy (CPU only)."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

RNG = np.random.default_rng(99)


def _case(T=6, H=8, V=40):
    return RNG.standard_normal((T, H)), RNG.standard_normal((V, H)) * 0.7, RNG.integers(0, V, T)


@pytest.mark.parametrize("chunk", [16, 40, 7, 64])
def test_chunked_equals_full_vocab_logsumexp_minus_target(chunk):
    hid, emb, tg = _case()
    loss_f, lse_f, mean_f = oracle.ce_full(hid, emb, tg)
    loss_c, lse_c, mean_c, _ = oracle.ce_chunked(hid, emb, tg, chunk)
    np.testing.assert_allclose(loss_c, loss_f, atol=1e-12)
    np.testing.assert_allclose(lse_c, lse_f, atol=1e-12)
    assert abs(mean_c - mean_f) <= 1e-12


def test_full_matches_torch_cross_entropy():
    hid, emb, tg = _case(T=9, V=33)
    loss, _, mean = oracle.ce_full(hid, emb, tg)
    ref = F.cross_entropy(torch.tensor(hid @ emb.T), torch.tensor(tg), reduction="none").numpy()
    np.testing.assert_allclose(loss, ref, rtol=1e-12)
    assert abs(mean - ref.mean()) < 1e-12


def test_zero_embedding_gives_log_vocab():
    V = 128256
    hid = RNG.standard_normal((3, 4))
    emb = np.zeros((V, 4))
    tg = np.array([0, 5, V - 1])
    loss, _, mean = oracle.ce_full(hid, emb, tg, row_block=1)
    np.testing.assert_allclose(loss, math.log(V), rtol=1e-14)
    np.testing.assert_allclose(mean, 11.761783545564427, rtol=1e-14)


def test_dominant_target_logit_closed_form():
    """E = alpha*I, hidden = onehot(target): l_target = alpha, others 0, so
    loss = log(1 + (V-1) exp(-alpha)) -> 0 as alpha grows."""
    V = 12
    tg = np.array([3, 0, 11])
    for alpha in (1.0, 10.0, 40.0):
        emb = alpha * np.eye(V)
        hid = np.eye(V)[tg]
        loss, _, _, _ = oracle.ce_chunked(hid, emb, tg, 5)
        # exact up to rounding of LSE ~ alpha (a few ULPs of alpha in float64)
        np.testing.assert_allclose(loss, math.log1p((V - 1) * math.exp(-alpha)), rtol=1e-12,
                                   atol=4 * alpha * np.finfo(float).eps)
    assert loss.max() < 1e-15


def test_grad_rows_sum_to_zero():
    """sum_v (softmax - onehot) = 0 per token: with all embedding rows equal
    the hidden gradient vanishes and the column sums of demb vanish."""
    hid, emb, tg = _case()
    _, lse, _ = oracle.ce_full(hid, emb, tg)
    _, d_emb = oracle.ce_grads(hid, emb, tg, lse, 1.0)
    assert np.abs(d_emb.sum(axis=0)).max() < 1e-12
    emb_eq = np.broadcast_to(emb[:1], emb.shape).copy()
    _, lse_eq, _ = oracle.ce_full(hid, emb_eq, tg)
    d_hid, _ = oracle.ce_grads(hid, emb_eq, tg, lse_eq, 1.0)
    assert np.abs(d_hid).max() < 1e-12


def test_grads_finite_differences_ragged_chunks():
    T, H, V, C = 4, 8, 40, 16
    hid, emb, tg = _case(T, H, V)
    scale = 1.0 / T
    _, lse, _, _ = oracle.ce_chunked(hid, emb, tg, C)
    d_hid, d_emb = oracle.ce_grads(hid, emb, tg, lse, scale)
    loss = lambda: float(oracle.ce_chunked(hid, emb, tg, C)[2])
    h = 1e-6
    for arr, grad in ((hid, d_hid), (emb, d_emb)):
        flat = arr.reshape(-1)
        for i in RNG.choice(arr.size, 30, replace=False):
            old = flat[i]
            flat[i] = old + h
            fp = loss()
            flat[i] = old - h
            fm = loss()
            flat[i] = old
            assert abs(grad.reshape(-1)[i] - (fp - fm) / (2 * h)) < 1e-8


def test_grads_match_torch_autograd():
    hid, emb, tg = _case(T=5, V=21)
    th = torch.tensor(hid, requires_grad=True)
    te = torch.tensor(emb, requires_grad=True)
    F.cross_entropy(th @ te.T, torch.tensor(tg)).backward()
    _, lse, _ = oracle.ce_full(hid, emb, tg)
    d_hid, d_emb = oracle.ce_grads(hid, emb, tg, lse, 1.0 / 5)
    np.testing.assert_allclose(d_hid, th.grad.numpy(), rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(d_emb, te.grad.numpy(), rtol=1e-11, atol=1e-14)


def test_rows_match_full():
    hid, emb, tg = _case(T=8)
    loss, lse, _ = oracle.ce_full(hid, emb, tg)
    d_hid, _ = oracle.ce_grads(hid, emb, tg, lse, 0.125)
    rows = np.array([1, 6])
    l_r, lse_r, dh_r = oracle.ce_rows(hid[rows], emb, tg[rows], 0.125)
    np.testing.assert_allclose(l_r, loss[rows], rtol=1e-13)
    np.testing.assert_allclose(lse_r, lse[rows], rtol=1e-13)
    np.testing.assert_allclose(dh_r, d_hid[rows], rtol=1e-12)


def test_emb_rows_match_full():
    """Selected rows of demb, including ids that are some token's target (the
    one-hot term) and ids that are none, equal those rows of ce_grads' demb,
    which torch autograd pins; dropping the one-hot term is caught."""
    hid, emb, tg = _case(T=8)
    _, lse, _ = oracle.ce_full(hid, emb, tg)
    _, d_emb = oracle.ce_grads(hid, emb, tg, lse, 0.125)
    ids = np.unique(np.concatenate([tg[:3], [0, emb.shape[0] - 1, 7]]))
    rows = oracle.ce_emb_rows(hid, emb, tg, lse, 0.125, ids)
    np.testing.assert_allclose(rows, d_emb[ids], rtol=1e-12, atol=1e-15)
    l = hid @ emb[ids].T
    no_onehot = (np.exp(l - lse[:, None]) * 0.125).T @ hid
    assert np.abs(no_onehot - d_emb[ids]).max() > 1e-3


def test_chunk_partials_planted_mistake_is_caught():
    """Combining chunk sums without rescaling to the global max is wrong."""
    hid, emb, tg = _case()
    loss_f, _, _ = oracle.ce_full(hid, emb, tg)
    _, _, _, (m, s, t) = oracle.ce_chunked(hid, emb, tg, 16)
    wrong = m.max(axis=0) + np.log(s.sum(axis=0)) - t.sum(axis=0)
    assert np.abs(wrong - loss_f).max() > 1e-3
