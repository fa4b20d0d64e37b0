"""Pins for the oracle's whole-layer forward/backward and the k-way split
invariant (CPU only)."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import shard
from megatron_transformer_layer_fwd_gb300.inputs import LayerShape, layer_inputs, WORKLOADS

TINY = {
    "pre_gelu": LayerShape(2, 5, 8, 2, 2, 4, 12, dtype="f32"),
    "pre_gelu_causal_gqa": LayerShape(1, 6, 8, 4, 2, 3, 10, dtype="f32", causal=True),
    "post_gelu": LayerShape(2, 4, 8, 2, 2, 4, 12, dtype="f32", norm_pos="post"),
    "pre_swiglu_causal_gqa": LayerShape(2, 4, 8, 4, 1, 2, 8, dtype="f32", act="swiglu",
                                        causal=True, glu_block=2),
    "post_swiglu_noaffine": LayerShape(1, 5, 6, 2, 2, 3, 4, dtype="f32", norm_pos="post",
                                       act="swiglu", glu_block=2, ln_affine=False, has_bias=False),
}

KEYS = ("w_qkv", "b_qkv", "w_o", "b_o", "w_1", "b_1", "w_2", "b_2", "ln1_g", "ln1_b", "ln2_g", "ln2_b")


def _weights(inp):
    return {k: inp[k] for k in KEYS}


def _inputs(shape, seed=0):
    inp = layer_inputs(shape, seed, random_affine=True, random_dy=True)
    # scale weights up so the tiny layer is far from linear (a stricter FD check)
    for k in ("w_qkv", "w_o", "w_1", "w_2"):
        inp[k] = inp[k] * 25.0
    return inp


@pytest.mark.parametrize("name", list(TINY))
def test_block_backward_finite_differences(name):
    shape = TINY[name]
    inp = _inputs(shape)
    w = _weights(inp)
    x, dy = inp["x"], inp["dy"]
    y, cache = oracle.block_fwd(shape, w, x)
    dx, grads = oracle.block_bwd(shape, w, cache, dy)
    loss = lambda: float((dy * oracle.block_fwd(shape, w, x)[0]).sum())
    h = 1e-6
    rng = np.random.default_rng(7)

    def check(arr, grad):
        n = arr.size
        idx = rng.choice(n, size=min(n, 24), replace=False)
        flat = arr.reshape(-1)
        for i in idx:
            old = flat[i]
            flat[i] = old + h
            fp = loss()
            flat[i] = old - h
            fm = loss()
            flat[i] = old
            fd = (fp - fm) / (2 * h)
            assert abs(grad.reshape(-1)[i] - fd) <= 1e-6 * max(1.0, abs(fd)), (i, grad.reshape(-1)[i], fd)

    check(x, dx)
    for k in KEYS:
        if w[k] is None:
            assert grads[k] is None
        else:
            check(w[k], grads[k])


def _torch_block(shape, w, x):
    """The same layer written with torch library ops, for autograd."""
    B, S, H = shape.batch, shape.seq, shape.hidden
    nq, nkv, d = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    eps = shape.ln_eps
    ln = lambda t, g, b: F.layer_norm(t, (H,), g, b, eps)
    a_in = ln(x, w["ln1_g"], w["ln1_b"]) if shape.norm_pos == "pre" else x
    qkv = F.linear(a_in, w["w_qkv"], w["b_qkv"])
    q, k, v = torch.split(qkv, [nq * d, nkv * d, nkv * d], dim=1)
    q = q.reshape(B, S, nq, d).transpose(1, 2)
    k = k.reshape(B, S, nkv, d).transpose(1, 2)
    v = v.reshape(B, S, nkv, d).transpose(1, 2)
    o = F.scaled_dot_product_attention(q, k, v, is_causal=shape.causal, enable_gqa=True)
    O = o.transpose(1, 2).reshape(B * S, nq * d)
    r1 = x + F.linear(O, w["w_o"], w["b_o"])
    if shape.norm_pos == "pre":
        h, f_in = r1, ln(r1, w["ln2_g"], w["ln2_b"])
    else:
        h = ln(r1, w["ln1_g"], w["ln1_b"])
        f_in = h
    u = F.linear(f_in, w["w_1"], w["b_1"])
    if shape.act == "swiglu":
        gb = shape.glu_block
        uu = u.reshape(B * S, -1, 2, gb)
        a = (F.silu(uu[:, :, 0, :]) * uu[:, :, 1, :]).reshape(B * S, -1)
    else:
        a = F.gelu(u)
    r2 = h + F.linear(a, w["w_2"], w["b_2"])
    return r2 if shape.norm_pos == "pre" else ln(r2, w["ln2_g"], w["ln2_b"])


@pytest.mark.parametrize("name", list(TINY))
def test_block_matches_torch_fp64_autograd(name):
    shape = TINY[name]
    inp = _inputs(shape, seed=3)
    w = _weights(inp)
    tw = {k: (torch.tensor(v, requires_grad=True) if v is not None else None) for k, v in w.items()}
    tx = torch.tensor(inp["x"], requires_grad=True)
    ty = _torch_block(shape, tw, tx)
    ty.backward(torch.tensor(inp["dy"]))
    y, cache = oracle.block_fwd(shape, w, inp["x"])
    np.testing.assert_allclose(y, ty.detach().numpy(), rtol=1e-10, atol=1e-11)
    dx, g = oracle.block_bwd(shape, w, cache, inp["dy"])
    np.testing.assert_allclose(dx, tx.grad.numpy(), rtol=1e-9, atol=1e-10)
    for k in KEYS:
        if w[k] is not None:
            np.testing.assert_allclose(g[k], tw[k].grad.numpy(), rtol=1e-9, atol=1e-10, err_msg=k)


def test_pre_ln_zero_weights_is_identity():
    shape = TINY["pre_swiglu_causal_gqa"]
    inp = layer_inputs(shape, 0)
    w = {k: (np.zeros_like(inp[k]) if k.startswith(("w_", "b_")) and inp[k] is not None else inp[k])
         for k in KEYS}
    y, _ = oracle.block_fwd(shape, w, inp["x"])
    np.testing.assert_array_equal(y, inp["x"])


def test_post_ln_mean_loss_is_zero_with_zero_grads():
    """Textbook Post-LN without affine: mean(LN(.)) == 0 for every row, so
    loss = mean(out) is identically 0 and every gradient vanishes."""
    shape = WORKLOADS["fp32_postln_b2s128h256"].replace(batch=1, seq=16)
    inp = layer_inputs(shape, 0)
    w = _weights(inp)
    y, cache = oracle.block_fwd(shape, w, inp["x"])
    assert abs(y.mean()) <= 1e-14
    dy = np.full_like(y, 1.0 / y.size)
    dx, g = oracle.block_bwd(shape, w, cache, dy)
    assert np.abs(dx).max() <= 1e-10
    for k in ("w_qkv", "w_o", "w_1", "w_2"):
        assert np.abs(g[k]).max() <= 1e-10, k


def test_fwd_rows_matches_full_forward():
    for name in ("pre_gelu_causal_gqa", "post_gelu", "pre_swiglu_causal_gqa"):
        shape = TINY[name]
        inp = _inputs(shape)
        w = _weights(inp)
        y, _ = oracle.block_fwd(shape, w, inp["x"])
        rows = np.array([0, shape.tokens - 1, shape.seq // 2])
        np.testing.assert_allclose(oracle.block_fwd_rows(shape, w, inp["x"], rows), y[rows],
                                   rtol=1e-13, atol=1e-13)


# ------------------------------------------------------ k-way split invariant

SPLIT_SHAPES = {
    "mha_gelu": LayerShape(1, 6, 8, 8, 8, 2, 16, dtype="f32"),
    "gqa_swiglu_causal": LayerShape(2, 5, 8, 8, 4, 2, 16, dtype="f32", act="swiglu",
                                    causal=True, glu_block=2),
}


@pytest.mark.parametrize("name", list(SPLIT_SHAPES))
@pytest.mark.parametrize("k", [2, 4, 8])
def test_sharded_partial_sums_equal_unsplit_layer(name, k):
    shape = SPLIT_SHAPES[name]
    if shape.n_kv_heads % k or (shape.act == "swiglu" and (shape.ffn // k) % shape.glu_block):
        pytest.skip("shard would split a KV head or a gate/up block")
    inp = _inputs(shape, seed=5)
    w = _weights(inp)
    y, c = oracle.block_fwd(shape, w, inp["x"])
    dx, g = oracle.block_bwd(shape, w, c, inp["dy"])
    # forward: sum of attention partials (+ bo once) == unsplit projection
    parts, caches = zip(*(shard.attn_partial_fwd(shape, w, c["a_in"], i, k) for i in range(k)))
    np.testing.assert_allclose(sum(parts) + w["b_o"], c["h"] - inp["x"], rtol=1e-12, atol=1e-12)
    fparts, fcaches = zip(*(shard.ffn_partial_fwd(shape, w, c["f_in"], i, k) for i in range(k)))
    np.testing.assert_allclose(sum(fparts) + w["b_2"] + c["h"], y, rtol=1e-12, atol=1e-12)
    # backward: weight grads are slices, input grads sum (pre-LN: dr1 / dr2 known)
    dr2 = inp["dy"]
    d_fin = 0
    for i, fc in enumerate(fcaches):
        dfi, dW1, db1, dW2 = shard.ffn_partial_bwd(shape, w, fc, dr2)
        np.testing.assert_allclose(dW1, g["w_1"][fc["r1"]], rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(db1, g["b_1"][fc["r1"]], rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(dW2, g["w_2"][:, fc["c2"]], rtol=1e-11, atol=1e-13)
        d_fin = d_fin + dfi
    _, mean2, rstd2 = oracle.ln_fwd(c["h"], w["ln2_g"], w["ln2_b"], shape.ln_eps)
    dr1 = dr2 + oracle.ln_bwd(d_fin, c["h"], mean2, rstd2, w["ln2_g"])[0]
    np.testing.assert_allclose(dr1.sum(axis=0), g["b_o"], rtol=1e-11, atol=1e-13)
    d_ain = 0
    for i, ac in enumerate(caches):
        dai, dWqkv, dbqkv, dWo = shard.attn_partial_bwd(shape, w, ac, dr1)
        np.testing.assert_allclose(dWqkv, g["w_qkv"][ac["rows"]], rtol=1e-10, atol=1e-13)
        np.testing.assert_allclose(dbqkv, g["b_qkv"][ac["rows"]], rtol=1e-10, atol=1e-13)
        np.testing.assert_allclose(dWo, g["w_o"][:, ac["o_cols"]], rtol=1e-11, atol=1e-13)
        d_ain = d_ain + dai
    _, mean1, rstd1 = oracle.ln_fwd(inp["x"], w["ln1_g"], w["ln1_b"], shape.ln_eps)
    dx_split = dr1 + oracle.ln_bwd(d_ain, inp["x"], mean1, rstd1, w["ln1_g"])[0]
    np.testing.assert_allclose(dx_split, dx, rtol=1e-10, atol=1e-12)


def test_shard_planted_mistake_is_caught():
    """A shard that drops one head's Wo columns must break the sum."""
    shape = SPLIT_SHAPES["mha_gelu"]
    inp = _inputs(shape, seed=5)
    w = _weights(inp)
    _, c = oracle.block_fwd(shape, w, inp["x"])
    parts = [shard.attn_partial_fwd(shape, w, c["a_in"], i, 2)[0] for i in range(2)]
    w_bad = dict(w)
    w_bad["w_o"] = w["w_o"].copy()
    w_bad["w_o"][:, :2] = 0.0
    bad = [shard.attn_partial_fwd(shape, w_bad, c["a_in"], i, 2)[0] for i in range(2)]
    good_err = np.abs(sum(parts) + w["b_o"] - (c["h"] - inp["x"])).max()
    bad_err = np.abs(sum(bad) + w["b_o"] - (c["h"] - inp["x"])).max()
    assert good_err < 1e-12 < 1e-3 < bad_err
