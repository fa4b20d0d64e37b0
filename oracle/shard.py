"""k-way column -> row split of the layer's two sublayers (the TP invariant).

"LLM Lab 06: build a Megatron-style Transformer Block from scratch",
sections 2-3, and "02 - How a whole Transformer block is split", sections
1-2: attention is split by head (linear_qkv column-parallel: a shard holds
the Q/K/V rows of its heads; linear_proj row-parallel: the matching input
columns of Wo) and the MLP column -> row (fc1's output columns, fc2's input
rows). Each shard produces a partial product of the sublayer output; the
all-reduce sums the partials. The biases of the row-parallel layers (bo, b2)
are added once, after the sum.

On one GPU this survives only as an invariant: the sum over shards of the
partial products equals the unsplit sublayer, and each shard's weight
gradients are the matching slices of the unsplit gradients while the input
gradients sum to the unsplit one.

Shard i of k takes query heads [i*nq/k, (i+1)*nq/k) and key/value heads
[i*nkv/k, (i+1)*nkv/k) (so GQA groups never straddle shards), and the fc1
output columns [i*W/k, (i+1)*W/k) with W = ffn (GELU) or 2*ffn (SwiGLU): with
the interleaved gate/up layout a contiguous range of fc1 columns holds whole
gate/up pairs, which is why the pages interleave (section 1 of "02 ...").

Test infrastructure only.
"""
import numpy as np

from .attention import attention_fwd, attention_bwd
from .activations import gelu, gelu_grad, swiglu_fwd, swiglu_bwd


def head_shard(cfg, i, k):
    """Index arrays (qkv_rows, o_cols) of shard i of k for the attention sublayer."""
    nq, nkv, d = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    assert nq % k == 0 and nkv % k == 0, "every shard needs whole KV heads"
    qh = np.arange(i * nq // k, (i + 1) * nq // k)
    kh = np.arange(i * nkv // k, (i + 1) * nkv // k)
    heads_rows = lambda base, hs: (base + hs[:, None] * d + np.arange(d)[None, :]).ravel()
    q_rows = heads_rows(0, qh)
    k_rows = heads_rows(nq * d, kh)
    v_rows = heads_rows((nq + nkv) * d, kh)
    return np.concatenate([q_rows, k_rows, v_rows]), q_rows


def ffn_shard(cfg, i, k):
    """Index arrays (w1_rows, w2_cols) of shard i of k for the MLP sublayer."""
    F = cfg.ffn
    gb = cfg.glu_block
    assert F % k == 0
    if cfg.act == "swiglu":
        assert (F // k) % gb == 0, "a shard must hold whole gate/up blocks"
        w1_rows = np.arange(2 * i * F // k, 2 * (i + 1) * F // k)
    else:
        w1_rows = np.arange(i * F // k, (i + 1) * F // k)
    return w1_rows, np.arange(i * F // k, (i + 1) * F // k)


def attn_partial_fwd(cfg, w, a_in, i, k):
    """Shard i's partial product of the attention sublayer: O_i Wo[:, cols_i]^T."""
    rows, o_cols = head_shard(cfg, i, k)
    B, S, d = cfg.batch, cfg.seq, cfg.head_dim
    nq_s, nkv_s = cfg.n_q_heads // k, cfg.n_kv_heads // k
    qkv = a_in @ w["w_qkv"][rows].T
    if w["b_qkv"] is not None:
        qkv = qkv + w["b_qkv"][rows][None, :]
    q = qkv[:, : nq_s * d].reshape(B, S, nq_s, d).transpose(0, 2, 1, 3)
    kk = qkv[:, nq_s * d: (nq_s + nkv_s) * d].reshape(B, S, nkv_s, d).transpose(0, 2, 1, 3)
    v = qkv[:, (nq_s + nkv_s) * d:].reshape(B, S, nkv_s, d).transpose(0, 2, 1, 3)
    o, _ = attention_fwd(q, kk, v, cfg.causal)
    O = o.transpose(0, 2, 1, 3).reshape(B * S, nq_s * d)
    part = O @ w["w_o"][:, o_cols].T
    return part, {"a_in": a_in, "q": q, "k": kk, "v": v, "O": O, "rows": rows, "o_cols": o_cols}


def attn_partial_bwd(cfg, w, c, dpart):
    """Given dL/d(total) (= dL/d(each partial)), shard gradients:
    (d a_in contribution, dWqkv[rows], dbqkv[rows] or None, dWo[:, o_cols])."""
    B, S, d = cfg.batch, cfg.seq, cfg.head_dim
    nq_s = c["q"].shape[1]
    dWo = dpart.T @ c["O"]
    dO = dpart @ w["w_o"][:, c["o_cols"]]
    do = dO.reshape(B, S, nq_s, d).transpose(0, 2, 1, 3)
    dq, dk, dv = attention_bwd(do, c["q"], c["k"], c["v"], cfg.causal)
    m = lambda t: t.transpose(0, 2, 1, 3).reshape(B * S, -1)
    dqkv = np.concatenate([m(dq), m(dk), m(dv)], axis=1)
    dW = dqkv.T @ c["a_in"]
    db = dqkv.sum(axis=0) if w["b_qkv"] is not None else None
    return dqkv @ w["w_qkv"][c["rows"]], dW, db, dWo


def ffn_partial_fwd(cfg, w, f_in, i, k):
    """Shard i's partial product of the MLP sublayer: act(f_in W1_i^T + b1_i) W2[:, cols_i]^T."""
    r1, c2 = ffn_shard(cfg, i, k)
    u = f_in @ w["w_1"][r1].T
    if w["b_1"] is not None:
        u = u + w["b_1"][r1][None, :]
    a = swiglu_fwd(u, cfg.glu_block) if cfg.act == "swiglu" else gelu(u)
    return a @ w["w_2"][:, c2].T, {"f_in": f_in, "u": u, "a": a, "r1": r1, "c2": c2}


def ffn_partial_bwd(cfg, w, c, dpart):
    """(d f_in contribution, dW1[rows], db1[rows] or None, dW2[:, cols])."""
    dW2 = dpart.T @ c["a"]
    da = dpart @ w["w_2"][:, c["c2"]]
    du = swiglu_bwd(da, c["u"], cfg.glu_block) if cfg.act == "swiglu" else da * gelu_grad(c["u"])
    db1 = du.sum(axis=0) if w["b_1"] is not None else None
    return du @ w["w_1"][c["r1"]], du.T @ c["f_in"], db1, dW2
