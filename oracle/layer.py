"""One Megatron-style transformer layer: forward and hand-derived backward.

Dataflow ("LLM Lab 06: build a Megatron-style Transformer Block from
scratch", section 2; "02 - How a whole Transformer block is split",
sections 1-2), tokens t = b*S + s as rows of [T, H] (batch-major, the
[batch, seq, hidden] layout of page 1), weights [out, in] (y = x W^T + b):

  Pre-LN ("pre"; page 1's code: the norm sits before each sublayer)
      xn = LN1(x);  qkv = xn Wqkv^T + bqkv;  O = Attn(qkv)
      h  = x + O Wo^T + bo
      hn = LN2(h);  u = hn W1^T + b1;  a = act(u)
      y  = h + a W2^T + b2
  Post-LN ("post"; textbook form: LN after each residual add)
      qkv = x Wqkv^T + bqkv;  O = Attn(qkv)
      h  = LN1(x + O Wo^T + bo)
      u  = h W1^T + b1;  a = act(u)
      y  = LN2(h + a W2^T + b2)

Wqkv rows are [Q heads | K heads | V heads] ("02 ...", section 2: linear_qkv
of width q_proj + 2*kv_proj); head n of Q is rows n*d .. n*d+d-1. The output
projection Wo (linear_proj, "02 ...", section 2) maps the nq*d concatenated
head outputs back to H. act is erf-GELU, or SwiGLU on the interleaved fc1
output (see activations.py).

Dropout ("02 - How a whole Transformer block is split", section 5), when
`drop` is given (masks from oracle/dropout.py): on the attention
probabilities (attention.py), and on the outputs of the output projection and
of fc2 before their residual adds:
      h = x + D_proj(O Wo^T + bo),   y = h + D_fc2(a W2^T + b2)   (Pre-LN)
(Post-LN likewise inside LN1 / LN2), D(z) = z o M s. The backward passes the
residual gradient through unchanged and multiplies the sublayer branch's
gradient by M s.

The backward is written out by hand (no autograd), in reverse order:
  fc2:  db2 = sum_t dr2, dW2 = dr2^T a, da = dr2 W2
  act:  du = da * gelu'(u)   |  swiglu_bwd(da, u)
  fc1:  db1 = sum_t du, dW1 = du^T f_in, df_in = du W1
  LN2 / LN1 backward (layernorm.py), residual grads added
  proj: dbo = sum_t dr1, dWo = dr1^T O, dO = dr1 Wo
  attention backward (attention.py)
  qkv:  dbqkv = sum_t dqkv, dWqkv = dqkv^T a_in, da_in = dqkv Wqkv

Test infrastructure only.
"""
import numpy as np

from .layernorm import ln_fwd, ln_bwd
from .activations import gelu, gelu_grad, swiglu_fwd, swiglu_bwd
from .attention import attention_fwd, attention_bwd

_WEIGHT_KEYS = ("w_qkv", "b_qkv", "w_o", "b_o", "w_1", "b_1", "w_2", "b_2",
                "ln1_g", "ln1_b", "ln2_g", "ln2_b")


def _lin(x, w, b):
    y = x @ w.T
    return y + b[None, :] if b is not None else y


def _split_heads(qkv, cfg):
    B, S = cfg.batch, cfg.seq
    nq, nkv, d = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    q = qkv[:, : nq * d].reshape(B, S, nq, d).transpose(0, 2, 1, 3)
    k = qkv[:, nq * d: (nq + nkv) * d].reshape(B, S, nkv, d).transpose(0, 2, 1, 3)
    v = qkv[:, (nq + nkv) * d:].reshape(B, S, nkv, d).transpose(0, 2, 1, 3)
    return q, k, v


def _merge_heads(o):
    B, nq, S, d = o.shape
    return o.transpose(0, 2, 1, 3).reshape(B * S, nq * d)


def _act(u, cfg):
    return swiglu_fwd(u, cfg.glu_block) if cfg.act == "swiglu" else gelu(u)


def _act_bwd(da, u, cfg):
    return swiglu_bwd(da, u, cfg.glu_block) if cfg.act == "swiglu" else da * gelu_grad(u)


def _drop(z, site):
    if site is None:
        return z
    keep, scale = site
    return np.where(keep, z * scale, 0.0)


def block_fwd(cfg, w, x, drop=None):
    """Forward of one layer. Returns (y [T, H], cache for block_bwd).
    drop: optional {"attn": (keep, scale) or None, "proj": ..., "fc2": ...}."""
    x = np.asarray(x, dtype=np.float64)
    eps = cfg.ln_eps
    drop = drop or {}
    c = {"x": x, "drop": drop}
    if cfg.norm_pos == "pre":
        xn, c["mu1"], c["rs1"] = ln_fwd(x, w["ln1_g"], w["ln1_b"], eps)
        a_in = xn
    else:
        a_in = x
    c["a_in"] = a_in
    qkv = _lin(a_in, w["w_qkv"], w["b_qkv"])
    q, k, v = _split_heads(qkv, cfg)
    ad = drop.get("attn")
    o, c["lse"] = attention_fwd(q, k, v, cfg.causal, *(ad if ad is not None else (None, 1.0)))
    c["q"], c["k"], c["v"] = q, k, v
    O = _merge_heads(o)
    c["O"] = O
    r1 = x + _drop(_lin(O, w["w_o"], w["b_o"]), drop.get("proj"))
    if cfg.norm_pos == "pre":
        h = r1
        f_in, c["mu2"], c["rs2"] = ln_fwd(h, w["ln2_g"], w["ln2_b"], eps)
    else:
        c["r1"] = r1
        h, c["mu1"], c["rs1"] = ln_fwd(r1, w["ln1_g"], w["ln1_b"], eps)
        f_in = h
    c["h"], c["f_in"] = h, f_in
    u = _lin(f_in, w["w_1"], w["b_1"])
    a = _act(u, cfg)
    c["u"], c["a"] = u, a
    r2 = h + _drop(_lin(a, w["w_2"], w["b_2"]), drop.get("fc2"))
    if cfg.norm_pos == "pre":
        y = r2
    else:
        c["r2"] = r2
        y, c["mu2"], c["rs2"] = ln_fwd(r2, w["ln2_g"], w["ln2_b"], eps)
    return y, c


def block_bwd(cfg, w, c, dy):
    """Backward of block_fwd given dL/dy. Returns (dx, grads dict).

    grads holds dW for every weight key present (None where the weight is None).
    """
    dy = np.asarray(dy, dtype=np.float64)
    g = {}
    if cfg.norm_pos == "pre":
        dr2 = dy
    else:
        dr2, g["ln2_g"], g["ln2_b"] = ln_bwd(dy, c["r2"], c["mu2"], c["rs2"], w["ln2_g"])
    drop = c.get("drop") or {}
    # fc2 (row-parallel linear in the pages; here the whole K range at once),
    # through its dropout
    dz2 = _drop(dr2, drop.get("fc2"))
    g["b_2"] = dz2.sum(axis=0) if w["b_2"] is not None else None
    g["w_2"] = dz2.T @ c["a"]
    da = dz2 @ w["w_2"]
    du = _act_bwd(da, c["u"], cfg)
    g["b_1"] = du.sum(axis=0) if w["b_1"] is not None else None
    g["w_1"] = du.T @ c["f_in"]
    df_in = du @ w["w_1"]
    if cfg.norm_pos == "pre":
        dhn_x, g["ln2_g"], g["ln2_b"] = ln_bwd(df_in, c["h"], c["mu2"], c["rs2"], w["ln2_g"])
        dr1 = dr2 + dhn_x            # residual: h feeds both LN2 and the fc2 add
    else:
        dh = df_in + dr2             # h feeds fc1 and the fc2 residual add
        dr1, g["ln1_g"], g["ln1_b"] = ln_bwd(dh, c["r1"], c["mu1"], c["rs1"], w["ln1_g"])
    dz1 = _drop(dr1, drop.get("proj"))
    g["b_o"] = dz1.sum(axis=0) if w["b_o"] is not None else None
    g["w_o"] = dz1.T @ c["O"]
    dO = dz1 @ w["w_o"]
    B, nq, S, d = c["q"].shape
    do = dO.reshape(B, S, nq, d).transpose(0, 2, 1, 3)
    ad = drop.get("attn")
    dq, dk, dv = attention_bwd(do, c["q"], c["k"], c["v"], cfg.causal,
                               *(ad if ad is not None else (None, 1.0)))
    dqkv = np.concatenate([_merge_heads(dq), _merge_heads(dk), _merge_heads(dv)], axis=1)
    g["b_qkv"] = dqkv.sum(axis=0) if w["b_qkv"] is not None else None
    g["w_qkv"] = dqkv.T @ c["a_in"]
    da_in = dqkv @ w["w_qkv"]
    if cfg.norm_pos == "pre":
        dxn_x, g["ln1_g"], g["ln1_b"] = ln_bwd(da_in, c["x"], c["mu1"], c["rs1"], w["ln1_g"])
        dx = dr1 + dxn_x
    else:
        dx = dr1 + da_in
    for k in _WEIGHT_KEYS:
        if w.get(k) is None:
            g[k] = None
    return dx, g


def block_fwd_rows(cfg, w, x, rows):
    """Forward output y for the given token rows only (same definition as
    block_fwd; keys/values are formed for every key position those rows see).

    Used to check full-size outputs one row at a time.
    """
    x = np.asarray(x, dtype=np.float64)
    rows = np.asarray(rows)
    S, H = cfg.seq, cfg.hidden
    nq, nkv, d = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    rep = nq // nkv
    eps = cfg.ln_eps
    out = np.empty((len(rows), H))
    wq, bq = w["w_qkv"][: nq * d], (w["b_qkv"][: nq * d] if w["b_qkv"] is not None else None)
    wkv = w["w_qkv"][nq * d:]
    bkv = w["b_qkv"][nq * d:] if w["b_qkv"] is not None else None
    kv_cache = {}
    for i, t in enumerate(rows):
        b, s = divmod(int(t), S)
        if b not in kv_cache:
            xb = x[b * S:(b + 1) * S]
            a_b = ln_fwd(xb, w["ln1_g"], w["ln1_b"], eps)[0] if cfg.norm_pos == "pre" else xb
            kv = _lin(a_b, wkv, bkv)
            kv_cache[b] = (kv[:, : nkv * d].reshape(S, nkv, d), kv[:, nkv * d:].reshape(S, nkv, d))
        kb, vb = kv_cache[b]
        xt = x[t:t + 1]
        a_t = ln_fwd(xt, w["ln1_g"], w["ln1_b"], eps)[0] if cfg.norm_pos == "pre" else xt
        qt = _lin(a_t, wq, bq).reshape(nq, d)
        n_keys = s + 1 if cfg.causal else S
        o = np.empty(nq * d)
        for h in range(nq):
            gi = h // rep
            sc = (kb[:n_keys, gi] @ qt[h]) / np.sqrt(d)
            p = np.exp(sc - sc.max())
            p /= p.sum()
            o[h * d:(h + 1) * d] = p @ vb[:n_keys, gi]
        r1 = xt + _lin(o[None, :], w["w_o"], w["b_o"])
        if cfg.norm_pos == "pre":
            h_t = r1
            f_in = ln_fwd(h_t, w["ln2_g"], w["ln2_b"], eps)[0]
        else:
            h_t = ln_fwd(r1, w["ln1_g"], w["ln1_b"], eps)[0]
            f_in = h_t
        a = _act(_lin(f_in, w["w_1"], w["b_1"]), cfg)
        r2 = h_t + _lin(a, w["w_2"], w["b_2"])
        y = r2 if cfg.norm_pos == "pre" else ln_fwd(r2, w["ln2_g"], w["ln2_b"], eps)[0]
        out[i] = y[0]
    return out
