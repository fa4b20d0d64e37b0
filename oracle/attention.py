"""Per-head scaled dot-product attention, dense, forward and backward.

Definition ("LLM Lab 06: build a Megatron-style Transformer Block from
scratch", section 2; "02 - How a whole Transformer block is split",
section 2): for batch b and query head h,
    S = Q_h K_g^T / sqrt(d),  P = softmax_rows(S),  O_h = P V_g.
GQA ("02 ...", section 2, GQA/MQA paragraph): with nkv < nq key/value heads,
query head h reads key/value head g = floor(h / (nq / nkv)) (contiguous
groups - the pages do not fix the mapping; this is the plain reading).
Causal (the causal workloads): key j is visible to query i iff j <= i; masked
scores are -inf before the softmax.

The full [S, S] matrix is formed per (b, h): no online softmax, no tiling.
LSE = log sum_j exp(S_ij) (max-shifted for range only) is returned because the
GPU path saves it for the backward.

Backward, hand-derived from the softmax Jacobian
dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik) with dP = dO V^T:
    dV_g += P^T dO,  dQ = dS K_g / sqrt(d),  dK_g += dS^T Q_h / sqrt(d),
summing over the query heads of each group.

Dropout on the probabilities ("02 - How a whole Transformer block is split",
section 5: inside the tensor-parallel region), given a keep mask M and scale
s: O_h = (P o M s) V_g; the LSE is that of P. Backward: dV_g += (P o M s)^T dO,
dP = (dO V_g^T) o M s, then dS as above.

Test infrastructure only.
"""
import numpy as np


def _scores(qh, kg, causal):
    d = qh.shape[-1]
    s = (qh @ kg.T) / np.sqrt(d)
    if causal:
        S = s.shape[0]
        s = np.where(np.tril(np.ones((S, S), dtype=bool)), s, -np.inf)
    return s


def _softmax(s):
    m = s.max(axis=-1, keepdims=True)
    p = np.exp(s - m)
    l = p.sum(axis=-1, keepdims=True)
    return p / l, (m + np.log(l))[:, 0]


def attention_fwd(q, k, v, causal=False, keep=None, scale=1.0):
    """q [B, nq, S, d]; k, v [B, nkv, S, d] -> (o [B, nq, S, d], lse [B, nq, S]).
    keep: optional dropout keep mask [B, nq, S, S] (kept probabilities x scale)."""
    B, nq, S, d = q.shape
    nkv = k.shape[1]
    assert nq % nkv == 0
    rep = nq // nkv
    o = np.empty_like(q, dtype=np.float64)
    lse = np.empty((B, nq, S))
    for b in range(B):
        for h in range(nq):
            g = h // rep
            p, lse[b, h] = _softmax(_scores(q[b, h], k[b, g], causal))
            if keep is not None:
                p = np.where(keep[b, h], p * scale, 0.0)
            o[b, h] = p @ v[b, g]
    return o, lse


def attention_bwd(do, q, k, v, causal=False, keep=None, scale=1.0):
    """Gradients (dq, dk, dv) of sum(do * attention_fwd(q, k, v, causal, keep, scale)[0])."""
    B, nq, S, d = q.shape
    nkv = k.shape[1]
    rep = nq // nkv
    dq = np.zeros_like(q, dtype=np.float64)
    dk = np.zeros_like(k, dtype=np.float64)
    dv = np.zeros_like(v, dtype=np.float64)
    for b in range(B):
        for h in range(nq):
            g = h // rep
            p, _ = _softmax(_scores(q[b, h], k[b, g], causal))
            pd = p if keep is None else np.where(keep[b, h], p * scale, 0.0)
            dv[b, g] += pd.T @ do[b, h]
            dp = do[b, h] @ v[b, g].T
            if keep is not None:
                dp = np.where(keep[b, h], dp * scale, 0.0)
            ds = p * (dp - (p * dp).sum(axis=-1, keepdims=True))
            dq[b, h] = ds @ k[b, g] / np.sqrt(d)
            dk[b, g] += ds.T @ q[b, h] / np.sqrt(d)
    return dq, dk, dv
