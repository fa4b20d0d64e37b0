"""Tied-embedding cross-entropy: full-vocab definition and the chunked form.

"02 - How a whole Transformer block is split", section 4 (vocab-parallel
cross entropy): with logits l = hidden E^T split by vocabulary into shards,
the loss is assembled from per-shard partials without gathering the full
[tokens, vocab] logits:
  (1) each shard's row max, combined by a global max (numerical stability),
  (2) the target logit, nonzero only on the shard that owns the target,
      combined by a sum,
  (3) each shard's sum of exp(l - max), combined by a sum,
  loss_t = log(sum_exp) - target_logit  (= -log softmax(l)[target]).
Backward is local per shard: grad = softmax - onehot(target).
Section 3 of the same page: the input and output embeddings share one
[vocab, h] matrix (weight tying), so E is the logits weight here.

Here the shards are vocab chunks of one GPU. Each chunk's max is its own
(m_c); the per-chunk sums are rescaled to the global max before adding,
which is the same combination written for unequal shard maxima:
  M = max_c m_c,  S = sum_c s_c exp(m_c - M),  LSE = M + log S.
Reduction over tokens: mean (the pages do not state it; plain reading),
so the gradient is scaled by 1/T. No ignore index, no label smoothing.

Test infrastructure only.
"""
import numpy as np


def _row_blocks(T, block):
    for r0 in range(0, T, block):
        yield r0, min(T, r0 + block)


def ce_full(hidden, emb, targets, row_block=512):
    """Definition: per-token loss_t = logsumexp_v(l_tv) - l_t,target.

    Returns (loss [T], lse [T], mean loss). Rows are streamed in blocks to
    bound memory; each row's LSE uses the whole vocabulary at once.
    """
    T = hidden.shape[0]
    lse = np.empty(T)
    tgt = np.empty(T)
    for r0, r1 in _row_blocks(T, row_block):
        l = hidden[r0:r1] @ emb.T
        m = l.max(axis=1)
        lse[r0:r1] = m + np.log(np.exp(l - m[:, None]).sum(axis=1))
        tgt[r0:r1] = l[np.arange(r1 - r0), targets[r0:r1]]
    loss = lse - tgt
    return loss, lse, loss.mean()


def ce_chunked(hidden, emb, targets, chunk):
    """The shard-partial algorithm with vocab chunks [c*chunk, min((c+1)*chunk, V)).

    Returns (loss [T], lse [T], mean loss, partials) with partials =
    (m [n_chunks, T], s [n_chunks, T], t [n_chunks, T]).
    """
    T = hidden.shape[0]
    V = emb.shape[0]
    n_chunks = (V + chunk - 1) // chunk
    m = np.empty((n_chunks, T))
    s = np.empty((n_chunks, T))
    t = np.zeros((n_chunks, T))
    rows = np.arange(T)
    for c in range(n_chunks):
        v0, v1 = c * chunk, min(V, (c + 1) * chunk)
        l = hidden @ emb[v0:v1].T                       # [T, C]
        m[c] = l.max(axis=1)                            # (1) local max
        s[c] = np.exp(l - m[c][:, None]).sum(axis=1)    # (3) local sum exp
        own = (targets >= v0) & (targets < v1)          # (2) masked target logit
        t[c, own] = l[rows[own], targets[own] - v0]
    M = m.max(axis=0)
    S = (s * np.exp(m - M[None, :])).sum(axis=0)
    lse = M + np.log(S)
    loss = lse - t.sum(axis=0)
    return loss, lse, loss.mean(), (m, s, t)


def ce_grads(hidden, emb, targets, lse, scale, row_block=512):
    """dL/dhidden and dL/demb for L = scale * sum_t loss_t.

    G = (softmax(l) - onehot(target)) * scale,  dhidden = G E,  demb = G^T hidden.
    """
    T = hidden.shape[0]
    d_hidden = np.empty_like(hidden, dtype=np.float64)
    d_emb = np.zeros_like(emb, dtype=np.float64)
    for r0, r1 in _row_blocks(T, row_block):
        l = hidden[r0:r1] @ emb.T
        G = np.exp(l - lse[r0:r1, None])
        G[np.arange(r1 - r0), targets[r0:r1]] -= 1.0
        G *= scale
        d_hidden[r0:r1] = G @ emb
        d_emb += G.T @ hidden[r0:r1]
    return d_hidden, d_emb


def ce_rows(hidden_rows, emb, targets_rows, scale):
    """Per-row loss, LSE and dhidden for selected tokens only (full-size checks).

    Each row's values depend on that row alone, so they equal the same rows
    of ce_full / ce_grads.
    """
    l = hidden_rows @ emb.T
    m = l.max(axis=1)
    lse = m + np.log(np.exp(l - m[:, None]).sum(axis=1))
    n = len(targets_rows)
    loss = lse - l[np.arange(n), targets_rows]
    G = np.exp(l - lse[:, None])
    G[np.arange(n), targets_rows] -= 1.0
    return loss, lse, (G * scale) @ emb


def ce_emb_rows(hidden, emb, targets, lse, scale, vocab_ids):
    """Selected rows of dL/demb for L = scale * sum_t loss_t (full-size checks).

    Row v of demb = G^T hidden is sum_t G[t, v] hidden[t] with
    G[t, v] = (exp(l_tv - LSE_t) - [targets_t = v]) * scale: it needs the
    logits of column v for every token and every token's LSE (from ce_full),
    and nothing else, so it equals those rows of ce_grads' demb.
    """
    vocab_ids = np.asarray(vocab_ids)
    l = hidden @ emb[vocab_ids].T                        # [T, n]
    G = np.exp(l - lse[:, None])
    G -= (targets[:, None] == vocab_ids[None, :])
    G *= scale
    return G.T @ hidden

