"""Vocab-parallel embedding lookup and its backward.

"02 - How a whole Transformer block is split", section 3 (vocab-parallel
embedding): the [vocab, h] table is split along the vocabulary; a rank holds
rows [v0, v1). For a token id outside its range the rank looks up a masked
row and zeroes the result, so every token's row comes from exactly one rank
and the all-reduce (a sum) over ranks yields the full lookup. The input and
output embeddings are usually tied (one table), so the table's gradient is
the sum of the lookup's gradient and the output projection's (the CE's)
gradient.

  embedding_fwd   out[t] = E_shard[ids[t] - v0] if v0 <= ids[t] < v1, else 0
  embedding_bwd   dE_shard[v - v0] = sum over t with ids[t] = v of dout[t]
                  (the adjoint of the lookup: <lookup(E), dout> = <E, bwd(dout)>)

Both are written out with explicit loops over tokens (the definition), no
library scatter. Test infrastructure only; pinned by
tests/test_oracle_embedding.py.
"""
import numpy as np


def embedding_fwd(ids, emb_shard, v0, v1):
    """Masked lookup of shard rows [v0, v1); float64 [T, H]."""
    ids = np.asarray(ids)
    E = np.asarray(emb_shard, dtype=np.float64)
    assert E.shape[0] == v1 - v0
    out = np.zeros((ids.shape[0], E.shape[1]))
    for t, v in enumerate(ids):
        if v0 <= v < v1:
            out[t] = E[v - v0]
    return out


def embedding_bwd(ids, dout, v0, v1):
    """Gradient of the shard's rows: float64 [v1 - v0, H]."""
    ids = np.asarray(ids)
    dout = np.asarray(dout, dtype=np.float64)
    dE = np.zeros((v1 - v0, dout.shape[1]))
    for t, v in enumerate(ids):
        if v0 <= v < v1:
            dE[v - v0] += dout[t]
    return dE
