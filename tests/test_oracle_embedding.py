"""Pins of the vocab-parallel embedding oracle against facts that do not
come from its own code: the unsharded lookup is plain row indexing, the
shard outputs sum to it, the backward is the adjoint of the lookup, and
closed forms for distinct / repeated / out-of-range ids."""
import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(41)


def _case(T=37, H=24, V=50):
    ids = RNG.integers(0, V, size=T)
    E = RNG.standard_normal((V, H))
    dout = RNG.standard_normal((T, H))
    return ids, E, dout


def test_full_lookup_is_row_indexing():
    ids, E, _ = _case()
    assert np.array_equal(oracle.embedding_fwd(ids, E, 0, E.shape[0]), E[ids])


@pytest.mark.parametrize("k", [2, 3, 5])
def test_shard_outputs_sum_to_full_lookup(k):
    """Vocab split in k contiguous ranges (the last one ragged): each token's
    row comes from exactly one shard."""
    ids, E, _ = _case()
    V = E.shape[0]
    bounds = np.linspace(0, V, k + 1).astype(int)
    tot = sum(oracle.embedding_fwd(ids, E[a:b], a, b) for a, b in zip(bounds[:-1], bounds[1:]))
    assert np.array_equal(tot, E[ids])
    # a shard's output is zero exactly on the rows of tokens it does not own
    a, b = bounds[1], bounds[2]
    part = oracle.embedding_fwd(ids, E[a:b], a, b)
    outside = (ids < a) | (ids >= b)
    assert np.all(part[outside] == 0) and np.array_equal(part[~outside], E[ids[~outside]])


def test_backward_is_adjoint_of_lookup():
    """<lookup(E), dout> == <E, bwd(dout)> for every shard."""
    ids, E, dout = _case()
    for a, b in ((0, 50), (10, 27), (49, 50)):
        lhs = np.sum(oracle.embedding_fwd(ids, E[a:b], a, b) * dout)
        rhs = np.sum(E[a:b] * oracle.embedding_bwd(ids, dout, a, b))
        assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(lhs))


def test_backward_closed_forms():
    H = 6
    dout = RNG.standard_normal((5, H))
    # distinct ids: the rows are the output gradients themselves
    ids = np.array([3, 0, 7, 1, 4])
    dE = oracle.embedding_bwd(ids, dout, 0, 8)
    assert np.array_equal(dE[ids], dout)
    assert np.all(dE[[2, 5, 6]] == 0)
    # repeated id: the sum of its tokens' gradients
    ids = np.array([2, 2, 5, 2, 5])
    dE = oracle.embedding_bwd(ids, dout, 0, 8)
    assert np.allclose(dE[2], dout[0] + dout[1] + dout[3], rtol=0, atol=1e-15)
    assert np.allclose(dE[5], dout[2] + dout[4], rtol=0, atol=1e-15)
    # shard [4, 8): only the tokens with id 5 land, at local row 1
    dE = oracle.embedding_bwd(ids, dout, 4, 8)
    assert dE.shape == (4, H) and np.allclose(dE[1], dout[2] + dout[4], rtol=0, atol=1e-15)
    assert np.all(dE[[0, 2, 3]] == 0)


def test_backward_column_sums_match_the_tokens():
    """Every in-range token's gradient lands in exactly one row."""
    ids, _, dout = _case()
    dE = oracle.embedding_bwd(ids, dout, 0, 50)
    assert np.allclose(dE.sum(axis=0), dout.sum(axis=0), rtol=1e-12, atol=1e-12)


def test_planted_error_is_caught():
    """A lookup that ignores the mask (clips ids into the shard instead) breaks
    the shard-sum invariant."""
    ids, E, _ = _case()
    a, b = 0, 25
    def wrong(ids, Es, v0, v1):
        return Es[np.clip(ids - v0, 0, v1 - v0 - 1)]
    tot = wrong(ids, E[a:b], a, b) + oracle.embedding_fwd(ids, E[b:], b, 50)
    assert not np.array_equal(tot, E[ids])
