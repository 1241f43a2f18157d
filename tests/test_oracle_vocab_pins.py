"""Pins of the oracle's vocabulary-parallel embedding and cross-entropy,
without the GPU: library routines (numpy indexing, scipy's logsumexp and
log_softmax), closed forms, invariants, finite differences, and planted
mistakes that the checks must catch."""
import numpy as np
import pytest
from scipy.special import log_softmax, logsumexp

from oracle import tp_oracle as O


@pytest.mark.parametrize("tp", [1, 2, 4, 8])
def test_embedding_equals_row_gather(tp):
    r = np.random.default_rng(1)
    V, H = 64, 5
    E = r.normal(size=(V, H))
    ids = r.integers(0, V, size=40)
    np.testing.assert_array_equal(O.vocab_embedding(ids, E, tp), E[ids])


def test_embedding_shard_boundaries_int_exact():
    """ids at both edges of every shard, integer table: exact."""
    V, H, tp = 32, 3, 4
    E = np.arange(V * H, dtype=np.int64).reshape(V, H)
    v = V // tp
    ids = np.array([s * v + d for s in range(tp) for d in (0, v - 1)])
    got = O.vocab_embedding(ids, E, tp)
    assert got.dtype == np.int64
    np.testing.assert_array_equal(got, E[ids])


def test_embedding_each_shard_contributes_only_its_ids():
    V, H, tp = 16, 2, 4
    E = np.ones((V, H))
    shards = O.vocab_shards(E, tp)
    assert [sh.shape for sh in shards] == [(4, 2)] * 4
    with pytest.raises(ValueError):
        O.vocab_shards(np.ones((10, 2)), 4)


def test_cross_entropy_against_library():
    r = np.random.default_rng(2)
    z = r.normal(size=(7, 50)) * 3
    y = r.integers(0, 50, size=7)
    want = logsumexp(z, axis=1) - z[np.arange(7), y]
    np.testing.assert_allclose(O.cross_entropy(z, y), want, rtol=1e-13)
    np.testing.assert_allclose(O.cross_entropy(z, y), -log_softmax(z, axis=1)[np.arange(7), y], rtol=1e-12)


def test_cross_entropy_closed_forms():
    V = 1000
    # uniform logits: the label has probability 1/V
    assert O.cross_entropy(np.zeros((1, V)), [3])[0] == pytest.approx(np.log(V), rel=1e-14)
    # the label's logit L above all others (0): log(1 + (V - 1) e^-L)
    for L in (0.5, 5.0, 40.0):
        z = np.zeros((1, V))
        z[0, 7] = L
        assert O.cross_entropy(z, [7])[0] == pytest.approx(np.log1p((V - 1) * np.exp(-L)), rel=1e-12)
    # two classes: softplus of the logit difference
    z = np.array([[1.5, -0.25]])
    assert O.cross_entropy(z, [1])[0] == pytest.approx(np.log1p(np.exp(1.75)), rel=1e-13)


def test_cross_entropy_shift_invariant_and_large_logits():
    r = np.random.default_rng(3)
    z = r.normal(size=(4, 30))
    y = r.integers(0, 30, size=4)
    np.testing.assert_allclose(O.cross_entropy(z + 1234.5, y), O.cross_entropy(z, y), atol=1e-10)
    assert np.isfinite(O.cross_entropy(z * 1000, y)).all()


@pytest.mark.parametrize("tp", [1, 2, 5, 10])
def test_vocab_parallel_cross_entropy_tp_invariant(tp):
    r = np.random.default_rng(4)
    z = r.normal(size=(6, 40))
    y = r.integers(0, 40, size=6)
    shards = O.split_columns(z, tp)
    np.testing.assert_allclose(O.vocab_parallel_cross_entropy(shards, y), O.cross_entropy(z, y), rtol=1e-14)


def test_cross_entropy_grad_finite_differences():
    r = np.random.default_rng(5)
    z = r.normal(size=(3, 9))
    y = r.integers(0, 9, size=3)
    g = O.cross_entropy_grad(z, y, scale=1.0 / 3)
    eps = 1e-6
    num = np.zeros_like(z)
    for i in range(z.shape[0]):
        for j in range(z.shape[1]):
            zp, zm = z.copy(), z.copy()
            zp[i, j] += eps
            zm[i, j] -= eps
            num[i, j] = (O.cross_entropy(zp, y).mean() - O.cross_entropy(zm, y).mean()) / (2 * eps)
    np.testing.assert_allclose(g, num, atol=1e-8)
    np.testing.assert_allclose(g.sum(axis=1), 0.0, atol=1e-14)


# --- planted mistakes --------------------------------------------------------

def test_planted_unshifted_normaliser_is_caught(monkeypatch):
    def wrong(z):
        return np.log(np.exp(np.asarray(z, np.float64)).sum(axis=1))
    monkeypatch.setattr(O, "log_softmax_normaliser", wrong)
    with np.errstate(over="ignore"):
        assert not np.isfinite(O.cross_entropy(np.full((1, 4), 1000.0), [0])).all()


def test_planted_shard_offset_is_caught(monkeypatch):
    real = O.vocab_shards

    def wrong(E, tp):  # shards shifted by one row
        return [np.roll(sh, 1, axis=0) for sh in real(E, tp)]
    monkeypatch.setattr(O, "vocab_shards", wrong)
    E = np.arange(16.0).reshape(8, 2)
    assert not np.array_equal(O.vocab_embedding([1, 5], E, 2), E[[1, 5]])


def test_planted_wrong_label_column_is_caught(monkeypatch):
    r = np.random.default_rng(6)
    z = r.normal(size=(2, 6))
    want = logsumexp(z, axis=1) - z[[0, 1], [2, 4]]
    monkeypatch.setattr(O, "cross_entropy", lambda zz, yy: O.log_softmax_normaliser(zz) - np.asarray(zz)[
        np.arange(len(yy)), (np.asarray(yy) + 1) % zz.shape[1]])
    assert not np.allclose(O.vocab_parallel_cross_entropy(O.split_columns(z, 2), [2, 4]), want)
