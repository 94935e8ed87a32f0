"""Pins of the lse-given oracle (row_lse, importance_given_lse).

The single-pass variant takes each row's softmax normaliser from the caller.
These tests fix the oracle's two halves against closed forms, hand-computed
values and exact properties, each computed here without the oracle:
- a row's weights over the prompt keys and its causal look-ahead keys sum to
  1 under its lse;
- equal keys give lse = s0 + ln(M + j + 1);
- a hand case has lse = ln 5;
- shifting lse by c scales importance by e^-c;
- two layers combine by max.
A missing scale, a non-causal look-ahead mask, an added instead of a
subtracted lse, or a mean over layers fails one of them.
"""
import math

import numpy as np
import pytest

import oracle


def _rand(rng, N, L, H, H_kv, M, d):
    return (rng.standard_normal((N, L, H, d)), rng.standard_normal((L, H_kv, M, d)),
            rng.standard_normal((L, H_kv, N, d)))


def test_row_lse_normalises_prompt_plus_causal_lookahead_keys():
    rng = np.random.default_rng(21)
    N, L, H, H_kv, M, d = 5, 2, 4, 2, 37, 8
    Q, K, Kla = _rand(rng, N, L, H, H_kv, M, d)
    lse = oracle.row_lse(Q, K, Kla)
    assert lse.shape == (L, H, N)
    G = H // H_kv
    for l in range(L):
        for h in range(H):
            g = h // G
            for j in range(N):
                q = Q[j, l, h]
                s = np.array([q @ K[l, g, i] for i in range(M)]) / math.sqrt(d)
                u = np.array([q @ Kla[l, g, k] for k in range(j + 1)]) / math.sqrt(d)
                tot = np.exp(s - lse[l, h, j]).sum() + np.exp(u - lse[l, h, j]).sum()
                assert abs(tot - 1.0) < 1e-12


def test_row_lse_hand_case():
    """d = 1, M = 2, N = 1: logits 0 and ln 3 plus the look-ahead key's 0 -> lse = ln 5."""
    Q = np.array([[[[1.0]]]])
    K = np.array([[[[0.0], [math.log(3.0)]]]])
    Kla = np.array([[[[0.0]]]])
    np.testing.assert_allclose(oracle.row_lse(Q, K, Kla), [[[math.log(5.0)]]], rtol=1e-14)
    np.testing.assert_allclose(oracle.importance_given_lse(Q, K, [[[math.log(5.0)]]]), [0.2, 0.6], rtol=1e-14)


@pytest.mark.parametrize("N,L,H,H_kv,M,d", [(1, 1, 1, 1, 9, 4), (4, 2, 4, 2, 25, 8)])
def test_closed_form_equal_keys(N, L, H, H_kv, M, d):
    rng = np.random.default_rng(5)
    Q = rng.standard_normal((N, L, H, d))
    v = rng.standard_normal(d)
    K = np.broadcast_to(v, (L, H_kv, M, d)).copy()
    Kla = np.broadcast_to(v, (L, H_kv, N, d)).copy()
    s0 = np.einsum("jlhd,d->lhj", Q, v) / math.sqrt(d)                 # every logit of row (l, h, j)
    want_lse = s0 + np.log(M + np.arange(N) + 1.0)[None, None, :]
    np.testing.assert_allclose(oracle.row_lse(Q, K, Kla), want_lse, rtol=1e-13)
    want = sum(1.0 / (M + j + 1) for j in range(N)) / N
    np.testing.assert_allclose(oracle.importance_given_lse(Q, K, want_lse), np.full(M, want), rtol=1e-12)


def test_shifting_lse_scales_importance():
    rng = np.random.default_rng(8)
    Q, K, Kla = _rand(rng, 3, 2, 2, 1, 20, 8)
    lse = oracle.row_lse(Q, K, Kla)
    base = oracle.importance_given_lse(Q, K, lse)
    for c in (0.5, -1.25, 3.0):
        np.testing.assert_allclose(oracle.importance_given_lse(Q, K, lse + c), base * math.exp(-c), rtol=1e-12)


def test_layers_combine_by_max():
    """Two layers, d = 1, M = 2, lse = ln 5 in each: weights [1/5, 3/5] and [4/5, 1/5] -> max [4/5, 3/5]."""
    Q = np.ones((1, 2, 1, 1))
    K = np.array([[[[0.0], [math.log(3.0)]]], [[[math.log(4.0)], [0.0]]]])
    lse = np.full((2, 1, 1), math.log(5.0))
    np.testing.assert_allclose(oracle.importance_given_lse(Q, K, lse), [0.8, 0.6], rtol=1e-14)


def test_given_lse_reproduces_importance():
    """The oracle's two routes agree: the lse-given aggregation of row_lse is importance()."""
    rng = np.random.default_rng(13)
    Q, K, Kla = _rand(rng, 4, 2, 4, 2, 45, 8)
    K[:, :, 0] *= 4.0
    np.testing.assert_allclose(oracle.importance_given_lse(Q, K, oracle.row_lse(Q, K, Kla)),
                               oracle.importance(Q, K, Kla), rtol=1e-12, atol=1e-15)


def test_zero_lookahead_gives_ones():
    K = np.zeros((1, 1, 6, 4))
    np.testing.assert_array_equal(oracle.importance_given_lse(np.zeros((0, 1, 1, 4)), K, np.zeros((1, 1, 0))),
                                  np.ones(6))
