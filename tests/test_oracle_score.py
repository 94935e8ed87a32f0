"""Pins of the scoring oracle against what the pages and the mathematics fix.

Hand-computed cases (tests/golden/hand_attention_cases.json), a closed form,
a library softmax special case, the softmax row-sum invariant and symmetries.
Each is chosen so that a plausible slip in the oracle fails one of them: a
missing 1/sqrt(d), a non-causal look-ahead mask, a mean instead of a max, a
wrong GQA pairing, a sum instead of a mean over look-ahead steps.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.special

import oracle
from conftest import GOLDEN


def _num(v):
    if isinstance(v, str):
        if v.startswith("ln(") and v.endswith(")"):
            return math.log(float(Fraction(v[3:-1])))
        return float(Fraction(v))
    return float(v)


def _arr(x):
    if isinstance(x, list):
        return np.array([_arr(v) for v in x], dtype=np.float64)
    return _num(x)


def _hand_cases():
    with open(os.path.join(GOLDEN, "hand_attention_cases.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _hand_cases(), ids=lambda c: c["name"])
def test_hand_cases(case):
    Q, K, Kla = _arr(case["Q_la"]), _arr(case["K_prompt"]), _arr(case["K_la"])
    assert Q.shape == (case["N"], case["L"], case["H"], case["d"])
    assert K.shape == (case["L"], case["H_kv"], case["M"], case["d"])
    assert Kla.shape == (case["L"], case["H_kv"], case["N"], case["d"])
    got = oracle.importance(Q, K, Kla)
    want = np.array([_num(v) for v in case["importance"]])
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-15)


def _rand(rng, N, L, H, H_kv, M, d):
    return (rng.standard_normal((N, L, H, d)), rng.standard_normal((L, H_kv, M, d)),
            rng.standard_normal((L, H_kv, N, d)))


@pytest.mark.parametrize("N,L,H,H_kv,M,d", [(1, 1, 1, 1, 7, 4), (3, 2, 4, 2, 33, 8), (5, 3, 6, 1, 50, 16)])
def test_closed_form_equal_keys(N, L, H, H_kv, M, d):
    """All keys equal -> every softmax row is uniform over M + j + 1 keys."""
    rng = np.random.default_rng(7)
    Q = rng.standard_normal((N, L, H, d))
    v = rng.standard_normal(d)
    K = np.broadcast_to(v, (L, H_kv, M, d)).copy()
    Kla = np.broadcast_to(v, (L, H_kv, N, d)).copy()
    want = sum(1.0 / (M + j + 1) for j in range(N)) / N
    np.testing.assert_allclose(oracle.importance(Q, K, Kla), np.full(M, want), rtol=1e-12)


def test_library_softmax_with_scale():
    """L = H = N = 1, q = (2, 0, 0, 0), d = 4: logits are K[:, 0] exactly iff scaled by 1/sqrt(d)."""
    rng = np.random.default_rng(3)
    M, d = 40, 4
    K = rng.standard_normal((1, 1, M, d))
    Kla = rng.standard_normal((1, 1, 1, d))
    Q = np.zeros((1, 1, 1, d))
    Q[0, 0, 0, 0] = 2.0
    ref = scipy.special.softmax(np.concatenate([K[0, 0, :, 0], Kla[0, 0, :, 0]]))[:M]
    np.testing.assert_allclose(oracle.importance(Q, K, Kla), ref, rtol=1e-12)


def test_rows_sum_to_one():
    rng = np.random.default_rng(11)
    N, L, H, H_kv, M, d = 6, 2, 4, 2, 64, 16
    Q, K, Kla = _rand(rng, N, L, H, H_kv, M, d)
    K[:, :, 0] *= 4.0
    for l in range(L):
        for h in range(H):
            a, a_la = oracle.attention_rows(Q, K, Kla, l, h)
            tot = a.sum(axis=1) + a_la.sum(axis=1)
            np.testing.assert_allclose(tot, 1.0, rtol=0, atol=1e-12)
            assert np.all(np.triu(a_la, k=1) == 0.0)     # causal: no weight on later steps
            assert np.all(np.diag(a_la) > 0.0)           # step j sees its own key


def test_bounds_and_zero_lookahead():
    rng = np.random.default_rng(5)
    Q, K, Kla = _rand(rng, 4, 2, 2, 1, 30, 8)
    imp = oracle.importance(Q, K, Kla)
    assert np.all(imp > 0) and np.all(imp < 1)
    # N = 0: nothing captured -> importance 1.0 everywhere (compute_imp's fallback)
    np.testing.assert_array_equal(oracle.importance(Q[:0], K, Kla[:, :, :0]), np.ones(30))


def test_token_permutation_equivariance():
    rng = np.random.default_rng(17)
    Q, K, Kla = _rand(rng, 3, 2, 4, 2, 45, 8)
    perm = rng.permutation(45)
    a = oracle.importance(Q, K, Kla)
    b = oracle.importance(Q, K[:, :, perm], Kla)
    np.testing.assert_allclose(b, a[perm], rtol=1e-12)


def test_layer_and_in_group_head_permutation_invariance():
    rng = np.random.default_rng(19)
    N, L, H, H_kv, M, d = 3, 3, 4, 2, 25, 8
    Q, K, Kla = _rand(rng, N, L, H, H_kv, M, d)
    a = oracle.importance(Q, K, Kla)
    lp = np.array([2, 0, 1])
    np.testing.assert_allclose(oracle.importance(Q[:, lp], K[lp], Kla[lp]), a, rtol=1e-12)
    hp = np.array([1, 0, 3, 2])                  # swap heads inside each KV group
    np.testing.assert_allclose(oracle.importance(Q[:, :, hp], K, Kla), a, rtol=1e-12)


def test_gqa_equals_mha_with_repeated_keys():
    rng = np.random.default_rng(23)
    N, L, H, H_kv, M, d = 2, 2, 6, 2, 20, 8
    G = H // H_kv
    Q, K, Kla = _rand(rng, N, L, H, H_kv, M, d)
    a = oracle.importance(Q, K, Kla)
    b = oracle.importance(Q, np.repeat(K, G, axis=1), np.repeat(Kla, G, axis=1))
    np.testing.assert_allclose(b, a, rtol=1e-12)


def test_max_is_not_diluted_by_extra_weak_layer():
    """A layer that attends uniformly leaves a dominant key's importance unchanged (max),
    where a mean over layers would pull it halfway to the uniform weight."""
    rng = np.random.default_rng(29)
    N, H, M, d = 2, 2, 16, 4
    Q, K, Kla = _rand(rng, N, 1, H, 1, M, d)
    Q[:, 0] = np.abs(Q[:, 0])
    K[0, 0, 3] = 10.0                               # every head and step puts most weight here
    a = oracle.importance(Q, K, Kla)
    assert a[3] > 0.5
    Q2 = np.concatenate([Q, np.zeros_like(Q)], axis=1)      # layer 1: q = 0 -> uniform rows
    K2 = np.concatenate([K, K], axis=0)
    Kla2 = np.concatenate([Kla, Kla], axis=0)
    b = oracle.importance(Q2, K2, Kla2)
    uni = np.mean([1.0 / (M + j + 1) for j in range(N)])
    assert b[3] == a[3]
    assert np.all(b >= a) and np.all(b >= uni * (1 - 1e-12))


def test_bf16_bits_read_exactly():
    from workloads import bf16_bits_from_f32, f32_from_bf16_bits
    rng = np.random.default_rng(31)
    Q, K, Kla = (x.astype(np.float32) for x in _rand(rng, 2, 1, 2, 1, 12, 8))
    bits = [bf16_bits_from_f32(x).reshape(x.shape) for x in (Q, K, Kla)]
    vals = [f32_from_bf16_bits(b) for b in bits]
    np.testing.assert_array_equal(oracle.importance(*bits), oracle.importance(*vals))
