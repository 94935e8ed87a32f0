"""Pins of the prefill-row capture (oracle shift = 1): row 0 is the prompt's last
query captured at prefill, whose softmax covers only the M prompt keys; row j >= 1
is decode step j - 1, which also sees look-ahead keys 0..j-1 (llama.cpp guide,
"How It Works": the prefill's last row, then the look-ahead decode steps)."""
import math

import numpy as np
import scipy.special

import oracle


def test_prefill_row_alone_is_a_softmax_over_the_prompt():
    rng = np.random.default_rng(2)
    M, d = 30, 4
    K = rng.standard_normal((1, 1, M, d))
    Q = np.zeros((1, 1, 1, d))
    Q[0, 0, 0, 0] = 2.0                      # scaled logits are exactly K[:, 0]
    Kla = np.zeros((1, 1, 0, d))
    ref = scipy.special.softmax(K[0, 0, :, 0])
    np.testing.assert_allclose(oracle.importance(Q, K, Kla, shift=1), ref, rtol=1e-12)
    lse = oracle.row_lse(Q, K, Kla, shift=1)
    np.testing.assert_allclose(lse[0, 0, 0], scipy.special.logsumexp(K[0, 0, :, 0]), rtol=1e-13)


def test_closed_form_equal_keys():
    """Row j sees M + j keys when they are all equal, so its weights are 1/(M + j)."""
    rng = np.random.default_rng(3)
    N_rows, L, H, H_kv, M, d = 5, 2, 4, 2, 21, 8
    Q = rng.standard_normal((N_rows, L, H, d))
    v = rng.standard_normal(d)
    K = np.broadcast_to(v, (L, H_kv, M, d)).copy()
    Kla = np.broadcast_to(v, (L, H_kv, N_rows - 1, d)).copy()
    want = sum(1.0 / (M + j) for j in range(N_rows)) / N_rows
    np.testing.assert_allclose(oracle.importance(Q, K, Kla, shift=1), np.full(M, want), rtol=1e-12)


def test_rows_sum_to_one_and_see_the_right_lookahead_keys():
    rng = np.random.default_rng(9)
    N_rows, M, d = 4, 17, 8
    Q = rng.standard_normal((N_rows, 1, 2, d))
    K = rng.standard_normal((1, 1, M, d))
    Kla = rng.standard_normal((1, 1, N_rows - 1, d))
    for h in range(2):
        a, a_la = oracle.attention_rows(Q, K, Kla, 0, h, shift=1)
        np.testing.assert_allclose(a.sum(1) + a_la.sum(1), 1.0, atol=1e-12)
        assert np.all(a_la[0] == 0)                                  # the prefill row sees no look-ahead key
        for j in range(1, N_rows):
            assert np.all(a_la[j, :j] > 0) and np.all(a_la[j, j:] == 0)
    # the lse route agrees
    np.testing.assert_allclose(oracle.importance_given_lse(Q, K, oracle.row_lse(Q, K, Kla, shift=1)),
                               oracle.importance(Q, K, Kla, shift=1), rtol=1e-12)
