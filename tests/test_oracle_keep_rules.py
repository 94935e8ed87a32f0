"""Pins of the guide's v2 keep rules (oracle.keep_rules): hand-computed cases
for the always-kept tokens, the minimum-token back-fill, the keep-all rule and
the strided cap, and properties on random selections."""
import numpy as np
import pytest

import oracle


def chunk_mask(M, chunk, kept_chunks):
    nc = (M + chunk - 1) // chunk
    m = np.zeros(nc, dtype=bool)
    m[list(kept_chunks)] = True
    return m


def sel(M, chunk, kept_chunks):
    m = chunk_mask(M, chunk, kept_chunks)
    return oracle.kept_positions(m, chunk, M), m


def test_always_kept_tokens():
    kept, m = sel(20, 4, {2})                                   # tokens 8..11
    got = oracle.keep_rules(kept, m, 20, 4, min_tok=128, always_keep=True)
    np.testing.assert_array_equal(got, [0, 1, 2, 3, 8, 9, 10, 11, 18, 19])


def test_backfill_from_unselected_chunks_in_order():
    # M = 100, chunk 4: eff_min = min(128, max(4, 10)) = 10; chunk 7 gives 4 tokens
    kept, m = sel(100, 4, {7})
    got = oracle.keep_rules(kept, m, 100, 4, min_tok=128)
    np.testing.assert_array_equal(got, [0, 1, 2, 3, 4, 5, 28, 29, 30, 31])


def test_always_kept_then_backfill_skips_tokens_already_kept():
    # M = 200, chunk 8: eff_min = 20; chunk 10 (8 tokens) + 6 always-kept = 14 -> 6 more
    kept, m = sel(200, 8, {10})
    got = oracle.keep_rules(kept, m, 200, 8, min_tok=128, always_keep=True)
    np.testing.assert_array_equal(got, list(range(10)) + list(range(80, 88)) + [198, 199])


def test_short_prompt_keeps_everything():
    kept, m = sel(4, 2, {1})
    np.testing.assert_array_equal(oracle.keep_rules(kept, m, 4, 2, min_tok=128), [0, 1, 2, 3])
    kept, m = sel(40, 4, {0})                                   # eff_min = min(128, max(4, 4)) = 4 < 40
    np.testing.assert_array_equal(oracle.keep_rules(kept, m, 40, 4, min_tok=128), [0, 1, 2, 3])


@pytest.mark.parametrize("n,cap,want_idx", [(10, 4, [0, 2, 4, 9]), (7, 3, [0, 2, 6]), (9, 4, [0, 2, 4, 8]),
                                            (5, 5, [0, 1, 2, 3, 4]), (12, 1, [11])])
def test_strided_cap_keeps_the_last_token(n, cap, want_idx):
    kept = np.arange(n, dtype=np.int32) * 3
    m = np.ones(n, dtype=bool)
    got = oracle.keep_rules(kept, m, 3 * n, 3, max_keep=cap)
    np.testing.assert_array_equal(got, kept[want_idx])


def test_rules_off_change_nothing():
    kept, m = sel(64, 8, {1, 5})
    np.testing.assert_array_equal(oracle.keep_rules(kept, m, 64, 8), kept)


def test_properties_on_random_selections():
    rng = np.random.default_rng(4)
    for _ in range(200):
        M = int(rng.integers(1, 400))
        chunk = int(rng.integers(1, 40))
        nc = (M + chunk - 1) // chunk
        chosen = set(rng.choice(nc, size=int(rng.integers(1, nc + 1)), replace=False).tolist())
        kept, m = sel(M, chunk, chosen)
        min_tok = int(rng.integers(0, 200))
        got = oracle.keep_rules(kept, m, M, chunk, min_tok=min_tok, always_keep=True)
        assert np.all(np.diff(got) > 0) and got[0] >= 0 and got[-1] < M          # ascending, unique, in range
        assert set(kept.tolist()) <= set(got.tolist())                          # the selection stays
        for a in [0, 1, 2, 3] + ([M - 2, M - 1] if M > 4 else []):
            if a < M:
                assert a in set(got.tolist())
        eff_min = min(min_tok, max(4, M // 10)) if min_tok > 0 else 0
        assert len(got) >= min(eff_min, M)
