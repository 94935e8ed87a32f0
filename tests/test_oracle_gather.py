"""Pins of the sparse-prefill gather oracle: the paper review's worked example of
position ID recovery (tests/golden/position_ids_example.json), batch packing
and empty requests."""
import json
import os

import numpy as np

import oracle
from conftest import GOLDEN


def test_review_worked_example():
    ex = json.load(open(os.path.join(GOLDEN, "position_ids_example.json")))
    M = len(ex["original_position_ids"])
    token_ids = np.arange(M) * 7 + 100                      # any token IDs
    tokens, positions, cu_kept, next_pos = oracle.gather_kept(token_ids, [0, M], [ex["kept_position_ids"]])
    np.testing.assert_array_equal(positions, ex["kept_position_ids"])
    np.testing.assert_array_equal(tokens, [100 + 7 * p for p in ex["kept_position_ids"]])
    np.testing.assert_array_equal(cu_kept, [0, 5])
    decode = next_pos[0] + np.arange(len(ex["decode_position_ids"]))
    np.testing.assert_array_equal(decode, ex["decode_position_ids"])


def test_batch_packs_requests_in_order():
    cu = [0, 4, 4, 9]                                       # request 1 is empty
    token_ids = np.array([10, 11, 12, 13, 20, 21, 22, 23, 24])
    kept = [np.array([1, 3]), np.array([], dtype=np.int32), np.array([0, 2, 4])]
    tokens, positions, cu_kept, next_pos = oracle.gather_kept(token_ids, cu, kept)
    np.testing.assert_array_equal(tokens, [11, 13, 20, 22, 24])
    np.testing.assert_array_equal(positions, [1, 3, 0, 2, 4])
    np.testing.assert_array_equal(cu_kept, [0, 2, 2, 5])
    np.testing.assert_array_equal(next_pos, [4, 0, 5])
