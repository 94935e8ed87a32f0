"""Pins of the selection oracle: the worked position-ID example, keep-count
closed forms, hand-computed chunk means and pools, brute force over all
subsets, and the cumulative-mass special cases."""
import itertools
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from conftest import GOLDEN


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_position_id_example():
    ex = _load("position_ids_example.json")
    M = len(ex["original_position_ids"])
    imp = np.full(M, 0.1, dtype=np.float32)
    for rank, p in enumerate(ex["kept_position_ids"]):
        imp[p] = 0.9 - 0.1 * rank
    pos, n = oracle.select(imp, ex["chunk"], ex["pool_k"], "topk", ex["keep_rate"])
    assert pos.tolist() == ex["kept_position_ids"] and n == 5
    assert list(range(M, M + len(ex["decode_position_ids"]))) == ex["decode_position_ids"]


@pytest.mark.parametrize("case", _load("keep_counts.json")["cases"], ids=lambda c: c["workload"])
def test_keep_counts(case):
    nc = (case["M"] + case["chunk"] - 1) // case["chunk"]
    assert nc == case["nc"]
    assert oracle.keep_count(nc, case["keep_rate"]) == case["kc"]
    rng = np.random.default_rng(case["M"])
    imp = rng.random(case["M"]).astype(np.float32)
    pos, n = oracle.select(imp, case["chunk"], 3, "topk", case["keep_rate"])
    last = case["M"] - (nc - 1) * case["chunk"]
    last_kept = bool(np.any(pos >= (nc - 1) * case["chunk"]))
    assert n == case["n_kept_if_last_chunk_full"] - (case["chunk"] - last if last_kept else 0)
    assert np.all(np.diff(pos) > 0)


def test_pool_and_chunk_means_hand():
    g = _load("selection_hand_cases.json")
    for c in g["pool"]:
        got = oracle.avg_pool(np.array(c["values"], dtype=np.float64), c["k"])
        np.testing.assert_array_equal(got, [float(Fraction(v)) for v in c["expected"]])
    for c in g["chunk_means"]:
        x = np.array(eval(f"[{c['scores']}]"), dtype=np.float64)   # noqa: S307 (fixture text)
        got = oracle.chunk_means(x, c["chunk"])
        np.testing.assert_array_equal(got, [float(Fraction(v)) for v in c["expected"]])


def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(41)
    for trial in range(60):
        nc = int(rng.integers(1, 11))
        p = rng.integers(0, 4, size=nc).astype(np.float64) / 4.0     # many exact ties
        for kc in range(1, nc + 1):
            mask = oracle.topk_chunks(p, kc)
            got = tuple(np.flatnonzero(mask))
            best = None
            for sub in itertools.combinations(range(nc), kc):
                key = (sum(Fraction(p[c]) for c in sub), tuple(-c for c in sub))
                if best is None or key > best[0]:
                    best = (key, sub)
            assert got == best[1], (p, kc, got, best)


def test_ties_go_to_lower_chunks():
    imp = np.full(320, 0.5, dtype=np.float32)
    pos, n = oracle.select(imp, 32, 3, "topk", 0.3)
    assert n == 3 * 32 and pos.tolist() == list(range(96))


def test_empty_prompt():
    pos, n = oracle.select(np.zeros(0, np.float32), 32, 3, "topk", 0.3)
    assert n == 0 and pos.size == 0
    pos, n = oracle.select(np.zeros(0, np.float32), 32, 1, "mass", 0.85, (64, 1.5, 128, 1.3, 1))
    assert n == 0


def test_mass_special_cases():
    rng = np.random.default_rng(43)
    imp = rng.random(1000).astype(np.float32)
    pos, n = oracle.select(imp, 32, 1, "mass", 1.0)
    assert n == 1000                                   # tau = 1 keeps every chunk
    imp2 = np.full(320, 1e-3, dtype=np.float32)
    imp2[64:96] = 1.0                                  # one chunk holds > 85% of the mass
    pos, n = oracle.select(imp2, 32, 1, "mass", 0.85)
    assert pos.tolist() == list(range(64, 96))


def test_mass_brute_force_minimal_cardinality():
    """Equal-size chunks and exact integer mass: the kept prefix is a smallest set reaching tau."""
    rng = np.random.default_rng(47)
    for trial in range(80):
        nc = int(rng.integers(1, 9))
        chunk = 4
        x = rng.integers(0, 6, size=nc * chunk).astype(np.float32)
        tau = float(rng.choice([0.25, 0.5, 0.75, 0.85, 1.0]))
        pos, n = oracle.select(x, chunk, 1, "mass", tau)
        sums = [Fraction(int(x[c * chunk:(c + 1) * chunk].sum())) for c in range(nc)]
        target = Fraction(tau) * sum(sums)
        kept = sorted(set(int(p) // chunk for p in pos))
        assert sum(sums[c] for c in kept) >= target
        k_min = next(k for k in range(0, nc + 1)
                     if any(sum(sums[c] for c in sub) >= target
                            for sub in itertools.combinations(range(nc), k)))
        assert len(kept) == max(1, k_min), (x, tau, kept, k_min)


def test_normalize_and_boost():
    imp = np.full(150, 0.25, dtype=np.float32)          # max == min -> all 1.0
    x = oracle.normalize_boost(imp, (64, 1.5, 128, 1.3, 1))
    want = np.ones(150)
    want[:64] *= 1.5
    want[150 - 128:] *= 1.3                              # positions 22..63 get both
    np.testing.assert_array_equal(x, want)
    rng = np.random.default_rng(53)
    imp = rng.random(500).astype(np.float32)
    x = oracle.normalize_boost(imp, (0, 1.0, 0, 1.0, 1))
    assert x.min() == 0.0 and x.max() == 1.0
    assert x[np.argmin(imp)] == 0.0 and x[np.argmax(imp)] == 1.0
    x = oracle.normalize_boost(imp, (64, 1.5, 128, 1.3, 0))   # no normalisation
    np.testing.assert_array_equal(x[64:372], imp[64:372].astype(np.float64))


def test_varlen_is_per_request():
    rng = np.random.default_rng(59)
    lens = [100, 0, 37, 64]
    cu = np.concatenate([[0], np.cumsum(lens)])
    imp = rng.random(int(cu[-1])).astype(np.float32)
    res = oracle.select_varlen(imp, cu, 16, 3, "topk", 0.3)
    for b, (pos, n) in enumerate(res):
        p2, n2 = oracle.select(imp[cu[b]:cu[b + 1]], 16, 3, "topk", 0.3)
        assert n == n2 and np.array_equal(pos, p2)
        assert pos.size == 0 or pos.max() < lens[b]


def test_varlen_hand_case():
    """Two requests packed back to back, worked by hand (the guide's per-request
    selection; positions are each request's own, from 0).  Request 0: scores
    [0.9, 0.1, 0.1, 0.8], chunk 1, no pool, keep 0.5 -> kc = ceil(4 * 0.5) = 2:
    chunks 0 and 3.  Request 1: [0.2, 0.7] -> kc = 1: chunk 1.  Mass mode,
    tau = 0.5: request 0's total 1.9, ranked 0.9 (0.9 < 0.95), then 0.8 (1.7):
    chunks 0 and 3; request 1's total 0.9, ranked 0.7 >= 0.45: chunk 1."""
    imp = np.array([0.9, 0.1, 0.1, 0.8, 0.2, 0.7], dtype=np.float32)
    cu = [0, 4, 6]
    res = oracle.select_varlen(imp, cu, 1, 1, "topk", 0.5)
    assert [list(p) for p, _ in res] == [[0, 3], [1]] and [n for _, n in res] == [2, 1]
    res = oracle.select_varlen(imp, cu, 1, 1, "mass", 0.5)
    assert [list(p) for p, _ in res] == [[0, 3], [1]]
