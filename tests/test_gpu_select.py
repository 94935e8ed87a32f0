"""Selection parity: sp_select / sp_select_varlen through the C ABI against the
oracle's selection, bit for bit, on the same fp32 importance vector (taken
from the oracle's scoring or from the seeded generator, never from the GPU),
plus end-to-end checks of the GPU pipeline on every workload."""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_helpers import to_device, workload_inputs, workload_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sp():
    import torch
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    from speculative_prefill_token_sp_gb300 import build
    build.build()
    import speculative_prefill_token_sp_gb300 as m
    m.lib()
    return m


def gpu_select(sp, imp: np.ndarray, chunk, pool_k, mode, rate, boost=None):
    import torch
    out = sp.select(torch.from_numpy(np.ascontiguousarray(imp, dtype=np.float32)).cuda(), chunk, pool_k, mode,
                    rate, boost)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def assert_same(sp, imp, chunk, pool_k, mode, rate, boost=None):
    got = gpu_select(sp, imp, chunk, pool_k, mode, rate, boost)
    want, n = oracle.select(imp, chunk, pool_k, mode, rate, boost)
    assert got.shape[0] == n and np.array_equal(got, want), (chunk, pool_k, mode, rate, got[:20], want[:20])


@pytest.mark.parametrize("name", ["tiny-f32-512", "llama8b-bf16-8k", "llama8b-bf16-32k", "llama8b-bf16-128k"])
def test_workload_selection_bit_exact(sp, name):
    """Oracle importance (rounded to fp32) -> GPU selection == oracle selection."""
    x = workload_inputs(name)
    wl = x.wl
    imp = workload_oracle(name).astype(np.float32)
    assert_same(sp, imp, wl.chunk, wl.pool_k, wl.mode, wl.keep_rate)


def test_v3_batch_selection_bit_exact(sp):
    import torch
    v = workload_inputs("v3-batch16-0.8b-bf16")
    wl = v.wl
    imps = [r.astype(np.float32) for r in workload_oracle("v3-batch16-0.8b-bf16")]
    packed = np.concatenate(imps)
    got = sp.select_varlen(torch.from_numpy(packed).cuda(), v.cu_M, wl.chunk, wl.pool_k, wl.mode, wl.mass,
                           wl.boost)
    torch.cuda.synchronize()
    for b, imp in enumerate(imps):
        want, n = oracle.select(imp, wl.chunk, wl.pool_k, wl.mode, wl.mass, wl.boost)
        assert np.array_equal(got[b].cpu().numpy(), want), b


RANDOM_CASES = [
    # (M, chunk, pool_k, mode, rate, boost, quantise)
    (1, 32, 3, "topk", 0.3, None, 0),
    (10, 1, 1, "topk", 0.5, None, 0),
    (31, 32, 3, "topk", 0.3, None, 0),
    (70, 32, 3, "topk", 0.5, None, 0),
    (1000, 7, 5, "topk", 0.25, None, 4),
    (4096, 16, 3, "topk", 0.1, None, 2),
    (5000, 1, 9, "topk", 0.05, None, 3),
    (65537, 32, 3, "topk", 0.1, None, 0),
    (300000, 64, 3, "topk", 0.2, None, 5),
    (9, 4, 1, "mass", 0.85, None, 0),
    (150, 32, 1, "mass", 0.85, W.V3_BOOST, 0),
    (2000, 32, 1, "mass", 0.5, (64, 1.5, 128, 1.3, 0), 3),
    (20000, 32, 1, "mass", 0.85, W.V3_BOOST, 0),
    (32768, 2, 1, "mass", 0.99, W.V3_BOOST, 2),
    (5000, 10, 1, "mass", 1.0, None, 0),
    (3000, 16, 3, "topk", 0.4, W.V3_BOOST, 0),
    (5000, 1, 101, "topk", 0.1, None, 2),      # wide pool window: 50 chunks of halo per block
    (3000, 1, 501, "topk", 0.2, None, 0),      # a halo beyond the fused kernel's: the separate pool pass
]


@pytest.mark.parametrize("case", RANDOM_CASES, ids=lambda c: f"M{c[0]}c{c[1]}k{c[2]}{c[3]}{c[4]}q{c[6]}")
def test_random_selection_bit_exact(sp, case):
    M, chunk, pool_k, mode, rate, boost, q = case
    rng = np.random.default_rng(M * 7 + chunk)
    imp = rng.random(M).astype(np.float32) * 1e-3
    if q:                                      # few distinct values -> many exact ties
        imp = (np.floor(imp * 1e3 * q) / q).astype(np.float32)
    assert_same(sp, imp, chunk, pool_k, mode, rate, boost)


def test_constant_importance_keeps_first_chunks(sp):
    imp = np.full(1000, 0.125, dtype=np.float32)
    assert_same(sp, imp, 32, 3, "topk", 0.3)
    assert_same(sp, imp, 32, 1, "mass", 0.85, W.V3_BOOST)


def test_empty_and_varlen_edges(sp):
    import torch
    rng = np.random.default_rng(5)
    lens = [0, 1, 33, 0, 500, 64]
    cu = np.concatenate([[0], np.cumsum(lens)])
    imp = rng.random(int(cu[-1])).astype(np.float32)
    for mode, rate, pool, boost in (("topk", 0.3, 3, None), ("mass", 0.7, 1, W.V3_BOOST)):
        got = sp.select_varlen(torch.from_numpy(imp).cuda(), cu, 16, pool, mode, rate, boost)
        torch.cuda.synchronize()
        want = oracle.select_varlen(imp, cu, 16, pool, mode, rate, boost)
        for b in range(len(lens)):
            assert np.array_equal(got[b].cpu().numpy(), want[b][0]), (mode, b)


@pytest.mark.parametrize("name", ["tiny-f32-512", "llama8b-bf16-8k", "llama8b-bf16-32k"])
def test_end_to_end_pipeline(sp, name):
    """GPU importance -> GPU selection: the count follows the kc rule exactly and
    every disagreement with the oracle's selection is a near-tie."""
    import torch
    x = workload_inputs(name)
    wl = x.wl
    Q, K, Kla = (to_device(getattr(x, n)) for n in ("Q_la", "K_prompt", "K_la"))
    imp_gpu = sp.score(Q, K, Kla)
    kept = sp.select(imp_gpu, wl.chunk, wl.pool_k, wl.mode, wl.keep_rate)
    torch.cuda.synchronize()
    kept = kept.cpu().numpy()
    ref_imp = workload_oracle(name)
    want, n = oracle.select(ref_imp.astype(np.float32), wl.chunk, wl.pool_k, wl.mode, wl.keep_rate)
    assert kept.shape[0] == n                   # same kc, and all chunks are full here
    assert np.all(np.diff(kept) > 0)
    means = oracle.chunk_means(ref_imp, wl.chunk)
    pooled = oracle.avg_pool(means, wl.pool_k)
    kc = oracle.keep_count(len(means), wl.keep_rate)
    thr = np.sort(pooled)[::-1][kc - 1]
    got_c = set((kept // wl.chunk).tolist())
    want_c = set((want // wl.chunk).tolist())
    for c in got_c ^ want_c:
        assert abs(pooled[c] - thr) <= 1e-2 * thr, (c, pooled[c], thr)
