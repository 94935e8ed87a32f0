"""Selection parity: sp_select / sp_select_varlen through the C ABI against the
oracle's selection, bit for bit, on the same fp32 importance vector: the
oracle's importance rounded to fp32, seeded random values, and, for the whole
path on every workload, the importance the GPU computed."""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_helpers import check_importance, to_device, workload_inputs, workload_oracle

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


PIPELINE = ["tiny-f32-512", "llama8b-bf16-8k", "llama8b-bf16-32k", "llama8b-bf16-128k", "v3-batch16-0.8b-bf16"]


@pytest.mark.parametrize("name", PIPELINE)
def test_pipeline_selection_bit_exact_on_gpu_importance(sp, name):
    """The whole path on the GPU (sp_score -> sp_select, or the varlen pair for
    the v3 batch), checked twice: the GPU importance against the oracle's
    importance of the seeded inputs (within the importance tolerance), and the
    GPU's kept positions against the oracle's selection run on that same GPU
    importance vector (bit for bit, per request).  The oracle is only the
    checker of the selection step here; ties go to the lower chunk index on
    both sides."""
    import torch
    x = workload_inputs(name)
    wl = x.wl
    rate = wl.keep_rate if wl.mode == "topk" else wl.mass
    if hasattr(x, "requests"):
        Q, K, Kla, cu = x.packed()
        imp_dev = sp.score_varlen(to_device(Q), to_device(K), to_device(Kla), cu, check=True)
        kept = sp.select_varlen(imp_dev, cu, wl.chunk, wl.pool_k, wl.mode, rate, wl.boost)
        torch.cuda.synchronize()
        imp = imp_dev.cpu().numpy()
        refs = workload_oracle(name)
        for b in range(len(x.requests)):
            part = imp[cu[b]:cu[b + 1]]
            check_importance(part, refs[b], wl.dtype, f"{name} request {b}")
            want, n = oracle.select(part, wl.chunk, wl.pool_k, wl.mode, rate, wl.boost)
            got = kept[b].cpu().numpy()
            assert got.shape[0] == n and np.array_equal(got, want), (name, b, got[:16], want[:16])
        return
    Q, K, Kla = (to_device(getattr(x, n)) for n in ("Q_la", "K_prompt", "K_la"))
    imp_dev = sp.score(Q, K, Kla, check=True)
    kept = sp.select(imp_dev, wl.chunk, wl.pool_k, wl.mode, rate, wl.boost)
    torch.cuda.synchronize()
    imp = imp_dev.cpu().numpy()
    check_importance(imp, workload_oracle(name), wl.dtype, name)
    want, n = oracle.select(imp, wl.chunk, wl.pool_k, wl.mode, rate, wl.boost)
    got = kept.cpu().numpy()
    assert got.shape[0] == n and np.array_equal(got, want), (name, got[:16], want[:16])
    if wl.mode == "topk":
        # the kept count of the top-K rule: kc full chunks (no partial chunk at these sizes)
        nc = -(-wl.M // wl.chunk)
        assert n == oracle.keep_count(nc, wl.keep_rate) * wl.chunk


# ---------------------------------------------------------------------------
# Chunk sums, means and pooled scores themselves, bit for bit.  Plain fp32
# chunks of up to 64 values are summed exactly in integers when every partial
# sum of the left-to-right chain is an fp64 number, and by the chain otherwise;
# these inputs reach both, and the edges between them.  The test reads the
# three arrays from the selection workspace: after the 256-byte status header,
# the per-prompt normalisation coefficients, then sums[nc], means[nc] and
# pooled[nc], each block aligned to 256 bytes.
# ---------------------------------------------------------------------------

def _ws_arrays(ws, nc, B=1):
    al = lambda x: (x + 255) // 256 * 256
    off = al(256 + 32 * max(B, 1))
    raw = ws.cpu().numpy()
    out = []
    for _ in range(3):
        out.append(raw[off: off + 8 * nc].view(np.float64).copy())
        off = al(off + 8 * nc)
    return out                                            # sums, means, pooled


def _edge53(M, chunk, rng):
    """Chunks whose exact total sits just below or just above 2^53 units of the
    smallest value's last place: one value 2^(q+23) and two or three values
    (2^24 - 1) * 2^(q+28), the rest zero."""
    x = np.zeros(M, dtype=np.float32)
    for c in range(M // chunk):
        q = int(rng.integers(-60, -30))
        big = np.float32(np.ldexp(float((1 << 24) - 1), q + 28))
        x[c * chunk] = np.float32(np.ldexp(1.0, q + 23))
        nbig = 2 + (c % 2)
        for t in range(nbig):
            x[c * chunk + 1 + t] = big
        rng.shuffle(x[c * chunk: (c + 1) * chunk])
    return x


def _chunk_inputs(kind, M, chunk, seed):
    rng = np.random.default_rng(seed)
    if kind == "narrow":        # within 2^10 of each other: the exact path
        return rng.uniform(1e-3, 1.0, M).astype(np.float32)
    if kind == "wide":          # log-uniform over 2^-100 .. 1: mostly the chain
        return np.exp2(rng.uniform(-100, 0, M)).astype(np.float32)
    if kind == "subnormal":     # fp32 subnormals beside small normals, some zeros
        x = (rng.integers(0, 1 << 23, M).astype(np.uint32)).view(np.float32).copy()
        x[rng.random(M) < 0.3] = np.float32(2.0 ** -120)
        x[rng.random(M) < 0.2] = 0.0
        return x
    if kind == "zeros":         # whole chunks of zeros and scattered zeros
        x = rng.uniform(0.0, 1.0, M).astype(np.float32)
        x[rng.random(M) < 0.5] = 0.0
        x[: 3 * chunk] = 0.0
        return x
    if kind == "signed":        # negative values and a negative zero: the chain
        x = rng.normal(0.0, 1.0, M).astype(np.float32)
        x[min(5, M - 1)] = np.float32(-0.0)
        return x
    if kind == "edge53":
        return _edge53(M, chunk, rng)
    raise ValueError(kind)


CHUNK_CASES = [
    # (kind, M, chunk, pool_k)
    ("narrow", 32 * 300, 32, 3),
    ("narrow", 64 * 200 + 17, 64, 3),
    ("narrow", 48 * 100 + 5, 48, 5),
    ("narrow", 17 * 99, 17, 7),
    ("narrow", 65 * 50 + 3, 65, 3),
    ("narrow", 1000, 1, 3),
    ("wide", 32 * 300 + 9, 32, 3),
    ("wide", 64 * 100, 64, 1),
    ("subnormal", 32 * 200, 32, 3),
    ("subnormal", 64 * 100 + 33, 64, 5),
    ("zeros", 32 * 100, 32, 3),
    ("signed", 32 * 100 + 1, 32, 3),
    ("signed", 64 * 60, 64, 3),
    ("edge53", 32 * 200, 32, 3),
    ("edge53", 64 * 100, 64, 3),
]


@pytest.mark.parametrize("case", CHUNK_CASES, ids=lambda c: f"{c[0]}-M{c[1]}c{c[2]}k{c[3]}")
def test_chunk_sums_means_pooled_bit_exact(sp, case):
    import torch
    kind, M, chunk, pool_k = case
    imp = _chunk_inputs(kind, M, chunk, seed=M + chunk)
    ws = torch.zeros(sp.sp_select_workspace_size(M, chunk), dtype=torch.uint8, device="cuda")
    sp.select(torch.from_numpy(imp).cuda(), chunk, pool_k, "topk", 0.3, ws=ws)
    torch.cuda.synchronize()
    nc = (M + chunk - 1) // chunk
    sums, means, pooled = _ws_arrays(ws, nc)
    want_sums, _ = oracle.chunk_sums(imp, chunk)
    want_means = oracle.chunk_means(imp, chunk)
    assert np.array_equal(sums.view(np.uint64), want_sums.view(np.uint64)), kind
    assert np.array_equal(means.view(np.uint64), want_means.view(np.uint64)), kind
    if pool_k > 1:
        want_pooled = oracle.avg_pool(want_means, pool_k)
        assert np.array_equal(pooled.view(np.uint64), want_pooled.view(np.uint64)), kind


# ---------------------------------------------------------------------------
# Cumulative-mass cut.  The kernel decides R_k >= target from parallel sums
# with an error margin and runs the two serial fp64 chains of the definition
# only when the margin does not decide; these inputs reach both: exact ties
# between the running mass and the target, a target reached only at the last
# chunk (tau = 1), all-zero and negative chunk sums, and ordinary prompts.
# ---------------------------------------------------------------------------

MASS_CASES = [
    # (kind, M, chunk, tau, boost)
    ("zeros", 3000, 32, 0.85, None),
    ("constant", 3200, 32, 0.5, None),
    ("constant", 3200, 32, 0.85, None),
    ("constant", 640, 32, 1.0, None),
    ("dyadic", 8000, 16, 0.75, None),
    ("negative", 5000, 32, 0.85, (0, 1.0, 0, 1.0, 0)),
    ("random", 20000, 32, 1.0, W.V3_BOOST),
    ("random", 200000, 16, 0.85, W.V3_BOOST),
    ("random", 30000, 32, 0.3, (64, 1.5, 128, 1.3, 0)),
]


def _mass_inputs(kind, M, seed):
    rng = np.random.default_rng(seed)
    if kind == "zeros":
        return np.zeros(M, dtype=np.float32)
    if kind == "constant":
        return np.full(M, 0.125, dtype=np.float32)
    if kind == "dyadic":
        return (rng.integers(0, 4, M) * 0.25).astype(np.float32)
    if kind == "negative":
        return rng.normal(0.0, 1.0, M).astype(np.float32)
    return (rng.random(M) * 1e-3).astype(np.float32)


@pytest.mark.parametrize("case", MASS_CASES, ids=lambda c: f"{c[0]}-M{c[1]}c{c[2]}t{c[3]}")
def test_mass_cut_bit_exact(sp, case):
    kind, M, chunk, tau, boost = case
    imp = _mass_inputs(kind, M, seed=M + chunk)
    assert_same(sp, imp, chunk, 1, "mass", tau, boost)


def test_many_prompts_varlen_bit_exact(sp):
    """A batch of 200 prompts (some empty): the selection kernels look prompts
    up in offset tables staged in shared memory; both modes against the oracle."""
    import torch
    rng = np.random.default_rng(11)
    lens = rng.integers(0, 3000, 200)
    lens[::17] = 0
    cu = np.concatenate([[0], np.cumsum(lens)])
    imp = (rng.random(int(cu[-1])) * 1e-3).astype(np.float32)
    for chunk, mode, rate, pool, boost in ((32, "topk", 0.2, 3, None), (16, "topk", 0.3, 5, W.V3_BOOST),
                                           (32, "mass", 0.85, 1, W.V3_BOOST), (64, "mass", 0.6, 1, None)):
        got = sp.select_varlen(torch.from_numpy(imp).cuda(), cu, chunk, pool, mode, rate, boost)
        torch.cuda.synchronize()
        want = oracle.select_varlen(imp, cu, chunk, pool, mode, rate, boost)
        for b in range(len(lens)):
            assert np.array_equal(got[b].cpu().numpy(), want[b][0]), (mode, chunk, b)
