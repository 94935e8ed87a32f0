"""Parity of sp_score_lse (single pass, each row's lse given) with the fp64
oracle, element by element.

The lse given to the kernel is the oracle's row_lse rounded to fp32, and the
oracle's importance_given_lse reads the same fp32 values.  The cases cover the
general path (fp32), the tensor-core path (bf16 8B shape) with 1 to 8 slab
classes, ragged tails, and N = 0.
"""
import functools

import numpy as np
import pytest

import oracle
import workloads as W
from gpu_helpers import check_importance, to_device, workload_inputs

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


def run_lse(sp, x, lse32):
    import torch
    Q, K = to_device(x.Q_la), to_device(x.K_prompt)
    imp = sp.score_lse(Q, K, torch.from_numpy(lse32).cuda(), check=True)
    torch.cuda.synchronize()
    return imp.cpu().numpy()


def check_case(sp, x, what):
    lse32 = oracle.row_lse(x.Q_la, x.K_prompt, x.K_la).astype(np.float32)
    got = run_lse(sp, x, lse32)
    ref = oracle.importance_given_lse(x.Q_la, x.K_prompt, lse32.astype(np.float64))
    check_importance(got, ref, x.wl.dtype, what)


@pytest.mark.parametrize("name", ["tiny-f32-512", "llama8b-bf16-8k"])
def test_workload_parity(sp, name):
    x = workload_inputs(name)
    check_case(sp, x, x.wl.name)


SHAPES = [
    # (L, H, H_kv, d, M, N, dtype)
    (1, 1, 1, 64, 1, 1, "bf16"),
    (2, 4, 2, 128, 129, 3, "bf16"),
    (3, 8, 8, 64, 300, 1, "bf16"),
    (1, 32, 4, 128, 4097, 8, "bf16"),
    (2, 6, 3, 72, 513, 5, "bf16"),         # general path (d = 72)
    (2, 32, 8, 128, 2500, 16, "bf16"),     # two tensor-core passes of 8 steps
    (1, 16, 2, 64, 900, 10, "bf16"),       # passes of 4, 4 and 2 steps
    (2, 40, 8, 128, 1200, 8, "bf16"),      # G = 5 padded to 8: two passes
    (1, 24, 8, 64, 1000, 6, "bf16"),       # G = 3 padded to 4
    (1, 16, 2, 256, 257, 4, "f32"),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "L{}H{}Hkv{}d{}M{}N{}{}".format(*s))
def test_random_shapes(sp, shape):
    L, H, H_kv, d, M, N, dt = shape
    wl = W.Workload("t", L=L, H=H, H_kv=H_kv, d=d, M=M, N=N, dtype=dt, chunk=16, pool_k=3, mode="topk",
                    keep_rate=0.3, needle_frac=0.05, run_min=2, run_max=8)
    check_case(sp, W.make_inputs(wl, seed=2000 + M), str(shape))


@pytest.mark.parametrize("M", [40960, 131072])
def test_long_prompts_few_layers(sp, M):
    wl = W.Workload("t", L=1, H=32, H_kv=8, d=128, M=M, N=8, dtype="bf16", chunk=64, pool_k=3, mode="topk",
                    keep_rate=0.1, needle_frac=0.01, run_min=16, run_max=128)
    check_case(sp, W.make_inputs(wl, seed=M + 1), f"M={M}")


def test_zero_lookahead_gives_ones(sp):
    import torch
    K = torch.randn(2, 2, 50, 64, device="cuda").to(torch.bfloat16)
    Q = torch.empty(0, 2, 4, 64, device="cuda", dtype=torch.bfloat16)
    lse = torch.empty(2, 4, 0, device="cuda")
    imp = sp.score_lse(Q, K, lse)
    torch.cuda.synchronize()
    assert torch.all(imp == 1.0)


def _lse_varlen_parity(sp, v, what):
    """sp_score_lse_varlen on a packed batch against the oracle prompt by prompt;
    returns the number of kernels the call launched."""
    import torch
    Q, K, _, cu = v.packed()
    lse32 = np.stack([oracle.row_lse(r.Q_la, r.K_prompt, r.K_la) for r in v.requests]).astype(np.float32)
    n0 = sp.sp_kernel_launches()
    got = sp.score_lse_varlen(to_device(Q), to_device(K), torch.from_numpy(lse32).cuda(), cu, check=True)
    torch.cuda.synchronize()
    launches = sp.sp_kernel_launches() - n0
    got = got.cpu().numpy()
    for b, r in enumerate(v.requests):
        if r.M:
            ref = oracle.importance_given_lse(r.Q_la, r.K_prompt, lse32[b].astype(np.float64))
            check_importance(got[cu[b]:cu[b + 1]], ref, v.wl.dtype, f"{what} req {b}")
    return launches


def test_varlen_v3_batch_parity(sp):
    """The 16-request 0.8B-shaped batch (2K to 32K tokens each) in one call."""
    _lse_varlen_parity(sp, workload_inputs("v3-batch16-0.8b-bf16"), "v3 batch")


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_varlen_ragged_with_empty_prompts(sp, dt):
    """Empty, one-token and ragged prompts; bf16 on the tensor-core path, fp32
    on the general path."""
    wl = W.Workload("t", L=2, H=8, H_kv=2, d=64, M=0, N=4, dtype=dt, chunk=16, pool_k=1, mode="mass",
                    mass=0.85, needle_frac=0.05, run_min=2, run_max=8)
    v = W.make_varlen_inputs(wl, 78, lengths=[300, 0, 1, 129, 1000, 0])
    _lse_varlen_parity(sp, v, f"ragged {dt}")


def test_varlen_more_prompts_than_one_wave_holds(sp):
    """40 short prompts: two waves of one preparation and one scoring launch each."""
    wl = W.Workload("t", L=2, H=8, H_kv=2, d=128, M=0, N=4, dtype="bf16", chunk=16, pool_k=1, mode="topk",
                    keep_rate=0.3, needle_frac=0.05, run_min=2, run_max=8)
    rng = np.random.default_rng(43)
    lengths = [int(m) if m > 20 else 0 for m in rng.integers(0, 400, size=40)]
    assert sum(1 for m in lengths if m) > 32
    v = W.make_varlen_inputs(wl, 44, lengths=lengths)
    assert _lse_varlen_parity(sp, v, "40 prompts") == 4


def test_varlen_one_prompt_equals_single_call(sp):
    """A batch of one prompt gives bit-identical importance to sp_score_lse."""
    import torch
    x = workload_inputs("llama8b-bf16-8k")
    lse = torch.from_numpy(oracle.row_lse(x.Q_la, x.K_prompt, x.K_la).astype(np.float32)).cuda()
    Q, K = to_device(x.Q_la), to_device(x.K_prompt)
    a = sp.score_lse(Q, K, lse)
    b = sp.score_lse_varlen(Q[None], K, lse[None], [0, x.wl.M])
    torch.cuda.synchronize()
    assert torch.equal(a, b)
