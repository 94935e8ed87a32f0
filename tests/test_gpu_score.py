"""Scoring parity: sp_score / sp_score_varlen through the C ABI against the fp64
oracle, element by element, on the seeded workloads (all five at full size)
and on random shapes with ragged tails and edge cases."""
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


def run_score(sp, x):
    import torch
    Q, K, Kla = (to_device(getattr(x, n)) for n in ("Q_la", "K_prompt", "K_la"))
    imp = sp.score(Q, K, Kla, check=True)
    torch.cuda.synchronize()
    return imp.cpu().numpy()


@pytest.mark.parametrize("name", ["tiny-f32-512", "llama8b-bf16-8k", "llama8b-bf16-32k", "llama8b-bf16-128k"])
def test_workload_parity(sp, name):
    x = workload_inputs(name)
    got = run_score(sp, x)
    ref = workload_oracle(name)
    check_importance(got, ref, x.wl.dtype, x.wl.name)


def test_tensor_core_path_serves_the_8b_workloads(sp):
    """The 8B-shaped bf16 prompts run on the tcgen05 path: one preparation
    kernel plus one persistent kernel per call (the general path launches 4)."""
    import torch
    x = workload_inputs("llama8b-bf16-8k")
    Q, K, Kla = (to_device(getattr(x, n)) for n in ("Q_la", "K_prompt", "K_la"))
    n0 = sp.sp_kernel_launches()
    sp.score(Q, K, Kla)
    torch.cuda.synchronize()
    assert sp.sp_kernel_launches() - n0 == 2


def test_varlen_v3_batch_parity(sp):
    import torch
    v = workload_inputs("v3-batch16-0.8b-bf16")
    Q, K, Kla, cu = v.packed()
    got = sp.score_varlen(to_device(Q), to_device(K), to_device(Kla), cu, check=True)
    torch.cuda.synchronize()
    got = got.cpu().numpy()
    refs = workload_oracle("v3-batch16-0.8b-bf16")
    for b, r in enumerate(v.requests):
        ref = refs[b]
        check_importance(got[cu[b]:cu[b + 1]], ref, v.wl.dtype, f"{v.wl.name} request {b}")


SHAPES = [
    # (L, H, H_kv, d, M, N, dtype)
    (1, 1, 1, 64, 1, 1, "bf16"),
    (1, 2, 1, 64, 7, 2, "f32"),
    (2, 4, 2, 128, 129, 3, "bf16"),
    (3, 8, 8, 64, 300, 1, "bf16"),
    (2, 8, 1, 128, 1000, 8, "bf16"),
    (1, 16, 2, 256, 257, 4, "f32"),
    (2, 6, 3, 72, 513, 5, "bf16"),
    (1, 32, 4, 128, 4097, 8, "bf16"),
    (2, 4, 4, 8, 77, 16, "f32"),
    (1, 64, 1, 64, 200, 4, "bf16"),
    # more query rows than one tensor-core pass takes (N * G > 32): passes of 32 / G steps
    (2, 32, 8, 128, 3000, 16, "bf16"),       # two passes of 8 steps
    (1, 16, 2, 64, 1500, 12, "bf16"),        # three passes of 4 steps
    (2, 8, 8, 64, 700, 48, "bf16"),          # G = 1: passes of 32 and 16 steps
    (1, 8, 4, 128, 5000, 30, "bf16"),        # G = 2: passes of 16 and 14 steps
    # query heads per KV head that are not a power of two: each step's rows padded to 4, 8 or 16
    (2, 24, 8, 128, 2000, 8, "bf16"),        # G = 3 (padded to 4): one pass
    (1, 40, 8, 128, 3000, 8, "bf16"),        # G = 5 (padded to 8): two passes
    (1, 28, 4, 128, 1500, 8, "bf16"),        # G = 7 (padded to 8): two passes
    (2, 12, 2, 64, 900, 3, "bf16"),          # G = 6 (padded to 8), d = 64
    (1, 128, 8, 128, 1000, 2, "bf16"),       # G = 16: one pass of 2 steps
    (1, 48, 4, 64, 700, 5, "bf16"),          # G = 12 (padded to 16): three passes
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "L{}H{}Hkv{}d{}M{}N{}{}".format(*s))
def test_random_shapes(sp, shape):
    L, H, H_kv, d, M, N, dt = shape
    wl = W.Workload("t", L=L, H=H, H_kv=H_kv, d=d, M=M, N=N, dtype=dt, chunk=16, pool_k=3, mode="topk",
                    keep_rate=0.3, needle_frac=0.05, run_min=2, run_max=8)
    x = W.make_inputs(wl, seed=1000 + M)
    got = run_score(sp, x)
    ref = oracle.importance(x.Q_la, x.K_prompt, x.K_la)
    check_importance(got, ref, dt, str(shape))


@pytest.mark.parametrize("M", [40960, 65536, 98305, 131072, 200000, 270000])
def test_long_prompts_few_layers(sp, M):
    """3 to 14 tiles of 128 tokens per CTA per slab and short look-behind (lag)
    windows (one held slab beyond about 155K tokens), on one layer of the 8B
    shape so that the oracle stays cheap; every length stays on the
    tensor-core path (one preparation and one scoring launch)."""
    wl = W.Workload("t", L=1, H=32, H_kv=8, d=128, M=M, N=8, dtype="bf16", chunk=64, pool_k=3, mode="topk",
                    keep_rate=0.1, needle_frac=0.01, run_min=16, run_max=128)
    x = W.make_inputs(wl, seed=M)
    n0 = sp.sp_kernel_launches()
    got = run_score(sp, x)
    assert sp.sp_kernel_launches() - n0 == 2
    check_importance(got, oracle.importance(x.Q_la, x.K_prompt, x.K_la), "bf16", f"M={M}")


@pytest.mark.parametrize("H,H_kv,passes", [(24, 8, 1), (40, 8, 2), (28, 4, 2), (128, 8, 4)])
def test_unpadded_group_sizes_run_on_tensor_cores(sp, H, H_kv, passes):
    """G = 3, 5, 7, 16 at d = 128 with N = 8: one preparation and one scoring
    launch per pass of 32 / G_padded steps (the general path launches 4 kernels once)."""
    import torch
    wl = W.Workload("t", L=2, H=H, H_kv=H_kv, d=128, M=2000, N=8, dtype="bf16", chunk=32, pool_k=3, mode="topk",
                    keep_rate=0.1, needle_frac=0.02, run_min=16, run_max=128)
    x = W.make_inputs(wl, seed=H * 10 + H_kv)
    Q, K, Kla = (to_device(getattr(x, n)) for n in ("Q_la", "K_prompt", "K_la"))
    n0 = sp.sp_kernel_launches()
    imp = sp.score(Q, K, Kla, check=True)
    torch.cuda.synchronize()
    assert sp.sp_kernel_launches() - n0 == 2 * passes
    check_importance(imp.cpu().numpy(), oracle.importance(x.Q_la, x.K_prompt, x.K_la), "bf16", f"H={H} H_kv={H_kv}")


def test_more_steps_than_one_pass_runs_on_tensor_cores(sp):
    """N = 16 look-ahead steps at the 8B head shape (64 query rows per KV head):
    two tensor-core passes of 8 steps, each one preparation and one scoring
    launch (the general path would launch 4 kernels once)."""
    import torch
    wl = W.Workload("t", L=2, H=32, H_kv=8, d=128, M=9000, N=16, dtype="bf16", chunk=32, pool_k=3, mode="topk",
                    keep_rate=0.1, needle_frac=0.02, run_min=16, run_max=128)
    x = W.make_inputs(wl, seed=16)
    Q, K, Kla = (to_device(getattr(x, n)) for n in ("Q_la", "K_prompt", "K_la"))
    n0 = sp.sp_kernel_launches()
    imp = sp.score(Q, K, Kla, check=True)
    torch.cuda.synchronize()
    assert sp.sp_kernel_launches() - n0 == 4
    check_importance(imp.cpu().numpy(), oracle.importance(x.Q_la, x.K_prompt, x.K_la), "bf16", "N=16")


def test_varlen_more_steps_than_one_pass(sp):
    """A ragged batch with N * G = 48 rows: every wave runs twice (steps 0-7, 8-11)."""
    import torch
    wl = W.Workload("t", L=2, H=16, H_kv=4, d=64, M=0, N=12, dtype="bf16", chunk=32, pool_k=1, mode="mass",
                    mass=0.85, needle_frac=0.05, run_min=8, run_max=64)
    v = W.make_varlen_inputs(wl, 48, lengths=[3000, 0, 700, 5000, 64])
    Q, K, Kla, cu = v.packed()
    got = sp.score_varlen(to_device(Q), to_device(K), to_device(Kla), cu, check=True)
    torch.cuda.synchronize()
    got = got.cpu().numpy()
    for b, r in enumerate(v.requests):
        if r.M:
            check_importance(got[cu[b]:cu[b + 1]], oracle.importance(r.Q_la, r.K_prompt, r.K_la), "bf16", f"req {b}")


def test_varlen_ragged_with_empty_prompts(sp):
    import torch
    wl = W.Workload("t", L=2, H=8, H_kv=2, d=64, M=0, N=4, dtype="bf16", chunk=16, pool_k=1, mode="mass",
                    mass=0.85, needle_frac=0.05, run_min=2, run_max=8)
    v = W.make_varlen_inputs(wl, 77, lengths=[300, 0, 1, 129, 1000, 0])
    Q, K, Kla, cu = v.packed()
    got = sp.score_varlen(to_device(Q), to_device(K), to_device(Kla), cu)
    torch.cuda.synchronize()
    got = got.cpu().numpy()
    for b, r in enumerate(v.requests):
        if r.M:
            check_importance(got[cu[b]:cu[b + 1]], oracle.importance(r.Q_la, r.K_prompt, r.K_la), "bf16", f"req {b}")


def _varlen_parity(sp, v, what):
    import torch
    Q, K, Kla, cu = v.packed()
    n0 = sp.sp_kernel_launches()
    got = sp.score_varlen(to_device(Q), to_device(K), to_device(Kla), cu, check=True)
    torch.cuda.synchronize()
    launches = sp.sp_kernel_launches() - n0
    got = got.cpu().numpy()
    for b, r in enumerate(v.requests):
        if r.M:
            check_importance(got[cu[b]:cu[b + 1]], oracle.importance(r.Q_la, r.K_prompt, r.K_la), "bf16",
                             f"{what} req {b}")
    return launches


def test_varlen_more_prompts_than_one_wave_holds(sp):
    """40 short prompts (some empty): a wave takes at most 32 prompts, so the
    batch runs as two waves of one preparation and one scoring launch each.
    N*G = 16 < 32 rows also takes P2's bounds-checked path."""
    wl = W.Workload("t", L=2, H=8, H_kv=2, d=64, M=0, N=4, dtype="bf16", chunk=16, pool_k=1, mode="topk",
                    keep_rate=0.3, needle_frac=0.05, run_min=2, run_max=8)
    rng = np.random.default_rng(40)
    lengths = [int(m) if m > 20 else 0 for m in rng.integers(0, 400, size=40)]
    assert sum(1 for m in lengths if m) > 32
    v = W.make_varlen_inputs(wl, 41, lengths=lengths)
    assert _varlen_parity(sp, v, "40 prompts") == 4


def test_varlen_prompts_split_over_waves(sp):
    """A 120K-token prompt needs 118 of the SMs at 8 tiles per CTA and slab, so
    the 40K-token one after it starts a second wave (with the 5-token one)."""
    wl = W.Workload("t", L=1, H=4, H_kv=1, d=64, M=0, N=2, dtype="bf16", chunk=64, pool_k=3, mode="topk",
                    keep_rate=0.1, needle_frac=0.01, run_min=16, run_max=128)
    v = W.make_varlen_inputs(wl, 42, lengths=[120000, 40000, 5])
    assert _varlen_parity(sp, v, "two waves") == 4


def test_zero_lookahead_gives_ones_and_empty_prompt_is_noop(sp):
    import torch
    K = torch.randn(2, 2, 50, 64, device="cuda").to(torch.bfloat16)
    Q = torch.empty(0, 2, 4, 64, device="cuda", dtype=torch.bfloat16)
    Kla = torch.empty(2, 2, 0, 64, device="cuda", dtype=torch.bfloat16)
    imp = sp.score(Q, K, Kla)
    torch.cuda.synchronize()
    assert torch.all(imp == 1.0)
    K0 = torch.empty(2, 2, 0, 64, device="cuda", dtype=torch.bfloat16)
    Q1 = torch.randn(3, 2, 4, 64, device="cuda").to(torch.bfloat16)
    Kla1 = torch.randn(2, 2, 3, 64, device="cuda").to(torch.bfloat16)
    imp = sp.score(Q1, K0, Kla1)
    torch.cuda.synchronize()
    assert imp.numel() == 0


def test_workspace_status_ok_after_call(sp):
    import torch
    x = W.make_workload_inputs("tiny-f32-512")
    Q, K, Kla = (to_device(getattr(x, n)) for n in ("Q_la", "K_prompt", "K_la"))
    wl = x.wl
    need = sp.sp_score_workspace_size(wl.L, wl.H, wl.H_kv, wl.d, wl.M, wl.N, sp.SP_F32)
    ws = torch.full((need,), 0xAB, dtype=torch.uint8, device="cuda")     # garbage workspace
    imp = torch.empty(wl.M, device="cuda")
    assert sp.sp_score(Q, K, Kla, wl.L, wl.H, wl.H_kv, wl.d, wl.M, wl.N, sp.SP_F32, imp, ws, need) == sp.SP_OK
    assert sp.sp_workspace_status(ws) == sp.SP_OK
    check_importance(imp.cpu().numpy(), oracle.importance(x.Q_la, x.K_prompt, x.K_la), "f32", "garbage ws")
