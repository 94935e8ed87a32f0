"""Failure detection without a GPU fault: a bounded wait that runs out.

The tensor-core scoring kernel exchanges softmax statistics and lse between
its CTAs through global memory, and every wait on another CTA's entry gives up
after a limit (4 s by default).  A test hook lowers that limit to 1 us, far
shorter than the time the first exchange entry needs to appear (its slab must
be streamed, multiplied and reduced first), so the wait runs out.  The kernel
must then record SP_ETIMEOUT in the workspace, stop every warp role, drain its
in-flight copies and MMAs, free its tensor memory and return: the call ends,
the context stays usable, and the next call with the default limit is correct.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_helpers import check_importance, to_device

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


@pytest.mark.parametrize("M", [4096, 40000])
def test_exchange_wait_that_runs_out_reports_timeout_and_recovers(sp, M):
    import torch
    # the 8B head shape (tensor-core path), two layers; 40000 tokens gives every CTA several tiles
    wl = W.Workload("t", L=2, H=32, H_kv=8, d=128, M=M, N=8, dtype="bf16", chunk=32, pool_k=3, mode="topk",
                    keep_rate=0.1, needle_frac=0.02, run_min=16, run_max=128)
    x = W.make_inputs(wl, seed=4242 + M)
    Q, K, Kla = (to_device(getattr(x, n)) for n in ("Q_la", "K_prompt", "K_la"))
    need = sp.sp_score_workspace_size(wl.L, wl.H, wl.H_kv, wl.d, M, wl.N, sp.SP_BF16)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    imp = torch.empty(M, dtype=torch.float32, device="cuda")
    n0 = sp.sp_kernel_launches()
    prev = sp.sp_test_set_exchange_wait_ns(1000)
    try:
        s = sp.sp_score(Q, K, Kla, wl.L, wl.H, wl.H_kv, wl.d, M, wl.N, sp.SP_BF16, imp, ws, need)
    finally:
        assert sp.sp_test_set_exchange_wait_ns(prev) == 1000
    assert s == sp.SP_OK, sp.sp_last_error()            # the launch itself is fine
    assert sp.sp_kernel_launches() - n0 == 2            # preparation + the tensor-core kernel
    torch.cuda.synchronize()                            # the kernel returned
    assert sp.sp_workspace_status(ws) == sp.SP_ETIMEOUT
    assert "status 5" in sp.sp_last_error()
    # the same workspace, the default limit: a clean, correct call
    s = sp.sp_score(Q, K, Kla, wl.L, wl.H, wl.H_kv, wl.d, M, wl.N, sp.SP_BF16, imp, ws, need)
    assert s == sp.SP_OK, sp.sp_last_error()
    torch.cuda.synchronize()
    assert sp.sp_workspace_status(ws) == sp.SP_OK
    check_importance(imp.cpu().numpy(), oracle.importance(x.Q_la, x.K_prompt, x.K_la), "bf16", f"M={M}")


def test_hook_restores_the_default(sp):
    prev = sp.sp_test_set_exchange_wait_ns(0)
    assert sp.sp_test_set_exchange_wait_ns(prev) == 4_000_000_000
