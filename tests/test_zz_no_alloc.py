"""sp_select_noalloc: selection for callers that cannot allocate device memory.

Code running inside an allocator or its out-of-memory handler, serving loops
that must not call cudaMalloc, and plug-ins handed only their input and output
buffers cannot provide sp_select's workspace.  sp_select_noalloc keeps that
scratch in a fixed device array inside the library.  These tests call it
through the C ABI twice in a row (the second call must not see the first
call's leftovers) and compare with sp_select, which uses a caller workspace,
and with the oracle's selection of the same importance vector; selection is
integer work, so the comparisons are exact.  A call after the first one must
not change the device's free memory.  This file is collected last on purpose.
"""
import numpy as np
import pytest

import oracle

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


def _with_workspace(sp, imp, chunk, pool_k, mode, rate, boost):
    import torch
    M = imp.numel()
    kept = torch.full((max(M, 1),), -1, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int64, device="cuda")
    need = sp.sp_select_workspace_size(M, chunk)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    assert sp.sp_select(imp, M, chunk, pool_k, mode, rate, boost, kept, n, ws, need) == sp.SP_OK, sp.sp_last_error()
    torch.cuda.synchronize()
    k = int(n.item())
    return kept[:k].cpu().numpy(), k


def _no_alloc(sp, imp, chunk, pool_k, mode, rate, boost):
    import torch
    M = imp.numel()
    kept = torch.full((max(M, 1),), -1, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int64, device="cuda")
    assert sp.sp_select_noalloc(imp, M, chunk, pool_k, mode, rate, boost, kept, n) == sp.SP_OK, sp.sp_last_error()
    torch.cuda.synchronize()
    k = int(n.item())
    return kept[:k].cpu().numpy(), k


def test_no_alloc_matches_workspace_entry_point_twice(sp):
    import torch
    rng = np.random.default_rng(2024)
    calls = [
        # (M, chunk, pool_k, mode, rate, boost): a top-K call, then a v3 mass call of another size
        (32768, 32, 3, sp.SP_SELECT_TOPK, 0.1, None),
        (20000, 32, 1, sp.SP_SELECT_MASS, 0.85, (64, 1.5, 128, 1.3, 1)),
    ]
    for M, chunk, pool_k, mode, rate, boost in calls:
        host = (rng.random(M) * 1e-3).astype(np.float32)
        imp = torch.from_numpy(host).cuda()
        want, n_want = _with_workspace(sp, imp, chunk, pool_k, mode, rate, boost)
        got, n_got = _no_alloc(sp, imp, chunk, pool_k, mode, rate, boost)
        assert n_got == n_want
        assert np.array_equal(got, want)
        ref, n_ref = oracle.select(host, chunk, pool_k, "topk" if mode == sp.SP_SELECT_TOPK else "mass", rate,
                                   boost)
        assert n_got == n_ref and np.array_equal(got, ref)


def test_no_alloc_call_leaves_free_device_memory_unchanged(sp):
    import torch
    M, chunk = 40000, 32
    imp = torch.from_numpy((np.random.default_rng(7).random(M) * 1e-3).astype(np.float32)).cuda()
    kept = torch.empty(M, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int64, device="cuda")
    # the first call on the device may load the library's module (and its array)
    assert sp.sp_select_noalloc(imp, M, chunk, 3, sp.SP_SELECT_TOPK, 0.1, None, kept, n) == sp.SP_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    assert sp.sp_select_noalloc(imp, M, chunk, 3, sp.SP_SELECT_TOPK, 0.1, None, kept, n) == sp.SP_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_no_alloc_rejects_requests_beyond_its_fixed_scratch(sp):
    import torch
    M = 65536 * 32 + 1                       # 65537 chunks of 32
    imp = torch.zeros(M, dtype=torch.float32, device="cuda")
    kept = torch.empty(M, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int64, device="cuda")
    s = sp.sp_select_noalloc(imp, M, 32, 3, sp.SP_SELECT_TOPK, 0.1, None, kept, n)
    assert s == sp.SP_EUNSUPPORTED
    assert "65536" in sp.sp_last_error()
    # the limit itself is accepted
    M = 65536 * 32
    s = sp.sp_select_noalloc(imp[:M], M, 32, 3, sp.SP_SELECT_TOPK, 0.1, None, kept, n)
    torch.cuda.synchronize()
    assert s == sp.SP_OK and int(n.item()) == 6554 * 32
