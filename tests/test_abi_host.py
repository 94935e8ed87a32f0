"""Host-side checks of the C ABI (no GPU): the library builds and loads, exports
every symbol include/specprefill.h declares, and rejects bad arguments before
touching the GPU."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "specprefill.h")


@pytest.fixture(scope="module")
def sp():
    from speculative_prefill_token_sp_gb300 import build
    build.build()
    import speculative_prefill_token_sp_gb300 as m
    m.lib()
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sp_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol(sp):
    names = declared_functions()
    assert len(names) >= 12
    handle = ctypes.CDLL(sp.lib_path)
    for n in names:
        assert hasattr(handle, n), n
    assert set(names) == set(sp._SIGS), "binding and header disagree"


def test_version_and_status_strings(sp):
    assert sp.sp_version() == 100
    assert sp.sp_status_string(sp.SP_ENOMEM) == "SP_ENOMEM"
    assert sp.sp_status_string(99) == "SP_UNKNOWN"


def test_workspace_sizes(sp):
    a = sp.sp_score_workspace_size(32, 32, 8, 128, 32768, 8, sp.SP_BF16)
    b = sp.sp_score_workspace_size(32, 32, 8, 128, 131072, 8, sp.SP_BF16)
    assert 0 < a < b
    assert sp.sp_score_workspace_size(32, 30, 8, 128, 1024, 8, sp.SP_BF16) == 0      # H % H_kv != 0
    assert sp.sp_select_workspace_size(32768, 32) > 0
    assert sp.sp_select_workspace_size(-1, 32) == 0
    assert sp.sp_score_varlen_workspace_size(3, [0, 5, 5, 9], 2, 4, 2, 64, 4, sp.SP_F32) > 0
    assert sp.sp_select_varlen_workspace_size(2, [0, 7, 3], 8) == 0                    # decreasing cu


@pytest.mark.parametrize("args,status", [
    (dict(L=0), "SP_EINVAL"), (dict(H=5), "SP_EINVAL"), (dict(d=12), "SP_EUNSUPPORTED"),
    (dict(d=512), "SP_EUNSUPPORTED"), (dict(N=-1), "SP_EINVAL"), (dict(N=200), "SP_EUNSUPPORTED"),
    (dict(M=-5), "SP_EINVAL"), (dict(dtype=7), "SP_EINVAL"),
])
def test_score_rejects_bad_shapes(sp, args, status):
    a = dict(L=2, H=4, H_kv=2, d=64, M=512, N=4, dtype=sp.SP_F32)
    a.update(args)
    s = sp.sp_score(16, 16, 16, a["L"], a["H"], a["H_kv"], a["d"], a["M"], a["N"], a["dtype"], 16, 16, 1 << 30, 0)
    assert sp.sp_status_string(s) == status
    assert sp.sp_last_error() != ""


def test_score_rejects_small_workspace_and_bad_pointers(sp):
    need = sp.sp_score_workspace_size(2, 4, 2, 64, 512, 4, sp.SP_F32)
    s = sp.sp_score(16, 16, 16, 2, 4, 2, 64, 512, 4, sp.SP_F32, 16, 16, need - 1, 0)
    assert s == sp.SP_ENOMEM and "smaller" in sp.sp_last_error()
    s = sp.sp_score(None, 16, 16, 2, 4, 2, 64, 512, 4, sp.SP_F32, 16, 16, need, 0)
    assert s == sp.SP_EINVAL
    s = sp.sp_score(18, 16, 16, 2, 4, 2, 64, 512, 4, sp.SP_F32, 16, 16, need, 0)
    assert s == sp.SP_EINVAL and "aligned" in sp.sp_last_error()


def test_varlen_rejects_bad_offsets(sp):
    f = sp.sp_score_varlen
    assert f(16, 16, 16, 2, [1, 3, 5], 2, 4, 2, 64, 4, sp.SP_F32, 16, 16, 1 << 30, 0) == sp.SP_EINVAL
    assert f(16, 16, 16, 2, [0, 5, 3], 2, 4, 2, 64, 4, sp.SP_F32, 16, 16, 1 << 30, 0) == sp.SP_EINVAL
    assert f(16, 16, 16, 0, [0], 2, 4, 2, 64, 4, sp.SP_F32, 16, 16, 1 << 30, 0) == sp.SP_EINVAL
    cu = list(range(0, 258))
    assert f(16, 16, 16, 257, cu, 2, 4, 2, 64, 4, sp.SP_F32, 16, 16, 1 << 30, 0) == sp.SP_EUNSUPPORTED


@pytest.mark.parametrize("kw,status", [
    (dict(chunk=0), "SP_EINVAL"), (dict(pool_k=2), "SP_EINVAL"), (dict(pool_k=0), "SP_EINVAL"),
    (dict(rate=0.0), "SP_EINVAL"), (dict(rate=1.5), "SP_EINVAL"), (dict(mode=5), "SP_EINVAL"),
    (dict(mode=1, pool_k=3), "SP_EINVAL"), (dict(boost=(-1, 1.5, 0, 1.0, 0)), "SP_EINVAL"),
])
def test_select_rejects_bad_parameters(sp, kw, status):
    a = dict(chunk=32, pool_k=3, mode=0, rate=0.3, boost=None)
    a.update(kw)
    s = sp.sp_select(16, 512, a["chunk"], a["pool_k"], a["mode"], a["rate"], a["boost"], 16, 16, 16, 1 << 30, 0)
    assert sp.sp_status_string(s) == status


def test_select_rejects_small_workspace(sp):
    need = sp.sp_select_workspace_size(512, 32)
    assert sp.sp_select(16, 512, 32, 3, 0, 0.3, None, 16, 16, 16, need - 1, 0) == sp.SP_ENOMEM


def test_calls_without_gpu_fail_cleanly(sp):
    """Valid arguments on a machine without a GPU: an error status, never a crash."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    need = sp.sp_select_workspace_size(512, 32)
    assert sp.sp_select(16, 512, 32, 3, 0, 0.3, None, 16, 16, 16, need, 0) == sp.SP_ECUDA


def test_score_lse_validation(sp):
    """sp_score_lse: same shape rules as sp_score; the lse pointer replaces K_la (4-byte aligned)."""
    need = sp.sp_score_lse_workspace_size(2, 4, 2, 64, 512, 4, sp.SP_F32)
    assert need > 0
    assert sp.sp_score_lse_workspace_size(2, 5, 2, 64, 512, 4, sp.SP_F32) == 0          # H % H_kv != 0
    f = sp.sp_score_lse
    assert f(16, 16, 16, 2, 4, 2, 12, 512, 4, sp.SP_F32, 16, 16, need, 0) == sp.SP_EUNSUPPORTED   # d
    assert f(16, 16, 16, 2, 4, 2, 64, -1, 4, sp.SP_F32, 16, 16, need, 0) == sp.SP_EINVAL          # M
    assert f(16, 16, 16, 2, 4, 2, 64, 512, 4, sp.SP_F32, 16, 16, need - 1, 0) == sp.SP_ENOMEM
    assert f(16, 16, None, 2, 4, 2, 64, 512, 4, sp.SP_F32, 16, 16, need, 0) == sp.SP_EINVAL       # null lse
    assert f(16, 16, 18, 2, 4, 2, 64, 512, 4, sp.SP_F32, 16, 16, need, 0) == sp.SP_EINVAL         # misaligned lse
    assert "aligned" in sp.sp_last_error()


def test_gather_validation(sp):
    f = sp.sp_gather_kept
    assert f(16, 0, [0], 16, 16, 16, 16, 16, 0) == sp.SP_EINVAL                 # B < 1
    assert f(16, 2, [0, 5, 3], 16, 16, 16, 16, 16, 0) == sp.SP_EINVAL           # decreasing offsets
    assert f(16, 1, [0, 5], None, 16, 16, 16, 16, 0) == sp.SP_EINVAL            # no kept_pos
    assert f(None, 1, [0, 5], 16, 16, 16, None, 16, 0) == sp.SP_EINVAL          # tokens wanted, no token_ids
    assert f(16, 1, [0, 5], 16, 16, None, None, 16, 0) == sp.SP_EINVAL          # no output at all


def test_select_rules_validation(sp):
    need = sp.sp_select_rules_workspace_size(512, 32)
    assert need > sp.sp_select_workspace_size(512, 32)          # scratch for the merged list
    f = sp.sp_select_rules
    assert f(16, 512, 32, 3, 0, 0.3, None, (-1, 1, 0), 16, 16, 16, need, 0) == sp.SP_EINVAL
    assert f(16, 512, 32, 3, 0, 0.3, None, (128, 1, -5), 16, 16, 16, need, 0) == sp.SP_EINVAL
    assert f(16, 512, 32, 3, 0, 0.3, None, (5000, 1, 0), 16, 16, 16, need, 0) == sp.SP_EUNSUPPORTED
    assert f(16, 512, 32, 3, 0, 0.3, None, sp.GUIDE_RULES, 16, 16, 16, need - 1, 0) == sp.SP_ENOMEM


def test_score_prefill_validation(sp):
    need = sp.sp_score_prefill_workspace_size(2, 4, 2, 64, 512, 3, sp.SP_F32)
    assert need > 0
    f = sp.sp_score_prefill
    assert f(16, 16, 16, 2, 4, 2, 64, 512, -1, sp.SP_F32, 16, 16, need, 0) == sp.SP_EINVAL       # N < 0
    assert f(16, 16, 16, 2, 4, 2, 64, 512, 200, sp.SP_F32, 16, 16, need, 0) == sp.SP_EUNSUPPORTED  # (N+1)*G > 256
    assert f(16, 16, 16, 2, 4, 2, 64, 512, 3, sp.SP_F32, 16, 16, need - 1, 0) == sp.SP_ENOMEM
    assert f(16, 16, None, 2, 4, 2, 64, 512, 3, sp.SP_F32, 16, 16, need, 0) == sp.SP_EINVAL       # keys needed


def test_score_lse_varlen_validation(sp):
    """sp_score_lse_varlen: the offsets rules of sp_score_varlen, the lse pointer rules of sp_score_lse."""
    cu = [0, 300, 300, 812]
    need = sp.sp_score_lse_varlen_workspace_size(3, cu, 2, 4, 2, 64, 4, sp.SP_F32)
    assert need > 0
    assert sp.sp_score_lse_varlen_workspace_size(3, [0, 300, 200, 812], 2, 4, 2, 64, 4, sp.SP_F32) == 0
    assert sp.sp_score_lse_varlen_workspace_size(3, cu, 2, 5, 2, 64, 4, sp.SP_F32) == 0     # H % H_kv != 0
    f = sp.sp_score_lse_varlen
    assert f(16, 16, 16, 3, [1, 300, 300, 812], 2, 4, 2, 64, 4, sp.SP_F32, 16, 16, need, 0) == sp.SP_EINVAL
    assert f(16, 16, 16, 3, cu, 2, 4, 2, 12, 4, sp.SP_F32, 16, 16, need, 0) == sp.SP_EUNSUPPORTED   # d
    assert f(16, 16, 16, 3, cu, 2, 4, 2, 64, 4, sp.SP_F32, 16, 16, need - 1, 0) == sp.SP_ENOMEM
    assert f(16, 16, None, 3, cu, 2, 4, 2, 64, 4, sp.SP_F32, 16, 16, need, 0) == sp.SP_EINVAL       # null lse
    assert f(16, 16, 18, 3, cu, 2, 4, 2, 64, 4, sp.SP_F32, 16, 16, need, 0) == sp.SP_EINVAL         # misaligned lse
    assert "aligned" in sp.sp_last_error()
    cu257 = list(range(0, 258))
    assert f(16, 16, 16, 257, cu257, 2, 4, 2, 64, 4, sp.SP_F32, 16, 16, 1 << 30, 0) == sp.SP_EUNSUPPORTED


def test_exchange_wait_hook_is_host_only(sp):
    """The test hook only stores the limit that later calls read when planned."""
    prev = sp.sp_test_set_exchange_wait_ns(1234)
    assert prev == 4_000_000_000
    assert sp.sp_test_set_exchange_wait_ns(0) == 1234
    assert sp.sp_test_set_exchange_wait_ns(prev) == 4_000_000_000
