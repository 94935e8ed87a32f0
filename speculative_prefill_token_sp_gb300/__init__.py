"""SpecPrefill token-importance scoring and chunk selection on one GB300.

Python binding of libspecprefill.so (C ABI in include/specprefill.h).  The
functions named ``sp_*`` mirror the C entry points one to one and only marshal
arguments (torch tensors or raw integer addresses become pointers, streams
become cudaStream_t handles).  ``score``/``score_varlen``/``select``/
``select_varlen`` additionally allocate outputs and workspaces with torch and
raise ``SpError`` on a non-zero status.  Every step of the computation runs in
the library's CUDA kernels; if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

__all__ = [
    "SP_OK", "SP_EINVAL", "SP_ENOMEM", "SP_ECUDA", "SP_EDEVICE", "SP_ETIMEOUT", "SP_EUNSUPPORTED",
    "SP_BF16", "SP_F32", "SP_SELECT_TOPK", "SP_SELECT_MASS", "SpBoost", "SpError", "lib", "lib_path",
    "sp_score_workspace_size", "sp_score", "sp_score_lse_workspace_size", "sp_score_lse",
    "sp_score_prefill_workspace_size", "sp_score_prefill",
    "sp_score_varlen_workspace_size", "sp_score_varlen",
    "sp_score_lse_varlen_workspace_size", "sp_score_lse_varlen",
    "sp_select_workspace_size", "sp_select", "sp_select_varlen_workspace_size", "sp_select_varlen",
    "sp_select_noalloc", "sp_select_rules_workspace_size", "sp_select_rules", "SpKeepRules", "GUIDE_RULES",
    "sp_gather_kept", "sp_workspace_status", "sp_last_error", "sp_status_string", "sp_version",
    "sp_kernel_launches", "sp_test_set_exchange_wait_ns", "sp_test_score_plan",
    "score", "score_lse", "score_prefill", "score_varlen", "score_lse_varlen", "select", "select_rules", "select_varlen", "gather_kept", "V3_BOOST",
]

SP_OK, SP_EINVAL, SP_ENOMEM, SP_ECUDA, SP_EDEVICE, SP_ETIMEOUT, SP_EUNSUPPORTED = range(7)
SP_BF16, SP_F32 = 0, 1
SP_SELECT_TOPK, SP_SELECT_MASS = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(_HERE, "libspecprefill.so")


class SpBoost(ctypes.Structure):
    """sp_boost: v3 normalisation and structural boost."""
    _fields_ = [("first_n", ctypes.c_int32), ("first_mult", ctypes.c_double),
                ("last_n", ctypes.c_int32), ("last_mult", ctypes.c_double),
                ("normalize", ctypes.c_int32)]


# The llama.cpp guide's v3 defaults: first 64 tokens x1.5, last 128 x1.3, normalised.
V3_BOOST = (64, 1.5, 128, 1.3, 1)


class SpKeepRules(ctypes.Structure):
    """sp_keep_rules: the guide's v2 keep rules after the chunk selection."""
    _fields_ = [("min_tok", ctypes.c_int32), ("always_keep", ctypes.c_int32), ("max_keep", ctypes.c_int64)]


# The rules the llama.cpp guide runs with: min_tok 128, always-kept tokens, SP_MAX_KEEP 2000.
GUIDE_RULES = (128, 1, 2000)


class SpError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_status_name(status)}: {message}")
        self.status = status


_lib = None
_c = ctypes
_vp, _sz, _i32, _i64, _dbl = _c.c_void_p, _c.c_size_t, _c.c_int, _c.c_int64, _c.c_double
_SIGS = {
    "sp_score_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i64, _i32, _i32]),
    "sp_score": (_i32, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i64, _i32, _i32, _vp, _vp, _sz, _vp]),
    "sp_score_lse_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i64, _i32, _i32]),
    "sp_score_prefill_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i64, _i32, _i32]),
    "sp_score_prefill": (_i32, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i64, _i32, _i32, _vp, _vp, _sz, _vp]),
    "sp_score_lse": (_i32, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i64, _i32, _i32, _vp, _vp, _sz, _vp]),
    "sp_score_varlen_workspace_size": (_sz, [_i32, _vp, _i32, _i32, _i32, _i32, _i32, _i32]),
    "sp_score_varlen": (_i32, [_vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _vp,
                               _sz, _vp]),
    "sp_score_lse_varlen_workspace_size": (_sz, [_i32, _vp, _i32, _i32, _i32, _i32, _i32, _i32]),
    "sp_score_lse_varlen": (_i32, [_vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _vp,
                                   _sz, _vp]),
    "sp_select_workspace_size": (_sz, [_i64, _i32]),
    "sp_select": (_i32, [_vp, _i64, _i32, _i32, _i32, _dbl, _vp, _vp, _vp, _vp, _sz, _vp]),
    "sp_select_varlen_workspace_size": (_sz, [_i32, _vp, _i32]),
    "sp_select_varlen": (_i32, [_vp, _i32, _vp, _i32, _i32, _i32, _dbl, _vp, _vp, _vp, _vp, _sz, _vp]),
    "sp_select_noalloc": (_i32, [_vp, _i64, _i32, _i32, _i32, _dbl, _vp, _vp, _vp, _vp]),
    "sp_select_rules_workspace_size": (_sz, [_i64, _i32]),
    "sp_select_rules": (_i32, [_vp, _i64, _i32, _i32, _i32, _dbl, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "sp_gather_kept": (_i32, [_vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "sp_workspace_status": (_i32, [_vp, _vp]),
    "sp_last_error": (_c.c_char_p, []),
    "sp_status_string": (_c.c_char_p, [_i32]),
    "sp_version": (_i32, []),
    "sp_kernel_launches": (_c.c_uint64, []),
    "sp_test_set_exchange_wait_ns": (_c.c_uint64, [_c.c_uint64]),
    "sp_test_score_plan": (_i32, [_i32, _i32, _i32, _i32, _c.c_int64, _i32, _i32, _c.POINTER(_c.c_int)]),
}


def lib():
    """The loaded libspecprefill.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(lib_path):
            raise ImportError(f"{lib_path} is missing: build it with "
                              "`python -m speculative_prefill_token_sp_gb300.build`")
        handle = ctypes.CDLL(lib_path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _status_name(s: int) -> str:
    names = ["SP_OK", "SP_EINVAL", "SP_ENOMEM", "SP_ECUDA", "SP_EDEVICE", "SP_ETIMEOUT", "SP_EUNSUPPORTED"]
    return names[s] if 0 <= s < len(names) else f"status {s}"


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, ctypes.Array):
        return ctypes.addressof(x)
    raise TypeError(f"cannot pass {type(x).__name__} as a pointer")


def _stream(s) -> Optional[int]:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _i64_array(values):
    arr = (ctypes.c_int64 * len(values))(*[int(v) for v in values])
    return arr


def _boost(b):
    if b is None:
        return None
    if isinstance(b, SpBoost):
        return ctypes.pointer(b)
    return ctypes.pointer(SpBoost(*b))


# ----------------------------------------------------------------------------
# One-to-one marshalling of the C entry points
# ----------------------------------------------------------------------------

def sp_score_workspace_size(L, H, H_kv, d, M, N, dtype) -> int:
    return lib().sp_score_workspace_size(L, H, H_kv, d, M, N, dtype)


def sp_score(Q_la, K_prompt, K_la, L, H, H_kv, d, M, N, dtype, importance, ws, ws_bytes, stream=None) -> int:
    return lib().sp_score(_ptr(Q_la), _ptr(K_prompt), _ptr(K_la), L, H, H_kv, d, M, N, dtype,
                          _ptr(importance), _ptr(ws), ws_bytes, _stream(stream))


def sp_score_prefill_workspace_size(L, H, H_kv, d, M, N, dtype) -> int:
    return lib().sp_score_prefill_workspace_size(L, H, H_kv, d, M, N, dtype)


def sp_score_prefill(Q_rows, K_prompt, K_la, L, H, H_kv, d, M, N, dtype, importance, ws, ws_bytes,
                     stream=None) -> int:
    return lib().sp_score_prefill(_ptr(Q_rows), _ptr(K_prompt), _ptr(K_la), L, H, H_kv, d, M, N, dtype,
                                  _ptr(importance), _ptr(ws), ws_bytes, _stream(stream))


def sp_score_lse_workspace_size(L, H, H_kv, d, M, N, dtype) -> int:
    return lib().sp_score_lse_workspace_size(L, H, H_kv, d, M, N, dtype)


def sp_score_lse(Q_la, K_prompt, lse, L, H, H_kv, d, M, N, dtype, importance, ws, ws_bytes, stream=None) -> int:
    return lib().sp_score_lse(_ptr(Q_la), _ptr(K_prompt), _ptr(lse), L, H, H_kv, d, M, N, dtype,
                              _ptr(importance), _ptr(ws), ws_bytes, _stream(stream))


def sp_score_varlen_workspace_size(B, cu_M_host, L, H, H_kv, d, N, dtype) -> int:
    cu = _i64_array(cu_M_host)
    return lib().sp_score_varlen_workspace_size(B, ctypes.addressof(cu), L, H, H_kv, d, N, dtype)


def sp_score_varlen(Q_la, K_prompt, K_la, B, cu_M_host, L, H, H_kv, d, N, dtype, importance, ws, ws_bytes,
                    stream=None) -> int:
    cu = _i64_array(cu_M_host)
    return lib().sp_score_varlen(_ptr(Q_la), _ptr(K_prompt), _ptr(K_la), B, ctypes.addressof(cu), L, H, H_kv,
                                 d, N, dtype, _ptr(importance), _ptr(ws), ws_bytes, _stream(stream))


def sp_score_lse_varlen_workspace_size(B, cu_M_host, L, H, H_kv, d, N, dtype) -> int:
    cu = _i64_array(cu_M_host)
    return lib().sp_score_lse_varlen_workspace_size(B, ctypes.addressof(cu), L, H, H_kv, d, N, dtype)


def sp_score_lse_varlen(Q_la, K_prompt, lse, B, cu_M_host, L, H, H_kv, d, N, dtype, importance, ws, ws_bytes,
                        stream=None) -> int:
    cu = _i64_array(cu_M_host)
    return lib().sp_score_lse_varlen(_ptr(Q_la), _ptr(K_prompt), _ptr(lse), B, ctypes.addressof(cu), L, H,
                                     H_kv, d, N, dtype, _ptr(importance), _ptr(ws), ws_bytes, _stream(stream))


def sp_select_workspace_size(M, chunk) -> int:
    return lib().sp_select_workspace_size(M, chunk)


def sp_select(importance, M, chunk, pool_k, mode, rate, boost, kept_pos, n_kept, ws, ws_bytes,
              stream=None) -> int:
    return lib().sp_select(_ptr(importance), M, chunk, pool_k, mode, rate, _boost(boost), _ptr(kept_pos),
                           _ptr(n_kept), _ptr(ws), ws_bytes, _stream(stream))


def _rules(rules):
    if rules is None:
        return None
    if isinstance(rules, SpKeepRules):
        return ctypes.pointer(rules)
    return ctypes.pointer(SpKeepRules(*rules))


def sp_select_rules_workspace_size(M, chunk) -> int:
    return lib().sp_select_rules_workspace_size(M, chunk)


def sp_select_rules(importance, M, chunk, pool_k, mode, rate, boost, rules, kept_pos, n_kept, ws, ws_bytes,
                    stream=None) -> int:
    return lib().sp_select_rules(_ptr(importance), M, chunk, pool_k, mode, rate, _boost(boost), _rules(rules),
                                 _ptr(kept_pos), _ptr(n_kept), _ptr(ws), ws_bytes, _stream(stream))


def sp_select_varlen_workspace_size(B, cu_M_host, chunk) -> int:
    cu = _i64_array(cu_M_host)
    return lib().sp_select_varlen_workspace_size(B, ctypes.addressof(cu), chunk)


def sp_select_varlen(importance, B, cu_M_host, chunk, pool_k, mode, rate, boost, kept_pos, n_kept, ws,
                     ws_bytes, stream=None) -> int:
    cu = _i64_array(cu_M_host)
    return lib().sp_select_varlen(_ptr(importance), B, ctypes.addressof(cu), chunk, pool_k, mode, rate,
                                  _boost(boost), _ptr(kept_pos), _ptr(n_kept), _ptr(ws), ws_bytes,
                                  _stream(stream))


def sp_select_noalloc(importance, M, chunk, pool_k, mode, rate, boost, kept_pos, n_kept, stream=None) -> int:
    """sp_select without a workspace (scratch in a fixed device array of the library)."""
    return lib().sp_select_noalloc(_ptr(importance), M, chunk, pool_k, mode, rate, _boost(boost), _ptr(kept_pos),
                                   _ptr(n_kept), _stream(stream))


def sp_gather_kept(token_ids, B, cu_M_host, kept_pos, n_kept, out_tokens, out_positions, cu_kept,
                   stream=None) -> int:
    cu = _i64_array(cu_M_host)
    return lib().sp_gather_kept(_ptr(token_ids), B, ctypes.addressof(cu), _ptr(kept_pos), _ptr(n_kept),
                                _ptr(out_tokens), _ptr(out_positions), _ptr(cu_kept), _stream(stream))


def sp_workspace_status(ws, stream=None) -> int:
    return lib().sp_workspace_status(_ptr(ws), _stream(stream))


def sp_last_error() -> str:
    return lib().sp_last_error().decode()


def sp_status_string(s: int) -> str:
    return lib().sp_status_string(s).decode()


def sp_version() -> int:
    return lib().sp_version()


def sp_kernel_launches() -> int:
    return lib().sp_kernel_launches()


def sp_test_set_exchange_wait_ns(ns: int) -> int:
    """Test hook: limit (ns) of the scoring kernel's waits on other CTAs' exchange
    entries; 0 restores the default.  Returns the previous limit."""
    return lib().sp_test_set_exchange_wait_ns(int(ns))


def sp_test_score_plan(L: int, H: int, H_kv: int, d: int, M: int, N: int, sms: int = 152):
    """Test hook: the tensor-core scoring plan of one bf16 prompt as a dict
    (F, Pc, P, tiles, tiles_per_group, land, held, lag, smem_bytes), or None when
    that path does not take the shape.  Host only."""
    out = (_c.c_int * 9)()
    if not lib().sp_test_score_plan(L, H, H_kv, d, int(M), N, sms, out):
        return None
    keys = ("F", "Pc", "P", "tiles", "tiles_per_group", "land", "held", "lag", "smem_bytes")
    return dict(zip(keys, list(out)))


# ----------------------------------------------------------------------------
# Helpers that allocate with torch
# ----------------------------------------------------------------------------

def _check(status: int) -> None:
    if status != SP_OK:
        raise SpError(status, sp_last_error())


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return SP_BF16
    if t.dtype == torch.float32:
        return SP_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _workspace(nbytes: int, device, ws=None):
    import torch
    if ws is not None:
        if ws.numel() * ws.element_size() < nbytes:
            raise SpError(SP_ENOMEM, f"workspace smaller than {nbytes} bytes")
        return ws
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def _check_device(ws, stream, check):
    if check:
        _check(sp_workspace_status(ws, stream))


def score(Q_la, K_prompt, K_la, *, importance=None, ws=None, stream=None, check=False):
    """Importance [M] (fp32) of one prompt: Q_la [N,L,H,d], K_prompt [L,H_kv,M,d], K_la [L,H_kv,N,d].
    check=True synchronises and raises if a kernel recorded a run-time error."""
    import torch
    N, L, H, d = Q_la.shape
    _, H_kv, M, _ = K_prompt.shape
    dt = _dtype_code(K_prompt)
    if importance is None:
        importance = torch.empty(M, dtype=torch.float32, device=K_prompt.device)
    need = sp_score_workspace_size(L, H, H_kv, d, M, N, dt)
    ws = _workspace(need, K_prompt.device, ws)
    _check(sp_score(Q_la, K_prompt, K_la, L, H, H_kv, d, M, N, dt, importance, ws, ws.numel(), stream))
    _check_device(ws, stream, check)
    return importance


def score_prefill(Q_rows, K_prompt, K_la, *, importance=None, ws=None, stream=None, check=False):
    """Importance [M] (fp32) from the prefill's last query (Q_rows[0]) and N decode steps (Q_rows[1:]):
    Q_rows [N+1,L,H,d], K_prompt [L,H_kv,M,d], K_la [L,H_kv,N,d]."""
    import torch
    N1, L, H, d = Q_rows.shape
    _, H_kv, M, _ = K_prompt.shape
    dt = _dtype_code(K_prompt)
    if importance is None:
        importance = torch.empty(M, dtype=torch.float32, device=K_prompt.device)
    need = sp_score_prefill_workspace_size(L, H, H_kv, d, M, N1 - 1, dt)
    ws = _workspace(need, K_prompt.device, ws)
    _check(sp_score_prefill(Q_rows, K_prompt, K_la, L, H, H_kv, d, M, N1 - 1, dt, importance, ws, ws.numel(),
                            stream))
    _check_device(ws, stream, check)
    return importance


def score_lse(Q_la, K_prompt, lse, *, importance=None, ws=None, stream=None, check=False):
    """Importance [M] (fp32) of one prompt from given row normalisers: Q_la [N,L,H,d],
    K_prompt [L,H_kv,M,d], lse [L,H,N] fp32 (device)."""
    import torch
    N, L, H, d = Q_la.shape
    _, H_kv, M, _ = K_prompt.shape
    dt = _dtype_code(K_prompt)
    if importance is None:
        importance = torch.empty(M, dtype=torch.float32, device=K_prompt.device)
    need = sp_score_lse_workspace_size(L, H, H_kv, d, M, N, dt)
    ws = _workspace(need, K_prompt.device, ws)
    _check(sp_score_lse(Q_la, K_prompt, lse, L, H, H_kv, d, M, N, dt, importance, ws, ws.numel(), stream))
    _check_device(ws, stream, check)
    return importance


def score_varlen(Q_la, K_prompt, K_la, cu_M, *, importance=None, ws=None, stream=None, check=False):
    """Packed importance [T] of B prompts: Q_la [B,N,L,H,d], K_prompt [L,H_kv,T,d], K_la [B,L,H_kv,N,d]."""
    import torch
    B, N, L, H, d = Q_la.shape
    H_kv, T = K_prompt.shape[1], K_prompt.shape[2]
    cu = [int(x) for x in cu_M]
    dt = _dtype_code(K_prompt)
    if importance is None:
        importance = torch.empty(T, dtype=torch.float32, device=K_prompt.device)
    need = sp_score_varlen_workspace_size(B, cu, L, H, H_kv, d, N, dt)
    ws = _workspace(need, K_prompt.device, ws)
    _check(sp_score_varlen(Q_la, K_prompt, K_la, B, cu, L, H, H_kv, d, N, dt, importance, ws, ws.numel(),
                           stream))
    _check_device(ws, stream, check)
    return importance


def score_lse_varlen(Q_la, K_prompt, lse, cu_M, *, importance=None, ws=None, stream=None, check=False):
    """Packed importance [T] of B prompts from given row normalisers: Q_la [B,N,L,H,d],
    K_prompt [L,H_kv,T,d], lse [B,L,H,N] fp32 (device)."""
    import torch
    B, N, L, H, d = Q_la.shape
    H_kv, T = K_prompt.shape[1], K_prompt.shape[2]
    cu = [int(x) for x in cu_M]
    dt = _dtype_code(K_prompt)
    if importance is None:
        importance = torch.empty(T, dtype=torch.float32, device=K_prompt.device)
    need = sp_score_lse_varlen_workspace_size(B, cu, L, H, H_kv, d, N, dt)
    ws = _workspace(need, K_prompt.device, ws)
    _check(sp_score_lse_varlen(Q_la, K_prompt, lse, B, cu, L, H, H_kv, d, N, dt, importance, ws, ws.numel(),
                               stream))
    _check_device(ws, stream, check)
    return importance


def _mode(mode) -> int:
    if mode in (SP_SELECT_TOPK, "topk"):
        return SP_SELECT_TOPK
    if mode in (SP_SELECT_MASS, "mass"):
        return SP_SELECT_MASS
    raise ValueError(f"unknown mode {mode!r}")


def select(importance, chunk, pool_k, mode, rate, boost=None, *, kept_pos=None, n_kept=None, ws=None,
           stream=None, trim=True):
    """Kept position IDs of one prompt.  With trim=True (synchronises) returns
    kept_pos[:n]; otherwise (kept_pos buffer, n_kept device tensor)."""
    import torch
    M = importance.shape[0]
    dev = importance.device
    if kept_pos is None:
        kept_pos = torch.empty(max(M, 1), dtype=torch.int32, device=dev)
    if n_kept is None:
        n_kept = torch.empty(1, dtype=torch.int64, device=dev)
    ws = _workspace(sp_select_workspace_size(M, chunk), dev, ws)
    _check(sp_select(importance, M, chunk, pool_k, _mode(mode), float(rate), boost, kept_pos, n_kept, ws,
                     ws.numel(), stream))
    if trim:
        return kept_pos[: int(n_kept.item())]
    return kept_pos, n_kept


def select_rules(importance, chunk, pool_k, mode, rate, boost=None, rules=GUIDE_RULES, *, ws=None, stream=None):
    """Kept position IDs of one prompt after the selection and the keep rules (synchronises)."""
    import torch
    M = importance.shape[0]
    dev = importance.device
    kept_pos = torch.empty(max(M, 1), dtype=torch.int32, device=dev)
    n_kept = torch.empty(1, dtype=torch.int64, device=dev)
    ws = _workspace(sp_select_rules_workspace_size(M, chunk), dev, ws)
    _check(sp_select_rules(importance, M, chunk, pool_k, _mode(mode), float(rate), boost, rules, kept_pos, n_kept,
                           ws, ws.numel(), stream))
    return kept_pos[: int(n_kept.item())]


def select_varlen(importance, cu_M, chunk, pool_k, mode, rate, boost=None, *, kept_pos=None, n_kept=None,
                  ws=None, stream=None, trim=True):
    """Per-prompt kept position IDs of a packed batch.  trim=True returns a list of tensors."""
    import torch
    cu = [int(x) for x in cu_M]
    B = len(cu) - 1
    dev = importance.device
    if kept_pos is None:
        kept_pos = torch.empty(max(cu[-1], 1), dtype=torch.int32, device=dev)
    if n_kept is None:
        n_kept = torch.empty(B, dtype=torch.int64, device=dev)
    ws = _workspace(sp_select_varlen_workspace_size(B, cu, chunk), dev, ws)
    _check(sp_select_varlen(importance, B, cu, chunk, pool_k, _mode(mode), float(rate), boost, kept_pos,
                            n_kept, ws, ws.numel(), stream))
    if trim:
        n = n_kept.tolist()
        return [kept_pos[cu[b]: cu[b] + n[b]] for b in range(B)]
    return kept_pos, n_kept


def gather_kept(token_ids, cu_M, kept_pos, n_kept, *, stream=None):
    """Sparse-prefill batch of packed prompts: (tokens int32, positions int32, cu_kept int64 [B+1]),
    each prompt's kept tokens packed after the previous prompt's (device tensors, capacity T)."""
    import torch
    cu = [int(x) for x in cu_M]
    B, T = len(cu) - 1, cu[-1]
    dev = kept_pos.device
    tokens = torch.empty(max(T, 1), dtype=torch.int32, device=dev)
    positions = torch.empty(max(T, 1), dtype=torch.int32, device=dev)
    cu_kept = torch.empty(B + 1, dtype=torch.int64, device=dev)
    _check(sp_gather_kept(token_ids, B, cu, kept_pos, n_kept, tokens, positions, cu_kept, stream))
    return tokens, positions, cu_kept
