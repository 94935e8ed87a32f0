"""Shared helpers of the GPU tests: device upload of generated inputs and the
parity tolerances."""
import numpy as np


def to_device(arr: np.ndarray, device="cuda"):
    """uint16 arrays are bf16 bit patterns; fp32 arrays stay fp32."""
    import torch
    if arr.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(arr)).to(device)


def check_importance(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = "") -> None:
    """Importance parity: fp32 inputs |d| <= 1e-5; bf16 inputs |d| <= 1e-3 and
    |d| <= 1e-2 |ref| (+1e-9 for values that underflow)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite importance"
    diff = np.abs(got - ref)
    if dtype == "f32":
        bad = diff > 1e-5
    else:
        bad = (diff > 1e-3) | (diff > 1e-2 * np.abs(ref) + 1e-9)
    if bad.any():
        i = int(np.argmax(np.where(bad, diff / (np.abs(ref) + 1e-12), 0)))
        raise AssertionError(f"{what}: {int(bad.sum())} of {got.size} importance values out of tolerance; "
                             f"worst at {i}: got {got[i]!r} ref {ref[i]!r}; max abs diff {diff.max():.3e}")


import functools  # noqa: E402


@functools.lru_cache(maxsize=None)
def workload_inputs(name: str):
    import workloads as W
    return W.make_workload_inputs(name)


@functools.lru_cache(maxsize=None)
def workload_oracle(name: str):
    """fp64 oracle importance of the named workload (a list per request for a batch)."""
    import oracle
    x = workload_inputs(name)
    if hasattr(x, "requests"):
        return [oracle.importance(r.Q_la, r.K_prompt, r.K_la) for r in x.requests]
    return oracle.importance(x.Q_la, x.K_prompt, x.K_la)
