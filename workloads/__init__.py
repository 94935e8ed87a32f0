"""Seeded synthetic inputs for SpecPrefill token-importance scoring and selection.

This module is shared by the tests, the benchmark and the smoke check. It holds
the five workload configurations and the input generator, and nothing of the
method's arithmetic (no attention, no aggregation, no selection).

Recipe (the pages print no inputs; these stand in for the long LongBench/RULER
style prompts of the paper review "Speculative Prefill: Turbocharging TTFT ...",
section 5 "experimental setup"):
  * Q_la[N, L, H, d], K_prompt[L, H_kv, M, d], K_la[L, H_kv, N, d] are i.i.d.
    N(0, 1) draws in fp32.
  * The key of prompt position 0 is multiplied by 4 (an attention sink).
  * "Needle" positions: for every layer l and KV head g, the mean mu[l, g] of
    the query vectors Q_la[j, l, h] over all look-ahead steps j and all query
    heads h of group g is computed, and 3 * mu[l, g] is added to K_prompt[l, g, i]
    for every needle position i.  Needles are either single positions or runs
    of consecutive positions whose lengths are uniform in [run_min, run_max],
    placed until the requested fraction of M is covered; position 0 is never a
    needle.
  * bf16 configurations round every fp32 value to the nearest bf16 (ties to
    even); the oracle reads exactly the rounded values.
  * Random streams: numpy PCG64, seeded by numpy SeedSequence([seed, request]),
    with one spawned child stream for the needles, one for Q_la, one for K_la
    and one per (layer, KV head) slab of K_prompt, so that slabs can be drawn
    independently and in parallel.

Query head h reads KV head g = h // (H // H_kv) (contiguous groups).
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Optional

import numpy as np

__all__ = [
    "WORKLOADS", "BY_NAME", "V3_BOOST", "Workload", "Inputs", "VarlenInputs", "make_inputs",
    "make_varlen_inputs", "make_workload_inputs", "bf16_bits_from_f32",
    "f32_from_bf16_bits", "needle_positions",
]


@dataclasses.dataclass(frozen=True)
class Workload:
    """One workload: model shape, prompt size, input recipe and selection settings."""
    name: str
    L: int
    H: int
    H_kv: int
    d: int
    M: int                      # prompt length (for a batch: the maximum)
    N: int                      # look-ahead queries
    dtype: str                  # "f32" or "bf16"
    chunk: int
    pool_k: int
    mode: str                   # "topk" or "mass"
    keep_rate: float = 0.0      # top-K mode
    mass: float = 0.0           # mass mode
    boost: Optional[tuple] = None   # (first_n, first_mult, last_n, last_mult, normalize)
    needle_kind: str = "runs"   # "single" or "runs"
    needle_count: int = 0       # single needles
    needle_frac: float = 0.0    # runs
    run_min: int = 0
    run_max: int = 0
    batch: int = 1
    M_min: int = 0              # batch: prompt lengths uniform in [M_min, M]
    seed: int = 0               # the workload's own seed for its inputs

    @property
    def G(self) -> int:
        return self.H // self.H_kv

    def k_bytes_per_token(self) -> int:
        """Bytes of K_prompt per prompt token (the minimum HBM traffic of the path)."""
        return self.L * self.H_kv * self.d * (4 if self.dtype == "f32" else 2)


# The five workloads, each with its own seed.
WORKLOADS = [
    Workload("tiny-f32-512", L=2, H=4, H_kv=2, d=64, M=512, N=4, dtype="f32",
             chunk=32, pool_k=3, mode="topk", keep_rate=0.3,
             needle_kind="single", needle_count=16, seed=0),
    Workload("llama8b-bf16-8k", L=32, H=32, H_kv=8, d=128, M=8192, N=8, dtype="bf16",
             chunk=32, pool_k=3, mode="topk", keep_rate=0.3,
             needle_frac=0.05, run_min=8, run_max=64, seed=1),
    Workload("llama8b-bf16-32k", L=32, H=32, H_kv=8, d=128, M=32768, N=8, dtype="bf16",
             chunk=32, pool_k=3, mode="topk", keep_rate=0.1,
             needle_frac=0.02, run_min=16, run_max=128, seed=2),
    Workload("llama8b-bf16-128k", L=32, H=32, H_kv=8, d=128, M=131072, N=8, dtype="bf16",
             chunk=64, pool_k=3, mode="topk", keep_rate=0.1,
             needle_frac=0.01, run_min=16, run_max=128, seed=3),
    Workload("v3-batch16-0.8b-bf16", L=24, H=16, H_kv=4, d=64, M=32768, N=8, dtype="bf16",
             chunk=32, pool_k=1, mode="mass", mass=0.85,
             boost=(64, 1.5, 128, 1.3, 1),
             needle_frac=0.05, run_min=8, run_max=64, batch=16, M_min=2048, seed=4),
]
BY_NAME = {w.name: w for w in WORKLOADS}
# the v3 structural boosts: first 64 tokens x1.5, last 128 x1.3, scores min-max normalised first
V3_BOOST = BY_NAME["v3-batch16-0.8b-bf16"].boost


# ---------------------------------------------------------------------------
# bf16 helpers (plain bit manipulation; round to nearest, ties to even)
# ---------------------------------------------------------------------------

def bf16_bits_from_f32(x: np.ndarray, out: Optional[np.ndarray] = None) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even) and return the uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).copy()
    t = u >> 16
    t &= 1
    t += 0x7FFF
    u += t
    u >>= 16
    if out is None:
        return u.astype(np.uint16)
    out[...] = u.reshape(out.shape)
    return out


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """The exact fp32 value of each bf16 bit pattern."""
    return (b.astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# Generator
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class Inputs:
    """One request.  For bf16 the arrays hold uint16 bit patterns, else fp32."""
    wl: Workload
    M: int
    Q_la: np.ndarray        # [N, L, H, d]
    K_prompt: np.ndarray    # [L, H_kv, M, d]
    K_la: np.ndarray        # [L, H_kv, N, d]
    needles: np.ndarray     # sorted int64 positions

    def f32(self, name: str) -> np.ndarray:
        a = getattr(self, name)
        return f32_from_bf16_bits(a) if a.dtype == np.uint16 else a


def needle_positions(rng: np.random.Generator, wl: Workload, M: int) -> np.ndarray:
    """Needle positions of one request (position 0, the sink, is never a needle)."""
    if M <= 1:
        return np.zeros(0, np.int64)
    if wl.needle_kind == "single":
        k = min(wl.needle_count, M - 1)
        return np.sort(rng.choice(np.arange(1, M), size=k, replace=False)).astype(np.int64)
    target = int(round(wl.needle_frac * M))
    mark = np.zeros(M, dtype=bool)
    count = 0
    while count < target:
        length = int(rng.integers(wl.run_min, wl.run_max + 1))
        length = min(length, M - 1)
        start = int(rng.integers(1, M - length + 1))
        before = int(mark[start:start + length].sum())
        mark[start:start + length] = True
        count += length - before
    return np.flatnonzero(mark).astype(np.int64)


def _threads() -> int:
    try:
        return max(1, min(16, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return max(1, min(16, os.cpu_count() or 1))


def make_inputs(wl: Workload, seed: int, M: Optional[int] = None, request: int = 0) -> Inputs:
    """Draw one request of workload ``wl`` (prompt length ``M``, default wl.M)."""
    M = wl.M if M is None else int(M)
    L, H, H_kv, d, N, G = wl.L, wl.H, wl.H_kv, wl.d, wl.N, wl.G
    ss = np.random.SeedSequence([int(seed), int(request)])
    kids = ss.spawn(3 + L * H_kv)
    rng_needle = np.random.Generator(np.random.PCG64(kids[0]))
    rng_q = np.random.Generator(np.random.PCG64(kids[1]))
    rng_kla = np.random.Generator(np.random.PCG64(kids[2]))

    needles = needle_positions(rng_needle, wl, M)
    Q = rng_q.standard_normal((N, L, H, d), dtype=np.float32)
    K_la = rng_kla.standard_normal((L, H_kv, N, d), dtype=np.float32)
    # mean query of each (layer, KV head) group, over look-ahead steps and heads
    mu = Q.reshape(N, L, H_kv, G, d).mean(axis=(0, 3), dtype=np.float64).astype(np.float32)

    bf16 = wl.dtype == "bf16"
    K = np.empty((L, H_kv, M, d), dtype=np.uint16 if bf16 else np.float32)

    def slab(idx: int) -> None:
        l, g = divmod(idx, H_kv)
        rng = np.random.Generator(np.random.PCG64(kids[3 + idx]))
        k = rng.standard_normal((M, d), dtype=np.float32)
        if M > 0:
            k[0] *= np.float32(4.0)
        if needles.size:
            k[needles] += np.float32(3.0) * mu[l, g]
        if bf16:
            bf16_bits_from_f32(k, out=K[l, g])
        else:
            K[l, g] = k

    n = L * H_kv
    if n * M * d >= (1 << 22):
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(slab, range(n)))
    else:
        for i in range(n):
            slab(i)

    if bf16:
        Q = bf16_bits_from_f32(Q).reshape(Q.shape)
        K_la = bf16_bits_from_f32(K_la).reshape(K_la.shape)
    return Inputs(wl, M, Q, K, K_la, needles)


@dataclasses.dataclass
class VarlenInputs:
    """A batch of independent requests, packed along the token axis."""
    wl: Workload
    requests: list          # list[Inputs]
    cu_M: np.ndarray        # [B+1] int64 prefix sums of the prompt lengths

    def packed(self):
        """(Q_la[B,N,L,H,d], K_prompt[L,H_kv,sum M,d], K_la[B,L,H_kv,N,d], cu_M)."""
        Q = np.stack([r.Q_la for r in self.requests])
        K_la = np.stack([r.K_la for r in self.requests])
        K = np.concatenate([r.K_prompt for r in self.requests], axis=2)
        return Q, K, K_la, self.cu_M


def make_varlen_inputs(wl: Workload, seed: int, lengths=None) -> VarlenInputs:
    """Draw a batch; lengths default to uniform integers in [wl.M_min, wl.M]."""
    if lengths is None:
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), 1 << 20])))
        lengths = rng.integers(wl.M_min, wl.M + 1, size=wl.batch)
    lengths = [int(x) for x in lengths]
    reqs = [make_inputs(wl, seed, M=m, request=b) for b, m in enumerate(lengths)]
    cu = np.zeros(len(lengths) + 1, np.int64)
    cu[1:] = np.cumsum(lengths)
    return VarlenInputs(wl, reqs, cu)


def make_workload_inputs(name: str):
    """Inputs of the named workload, drawn with its own seed."""
    wl = BY_NAME[name]
    if wl.batch > 1:
        return make_varlen_inputs(wl, wl.seed)
    return make_inputs(wl, wl.seed)
