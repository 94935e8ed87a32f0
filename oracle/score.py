"""fp64 oracle of look-ahead attention scoring and max/max/mean aggregation.

TEST INFRASTRUCTURE (see the package docstring for who may call it).

Definitions followed:
  * attention score a_ij = softmax(Q_{M+j} K^T / sqrt(d))_i for prompt token i
    and look-ahead step j, per layer and query head -- paper review "Speculative
    Prefill ...", section "core algorithm: token importance speculation" and the
    first formula of section "core formulas";
  * aggregation: max over heads, then max over layers, then mean over the N
    look-ahead steps -- paper review, section "aggregate attention scores as
    token importance" (max-mean aggregation over the [N, L, S, H] tensor), and
    the llama.cpp guide "SpecPrefill -- Implementation Guide", section "Token
    Importance" and its function compute_imp.

Inputs are numpy arrays of real values (fp32 or fp64) or uint16 arrays, which
are read as bf16 bit patterns (value = the bits shifted into the high half of
an fp32).  All arithmetic is fp64.
"""
from __future__ import annotations

import math

import numpy as np


def _f64(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.uint16:                        # bf16 bit patterns
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def lookahead_rows(Q_la, K_la, l: int, h: int, G: int, shift: int = 0) -> np.ndarray:
    """Causal look-ahead logits u[j, k] = Q_la[j,l,h] . K_la[l,g,k] / sqrt(d), k <= j - shift.

    Entries with k > j - shift are -inf (row j has not seen later steps).
    shift = 1 is the capture with the prompt's last query as row 0 (it sees
    no look-ahead key) followed by the decode steps (row j sees keys 0..j-1).
    """
    d = Q_la.shape[3]
    g = h // G
    q = _f64(Q_la[:, l, h, :])                      # [N_rows, d]
    kla = _f64(K_la[l, g])                          # [N_la, d]
    u = (q @ kla.T) / math.sqrt(d)                  # [N_rows, N_la]
    for j in range(u.shape[0]):
        u[j, max(0, j - shift + 1):] = -np.inf
    return u


def _softmax_rows(s: np.ndarray, u: np.ndarray, shift: int = 0):
    """Row-wise softmax over [prompt logits s[j] | look-ahead logits u[j, :j-shift+1]]."""
    N = s.shape[0]
    a = np.empty_like(s)
    a_la = np.zeros_like(u)
    for j in range(N):
        nl = max(0, j - shift + 1)
        row = np.concatenate([s[j], u[j, :nl]])
        m = row.max()
        lse = m + math.log(np.exp(row - m).sum())
        a[j] = np.exp(s[j] - lse)
        a_la[j, :nl] = np.exp(u[j, :nl] - lse)
    return a, a_la


def attention_rows(Q_la, K_prompt, K_la, l: int, h: int, k64=None, shift: int = 0):
    """Post-softmax attention of every look-ahead query of (layer l, head h).

    Returns (a[N, M], a_la[N, N]): a[j, i] is the weight of prompt token i and
    a_la[j, k] that of look-ahead key k (zero for k > j).  Every row of
    [a | a_la] sums to 1.  ``k64`` may pass K_prompt[l, g] already in fp64.
    """
    N, L, H, d = Q_la.shape
    H_kv = K_prompt.shape[1]
    G = H // H_kv
    g = h // G
    q = _f64(Q_la[:, l, h, :])                      # [N, d]
    k = _f64(K_prompt[l, g]) if k64 is None else k64   # [M, d]
    s = (q @ k.T) / math.sqrt(d)                    # [N, M] prompt logits
    u = lookahead_rows(Q_la, K_la, l, h, G, shift)  # [N, N_la] look-ahead logits
    return _softmax_rows(s, u, shift)


def importance(Q_la, K_prompt, K_la, shift: int = 0) -> np.ndarray:
    """importance_i = (1/N) sum_j max_{l,h} a[l,h,j,i]   (fp64, shape [M]).

    Q_la[N, L, H, d], K_prompt[L, H_kv, M, d], K_la[L, H_kv, N - shift, d].
    shift = 1: row 0 is the prompt's last query captured at prefill (its
    softmax covers only the prompt keys), rows 1..N-1 the decode steps (the
    llama.cpp guide captures the prefill's last row and then the decode
    steps).  With N = 0 every token gets importance 1.0 (compute_imp's
    fallback when no step was captured).
    """
    N, L, H, d = Q_la.shape
    H_kv, M = K_prompt.shape[1], K_prompt.shape[2]
    G = H // H_kv
    if N == 0:
        return np.ones(M, dtype=np.float64)
    best = np.zeros((N, M), dtype=np.float64)       # max over (l, h) so far; weights are >= 0
    for l in range(L):
        for g in range(H_kv):
            k64 = _f64(K_prompt[l, g])
            for h in range(g * G, (g + 1) * G):
                a, _ = attention_rows(Q_la, K_prompt, K_la, l, h, k64=k64, shift=shift)
                np.maximum(best, a, out=best)
    total = np.zeros(M, dtype=np.float64)
    for j in range(N):                              # mean over look-ahead steps, j in order
        total += best[j]
    return total / N


def row_lse(Q_la, K_prompt, K_la, shift: int = 0) -> np.ndarray:
    """lse[l, h, j] = log(sum_i exp(s[l,h,j,i]) + sum_{k<=j} exp(u[l,h,j,k]))  (fp64, [L, H, N]).

    The normaliser of look-ahead query j's softmax over the M prompt keys and
    look-ahead keys 0..j: the quantity the speculator's own look-ahead decode
    attention already holds.  Computed with the max shift, row by row.
    """
    N, L, H, d = Q_la.shape
    H_kv = K_prompt.shape[1]
    G = H // H_kv
    out = np.empty((L, H, N), dtype=np.float64)
    for l in range(L):
        for g in range(H_kv):
            k = _f64(K_prompt[l, g])
            for h in range(g * G, (g + 1) * G):
                q = _f64(Q_la[:, l, h, :])
                s = (q @ k.T) / math.sqrt(d)
                u = lookahead_rows(Q_la, K_la, l, h, G, shift)
                for j in range(N):
                    row = np.concatenate([s[j], u[j, :max(0, j - shift + 1)]])
                    m = row.max()
                    out[l, h, j] = m + math.log(np.exp(row - m).sum())
    return out


def importance_given_lse(Q_la, K_prompt, lse) -> np.ndarray:
    """importance_i = (1/N) sum_j max_{l,h} exp(s[l,h,j,i] - lse[l,h,j])  (fp64, [M]).

    The same max/max/mean aggregation as importance(), with each row's softmax
    normaliser lse[L, H, N] given by the caller instead of computed from the
    keys (the single-pass variant: K is read once).
    """
    N, L, H, d = Q_la.shape
    H_kv, M = K_prompt.shape[1], K_prompt.shape[2]
    G = H // H_kv
    lse = np.asarray(lse, dtype=np.float64)
    if N == 0:
        return np.ones(M, dtype=np.float64)
    best = np.zeros((N, M), dtype=np.float64)
    for l in range(L):
        for g in range(H_kv):
            k = _f64(K_prompt[l, g])
            for h in range(g * G, (g + 1) * G):
                q = _f64(Q_la[:, l, h, :])
                s = (q @ k.T) / math.sqrt(d)        # [N, M]
                a = np.exp(s - lse[l, h][:, None])
                np.maximum(best, a, out=best)
    total = np.zeros(M, dtype=np.float64)
    for j in range(N):
        total += best[j]
    return total / N
