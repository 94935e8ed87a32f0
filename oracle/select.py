"""fp64 oracle of chunk scoring, pooling, chunk selection and position-ID output.

TEST INFRASTRUCTURE (see the package docstring for who may call it).

Definitions followed:
  * chunk_score_k = (1/|C_k|) sum_{i in C_k} importance_i over contiguous chunks;
    a last partial chunk is averaged over its real size -- paper review
    "Speculative Prefill ...", section "chunk selection and pooling denoising"
    and its chunk formula; llama.cpp guide "SpecPrefill -- Implementation
    Guide", function select_chunks (nc = ceil(M / chunk), sums in double);
  * 1D average pooling of the chunk scores, then top-K chunks -- paper review,
    same section (pooling is read as applied before the top-K choice);
  * kc = max(1, ceil(nc * keep_rate)) with an fp32 product -- select_chunks;
  * v3: min-max normalisation to [0, 1] (guide, "v3.1 Optimizations: Score
    Normalization"), structural boost x1.5 on the first 64 and x1.3 on the last
    128 positions (guide, "v3 Improvements: Structural Token Boosting"),
    chunks kept from the highest score until the cumulative attention mass
    reaches tau (guide, "v3 Improvements: Cumulative Attention Mass Selection");
  * output: kept tokens' original position IDs, ascending; decoding continues
    at M, M+1, ... -- paper review, section "position ID recovery" example
    [0..9] -> [0, 1, 3, 6, 7], decode 10, 11, 12; select_chunks sorts its output.

Operation order (fixed, so that an implementation can reproduce every fp64
rounding): token scores are fp64; chunk sums add left to right starting at 0.0
and are divided once by the chunk's size; pooled values add the in-range window
left to right from 0.0 and divide once by the window's count; normalisation is
(x - mn) / (mx - mn); each boost is one multiply, first-N then last-N; the
total mass adds chunk sums in chunk order; the running mass adds chunk sums in
ranked order.
"""
from __future__ import annotations

import math

import numpy as np


def token_scores(importance, boost=None) -> np.ndarray:
    """fp64 token scores, after optional min-max normalisation and boosts.

    boost = (first_n, first_mult, last_n, last_mult, normalize) or None.
    """
    imp = np.asarray(importance, dtype=np.float32)
    x = imp.astype(np.float64)
    if boost is None:
        return x
    return normalize_boost(imp, boost)


def normalize_boost(importance, boost) -> np.ndarray:
    """v3 token scores: min-max normalise (if asked) then multiply the boosts.

    If max == min every normalised score is 1.0 (the guide's fallback value).
    Overlapping boost ranges (M < first_n + last_n) get both multipliers.
    """
    first_n, first_mult, last_n, last_mult, normalize = boost
    imp = np.asarray(importance, dtype=np.float32)
    M = imp.shape[0]
    x = imp.astype(np.float64)
    if normalize and M > 0:
        mn = float(imp.min())
        mx = float(imp.max())
        if mx > mn:
            x = np.array([(float(v) - mn) / (mx - mn) for v in imp], dtype=np.float64)
        else:
            x = np.ones(M, dtype=np.float64)
    x = x.copy()
    for i in range(min(first_n, M)):
        x[i] = x[i] * first_mult
    for i in range(max(0, M - last_n), M):
        x[i] = x[i] * last_mult
    return x


def chunk_sums(x, chunk: int):
    """(sums[nc], counts[nc]) of contiguous chunks; nc = ceil(M / chunk)."""
    x = np.asarray(x, dtype=np.float64)
    M = x.shape[0]
    nc = (M + chunk - 1) // chunk
    sums = np.zeros(nc, dtype=np.float64)
    counts = np.zeros(nc, dtype=np.int64)
    for c in range(nc):
        s = 0.0
        lo, hi = c * chunk, min((c + 1) * chunk, M)
        for i in range(lo, hi):
            s = s + float(x[i])
        sums[c] = s
        counts[c] = hi - lo
    return sums, counts


def chunk_means(x, chunk: int) -> np.ndarray:
    """chunk_score_c = (sum of the chunk's scores) / (its real size)."""
    sums, counts = chunk_sums(x, chunk)
    return np.array([float(s) / float(n) for s, n in zip(sums, counts)], dtype=np.float64)


def avg_pool(v, k: int) -> np.ndarray:
    """Stride-1, centred, length-preserving average pool; edges average in-range values."""
    if k < 1 or k % 2 == 0:
        raise ValueError("pool kernel must be odd and >= 1")
    v = np.asarray(v, dtype=np.float64)
    n = v.shape[0]
    r = (k - 1) // 2
    out = np.zeros(n, dtype=np.float64)
    for c in range(n):
        lo, hi = max(0, c - r), min(n - 1, c + r)
        s = 0.0
        for t in range(lo, hi + 1):
            s = s + float(v[t])
        out[c] = s / float(hi - lo + 1)
    return out


def keep_count(nc: int, keep_rate: float) -> int:
    """kc = max(1, ceil(f32(nc) * f32(keep_rate))), at most nc (0 when nc == 0)."""
    if nc == 0:
        return 0
    prod = np.float32(nc) * np.float32(keep_rate)
    kc = max(1, int(math.ceil(float(prod))))
    return min(kc, nc)


def _ranked(scores) -> list:
    """Chunk indices by score descending, ties to the lower index."""
    scores = np.asarray(scores, dtype=np.float64)
    return sorted(range(scores.shape[0]), key=lambda c: (-float(scores[c]), c))


def topk_chunks(scores, kc: int) -> np.ndarray:
    """Boolean mask of exactly kc chunks with the largest scores (ties: lower index)."""
    n = len(scores)
    mask = np.zeros(n, dtype=bool)
    for c in _ranked(scores)[:kc]:
        mask[c] = True
    return mask


def mass_chunks(sums, means, tau: float) -> np.ndarray:
    """Cumulative-mass cut: rank by mean, keep the shortest prefix with mass >= tau*total."""
    n = len(sums)
    mask = np.zeros(n, dtype=bool)
    if n == 0:
        return mask
    total = 0.0
    for c in range(n):
        total = total + float(sums[c])
    target = float(tau) * total
    cum = 0.0
    for c in _ranked(means):
        cum = cum + float(sums[c])
        mask[c] = True
        if cum >= target:
            break
    return mask


def kept_positions(mask, chunk: int, M: int) -> np.ndarray:
    """Original position IDs of the kept chunks' tokens, ascending (int32)."""
    out = []
    for c in range(len(mask)):
        if mask[c]:
            out.extend(range(c * chunk, min((c + 1) * chunk, M)))
    return np.asarray(out, dtype=np.int32)


def select_mask(importance, chunk: int, pool_k: int, mode: str, rate: float, boost=None):
    """The chunk mask of the selection step (see select) and the prompt length.

    mode "topk": rate = keep_rate; chunk means -> avg pool (pool_k) -> top-kc.
    mode "mass": rate = tau; chunk means rank the chunks, chunk sums are the
    mass; pool_k must be 1.
    """
    imp = np.asarray(importance, dtype=np.float32)
    M = imp.shape[0]
    x = token_scores(imp, boost)
    sums, counts = chunk_sums(x, chunk)
    means = np.array([float(s) / float(n) for s, n in zip(sums, counts)], dtype=np.float64)
    nc = means.shape[0]
    if mode == "topk":
        p = avg_pool(means, pool_k)
        mask = topk_chunks(p, keep_count(nc, rate))
    elif mode == "mass":
        if pool_k != 1:
            raise ValueError("mass mode takes no pooling")
        mask = mass_chunks(sums, means, rate)
    else:
        raise ValueError(mode)
    return mask, M


def select(importance, chunk: int, pool_k: int, mode: str, rate: float, boost=None):
    """Whole selection step.  Returns (kept_pos int32[n_kept], n_kept).

    mode "topk": rate = keep_rate; chunk means -> avg pool (pool_k) -> top-kc.
    mode "mass": rate = tau; chunk means rank the chunks, chunk sums are the
    mass; pool_k must be 1.
    """
    mask, M = select_mask(importance, chunk, pool_k, mode, rate, boost)
    pos = kept_positions(mask, chunk, M)
    return pos, int(pos.shape[0])


def select_rules(importance, chunk: int, pool_k: int, mode: str, rate: float, boost=None, *,
                 min_tok: int = 0, always_keep: bool = False, max_keep: int = 0):
    """select() followed by keep_rules(): (kept_pos int32[n_kept], n_kept)."""
    mask, M = select_mask(importance, chunk, pool_k, mode, rate, boost)
    pos = keep_rules(kept_positions(mask, chunk, M), mask, M, chunk, min_tok, always_keep, max_keep)
    return pos, int(pos.shape[0])


def select_varlen(importance_packed, cu_M, chunk, pool_k, mode, rate, boost=None):
    """Per-request selection of a packed batch; returns a list of (kept_pos, n_kept)."""
    cu = np.asarray(cu_M, dtype=np.int64)
    return [select(importance_packed[cu[b]:cu[b + 1]], chunk, pool_k, mode, rate, boost)
            for b in range(cu.shape[0] - 1)]


def keep_rules(kept, mask, M: int, chunk: int, min_tok: int = 0, always_keep: bool = False,
               max_keep: int = 0) -> np.ndarray:
    """The guide's v2 keep rules on top of a chunk selection (llama.cpp guide,
    "Full Source Code": select_chunks' always-kept tokens and minimum-token
    back-fill, and the sparse-prefill cap SP_MAX_KEEP of its main program).

    kept: the selection's ascending positions; mask: its chunk mask.
      * min_tok > 0: eff_min = min(min_tok, max(4, M // 10)); a prompt of at
        most eff_min tokens keeps every token;
      * always_keep: tokens 0, 1, 2, 3 and, if M > 4, M - 2 and M - 1 are kept;
      * while fewer than eff_min tokens are kept, tokens of the chunks the
        selection left out join, chunk by chunk in index order and token by
        token, skipping tokens already kept;
      * the result is ascending;
      * max_keep > 0 and n > max_keep kept: every step-th kept token, step =
        n // max_keep, at most max_keep of them, the last of which is replaced
        by the last kept token.
    """
    mask = np.asarray(mask, dtype=bool)
    out = [int(p) for p in kept]
    eff_min = min(min_tok, max(4, M // 10)) if min_tok > 0 else 0
    if M <= eff_min:
        out = list(range(M))
    else:
        have = set(out)
        if always_keep:
            for a in [0, 1, 2, 3] + ([M - 2, M - 1] if M > 4 else []):
                if a < M and a not in have:
                    out.append(a)
                    have.add(a)
        if len(out) < eff_min:
            for c in range(len(mask)):
                if len(out) >= eff_min:
                    break
                if mask[c]:
                    continue
                for i in range(c * chunk, min((c + 1) * chunk, M)):
                    if len(out) >= eff_min:
                        break
                    if i not in have:
                        out.append(i)
                        have.add(i)
        out.sort()
    if max_keep > 0 and len(out) > max_keep:
        step = len(out) // max_keep
        capped = [out[i] for i in range(0, len(out), step)][:max_keep]
        if capped[-1] != out[-1]:
            capped[-1] = out[-1]
        out = capped
    return np.asarray(out, dtype=np.int32)
