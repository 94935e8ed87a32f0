"""Oracle of the sparse-prefill input gather (integer work only).

TEST INFRASTRUCTURE (see the package docstring for who may call it).

Definition followed (paper review "Speculative Prefill ...", section "core
algorithm: position ID recovery"; llama.cpp guide, "How It Works: sparse
prefill"): the target prefills only the kept tokens, each with its original
position ID, and decoding continues at position M, M + 1, ... of the full
prompt.  For a batch, the requests' kept tokens are packed one request after
another, each request's in ascending position order.
"""
from __future__ import annotations

import numpy as np


def gather_kept(token_ids, cu_M, kept):
    """token_ids [T] (packed by cu_M), kept: per request an ascending array of
    kept positions (relative to the request's start).

    Returns (tokens int32 [sum n_b], positions int32 [sum n_b], cu_kept int64
    [B + 1], next_pos int64 [B]) where request b's entries are
    tokens[cu_kept[b] + i] = token_ids[cu_M[b] + kept[b][i]],
    positions[cu_kept[b] + i] = kept[b][i], and next_pos[b] = M_b is the first
    decode position.
    """
    token_ids = np.asarray(token_ids)
    cu = np.asarray(cu_M, dtype=np.int64)
    B = cu.shape[0] - 1
    tokens, positions = [], []
    cu_kept = [0]
    for b in range(B):
        for p in kept[b]:
            p = int(p)
            assert 0 <= p < cu[b + 1] - cu[b]
            tokens.append(int(token_ids[cu[b] + p]))
            positions.append(p)
        cu_kept.append(len(tokens))
    return (np.asarray(tokens, dtype=np.int32), np.asarray(positions, dtype=np.int32),
            np.asarray(cu_kept, dtype=np.int64), (cu[1:] - cu[:-1]).astype(np.int64))
