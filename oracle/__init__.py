"""Plain, slow fp64 CPU oracle of SpecPrefill token-importance scoring and selection.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or run
anything in this package.  The product path (the CUDA library and its Python
binding) never does, and shares no code with it.

Sources (the three pages this method is described on):
  * [paper review] "Speculative Prefill: Turbocharging TTFT with Lightweight and
    Training-Free Token Importance Estimation" (xllm-io paper review of Liu,
    Chen, Zhang, arXiv 2502.02789), sections "core algorithm" and "core
    formulas".
  * [llama.cpp guide] "SpecPrefill -- Implementation Guide" (sliding-specprefill,
    specprefill.md), sections "How It Works", "v3 Improvements", "v3.1
    Optimizations & Bug Fixes", and the functions compute_imp / select_chunks
    in its "Full Source Code" section.

Readings taken where the pages are silent, garbled or at odds (each one is
pinned by the tests only as far as the mathematics allows):
  * logits are scaled by 1/sqrt(d) (the formula on the paper review omits it;
    the attention the guide captures is the model's scaled softmax);
  * look-ahead query j's softmax runs over all M prompt keys plus look-ahead
    keys 0..j (causal); importance reads only the prompt columns;
  * importance_i = (1/N) sum_j max_{l,h} a[l,h,j,i] (the formula on the paper
    review has a garbled index; its prose and the guide fix this order);
  * query head h reads KV head h // (H / H_kv)            -- parity unpinned by the pages
  * pooling: stride 1, centred window of pool_k chunks, edge windows average
    only their in-range chunks                              -- parity unpinned by the pages
  * top-K keeps exactly kc = max(1, ceil(f32(nc) * f32(keep_rate))) chunks,
    ties to the lower chunk index;
  * cumulative-mass mode ranks chunks by mean boosted score, a chunk's mass is
    the sum of its boosted token scores, and the shortest ranked prefix whose
    running mass reaches tau * total is kept             -- parity unpinned by the pages
  * N = 0 look-ahead steps gives importance 1.0 everywhere (the guide's
    compute_imp fallback when nothing was captured).
"""
from .score import importance, attention_rows, lookahead_rows, row_lse, importance_given_lse  # noqa: F401
from .select import (  # noqa: F401
    chunk_sums, chunk_means, avg_pool, keep_count, topk_chunks, normalize_boost,
    mass_chunks, kept_positions, select, select_varlen, keep_rules, select_mask, select_rules,
)
from .gather import gather_kept  # noqa: F401,E402
