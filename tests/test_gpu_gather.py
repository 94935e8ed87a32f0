"""sp_gather_kept against the gather oracle, bit-exact: the kept positions come
from sp_select_varlen on fp32 importance (selection itself is checked bit-exact
elsewhere), the oracle gathers from the same kept lists."""
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


@pytest.mark.parametrize("lengths", [[10], [300, 0, 1, 129, 1000, 0], [5000, 2048, 77]])
def test_gather_matches_oracle(sp, lengths):
    import torch
    rng = np.random.default_rng(len(lengths) * 1000 + sum(lengths))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    T = int(cu[-1])
    imp = rng.random(T).astype(np.float32)
    token_ids = rng.integers(0, 150000, T).astype(np.int32)
    imp_d = torch.from_numpy(imp).cuda()
    kept_d, n_d = sp.select_varlen(imp_d, cu, 16, 3, "topk", 0.3, trim=False)
    kept = kept_d.cpu().numpy()
    n = n_d.cpu().numpy()
    lists = [kept[cu[b]:cu[b] + n[b]] for b in range(len(lengths))]
    tokens, positions, cu_kept = sp.gather_kept(torch.from_numpy(token_ids).cuda(), cu, kept_d, n_d)
    torch.cuda.synchronize()
    w_tok, w_pos, w_cu, w_next = oracle.gather_kept(token_ids, cu, lists)
    tot = int(w_cu[-1])
    np.testing.assert_array_equal(cu_kept.cpu().numpy(), w_cu)
    np.testing.assert_array_equal(tokens.cpu().numpy()[:tot], w_tok)
    np.testing.assert_array_equal(positions.cpu().numpy()[:tot], w_pos)
    np.testing.assert_array_equal(w_next, lengths)
