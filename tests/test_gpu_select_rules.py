"""sp_select_rules bit-exact against the oracle's select_rules on the same fp32
importance: the guide's rules (128, always-kept tokens, cap 2000) and variants
on prompts that exercise the keep-all rule, the back-fill and the cap."""
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


CASES = [
    # (M, chunk, pool_k, mode, rate, rules)
    (3, 32, 1, "topk", 0.3, (128, 1, 2000)),          # M <= eff_min: everything
    (100, 4, 3, "topk", 0.05, (128, 1, 0)),           # back-fill
    (1000, 32, 3, "topk", 0.1, (128, 1, 2000)),
    (32768, 32, 3, "topk", 0.1, (128, 1, 2000)),      # cap 3296 -> 2000
    (32768, 32, 3, "topk", 0.1, (0, 0, 1000)),        # cap only
    (5000, 16, 1, "mass", 0.85, (128, 1, 0)),
    (77, 8, 1, "topk", 0.01, (4096, 1, 50)),          # back-fill to everything, then cap
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "M{}c{}p{}{}r{}-{}".format(*c[:5], "_".join(map(str, c[5]))))
def test_rules_match_oracle(sp, case):
    import torch
    M, chunk, pool_k, mode, rate, rules = case
    rng = np.random.default_rng(M + chunk)
    imp = rng.random(M).astype(np.float32)
    boost = (64, 1.5, 128, 1.3, 1) if mode == "mass" else None
    got = sp.select_rules(torch.from_numpy(imp).cuda(), chunk, pool_k, mode, rate, boost, rules).cpu().numpy()
    want, n = oracle.select_rules(imp, chunk, pool_k, mode, rate, boost, min_tok=rules[0],
                                  always_keep=bool(rules[1]), max_keep=rules[2])
    assert got.shape[0] == n
    np.testing.assert_array_equal(got, want)
