"""sp_score_prefill (the prefill's last query as row 0, then N decode steps)
against the oracle's shift = 1 aggregation, element by element, on both
paths (bf16 tensor cores, fp32 general path), with N = 0 (only the prefill row)."""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_helpers import check_importance, to_device

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


SHAPES = [
    # (L, H, H_kv, d, M, N_decode, dtype)
    (2, 32, 8, 128, 8192, 7, "bf16"),      # 8 rows x G 4 = 32: tensor cores
    (1, 32, 8, 128, 40960, 7, "bf16"),
    (2, 4, 2, 64, 300, 0, "bf16"),         # only the prefill row
    (2, 32, 8, 128, 3000, 11, "bf16"),     # 12 rows: passes of 8 and 4 steps (the second sees keys 0..10)
    (2, 4, 2, 64, 513, 3, "f32"),          # general path
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "L{}H{}Hkv{}d{}M{}N{}{}".format(*s))
def test_prefill_row_parity(sp, shape):
    import torch
    L, H, H_kv, d, M, Nd, dt = shape
    wl = W.Workload("t", L=L, H=H, H_kv=H_kv, d=d, M=M, N=Nd + 1, dtype=dt, chunk=32, pool_k=3, mode="topk",
                    keep_rate=0.1, needle_frac=0.02, run_min=8, run_max=64)
    x = W.make_inputs(wl, seed=3000 + M)
    Kla = np.ascontiguousarray(x.K_la[:, :, :Nd])            # the decode steps' keys
    imp = sp.score_prefill(to_device(x.Q_la), to_device(x.K_prompt), to_device(Kla), check=True)
    torch.cuda.synchronize()
    ref = oracle.importance(x.Q_la, x.K_prompt, Kla, shift=1)
    check_importance(imp.cpu().numpy(), ref, dt, str(shape))
