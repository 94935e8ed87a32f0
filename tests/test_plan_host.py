"""Host-side checks of the tensor-core scoring planner (no GPU): the plans of the
benchmark shapes, and invariants every plan must keep over a sweep of prompt
lengths and shapes (CTAs on the SMs, every token in some CTA's range, ranges
within the tile limits, TMEM and shared memory within the GB300's)."""
import pytest

SMS = 152
TMEM_COLS = 512
SMEM_PER_CTA = 227 * 1024


@pytest.fixture(scope="module")
def sp():
    from speculative_prefill_token_sp_gb300 import build
    build.build()
    import speculative_prefill_token_sp_gb300 as m
    m.lib()
    return m


def test_benchmark_shapes(sp):
    # 8B shape: L = 32, H = 32, H_kv = 8, d = 128, N = 8
    p = sp.sp_test_score_plan(32, 32, 8, 128, 32768, 8)
    assert (p["F"], p["Pc"], p["tiles"], p["lag"]) == (4, 38, 7, 2)
    p = sp.sp_test_score_plan(32, 32, 8, 128, 131072, 8)
    assert (p["F"], p["Pc"], p["tiles"], p["lag"]) == (1, 152, 7, 2)
    # 8K: ranges of whole tiles (13 classes of 11 CTAs, six full tiles) rather
    # than 16 classes of 9 with a nearly empty eighth tile
    p = sp.sp_test_score_plan(32, 32, 8, 128, 8192, 8)
    assert (p["F"], p["Pc"], p["tiles"]) == (13, 11, 6)
    # 0.8B shape at d = 64
    p = sp.sp_test_score_plan(24, 16, 4, 64, 131072, 8)
    assert (p["F"], p["Pc"], p["tiles"]) == (1, 152, 7)


def test_shapes_outside_the_path(sp):
    assert sp.sp_test_score_plan(32, 32, 8, 96, 32768, 8) is None      # d not 64 or 128
    assert sp.sp_test_score_plan(32, 136, 8, 128, 32768, 8) is None    # 17 query heads per KV head
    assert sp.sp_test_score_plan(32, 32, 8, 128, 310000, 8) is None    # over 16 tiles per CTA and slab
    assert sp.sp_test_score_plan(32, 30, 8, 128, 4096, 8) is None      # H not a multiple of H_kv


@pytest.mark.parametrize("shape", [(32, 32, 8, 128, 8), (24, 16, 4, 64, 8), (2, 4, 2, 64, 4), (32, 32, 8, 128, 16),
                                   (32, 96, 8, 128, 8), (28, 28, 4, 128, 4), (16, 64, 4, 64, 2)])
def test_plan_invariants(sp, shape):
    L, H, H_kv, d, N = shape
    S = L * H_kv
    lengths = sorted({1, 31, 32, 33, 127, 128, 129, 1000, 4096, 4097, 8192, 12345, 16384, 32768, 50000,
                      65536, 100000, 131072, 200000, 262144})
    for M in lengths:
        p = sp.sp_test_score_plan(L, H, H_kv, d, M, N, SMS)
        if p is None:
            continue
        F, Pc, P, tiles, tpg, land, held, lag = (p[k] for k in ("F", "Pc", "P", "tiles", "tiles_per_group",
                                                                 "land", "held", "lag"))
        units = (M + 31) // 32
        assert P == F * Pc and 1 <= P <= SMS and 1 <= F <= min(16, S), (M, p)
        assert Pc * ((units + Pc - 1) // Pc) >= units, (M, p)            # every token has a CTA
        per_cta = (units + Pc - 1) // Pc * 32
        assert tiles == (per_cta + 127) // 128 and tiles <= 16, (M, p)
        assert F == 1 or tiles <= 8, (M, p)                               # classes keep ranges short
        assert tpg == (tiles + 1) // 2, (M, p)
        assert lag == held - 1 and held >= 1 and held * tpg <= 32, (M, p)
        # TMEM: both groups' landing tiles (32 columns each) and held fp16 slabs (16 per tile)
        assert 2 * land * 32 + 2 * held * tpg * 16 <= TMEM_COLS, (M, p)
        assert p["smem_bytes"] <= SMEM_PER_CTA, (M, p)

