"""The seeded generator: determinism, shapes and the stated recipe."""
import numpy as np

import workloads as W


def test_deterministic_and_shapes():
    a = W.make_workload_inputs("tiny-f32-512")
    b = W.make_workload_inputs("tiny-f32-512")
    wl = W.BY_NAME["tiny-f32-512"]
    assert a.Q_la.shape == (wl.N, wl.L, wl.H, wl.d)
    assert a.K_prompt.shape == (wl.L, wl.H_kv, wl.M, wl.d)
    assert a.K_la.shape == (wl.L, wl.H_kv, wl.N, wl.d)
    for name in ("Q_la", "K_prompt", "K_la"):
        assert np.array_equal(getattr(a, name), getattr(b, name))
    assert a.needles.size == 16 and 0 not in a.needles


def test_needle_runs_fraction():
    wl = W.BY_NAME["llama8b-bf16-8k"]
    rng = np.random.default_rng(0)
    pos = W.needle_positions(rng, wl, wl.M)
    assert pos.size >= round(0.05 * wl.M) and pos.size < round(0.05 * wl.M) + wl.run_max
    assert pos.min() >= 1


def test_bf16_rounding_ties_to_even():
    x = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e-5], dtype=np.float32)
    b = W.bf16_bits_from_f32(x)
    back = W.f32_from_bf16_bits(b)
    # 1 + 2^-8 is half-way between 1 and 1 + 2^-7: ties to even -> 1.0
    assert back[1] == 1.0
    # 1 + 3*2^-8 is half-way between 1 + 2^-7 and 1 + 2^-6: ties to even -> 1 + 2^-6
    assert back[2] == 1.015625
    assert back[3] == -2.5
    assert abs(back[4] - 3.0e-5) <= 3.0e-5 * 2 ** -8


def test_varlen_packing():
    wl = W.BY_NAME["v3-batch16-0.8b-bf16"]
    v = W.make_varlen_inputs(wl, 4, lengths=[5, 0, 9])
    Q, K, Kla, cu = v.packed()
    assert cu.tolist() == [0, 5, 5, 14]
    assert K.shape == (wl.L, wl.H_kv, 14, wl.d)
    assert Q.shape == (3, wl.N, wl.L, wl.H, wl.d)
    assert np.array_equal(K[:, :, 5:14], v.requests[2].K_prompt)
