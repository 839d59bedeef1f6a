"""The seeded input generator: determinism, sampling consistency, bf16 rounding, moments."""
import numpy as np
import torch

from tensor_transformer_mlp_tp_gb300 import inputs


def test_splitmix64_reference_values():
    # splitmix64 with state 0: the first outputs published with the generator's reference code
    # (Vigna, "splitmix64.c", xoshiro/xoroshiro page): 0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F
    states = np.array([0, 0x9E3779B97F4A7C15, (2 * 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    out = inputs._splitmix64(states)
    assert [int(v) for v in out] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_deterministic_and_per_tensor():
    w = inputs.small_workload(32, 16, 2)
    a1, _ = inputs.draw(w, "X", seed=0)
    a2, _ = inputs.draw(w, "X", seed=0)
    a3, _ = inputs.draw(w, "X", seed=1)
    b1, _ = inputs.draw(w, "A", seed=0)
    assert np.array_equal(a1, a2)
    assert not np.array_equal(a1, a3)
    assert not np.array_equal(a1.ravel()[:100], b1.ravel()[:100])


def test_row_sample_equals_full_rows():
    w = inputs.small_workload(40, 24, 2)
    full_bits, full_vals = inputs.draw(w, "X")
    rows = np.array([0, 3, 17, 39])
    sb, sv = inputs.draw(w, "X", rows=rows)
    assert np.array_equal(sb, full_bits[rows])
    assert np.array_equal(sv, full_vals[rows])
    # odd row length: pairs of counters straddle rows
    w2 = inputs.small_workload(9, 7, 1, F=28)
    fb, _ = inputs.draw(w2, "X", shape=(9, 7))
    sb2, _ = inputs.draw(w2, "X", rows=np.arange(9), shape=(9, 7))
    assert np.array_equal(fb, sb2)


def test_bf16_round_nearest_even_matches_torch():
    x = np.concatenate([np.random.default_rng(0).normal(0, 10, 100000).astype(np.float32),
                        np.array([1.00390625, 1.01171875, -1.00390625, 0.0, -0.0, 3.0e38], dtype=np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(inputs.f32_to_bf16_bits(x), ref)
    back = inputs.bf16_bits_to_f32(ref)
    assert np.array_equal(back, torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_normal_moments():
    z = inputs.normals(inputs.stream_key(0, "w", "t"), 400000)
    assert abs(z.mean()) < 0.01
    assert abs(z.std() - 1.0) < 0.01
    assert abs(np.mean(z ** 4) - 3.0) < 0.05


def test_workload_recipes():
    w = inputs.WORKLOADS["sp_block_fwd_bwd"]
    assert (w.T, w.d, w.F, w.N, w.rows_per_chunk) == (8192, 4096, 16384, 8, 1024)
    assert w.dists["bias"] is None
    assert inputs.WORKLOADS["sp_large_fwd"].rows_per_chunk == 512
    for w in inputs.WORKLOADS.values():
        assert w.F == 4 * w.d and w.F % w.N == 0 and w.T % w.N == 0
