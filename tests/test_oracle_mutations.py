"""Planted mistakes: each plausible slip in the oracle must make at least one pin fail.

Every case swaps one oracle function for a subtly wrong copy (on the CPU,
for the duration of the test) and runs a pin from ``test_oracle_pins``;
the pin has to raise.  This guards against pins that would pass whatever
the oracle computes.
"""
import numpy as np
import pytest

import oracle
import test_oracle_pins as pins

_orig = {name: getattr(oracle, name) for name in dir(oracle) if not name.startswith("__")}


def _gelu_tanh(x):
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1 + np.tanh(np.sqrt(2 / np.pi) * (x + 0.044715 * x ** 3)))


def _gelu_prime_no_pdf(x):
    return 0.5 * (1.0 + oracle._erf(np.asarray(x, dtype=np.float64) * oracle.SQRT_HALF))


def _mlp_reference_no_bias(X, A, B, b=None):
    return _orig["mlp_reference"](X, A, B, None)


def _shard_ranges_overlap(F, N):
    r = _orig["shard_ranges"](F, N)
    return [(max(lo - 1, 0), hi) for lo, hi in r]


def _layer_norm_unbiased(x, gamma, beta, eps=1e-5):
    x = np.asarray(x, dtype=np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    var = x.var(axis=-1, ddof=1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * gamma + beta


def _layer_norm_eps_outside(x, gamma, beta, eps=1e-5):
    x = np.asarray(x, dtype=np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / (np.sqrt(var) + eps) * gamma + beta


def _reduce_scatter_reversed(parts, N):
    return _orig["reduce_scatter"](parts, N)[::-1]


def _mlp_partials_transposed_shard(X, A, B, b, N):
    # uses the *last* shard's rows of B for every shard (a wrong index)
    F = np.asarray(A).shape[1]
    bias = oracle._bias_or_zero(b, F)
    r = oracle.shard_ranges(F, N)
    lo_last, hi_last = r[-1]
    return [oracle.row_parallel_partial(oracle.column_parallel(X, np.asarray(A)[:, lo:hi], bias[lo:hi]),
                                        np.asarray(B)[lo_last:hi_last, :]) for lo, hi in r]


def _mlp_backward_dA_uses_dH(X, A, B, b, dY):
    g = _orig["mlp_backward"](X, A, B, b, dY)
    dH = np.asarray(dY, dtype=np.float64) @ np.asarray(B, dtype=np.float64).T
    g["dA"] = np.asarray(X, dtype=np.float64).T @ dH          # dropped GeLU' factor
    return g


def _mlp_backward_sign(X, A, B, b, dY):
    g = _orig["mlp_backward"](X, A, B, b, dY)
    g["dX"] = -g["dX"]
    return g


def _ln_backward_no_mean_g(x, gamma, eps, dy):
    x = np.asarray(x, dtype=np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    rstd = 1.0 / np.sqrt(var + eps)
    xhat = (x - mu) * rstd
    g = dy * gamma
    dx = rstd * (g - xhat * (g * xhat).mean(axis=-1, keepdims=True))
    return dx, (dy * xhat).sum(axis=0), dy.sum(axis=0)


def _sp_backward_last_chunk_dgamma(*args, **kw):
    out = _orig["sp_backward"](*args, **kw)
    out["dgamma"] = out["dgamma"] / len(out["dX_chunks"])
    return out


def _rms_norm_no_rounding(x, weight, eps=1e-5):
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps) * weight


def _round_bf16_truncate(x):
    m, e = np.frexp(np.asarray(x, dtype=np.float64))
    return np.ldexp(np.trunc(m * 256.0), e - 8)


def _philox_bump_first(counter, key, rounds=10):
    k = ((int(key[0]) + oracle.PHILOX4X64_W[0]) % 2 ** 64, (int(key[1]) + oracle.PHILOX4X64_W[1]) % 2 ** 64)
    return _orig["philox4x64"](counter, k, rounds)


def _dropout_keep_halves_swapped(rows, d, row0, p, seed, offset):
    # odd elements take the low half and even ones the high half: flip each pair of columns
    base = _orig["dropout_keep"](rows, d, row0, p, seed, offset)
    return base.reshape(rows, d // 2, 2)[:, :, ::-1].reshape(rows, d)


def _sp_block_forward_unscaled(X_chunks, gamma, beta, eps, A, B, b, b2, p, seed, offset, N):
    Y = _orig["sp_block_forward"](X_chunks, gamma, beta, eps, A, B, b, b2, p, seed, offset, N)
    s = 1.0 - float(np.float32(p))
    return [x + (y - x) * s for x, y in zip(X_chunks, Y)]


def _sp_block_backward_no_residual(X_chunks, gamma, beta, eps, A, B, b, p, seed, offset, dY_chunks, N):
    g = _orig["sp_block_backward"](X_chunks, gamma, beta, eps, A, B, b, p, seed, offset, dY_chunks, N)
    g["dX_chunks"] = [dx - dy for dx, dy in zip(g["dX_chunks"], dY_chunks)]
    return g


def _round_e4m3_ties_away(x):
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, e = np.frexp(a)
    q = np.ldexp(1.0, np.maximum(e - 1, -6) - 3)
    return np.copysign(np.minimum(np.floor(a / q + 0.5) * q, 448.0), x)


def _fp8_scale_max(h, fp8_max=448.0, margin=0):
    m = float(np.max(h))
    return 1.0 if m <= 0 else fp8_max / m / 2.0 ** margin


def _mlp_fp8_one_descale(X, A, B, b, N, scales):
    sx, sa, sb, sh = scales
    return _orig["mlp_fp8"](X, A, B, b, N, (sx, sa, sb * 2.0, sh))


def _round_e5m2_three_bits(x):
    return _orig["round_e4m3"](x)


def _mlp_backward_fp8_wrong_dB_scale(X, A, B, b, dY, N, scales, grad_scales):
    g = _orig["mlp_backward_fp8"](X, A, B, b, dY, N, scales, grad_scales)
    g["dB"] = g["dB"] * float(np.float32(scales[3]))      # the H scale left out of the dequantisation
    return g


def _attention_head_unscaled(Q, K, V, causal):
    Q = np.asarray(Q, dtype=np.float64)
    return _orig["attention_head"](Q * np.sqrt(Q.shape[1]), K, V, causal)


def _attention_head_mask_off_by_one(Q, K, V, causal):
    Q, K, V = (np.asarray(a, dtype=np.float64) for a in (Q, K, V))
    if not causal:
        return _orig["attention_head"](Q, K, V, False)
    S = Q.shape[0]
    sc = Q @ K.T / np.sqrt(Q.shape[1])
    sc = np.where(np.tril(np.ones((S, S), dtype=bool), k=1), sc, -np.inf)   # also sees the next token
    w = np.exp(sc - sc.max(axis=1, keepdims=True))
    return (w / w.sum(axis=1, keepdims=True)) @ V


def _attention_head_backward_no_D(Q, K, V, dO, causal):
    Q, K, V, dO = (np.asarray(a, dtype=np.float64) for a in (Q, K, V, dO))
    hd = Q.shape[1]
    sc = Q @ K.T / np.sqrt(hd)
    if causal:
        sc = np.where(np.tril(np.ones(sc.shape, dtype=bool)), sc, -np.inf)
    P = np.exp(sc - sc.max(axis=1, keepdims=True))
    P /= P.sum(axis=1, keepdims=True)
    dS = P * (dO @ V.T)                                    # the softmax Jacobian's -D term dropped
    return dS @ K / np.sqrt(hd), dS.T @ Q / np.sqrt(hd), P.T @ dO


CASES = [
    ("attention_head_backward", _attention_head_backward_no_D,
     lambda: pins.test_attention_head_backward_autograd_witness(True)),
    ("attention_head", _attention_head_unscaled, lambda: pins.test_attention_head_torch_witness(False)),
    ("attention_head", _attention_head_mask_off_by_one, lambda: pins.test_attention_head_bruteforce()),
    ("head_ranges", lambda H, N: [(lo, hi) for lo, hi in _orig["head_ranges"](H, N)][::-1],
     lambda: pins.test_attention_tp_shard_sum_is_the_unsharded_block()),
    ("round_e5m2", _round_e5m2_three_bits, lambda: pins.test_round_e5m2_bruteforce_and_torch()),
    ("mlp_backward_fp8", _mlp_backward_fp8_wrong_dB_scale,
     lambda: pins.test_mlp_backward_fp8_error_is_the_formats_size()),
    ("round_e4m3", _round_e4m3_ties_away, lambda: pins.test_round_e4m3_bruteforce_and_ties()),
    ("fp8_scale", _fp8_scale_max, lambda: pins.test_fp8_delayed_scale_closed_forms()),
    ("mlp_fp8", _mlp_fp8_one_descale, lambda: pins.test_mlp_fp8_torch_witness()),
    ("philox4x64", _philox_bump_first, lambda: pins.test_philox_matches_numpy_bit_generator()),
    ("dropout_keep", _dropout_keep_halves_swapped, lambda: pins.test_dropout_keep_bits_come_from_the_stated_block_and_half(0.5)),
    ("sp_block_forward", _sp_block_forward_unscaled, lambda: pins.test_sp_block_forward_torch_witness(2, 0.25)),
    ("sp_block_backward", _sp_block_backward_no_residual, lambda: pins.test_sp_block_backward_autograd_witness(2, 0.25)),
    ("rms_norm", _rms_norm_no_rounding, lambda: pins.test_rms_norm_bruteforce_rows()),
    ("round_bf16", _round_bf16_truncate, lambda: pins.test_round_bf16_ties_and_witnesses()),
    ("gelu", _gelu_tanh, lambda: pins.test_gelu_textbook_values()),
    ("gelu", _gelu_tanh, lambda: pins.test_mlp_bruteforce_d8(3, 2)),
    ("gelu_prime", _gelu_prime_no_pdf, lambda: pins.test_gelu_prime_finite_difference()),
    ("gelu_prime", _gelu_prime_no_pdf, lambda: pins.test_backward_autograd_witness(2)),
    ("mlp_reference", _mlp_reference_no_bias, lambda: pins.test_mlp_torch_witness()),
    ("shard_ranges", _shard_ranges_overlap, lambda: pins.test_shard_ranges_partition_exactly(32)),
    ("shard_ranges", _shard_ranges_overlap, lambda: pins.test_tp2_split_matches_pages()),
    ("layer_norm", _layer_norm_unbiased, lambda: pins.test_layer_norm_identities()),
    ("layer_norm", _layer_norm_eps_outside, lambda: pins.test_layer_norm_torch_witness()),
    ("reduce_scatter", _reduce_scatter_reversed, lambda: pins.test_reduce_scatter_chunks_are_row_ranges()),
    ("reduce_scatter", _reduce_scatter_reversed, lambda: pins.test_sp_forward_equals_layernorm_then_mlp(4)),
    ("mlp_partials", _mlp_partials_transposed_shard, lambda: pins.test_shard_sum_equals_unsharded(4)),
    ("mlp_backward", _mlp_backward_dA_uses_dH, lambda: pins.test_backward_finite_difference_d8()),
    ("mlp_backward", _mlp_backward_sign, lambda: pins.test_backward_autograd_witness(1)),
    ("layer_norm_backward", _ln_backward_no_mean_g, lambda: pins.test_layer_norm_backward_autograd_and_fd()),
    ("sp_backward", _sp_backward_last_chunk_dgamma, lambda: pins.test_sp_backward_autograd_witness(4)),
]


@pytest.mark.parametrize("case", range(len(CASES)), ids=[f"{c[0]}-{i}" for i, c in enumerate(CASES)])
def test_planted_mistake_is_caught(case, monkeypatch):
    name, bad, pin = CASES[case]
    monkeypatch.setattr(oracle, name, bad)
    with pytest.raises((AssertionError, ValueError)):
        pin()


def test_unmutated_pins_pass():
    for _, _, pin in CASES:
        pin()
