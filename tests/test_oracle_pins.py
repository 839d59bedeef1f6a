"""Pins of the CPU oracle to facts fixed outside the oracle itself.

Each test checks an oracle function against one of: values the pages print
(golden files), closed forms and textbook constants, identities stated on the
pages, brute force with pure-Python loops on tiny inputs, library witnesses
(torch fp64 on the CPU: ``gelu(approximate='none')``, ``layer_norm``,
autograd) and finite differences.  Sizes keep the whole module to seconds.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden
from tensor_transformer_mlp_tp_gb300 import inputs

RNG = np.random.default_rng(1234)


def rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# --------------------------------------------------------------------------- partition

def test_tp2_split_matches_pages():
    for d, F, shard, lo, hi in (map(int, r) for r in read_golden("tp2_split.txt")):
        assert F == 4 * d
        assert oracle.shard_ranges(F, 2)[shard] == (lo, hi)


@pytest.mark.parametrize("F", [4, 8, 12, 32, 48, 64, 96, 256, 4096, 16384, 32768])
def test_shard_ranges_partition_exactly(F):
    for N in range(1, 17):
        if F % N:
            with pytest.raises(ValueError):
                oracle.shard_ranges(F, N)
            continue
        r = oracle.shard_ranges(F, N)
        assert len(r) == N
        covered = np.zeros(F, dtype=np.int64)
        for lo, hi in r:
            assert hi - lo == F // N
            covered[lo:hi] += 1
        assert np.all(covered == 1)                      # disjoint and complete, bit-exact
        assert r[0][0] == 0 and r[-1][1] == F
        assert all(r[i][1] == r[i + 1][0] for i in range(N - 1))


def test_chunk_ranges_partition_rows():
    for T, N in [(8192, 8), (4096, 8), (24, 3), (7, 7)]:
        r = oracle.chunk_ranges(T, N)
        assert [hi - lo for lo, hi in r] == [T // N] * N
        assert r[0][0] == 0 and r[-1][1] == T
    with pytest.raises(ValueError):
        oracle.chunk_ranges(10, 4)


# --------------------------------------------------------------------------- GeLU

def test_gelu_textbook_values():
    for x, Phi, phi in (map(float, r) for r in read_golden("normal_cdf.txt")):
        assert oracle.gelu(x) == pytest.approx(x * Phi, abs=2e-15)
        assert oracle.gelu_prime(x) == pytest.approx(Phi + x * phi, abs=2e-15)


def test_gelu_closed_forms():
    x = np.linspace(-8, 8, 2001)
    g = oracle.gelu(x)
    assert oracle.gelu(0.0) == 0.0
    np.testing.assert_allclose(g - oracle.gelu(-x), x, rtol=0, atol=1e-14)   # x·Φ(x) - (-x)·Φ(-x) = x
    big = np.array([10.0, 20.0, 40.0])
    np.testing.assert_allclose(oracle.gelu(big), big, rtol=1e-15)
    np.testing.assert_allclose(oracle.gelu(-big), 0.0, atol=1e-20)
    assert oracle.gelu_prime(0.0) == 0.5


def test_gelu_matches_math_erf_bruteforce():
    xs = RNG.normal(0, 3, 500)
    ref = [0.5 * v * (1 + math.erf(v / math.sqrt(2))) for v in xs]
    np.testing.assert_allclose(oracle.gelu(xs), ref, rtol=1e-15, atol=1e-15)


def test_gelu_torch_witness():
    xs = RNG.normal(0, 3, 4096)
    ref = torch.nn.functional.gelu(torch.from_numpy(xs), approximate="none").numpy()
    np.testing.assert_allclose(oracle.gelu(xs), ref, rtol=1e-14, atol=1e-15)  # 1+erf cancels in the left tail


def test_gelu_prime_finite_difference():
    xs = np.linspace(-6, 6, 241)
    h = 1e-5
    fd = (oracle.gelu(xs + h) - oracle.gelu(xs - h)) / (2 * h)
    np.testing.assert_allclose(oracle.gelu_prime(xs), fd, rtol=0, atol=1e-9)


# --------------------------------------------------------------------------- forward

def _rand_block(T, d, F, bias=True):
    X = RNG.normal(0, 1, (T, d))
    A = RNG.normal(0, 0.3, (d, F))
    B = RNG.normal(0, 0.3, (F, d))
    b = RNG.normal(0, 0.3, F) if bias else None
    return X, A, B, b


def test_worked_example_d1():
    g = {k: float(v) for k, v in read_golden("worked_mlp_d1.txt")}
    X = np.array([[1.0]])
    A = np.array([[1.0, -1.0, 2.0, 0.0]])
    B = np.ones((4, 1))
    parts = oracle.mlp_partials(X, A, B, None, 2)
    assert parts[0][0, 0] == pytest.approx(g["Y0"], abs=2e-15)
    assert parts[1][0, 0] == pytest.approx(g["Y1"], abs=2e-15)
    assert oracle.mlp_tp(X, A, B, None, 2)[0, 0] == pytest.approx(g["Y"], abs=4e-15)
    assert oracle.mlp_reference(X, A, B)[0, 0] == pytest.approx(g["Y"], abs=4e-15)


def _bruteforce_mlp(X, A, B, b):
    T, d = len(X), len(X[0])
    F = len(A[0])
    Y = [[0.0] * d for _ in range(T)]
    for t in range(T):
        z = []
        for f in range(F):
            s = 0.0 if b is None else b[f]
            for k in range(d):
                s += X[t][k] * A[k][f]
            z.append(0.5 * s * (1.0 + math.erf(s / math.sqrt(2.0))))
        for j in range(d):
            acc = 0.0
            for f in range(F):
                acc += z[f] * B[f][j]
            Y[t][j] = acc
    return np.array(Y)


@pytest.mark.parametrize("T", [1, 3, 16])
@pytest.mark.parametrize("N", [1, 2, 4, 8])
def test_mlp_bruteforce_d8(T, N):
    X, A, B, b = _rand_block(T, 8, 32)
    ref = _bruteforce_mlp(X.tolist(), A.tolist(), B.tolist(), b.tolist())
    assert rel(oracle.mlp_tp(X, A, B, b, N), ref) < 1e-13
    assert rel(oracle.mlp_reference(X, A, B, b), ref) < 1e-13


def test_mlp_torch_witness():
    X, A, B, b = _rand_block(37, 24, 96)
    t = lambda a: torch.from_numpy(a)
    ref = torch.nn.functional.linear(
        torch.nn.functional.gelu(torch.nn.functional.linear(t(X), t(A).T, t(b)), approximate="none"),
        t(B).T).numpy()
    assert rel(oracle.mlp_reference(X, A, B, b), ref) < 1e-13


@pytest.mark.parametrize("N", [1, 2, 3, 4, 6, 8, 12, 16, 24, 48])
def test_shard_sum_equals_unsharded(N):
    """Output = Z·W2 = Σ_i Z_i·W2_i (column-parallel / row-parallel section of the deep-dive page)."""
    X, A, B, b = _rand_block(19, 16, 48)
    assert rel(oracle.mlp_tp(X, A, B, b, N), oracle.mlp_reference(X, A, B, b)) < 1e-12


def test_n1_is_textbook_mlp():
    X, A, B, b = _rand_block(5, 8, 32)
    parts = oracle.mlp_partials(X, A, B, b, 1)
    assert len(parts) == 1
    assert rel(parts[0], oracle.mlp_reference(X, A, B, b)) < 1e-15


def test_partials_are_the_column_row_blocks():
    """Shard i of the partials uses exactly A[:, s_i], b[s_i] and B[s_i, :]."""
    X, A, B, b = _rand_block(4, 8, 32)
    parts = oracle.mlp_partials(X, A, B, b, 4)
    for i, (lo, hi) in enumerate(oracle.shard_ranges(32, 4)):
        ref = _bruteforce_mlp(X.tolist(), A[:, lo:hi].tolist(), B[lo:hi].tolist(), b[lo:hi].tolist())
        assert rel(parts[i], ref) < 1e-13


# --------------------------------------------------------------------------- collectives

@pytest.mark.parametrize("N", [1, 2, 4, 8])
def test_allreduce_is_allgather_of_reducescatter_integers(N):
    """AllReduce(X) = AllGather(ReduceScatter(X)), bit-exact on integer-valued partials."""
    T, d = 16 * N, 24
    parts = [RNG.integers(-3, 4, (T, d)).astype(np.float64) for _ in range(N)]
    ar = oracle.all_reduce(parts)
    ag = oracle.all_gather(oracle.reduce_scatter(parts, N))
    assert np.array_equal(ar, ag)
    assert np.array_equal(ar, np.sum(np.stack(parts), axis=0))   # integers: order-free


def test_reduce_scatter_chunks_are_row_ranges():
    N, T, d = 4, 12, 5
    parts = [RNG.normal(size=(T, d)) for _ in range(N)]
    chunks = oracle.reduce_scatter(parts, N)
    total = sum(parts[i] for i in range(N))
    for j, (lo, hi) in enumerate(oracle.chunk_ranges(T, N)):
        np.testing.assert_allclose(chunks[j], total[lo:hi], rtol=1e-15, atol=0)


# --------------------------------------------------------------------------- LayerNorm

def test_layer_norm_identities():
    x = RNG.normal(2.0, 3.0, (64, 128))
    y = oracle.layer_norm(x, np.ones(128), np.zeros(128), 1e-5)
    np.testing.assert_allclose(y.mean(axis=1), 0.0, atol=1e-13)
    var = x.var(axis=1)                                       # numpy var is the biased (1/d) variance
    np.testing.assert_allclose(y.var(axis=1), var / (var + 1e-5), rtol=1e-12)
    # affine invariance: LN(a·x + c) = LN(x) for a > 0, up to the eps term
    y2 = oracle.layer_norm(7.0 * x - 3.0, np.ones(128), np.zeros(128), 0.0)
    y3 = oracle.layer_norm(x, np.ones(128), np.zeros(128), 0.0)
    np.testing.assert_allclose(y2, y3, rtol=1e-12, atol=1e-12)


def test_layer_norm_torch_witness():
    x = RNG.normal(0, 1, (33, 96))
    g = 1 + 0.1 * RNG.normal(size=96)
    bt = 0.1 * RNG.normal(size=96)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (96,), torch.from_numpy(g),
                                         torch.from_numpy(bt), eps=1e-5).numpy()
    np.testing.assert_allclose(oracle.layer_norm(x, g, bt, 1e-5), ref, rtol=1e-13, atol=1e-13)


def test_layer_norm_single_row_bruteforce():
    x = [3.0, -1.0, 0.5, 2.5]
    mu = sum(x) / 4
    var = sum((v - mu) ** 2 for v in x) / 4
    ref = [(v - mu) / math.sqrt(var + 1e-5) * 2.0 + 0.25 for v in x]
    np.testing.assert_allclose(oracle.layer_norm(np.array([x]), 2.0 * np.ones(4), 0.25 * np.ones(4))[0], ref,
                               rtol=1e-15)


# --------------------------------------------------------------------------- SP forward

@pytest.mark.parametrize("N", [1, 2, 4, 8])
def test_sp_forward_equals_layernorm_then_mlp(N):
    T, d, F = 8 * N, 16, 64
    X = RNG.normal(size=(T, d))
    g = 1 + 0.1 * RNG.normal(size=d)
    bt = 0.1 * RNG.normal(size=d)
    _, A, B, b = _rand_block(1, d, F)
    chunks = [X[lo:hi] for lo, hi in oracle.chunk_ranges(T, N)]
    Yc = oracle.sp_forward(chunks, g, bt, 1e-5, A, B, b, N)
    ref = oracle.mlp_reference(oracle.layer_norm(X, g, bt, 1e-5), A, B, b)
    assert len(Yc) == N and all(c.shape == (T // N, d) for c in Yc)
    assert rel(np.concatenate(Yc), ref) < 1e-12


# --------------------------------------------------------------------------- backward

def _torch_block_grads(X, A, B, b, dY):
    t = [torch.tensor(v, dtype=torch.float64, requires_grad=True) for v in (X, A, B, b)]
    Y = torch.nn.functional.gelu(t[0] @ t[1] + t[3], approximate="none") @ t[2]
    Y.backward(torch.from_numpy(dY))
    return [v.grad.numpy() for v in t]


@pytest.mark.parametrize("N", [1, 2, 4])
def test_backward_autograd_witness(N):
    X, A, B, b = _rand_block(11, 12, 48)
    dY = RNG.normal(size=(11, 12))
    gX, gA, gB, gb = _torch_block_grads(X, A, B, b, dY)
    g = oracle.mlp_backward_tp(X, A, B, b, dY, N)
    for mine, ref in [(g["dX"], gX), (g["dA"], gA), (g["dB"], gB), (g["db"], gb)]:
        assert rel(mine, ref) < 1e-12
    g1 = oracle.mlp_backward(X, A, B, b, dY)
    for k in ("dX", "dA", "dB", "db"):
        assert rel(g1[k], g[k]) < 1e-12


def test_backward_finite_difference_d8():
    X, A, B, b = _rand_block(3, 8, 32)
    dY = RNG.normal(size=(3, 8))
    g = oracle.mlp_backward(X, A, B, b, dY)
    loss = lambda X_, A_, B_, b_: float(np.sum(oracle.mlp_reference(X_, A_, B_, b_) * dY))
    h = 1e-6
    for name, arr, idx in [("dX", X, (1, 3)), ("dA", A, (2, 17)), ("dB", B, (30, 5)), ("db", b, (9,))]:
        args = {"dX": [X, A, B, b], "dA": [X, A, B, b], "dB": [X, A, B, b], "db": [X, A, B, b]}[name]
        pos = {"dX": 0, "dA": 1, "dB": 2, "db": 3}[name]
        plus = [a.copy() for a in args]
        minus = [a.copy() for a in args]
        plus[pos][idx] += h
        minus[pos][idx] -= h
        fd = (loss(*plus) - loss(*minus)) / (2 * h)
        assert g[name][idx] == pytest.approx(fd, rel=1e-7, abs=1e-9)


def test_layer_norm_backward_autograd_and_fd():
    x = RNG.normal(0.5, 2.0, (7, 24))
    gam = 1 + 0.2 * RNG.normal(size=24)
    bet = 0.2 * RNG.normal(size=24)
    dy = RNG.normal(size=(7, 24))
    tx = torch.tensor(x, requires_grad=True)
    tg = torch.tensor(gam, requires_grad=True)
    tb = torch.tensor(bet, requires_grad=True)
    torch.nn.functional.layer_norm(tx, (24,), tg, tb, eps=1e-5).backward(torch.from_numpy(dy))
    dx, dga, dbe = oracle.layer_norm_backward(x, gam, 1e-5, dy)
    assert rel(dx, tx.grad.numpy()) < 1e-12
    assert rel(dga, tg.grad.numpy()) < 1e-12
    assert rel(dbe, tb.grad.numpy()) < 1e-12
    h = 1e-6
    xp, xm = x.copy(), x.copy()
    xp[2, 5] += h
    xm[2, 5] -= h
    f = lambda v: float(np.sum(oracle.layer_norm(v, gam, bet, 1e-5) * dy))
    assert dx[2, 5] == pytest.approx((f(xp) - f(xm)) / (2 * h), rel=1e-7, abs=1e-9)


@pytest.mark.parametrize("N", [1, 2, 4])
def test_sp_backward_autograd_witness(N):
    T, d, F = 4 * N, 8, 32
    X = RNG.normal(size=(T, d))
    gam = 1 + 0.1 * RNG.normal(size=d)
    bet = 0.1 * RNG.normal(size=d)
    _, A, B, b = _rand_block(1, d, F)
    dY = RNG.normal(size=(T, d))
    tt = [torch.tensor(v, requires_grad=True) for v in (X, gam, bet, A, B, b)]
    xn = torch.nn.functional.layer_norm(tt[0], (d,), tt[1], tt[2], eps=1e-5)
    Y = torch.nn.functional.gelu(xn @ tt[3] + tt[5], approximate="none") @ tt[4]
    Y.backward(torch.from_numpy(dY))
    cr = oracle.chunk_ranges(T, N)
    g = oracle.sp_backward([X[lo:hi] for lo, hi in cr], gam, bet, 1e-5, A, B, b,
                           [dY[lo:hi] for lo, hi in cr], N)
    assert rel(np.concatenate(g["dX_chunks"]), tt[0].grad.numpy()) < 1e-12
    assert rel(g["dgamma"], tt[1].grad.numpy()) < 1e-12
    assert rel(g["dbeta"], tt[2].grad.numpy()) < 1e-12
    assert rel(g["dA"], tt[3].grad.numpy()) < 1e-12
    assert rel(g["dB"], tt[4].grad.numpy()) < 1e-12
    assert rel(g["db"], tt[5].grad.numpy()) < 1e-12


# --------------------------------------------------------------------------- inputs feed the oracle exactly

def test_bf16_inputs_are_exact_in_fp64():
    w = inputs.small_workload(64, 32, 4)
    bits, vals = inputs.draw(w, "X")
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(vals, ref)


# --------------------------------------------------------------------------- bf16 rounding and the RMS norm of the listing

def _bf16_bruteforce(v):
    """Round a Python float to bf16 through its float32 bit pattern (RNE on the low 16 bits)."""
    import struct
    b = struct.unpack("<I", struct.pack("<f", v))[0]
    low = b & 0xFFFF
    hi = b >> 16
    if low > 0x8000 or (low == 0x8000 and (hi & 1)):
        hi += 1
    return struct.unpack("<f", struct.pack("<I", hi << 16))[0]


def test_round_bf16_ties_and_witnesses():
    assert oracle.round_bf16(1.0 + 2.0 ** -8) == 1.0                # tie, even neighbour below
    assert oracle.round_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6  # tie, even neighbour above
    assert oracle.round_bf16(-(1.0 + 2.0 ** -7)) == -(1.0 + 2.0 ** -7)  # representable
    xs = RNG.normal(0, 10, 2000).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.bfloat16).double().numpy()
    assert np.array_equal(oracle.round_bf16(xs.astype(np.float64)), ref)
    assert np.array_equal(oracle.round_bf16(xs.astype(np.float64)), [_bf16_bruteforce(float(v)) for v in xs])


def test_rms_norm_bruteforce_rows():
    x = RNG.normal(0.3, 2.0, (5, 12))
    w = oracle.round_bf16(1 + 0.1 * RNG.normal(size=12))
    got = oracle.rms_norm(x, w, 1e-5)
    for r in range(5):
        ms = sum(v * v for v in x[r]) / 12
        rs = 1.0 / math.sqrt(ms + 1e-5)
        ref = [_bf16_bruteforce(float(np.float32(v * rs))) * w[c] for c, v in enumerate(x[r])]
        np.testing.assert_allclose(got[r], ref, rtol=0, atol=1e-12)


def test_rms_norm_torch_witness_and_closed_form():
    x = RNG.normal(0, 1, (64, 256))
    w = oracle.round_bf16(1 + 0.02 * RNG.normal(size=256))
    xt = torch.from_numpy(x)
    rstd = torch.rsqrt((xt * xt).mean(-1, keepdim=True) + 1e-5)
    ref = (xt * rstd).to(torch.bfloat16).double() * torch.from_numpy(w)
    np.testing.assert_allclose(oracle.rms_norm(x, w, 1e-5), ref.numpy(), rtol=0, atol=1e-12)
    # a constant row c: x / rms = sign(c) / sqrt(1 + eps/c^2), which rounds to +-1 in bf16
    c = np.full((1, 256), -3.0)
    np.testing.assert_array_equal(oracle.rms_norm(c, w, 1e-5)[0], -w)


# --------------------------------------------------------------------------- dropout generator and the whole SP region

def _numpy_philox_block(counter, key):
    """One Philox4x64-10 block from numpy's bit generator, which advances its counter before each block."""
    c = [int(v) for v in counter]
    assert c[0] >= 1, "the witness steps counter word 0 back by one"
    c[0] -= 1
    g = np.random.Philox(key=np.array(key, dtype=np.uint64), counter=np.array(c, dtype=np.uint64))
    return g.random_raw(4)


def test_philox_matches_numpy_bit_generator():
    rng = np.random.default_rng(11)
    ctrs = rng.integers(1, 2 ** 63, size=(24, 4), dtype=np.uint64)
    ctrs[:4, 1:] = 0
    keys = rng.integers(0, 2 ** 63, size=(24, 2), dtype=np.uint64)
    keys[0] = 0
    for c, k in zip(ctrs, keys):
        got = oracle.philox4x64(c[None, :], (int(k[0]), int(k[1])))[0]
        assert np.array_equal(got, _numpy_philox_block(c, k)), (c, k)
    # a vector of counters under one key equals the blocks one by one
    many = oracle.philox4x64(ctrs, (7, 9))
    for c, row in zip(ctrs, many):
        assert np.array_equal(row, _numpy_philox_block(c, (7, 9)))


@pytest.mark.parametrize("p", [0.1, 0.5, 0.875])
def test_dropout_keep_bits_come_from_the_stated_block_and_half(p):
    """Each element's keep bit, recomputed from numpy's Philox blocks by the stated word/half rule."""
    rows, d, row0, seed, offset = 5, 24, 3, 1234567, 42
    keep = oracle.dropout_keep(rows, d, row0, p, seed, offset)
    thr = math.floor((1.0 - float(np.float32(p))) * 2 ** 32)
    for r in range(rows):
        for c in range(d):
            e = (row0 + r) * d + c
            w = int(_numpy_philox_block((e // 8, offset, 0, 0), (seed, 0))[(e % 8) // 2])
            u = (w >> (32 * (e % 2))) & 0xFFFFFFFF
            assert keep[r, c] == (u < thr), (r, c)


def test_dropout_keep_invariants():
    assert oracle.dropout_threshold(0.0) == 2 ** 32
    assert oracle.dropout_threshold(0.5) == 2 ** 31
    assert oracle.dropout_threshold(0.25) == 3 * 2 ** 30
    with pytest.raises(ValueError):
        oracle.dropout_threshold(1.0)
    assert oracle.dropout_keep(16, 64, 0, 0.0, 3, 0).all()
    T, d, p = 512, 256, 0.1
    full = oracle.dropout_keep(T, d, 0, p, 99, 5)
    n = full.size
    assert abs(full.mean() - (1 - p)) < 6 * math.sqrt(p * (1 - p) / n)
    # the mask of a chunk is the slice of the whole output's mask (global element index)
    assert np.array_equal(full[128:256], oracle.dropout_keep(128, d, 128, p, 99, 5))
    # another offset (the next step) draws an independent mask
    other = oracle.dropout_keep(T, d, 0, p, 99, 6)
    agree = (full == other).mean()
    expect = p * p + (1 - p) * (1 - p)
    assert abs(agree - expect) < 6 * math.sqrt(expect * (1 - expect) / n)


def _block_problem(T, d, F):
    X = RNG.normal(size=(T, d))
    gam = 1 + 0.1 * RNG.normal(size=d)
    bet = 0.1 * RNG.normal(size=d)
    _, A, B, b = _rand_block(1, d, F)
    b2 = 0.1 * RNG.normal(size=d)
    return X, gam, bet, A, B, b, b2


def _torch_block(tt, keep, p, d):
    X, gam, bet, A, B, b, b2 = tt
    xn = torch.nn.functional.layer_norm(X, (d,), gam, bet, eps=1e-5)
    Z = torch.nn.functional.gelu(xn @ A + b, approximate="none") @ B + b2
    return X + Z * torch.from_numpy(keep.astype(np.float64)) / (1.0 - float(np.float32(p)))


@pytest.mark.parametrize("N,p", [(1, 0.1), (2, 0.25), (4, 0.5)])
def test_sp_block_forward_torch_witness(N, p):
    T, d, F = 4 * N, 16, 64
    X, gam, bet, A, B, b, b2 = _block_problem(T, d, F)
    keep = oracle.dropout_keep(T, d, 0, p, 77, 3)
    ref = _torch_block([torch.tensor(v) for v in (X, gam, bet, A, B, b, b2)], keep, p, d).numpy()
    cr = oracle.chunk_ranges(T, N)
    Y = oracle.sp_block_forward([X[lo:hi] for lo, hi in cr], gam, bet, 1e-5, A, B, b, b2, p, 77, 3, N)
    assert rel(np.concatenate(Y), ref) < 1e-12


def test_sp_block_forward_without_dropout_is_residual_plus_sp_forward():
    T, d, F, N = 16, 8, 32, 4
    X, gam, bet, A, B, b, _ = _block_problem(T, d, F)
    cr = oracle.chunk_ranges(T, N)
    Xc = [X[lo:hi] for lo, hi in cr]
    Y = oracle.sp_block_forward(Xc, gam, bet, 1e-5, A, B, b, None, 0.0, 1, 0, N)
    Z = oracle.sp_forward(Xc, gam, bet, 1e-5, A, B, b, N)
    for y, x, z in zip(Y, Xc, Z):
        assert np.array_equal(y, x + z)


@pytest.mark.parametrize("N,p", [(1, 0.0), (2, 0.25), (4, 0.5)])
def test_sp_block_backward_autograd_witness(N, p):
    T, d, F = 4 * N, 16, 64
    X, gam, bet, A, B, b, b2 = _block_problem(T, d, F)
    dY = RNG.normal(size=(T, d))
    keep = oracle.dropout_keep(T, d, 0, p, 5, 8)
    tt = [torch.tensor(v, requires_grad=True) for v in (X, gam, bet, A, B, b, b2)]
    _torch_block(tt, keep, p, d).backward(torch.from_numpy(dY))
    cr = oracle.chunk_ranges(T, N)
    g = oracle.sp_block_backward([X[lo:hi] for lo, hi in cr], gam, bet, 1e-5, A, B, b, p, 5, 8,
                                 [dY[lo:hi] for lo, hi in cr], N)
    assert rel(np.concatenate(g["dX_chunks"]), tt[0].grad.numpy()) < 1e-12
    for key, i in (("dgamma", 1), ("dbeta", 2), ("dA", 3), ("dB", 4), ("db", 5), ("db2", 6)):
        assert rel(g[key], tt[i].grad.numpy()) < 1e-12, key


# --------------------------------------------------------------------------- E4M3 and the FP8 forward

def _e4m3_table():
    """Every finite E4M3 value with its code, decoded from the format's definition (bias 7, 3 mantissa bits,
    exponent field 0 = subnormal, code S.1111.111 = NaN)."""
    vals = []
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        ex, man = (code >> 3) & 0xF, code & 0x7
        if ex == 0xF and man == 0x7:
            continue
        v = man / 8.0 * 2.0 ** -6 if ex == 0 else (1.0 + man / 8.0) * 2.0 ** (ex - 7)
        vals.append((sign * v, code))
    return vals


def _e4m3_bruteforce(x):
    if abs(x) > 448.0:
        return math.copysign(448.0, x)
    best = None
    for v, code in _e4m3_table():
        dist = abs(v - x)
        if best is None or dist < best[0] or (dist == best[0] and (code & 1) == 0 and (best[1] & 1) == 1):
            best = (dist, code, v)
    return best[2]


def test_round_e4m3_bruteforce_and_ties():
    table = sorted({v for v, _ in _e4m3_table()})
    assert len(table) == 253 and max(table) == 448.0 and min(v for v in table if v > 0) == 2.0 ** -9
    rng = np.random.default_rng(21)
    xs = list(rng.normal(size=300) * 10.0 ** rng.uniform(-3.5, 2.8, size=300))
    pos = [v for v in table if v >= 0]
    xs += [(a + b) / 2 for a, b in zip(pos[:-1], pos[1:])]          # every midpoint: ties to even
    xs += [-(a + b) / 2 for a, b in zip(pos[:-1], pos[1:])]
    xs += [449.0, 465.0, 1e6, -1e6, 0.0, 2.0 ** -10, 3 * 2.0 ** -11]
    got = oracle.round_e4m3(np.array(xs))
    for x, g in zip(xs, got):
        assert g == _e4m3_bruteforce(x), x


def test_round_e4m3_torch_witness():
    rng = np.random.default_rng(22)
    x = (rng.normal(size=4000) * 10.0 ** rng.uniform(-3, 2.6, size=4000)).astype(np.float32)
    x = x[np.abs(x) <= 448.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(oracle.round_e4m3(x), ref)
    q = oracle.quantize_e4m3(x, 0.75)
    assert np.array_equal(q, torch.from_numpy(x * np.float32(0.75)).to(torch.float8_e4m3fn).to(torch.float64).numpy())


def test_fp8_delayed_scale_closed_forms():
    assert oracle.fp8_scale(np.full(16, 3.5)) == 448.0 / 3.5
    assert oracle.fp8_scale(np.full(16, 3.5), margin=2) == 448.0 / 3.5 / 4
    assert oracle.fp8_scale([1.0, 2.0, 3.0, 6.0]) == 448.0 / 3.0        # the mean, not the max
    assert oracle.fp8_scale(np.zeros(8)) == 1.0
    h = oracle.roll_amax_history([1.0, 2.0, 3.0], 7.0)
    assert list(h) == [2.0, 3.0, 7.0]


def test_mlp_fp8_is_exact_on_representable_inputs():
    """Inputs on the E4M3 grid with power-of-two scales quantise to themselves, H = GeLU(...) does not, so
    compare the first layer exactly and the whole block against the textbook MLP on the quantised H."""
    rng = np.random.default_rng(23)
    grid = np.array(sorted({v for v, _ in _e4m3_table() if abs(v) <= 4.0}))
    T, d, F, N = 8, 16, 32, 4
    X = rng.choice(grid, size=(T, d))
    A = rng.choice(grid, size=(d, F)) / 8.0
    B = rng.choice(grid, size=(F, d)) / 16.0
    b = rng.choice(grid, size=F)
    scales = (2.0, 8.0, 16.0, 4.0)
    out = oracle.mlp_fp8(X, A, B, b, N, scales)
    assert np.allclose(out["H"], oracle.gelu(X @ A + b), rtol=0, atol=1e-12)
    assert np.allclose(out["Y"], out["qH"] @ B / 4.0, rtol=1e-13, atol=1e-13)
    assert out["amax"]["A"] == np.max(np.abs(A)) and out["amax"]["H"] == np.max(np.abs(out["H"]))


def test_mlp_fp8_torch_witness():
    """The FP8 MLP against torch: float32 products, torch's float8_e4m3fn cast, float64 matmuls."""
    T, d, F, N = 12, 16, 64, 4
    X, A, B, b = _rand_block(T, d, F)
    scales = (448.0 / np.max(np.abs(X)), 448.0 / np.max(np.abs(A)), 448.0 / np.max(np.abs(B)), 40.0)

    def q(v, s):
        return (torch.from_numpy(np.asarray(v, dtype=np.float32)) * torch.tensor(np.float32(s))).to(
            torch.float8_e4m3fn).to(torch.float64)

    f32 = lambda s: float(np.float32(s))
    H = torch.nn.functional.gelu(q(X, scales[0]) @ q(A, scales[1]) / (f32(scales[0]) * f32(scales[1])) +
                                 torch.from_numpy(b), approximate="none")
    Y = q(H.numpy(), scales[3]) @ q(B, scales[2]) / (f32(scales[3]) * f32(scales[2]))
    out = oracle.mlp_fp8(X, A, B, b, N, scales)
    assert rel(out["H"], H.numpy()) < 1e-12
    assert rel(out["Y"], Y.numpy()) < 1e-12
    # and the quantisation error is of the format's size: a few 2**-4 relative steps, not more
    assert 1e-3 < rel(out["Y"], oracle.mlp_reference(X, A, B, b)) < 0.1


@pytest.mark.parametrize("N", [1, 2, 4])
def test_sp_forward_fp8_is_mlp_fp8_on_the_gathered_norm(N):
    T, d, F = 4 * N, 16, 64
    X = RNG.normal(size=(T, d))
    gam, bet = 1 + 0.1 * RNG.normal(size=d), 0.1 * RNG.normal(size=d)
    _, A, B, b = _rand_block(1, d, F)
    scales = (100.0, 2000.0, 2000.0, 50.0)
    cr = oracle.chunk_ranges(T, N)
    out = oracle.sp_forward_fp8([X[lo:hi] for lo, hi in cr], gam, bet, 1e-5, A, B, b, N, scales)
    ref = oracle.mlp_fp8(oracle.layer_norm(X, gam, bet, 1e-5), A, B, b, N, scales)
    assert np.array_equal(np.concatenate(out["Y_chunks"]), ref["Y"])


# --------------------------------------------------------------------------- E5M2 and the FP8 backward

def _e5m2_table():
    """Every finite E5M2 value with its code: bias 15, 2 mantissa bits, exponent field 0 = subnormal,
    exponent field 31 = infinities and NaNs (excluded)."""
    vals = []
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        ex, man = (code >> 2) & 0x1F, code & 0x3
        if ex == 0x1F:
            continue
        v = man / 4.0 * 2.0 ** -14 if ex == 0 else (1.0 + man / 4.0) * 2.0 ** (ex - 15)
        vals.append((sign * v, code))
    return vals


def test_round_e5m2_bruteforce_and_torch():
    table = _e5m2_table()
    pos = sorted({v for v, _ in table if v >= 0})
    assert max(pos) == 57344.0 and pos[1] == 2.0 ** -16

    def brute(x):
        if abs(x) > 57344.0:
            return math.copysign(57344.0, x)
        best = None
        for v, code in table:
            dist = abs(v - x)
            if best is None or dist < best[0] or (dist == best[0] and (code & 1) == 0 and (best[1] & 1) == 1):
                best = (dist, code, v)
        return best[2]

    rng = np.random.default_rng(24)
    xs = list(rng.normal(size=200) * 10.0 ** rng.uniform(-5, 4.5, size=200))
    xs += [(a + b) / 2 for a, b in zip(pos[:-1], pos[1:])] + [6e4, -1e7, 0.0]
    got = oracle.round_e5m2(np.array(xs))
    for x, g in zip(xs, got):
        assert g == brute(x), x
    x = (rng.normal(size=3000) * 10.0 ** rng.uniform(-4, 4, size=3000)).astype(np.float32)
    assert np.array_equal(oracle.round_e5m2(x), torch.from_numpy(x).to(torch.float8_e5m2).to(torch.float64).numpy())


def _fp8_backward_problem(T=12, d=16, F=64):
    """A problem with every scale set from its tensor's amax, as delayed scaling settles to."""
    X, A, B, b = _rand_block(T, d, F)
    dY = RNG.normal(size=(T, d))
    s3 = (448.0 / np.max(np.abs(X)), 448.0 / np.max(np.abs(A)), 448.0 / np.max(np.abs(B)))
    scales = (*s3, 448.0 / oracle.mlp_fp8(X, A, B, b, 1, (*s3, 1.0))["amax"]["H"])
    first = oracle.mlp_backward_fp8(X, A, B, b, dY, 1, scales, (1.0, 1.0))["amax"]
    return X, A, B, b, dY, scales, (57344.0 / first["dY"], 57344.0 / first["dHpre"])


@pytest.mark.parametrize("N", [1, 2, 4])
def test_mlp_backward_fp8_with_exact_casts_is_the_chain_rule(N, monkeypatch):
    """With the casts made exact (identity rounding) the scales must cancel and the FP8 backward must be
    the pinned chain-rule backward: any wrong scale, transposed operand or misplaced factor shows."""
    X, A, B, b, dY, scales, gscales = _fp8_backward_problem()
    monkeypatch.setattr(oracle, "round_e4m3", lambda v: np.asarray(v, dtype=np.float64))
    monkeypatch.setattr(oracle, "round_e5m2", lambda v: np.asarray(v, dtype=np.float64))
    g = oracle.mlp_backward_fp8(X, A, B, b, dY, N, scales, gscales)
    # the only roundings left are the float32 products x*S; compare at float32 precision
    ref = oracle.mlp_backward(X.astype(np.float32), A.astype(np.float32), B.astype(np.float32), b,
                              dY.astype(np.float32))
    for k in ("dX", "dA", "dB", "db"):
        assert rel(g[k], ref[k]) < 1e-5, k


def test_fp8_backward_cast_formats_follow_the_page():
    """E4M3 for activations and weights, E5M2 for the gradients entering GEMMs: spy on the two casts."""
    X, A, B, b, dY, scales, gscales = _fp8_backward_problem()
    seen = {"e4m3": [], "e5m2": []}
    r4, r5 = oracle.round_e4m3, oracle.round_e5m2
    try:
        oracle.round_e4m3 = lambda v: (seen["e4m3"].append(np.shape(v)), r4(v))[1]
        oracle.round_e5m2 = lambda v: (seen["e5m2"].append(np.shape(v)), r5(v))[1]
        oracle.mlp_backward_fp8(X, A, B, b, dY, 2, scales, gscales)
    finally:
        oracle.round_e4m3, oracle.round_e5m2 = r4, r5
    T, d = X.shape
    F = A.shape[1]
    assert sorted(seen["e4m3"]) == sorted([(T, d), (d, F), (F, d), (T, F)])     # X, A, B, H
    assert sorted(seen["e5m2"]) == sorted([(T, d), (T, F)])                     # dY, dHpre


def test_mlp_backward_fp8_error_is_the_formats_size():
    X, A, B, b, dY, scales, gscales = _fp8_backward_problem(T=32, d=32, F=128)
    g = oracle.mlp_backward_fp8(X, A, B, b, dY, 4, scales, gscales)
    ref = oracle.mlp_backward(X, A, B, b, dY)
    # E5M2 keeps 2 mantissa bits (up to 12.5% per element); through two GEMMs the errors stay near 10%
    for k in ("dX", "dA", "dB"):
        assert 1e-3 < rel(g[k], ref[k]) < 0.2, k
    assert rel(g["db"], ref["db"]) < 0.2


def test_mlp_backward_fp8_saved_operands_enter_where_the_chain_rule_puts_them():
    """Saved codes replace the oracle's own ones tensor by tensor: its own values change nothing, and one
    code moved by delta moves exactly the gradients that contain it, by the product the formulas give
    (dA = q_Xᵀ q_g/(S_X S_g), dB = q_Hᵀ q_dY/(S_H S_dY), dX = q_g q_Aᵀ/(S_g S_A), db = Σ dHpre)."""
    X, A, B, b, dY, scales, gscales = _fp8_backward_problem(T=12, d=16, F=64)
    N = 2
    sx, sa, sb, sh = (float(np.float32(v)) for v in scales)
    sdy, sg = (float(np.float32(v)) for v in gscales)
    base = oracle.mlp_backward_fp8(X, A, B, b, dY, N, scales, gscales)
    qx = oracle.quantize_e4m3(X, scales[0])
    qa = oracle.quantize_e4m3(A, scales[1])
    qb = oracle.quantize_e4m3(B, scales[2])
    Hpre = (qx @ qa) / (sx * sa) + b
    qh = oracle.quantize_e4m3(oracle.gelu(Hpre), scales[3])
    qdy = oracle.quantize_e5m2(dY, gscales[0])
    own = {"qX": qx, "qH": qh, "Hpre": Hpre, "qdHpre": base["qdHpre"]}
    same = oracle.mlp_backward_fp8(X, A, B, b, dY, N, scales, gscales, saved=own)
    for k in ("dX", "dA", "dB", "db"):
        assert np.array_equal(same[k], base[k]), k
    delta = 0.5
    for name, r, c in (("qX", 3, 5), ("qH", 4, 7), ("qdHpre", 2, 9), ("Hpre", 1, 11)):
        moved = dict(own)
        moved[name] = own[name].copy()
        moved[name][r, c] += delta
        g = oracle.mlp_backward_fp8(X, A, B, b, dY, N, scales, gscales, saved=moved)
        diff = {k: g[k] - base[k] for k in ("dX", "dA", "dB", "db")}
        expect = {k: np.zeros_like(base[k]) for k in diff}
        if name == "qX":
            expect["dA"][c, :] = delta * base["qdHpre"][r, :] / (sx * sg)
        elif name == "qH":
            expect["dB"][c, :] = delta * qdy[r, :] / (sh * sdy)
        elif name == "qdHpre":
            expect["dA"][:, c] = qx[r, :] * delta / (sx * sg)
            expect["dX"][r, :] = delta * qa[:, c] / (sg * sa)
        else:
            g_up = (qdy @ qb.T)[r, c] / (sdy * sb)
            expect["db"][c] = g_up * (oracle.gelu_prime(Hpre[r, c] + delta) - oracle.gelu_prime(Hpre[r, c]))
        for k in diff:
            np.testing.assert_allclose(diff[k], expect[k], rtol=1e-9, atol=1e-12 * max(1.0, np.abs(base[k]).max()),
                                       err_msg=f"{name} -> {k}")


@pytest.mark.parametrize("N", [1, 2, 4])
def test_sp_backward_fp8_is_mlp_backward_fp8_on_the_gathered_norm(N):
    T, d, F = 4 * N, 16, 64
    X = RNG.normal(size=(T, d))
    gam, bet = 1 + 0.1 * RNG.normal(size=d), 0.1 * RNG.normal(size=d)
    _, A, B, b = _rand_block(1, d, F)
    dY = RNG.normal(size=(T, d))
    scales, gscales = (100.0, 2000.0, 2000.0, 50.0), (1000.0, 2.0 ** 12)
    cr = oracle.chunk_ranges(T, N)
    g = oracle.sp_backward_fp8([X[lo:hi] for lo, hi in cr], gam, bet, 1e-5, A, B, b, [dY[lo:hi] for lo, hi in cr],
                               N, scales, gscales)
    ref = oracle.mlp_backward_fp8(oracle.layer_norm(X, gam, bet, 1e-5), A, B, b, dY, N, scales, gscales)
    for k in ("dA", "dB", "db"):
        assert np.array_equal(g[k], ref[k]), k
    for (lo, hi), dx in zip(cr, g["dX_chunks"]):
        assert np.array_equal(dx, oracle.layer_norm_backward(X[lo:hi], gam, 1e-5, ref["dX"][lo:hi])[0])


# --------------------------------------------------------------------------- tensor-parallel attention

def _attn_problem(S=6, B=2, d=16, H=4, seed=0):
    rng = np.random.default_rng(seed)
    X = rng.normal(size=(S * B, d))
    Wqkv = rng.normal(size=(d, 3 * d)) * 0.4
    bqkv = rng.normal(size=3 * d) * 0.1
    Wo = rng.normal(size=(d, d)) * 0.3
    bo = rng.normal(size=d) * 0.1
    return X, Wqkv, bqkv, Wo, bo


@pytest.mark.parametrize("causal", [False, True])
def test_attention_head_torch_witness(causal):
    rng = np.random.default_rng(5)
    Q, K, V = (rng.normal(size=(7, 4)) for _ in range(3))
    ref = torch.nn.functional.scaled_dot_product_attention(
        *(torch.from_numpy(a)[None, None] for a in (Q, K, V)), is_causal=causal)[0, 0].numpy()
    assert rel(oracle.attention_head(Q, K, V, causal), ref) < 1e-13


def test_attention_head_bruteforce():
    """Pure-Python loops over a 3 x 2 head: scaled scores, max-subtracted exponentials, weighted sum."""
    Q = [[0.5, -1.0], [1.5, 0.25], [-0.75, 2.0]]
    K = [[1.0, 0.5], [-0.5, 1.0], [0.25, -1.5]]
    V = [[1.0, 2.0], [-3.0, 0.5], [0.0, -1.0]]
    for causal in (False, True):
        out = []
        for s in range(3):
            keys = range(s + 1) if causal else range(3)
            sc = [sum(Q[s][e] * K[t][e] for e in range(2)) / math.sqrt(2) for t in keys]
            m = max(sc)
            w = [math.exp(x - m) for x in sc]
            z = sum(w)
            out.append([sum(w[i] * V[t][e] for i, t in enumerate(keys)) / z for e in range(2)])
        assert np.allclose(oracle.attention_head(np.array(Q), np.array(K), np.array(V), causal), out,
                           rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_attention_tp_torch_witness(causal):
    """The whole block against torch: linear projections, SDPA per (batch, head), output projection."""
    S, B, d, H = 6, 2, 16, 4
    X, Wqkv, bqkv, Wo, bo = _attn_problem(S, B, d, H)
    hd = d // H
    x = torch.from_numpy(X).reshape(S, B, d)
    qkv = x @ torch.from_numpy(Wqkv) + torch.from_numpy(bqkv)               # [S, B, 3d]
    q, k, v = (qkv[..., p * d:(p + 1) * d].reshape(S, B, H, hd).permute(1, 2, 0, 3) for p in range(3))
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=causal)  # [B, H, S, hd]
    o = o.permute(2, 0, 1, 3).reshape(S * B, d)
    ref = (o @ torch.from_numpy(Wo) + torch.from_numpy(bo)).numpy()
    for N in (1, 2, 4):
        assert rel(oracle.attention_tp(X, Wqkv, bqkv, Wo, bo, H, N, B, causal), ref) < 1e-12


def test_attention_tp_shard_sum_is_the_unsharded_block():
    X, Wqkv, bqkv, Wo, bo = _attn_problem(S=5, B=3, d=24, H=6)
    one = oracle.attention_tp(X, Wqkv, bqkv, Wo, bo, 6, 1, 3, True)
    for N in (2, 3, 6):
        Y, parts = oracle.attention_tp(X, Wqkv, bqkv, Wo, bo, 6, N, 3, True, return_parts=True)
        assert rel(Y, one) < 1e-13
        assert len(parts["partials"]) == N
    assert oracle.head_ranges(32, 8)[3] == (12, 16)
    with pytest.raises(ValueError):
        oracle.head_ranges(6, 4)


def test_attention_causal_outputs_ignore_later_tokens():
    S, B, d, H = 6, 2, 16, 4
    X, Wqkv, bqkv, Wo, bo = _attn_problem(S, B, d, H)
    Y = oracle.attention_tp(X, Wqkv, bqkv, Wo, bo, H, 2, B, True)
    X2 = X.copy()
    X2[4 * B:] += 3.0                                  # change positions 4 and 5 of every batch element
    Y2 = oracle.attention_tp(X2, Wqkv, bqkv, Wo, bo, H, 2, B, True)
    assert np.array_equal(Y[:4 * B], Y2[:4 * B])
    assert not np.allclose(Y[4 * B:], Y2[4 * B:])
    # and batch elements do not see each other
    X3 = X.copy()
    X3[1::B] += 1.0                                    # batch element 1 only
    Y3 = oracle.attention_tp(X3, Wqkv, bqkv, Wo, bo, H, 2, B, False)
    Y0 = oracle.attention_tp(X, Wqkv, bqkv, Wo, bo, H, 2, B, False)
    assert np.array_equal(Y3[0::B], Y0[0::B])


@pytest.mark.parametrize("causal", [False, True])
def test_attention_head_backward_autograd_witness(causal):
    rng = np.random.default_rng(9)
    Q, K, V, dO = (rng.normal(size=(7, 4)) for _ in range(4))
    tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (Q, K, V))
    torch.nn.functional.scaled_dot_product_attention(tq[None, None], tk[None, None], tv[None, None],
                                                     is_causal=causal)[0, 0].backward(torch.from_numpy(dO))
    dq, dk, dv = oracle.attention_head_backward(Q, K, V, dO, causal)
    assert rel(dq, tq.grad.numpy()) < 1e-12
    assert rel(dk, tk.grad.numpy()) < 1e-12
    assert rel(dv, tv.grad.numpy()) < 1e-12


@pytest.mark.parametrize("causal,N", [(True, 2), (False, 4)])
def test_attention_tp_backward_autograd_witness(causal, N):
    S, B, d, H = 6, 2, 16, 4
    X, Wqkv, bqkv, Wo, bo = _attn_problem(S, B, d, H, seed=3)
    dY = np.random.default_rng(4).normal(size=(S * B, d))
    hd = d // H
    tt = [torch.tensor(a, requires_grad=True) for a in (X, Wqkv, bqkv, Wo, bo)]
    qkv = (tt[0] @ tt[1] + tt[2]).reshape(S, B, 3 * d)
    q, k, v = (qkv[..., p * d:(p + 1) * d].reshape(S, B, H, hd).permute(1, 2, 0, 3) for p in range(3))
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=causal).permute(2, 0, 1, 3)
    (o.reshape(S * B, d) @ tt[3] + tt[4]).backward(torch.from_numpy(dY))
    g = oracle.attention_tp_backward(X, Wqkv, bqkv, Wo, bo, H, N, B, causal, dY)
    for key, i in (("dX", 0), ("dWqkv", 1), ("dbqkv", 2), ("dWo", 3), ("dbo", 4)):
        assert rel(g[key], tt[i].grad.numpy()) < 1e-12, key


def test_attention_head_backward_saved_output():
    """D formed from a saved (perturbed) output O': the exact gradients' softmax rows sum to zero, so with
    a key column held at a constant c, dQ's column is then -c·rowsum(dO ⊙ (O' - O))/√hd; dV does not
    depend on D; passing the exact output reproduces the default."""
    rng = np.random.default_rng(11)
    Q, K, V, dO = (rng.normal(size=(6, 4)) for _ in range(4))
    c = 1.5
    K[:, 0] = c
    O = oracle.attention_head(Q, K, V, True)
    exact = oracle.attention_head_backward(Q, K, V, dO, True)
    same = oracle.attention_head_backward(Q, K, V, dO, True, O=O)
    for a, b in zip(exact, same):
        assert rel(a, b) < 1e-13
    assert np.max(np.abs(exact[0][:, 0])) < 1e-12
    O_saved = O + 0.01 * rng.normal(size=O.shape)
    dq, dk, dv = oracle.attention_head_backward(Q, K, V, dO, True, O=O_saved)
    delta = (dO * (O_saved - O)).sum(axis=1)
    assert np.allclose(dq[:, 0], -c * delta / 2.0, atol=1e-12, rtol=0)  # sqrt(hd) = 2
    assert rel(dv, exact[2]) < 1e-14


def test_attention_head_backward_finite_difference():
    """Central differences of a scalar loss <dO, O> for a few entries of Q, K and V."""
    rng = np.random.default_rng(10)
    Q, K, V, dO = (rng.normal(size=(5, 3)) for _ in range(4))
    dq, dk, dv = oracle.attention_head_backward(Q, K, V, dO, True)
    loss = lambda q, k, v: float((oracle.attention_head(q, k, v, True) * dO).sum())
    eps = 1e-6
    for name, A, G in (("Q", Q, dq), ("K", K, dk), ("V", V, dv)):
        for (i, j) in ((0, 0), (2, 1), (4, 2)):
            Ap, Am = A.copy(), A.copy()
            Ap[i, j] += eps
            Am[i, j] -= eps
            args_p = [Ap if n == name else M for n, M in (("Q", Q), ("K", K), ("V", V))]
            args_m = [Am if n == name else M for n, M in (("Q", Q), ("K", K), ("V", V))]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(fd - G[i, j]) < 1e-7 * max(1.0, abs(fd)), (name, i, j)
