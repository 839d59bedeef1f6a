"""GPU parity of the tensor-parallel attention block against the CPU oracle: the attention core on its
own (QKV drawn directly) and the whole block (projection GEMM, attention core, output projection with
the shard sum).  Sequences span several 128-query and 128-key tiles with ragged tails, several batch
elements and heads, causal and not."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import Guarded, assert_bf16_close, dev, f64
from tensor_transformer_mlp_tp_gb300 import binding, inputs

pytestmark = pytest.mark.gpu
HD = 128


@pytest.fixture(autouse=True)
def _device_status_clean():
    yield
    st, site = binding.tpmlp_get_device_status()
    assert st == binding.OK, f"device status {binding.status_string(st)} (wait site {site})"


def _core_reference(qkv, S, B, H, causal):
    """The oracle's attention per (batch element, head) from the [S B x 3 H hd] projection output."""
    d = H * HD
    out = np.zeros((S * B, d))
    for b in range(B):
        rows = slice(b, S * B, B)
        for h in range(H):
            q, k, v = (qkv[rows, part * d + h * HD:part * d + (h + 1) * HD] for part in range(3))
            out[rows, h * HD:(h + 1) * HD] = oracle.attention_head(q, k, v, causal)
    return out


@pytest.mark.parametrize("S,B,H", [(256, 1, 2), (200, 2, 2), (384, 1, 3), (64, 3, 1), (129, 1, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_attention_core(S, B, H, causal):
    w = inputs.small_workload(64, 64, 2, name=f"attn_{S}_{B}_{H}")
    qkv = inputs.draw(w, "QKV", shape=(S * B, 3 * H * HD), dist=(0.0, 1.0))
    O = Guarded((S * B, H * HD))
    binding.tpmlp_attention_core(dev(qkv[0]), S, B, H, O.t, causal=causal)
    torch.cuda.synchronize()
    assert_bf16_close("O", f64(O.t), _core_reference(qkv[1], S, B, H, causal))
    assert O.intact()


def test_attention_core_peaked_scores():
    """Large scores (a few keys dominate each row): the running maximum and the rescaling carry the result."""
    S, B, H = 320, 1, 1
    w = inputs.small_workload(64, 64, 2, name="attn_peaked")
    qkv = inputs.draw(w, "QKV", shape=(S * B, 3 * H * HD), dist=(0.0, 3.0))
    O = Guarded((S * B, H * HD))
    binding.tpmlp_attention_core(dev(qkv[0]), S, B, H, O.t, causal=True)
    torch.cuda.synchronize()
    assert_bf16_close("O", f64(O.t), _core_reference(qkv[1], S, B, H, True))


@pytest.mark.parametrize("S,B,H,N,causal", [(256, 2, 4, 2, True), (200, 1, 4, 4, False), (512, 1, 8, 8, True)])
def test_attention_tp_forward_block(S, B, H, N, causal):
    d = H * HD
    T = S * B
    w = inputs.small_workload(T, d, N, name=f"attnblk_{S}_{B}_{H}")
    X = inputs.draw(w, "X")
    Wqkv = inputs.draw(w, "Wqkv", shape=(d, 3 * d), dist=(0.0, 1.0 / np.sqrt(d)))
    bqkv = inputs.draw(w, "bqkv", shape=(3 * d,), dist=(0.0, 0.1))
    Wo = inputs.draw(w, "Wo", shape=(d, d), dist=(0.0, 1.0 / np.sqrt(d)))
    bo = inputs.draw(w, "bo", shape=(d,), dist=(0.0, 0.1))
    Y = Guarded((T, d))
    qkv = torch.empty(T, 3 * d, dtype=torch.bfloat16, device="cuda")
    O = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    binding.tpmlp_attention_tp_forward(dev(X[0]), dev(Wqkv[0]), dev(Wo[0]), S, B, H, N, Y.t, bqkv=dev(bqkv[0]),
                                       bo=dev(bo[0]), causal=causal, QKV_out=qkv, O_out=O)
    torch.cuda.synchronize()
    ref, parts = oracle.attention_tp(X[1], Wqkv[1], bqkv[1], Wo[1], bo[1], H, N, B, causal, return_parts=True)
    assert_bf16_close("QKV", f64(qkv), X[1] @ Wqkv[1] + bqkv[1])
    assert_bf16_close("O", f64(O), parts["O"])
    assert_bf16_close("Y", f64(Y.t), ref)
    assert Y.intact()


# ----------------------------------------------------------------------------- backward

LN2 = np.log(2.0)


def _lse_reference(qkv, S, B, H, causal):
    """Each row's log2-domain log-sum-exp of the scaled scores, [B·H x S]."""
    d = H * HD
    out = np.zeros((B * H, S))
    for b in range(B):
        rows = slice(b, S * B, B)
        for h in range(H):
            q, k = (qkv[rows, part * d + h * HD:part * d + (h + 1) * HD] for part in range(2))
            s = q @ k.T / np.sqrt(HD)
            if causal:
                s = np.where(np.tril(np.ones((S, S), dtype=bool)), s, -np.inf)
            m = s.max(axis=1)
            out[b * H + h] = (m + np.log(np.exp(s - m[:, None]).sum(axis=1))) / LN2
    return out


def _core_backward_reference(qkv, dO, S, B, H, causal):
    d = H * HD
    dqkv = np.zeros((S * B, 3 * d))
    for b in range(B):
        rows = slice(b, S * B, B)
        for h in range(H):
            c = [slice(part * d + h * HD, part * d + (h + 1) * HD) for part in range(3)]
            dq, dk, dv = oracle.attention_head_backward(qkv[rows, c[0]], qkv[rows, c[1]], qkv[rows, c[2]],
                                                        dO[rows, h * HD:(h + 1) * HD], causal)
            dqkv[rows, c[0]], dqkv[rows, c[1]], dqkv[rows, c[2]] = dq, dk, dv
    return dqkv


@pytest.mark.parametrize("S,B,H", [(256, 1, 2), (200, 2, 2), (129, 1, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_attention_core_lse(S, B, H, causal):
    """The forward's saved statistics: log2 of each row's softmax denominator (scores in log2 units)."""
    w = inputs.small_workload(64, 64, 2, name=f"attn_{S}_{B}_{H}")
    qkv = inputs.draw(w, "QKV", shape=(S * B, 3 * H * HD), dist=(0.0, 1.0))
    O = torch.empty(S * B, H * HD, dtype=torch.bfloat16, device="cuda")
    lse = torch.full(binding.attention_lse_shape(S, B, H), float("nan"), dtype=torch.float32, device="cuda")
    binding.tpmlp_attention_core(dev(qkv[0]), S, B, H, O, causal=causal, LSE=lse)
    torch.cuda.synchronize()
    got = lse[:, :S].double().cpu().numpy()
    ref = _lse_reference(qkv[1], S, B, H, causal)
    assert np.max(np.abs(got - ref)) <= 1e-3 * max(1.0, np.max(np.abs(ref)))
    assert_bf16_close("O", f64(O), _core_reference(qkv[1], S, B, H, causal))


@pytest.mark.parametrize("S,B,H", [(256, 1, 2), (200, 2, 2), (384, 1, 3), (64, 3, 1), (129, 1, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_attention_core_backward(S, B, H, causal):
    """dQ, dK, dV of every (batch, head) against the oracle's chain rule, from the forward's saved O and
    statistics; ragged tails pad the last query and key tiles."""
    w = inputs.small_workload(64, 64, 2, name=f"attnbwd_{S}_{B}_{H}")
    qkv = inputs.draw(w, "QKV", shape=(S * B, 3 * H * HD), dist=(0.0, 1.0))
    dO = inputs.draw(w, "dO", shape=(S * B, H * HD), dist=(0.0, 1.0))
    QKV = dev(qkv[0])
    O = torch.empty(S * B, H * HD, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(binding.attention_lse_shape(S, B, H), dtype=torch.float32, device="cuda")
    binding.tpmlp_attention_core(QKV, S, B, H, O, causal=causal, LSE=lse)
    dQKV = Guarded((S * B, 3 * H * HD))
    binding.tpmlp_attention_core_backward(QKV, O, dev(dO[0]), lse, S, B, H, dQKV.t, causal=causal)
    torch.cuda.synchronize()
    ref = _core_backward_reference(qkv[1], dO[1], S, B, H, causal)
    got = f64(dQKV.t)
    d = H * HD
    for part, name in enumerate(("dQ", "dK", "dV")):
        assert_bf16_close(name, got[:, part * d:(part + 1) * d], ref[:, part * d:(part + 1) * d])
    assert dQKV.intact()


def test_attention_core_backward_peaked_scores():
    """Peaked softmax rows (scores with a standard deviation near 9): dS = P (dP - D) cancels for the
    dominant keys, so D is formed on both sides from the same saved output, the exact O rounded to bf16
    as the forward returns it."""
    S, B, H = 320, 1, 1
    w = inputs.small_workload(64, 64, 2, name="attnbwd_peaked")
    qkv = inputs.draw(w, "QKV", shape=(S * B, 3 * H * HD), dist=(0.0, 3.0))
    dO = inputs.draw(w, "dO", shape=(S * B, H * HD), dist=(0.0, 1.0))
    q, k, v = qkv[1][:, :HD], qkv[1][:, HD:2 * HD], qkv[1][:, 2 * HD:]
    O_saved = oracle.round_bf16(oracle.attention_head(q, k, v, True))
    QKV = dev(qkv[0])
    O = dev(inputs.f32_to_bf16_bits(O_saved.astype(np.float32)))  # exact: O_saved holds bf16 values
    lse = torch.empty(binding.attention_lse_shape(S, B, H), dtype=torch.float32, device="cuda")
    binding.tpmlp_attention_core(QKV, S, B, H, torch.empty_like(O), causal=True, LSE=lse)
    dQKV = torch.empty(S * B, 3 * H * HD, dtype=torch.bfloat16, device="cuda")
    binding.tpmlp_attention_core_backward(QKV, O, dev(dO[0]), lse, S, B, H, dQKV, causal=True)
    torch.cuda.synchronize()
    ref = np.concatenate(oracle.attention_head_backward(q, k, v, dO[1], True, O=O_saved), axis=1)
    got = f64(dQKV)
    for part, name in enumerate(("dQ", "dK", "dV")):
        assert_bf16_close(name, got[:, part * HD:(part + 1) * HD], ref[:, part * HD:(part + 1) * HD])


def test_attention_core_backward_deterministic():
    """No atomics: two runs give the same bits."""
    S, B, H = 384, 2, 2
    w = inputs.small_workload(64, 64, 2, name="attnbwd_det")
    qkv = inputs.draw(w, "QKV", shape=(S * B, 3 * H * HD), dist=(0.0, 1.0))
    dO = dev(inputs.draw(w, "dO", shape=(S * B, H * HD), dist=(0.0, 1.0))[0])
    QKV = dev(qkv[0])
    O = torch.empty(S * B, H * HD, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(binding.attention_lse_shape(S, B, H), dtype=torch.float32, device="cuda")
    binding.tpmlp_attention_core(QKV, S, B, H, O, causal=True, LSE=lse)
    outs = []
    for _ in range(2):
        dQKV = torch.empty(S * B, 3 * H * HD, dtype=torch.bfloat16, device="cuda")
        binding.tpmlp_attention_core_backward(QKV, O, dO, lse, S, B, H, dQKV, causal=True)
        outs.append(dQKV)
    torch.cuda.synchronize()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


@pytest.mark.parametrize("S,B,H,N,causal", [(256, 2, 4, 2, True), (200, 1, 4, 4, False), (384, 1, 8, 8, True)])
def test_attention_tp_backward_block(S, B, H, N, causal):
    """The whole block's gradients (dX with the backward shard sum, dWqkv, dbqkv, dWo, dbo) against the
    oracle, from the forward's saved QKV, O and statistics."""
    d = H * HD
    T = S * B
    w = inputs.small_workload(T, d, N, name=f"attnblkbwd_{S}_{B}_{H}")
    X = inputs.draw(w, "X")
    Wqkv = inputs.draw(w, "Wqkv", shape=(d, 3 * d), dist=(0.0, 1.0 / np.sqrt(d)))
    bqkv = inputs.draw(w, "bqkv", shape=(3 * d,), dist=(0.0, 0.1))
    Wo = inputs.draw(w, "Wo", shape=(d, d), dist=(0.0, 1.0 / np.sqrt(d)))
    bo = inputs.draw(w, "bo", shape=(d,), dist=(0.0, 0.1))
    dY = inputs.draw(w, "dY", shape=(T, d), dist=(0.0, 1.0))
    Xd, Wqkvd, Wod = dev(X[0]), dev(Wqkv[0]), dev(Wo[0])
    Y = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    qkv = torch.empty(T, 3 * d, dtype=torch.bfloat16, device="cuda")
    O = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(binding.attention_lse_shape(S, B, H), dtype=torch.float32, device="cuda")
    binding.tpmlp_attention_tp_forward(Xd, Wqkvd, Wod, S, B, H, N, Y, bqkv=dev(bqkv[0]), bo=dev(bo[0]), causal=causal,
                                       QKV_out=qkv, O_out=O, LSE_out=lse)
    dX = Guarded((T, d))
    dWqkv = Guarded((d, 3 * d))
    dbqkv = Guarded((3 * d,))
    dWo = Guarded((d, d))
    dbo = Guarded((d,))
    dQKV = torch.empty(T, 3 * d, dtype=torch.bfloat16, device="cuda")
    binding.tpmlp_attention_tp_backward(Xd, Wqkvd, Wod, qkv, O, lse, dev(dY[0]), S, B, H, N, dX.t, dWqkv.t, dWo.t,
                                        dbqkv=dbqkv.t, dbo=dbo.t, causal=causal, dQKV_out=dQKV)
    torch.cuda.synchronize()
    ref = oracle.attention_tp_backward(X[1], Wqkv[1], bqkv[1], Wo[1], bo[1], H, N, B, causal, dY[1])
    assert_bf16_close("dQKV", f64(dQKV), ref["dQKV"])
    for name, buf in (("dX", dX), ("dWqkv", dWqkv), ("dbqkv", dbqkv), ("dWo", dWo), ("dbo", dbo)):
        assert_bf16_close(name, f64(buf.t), ref[name])
        assert buf.intact(), name


# ----------------------------------------------------------------------------- the bench's attention shape

def test_attention_core_forward_backward_bench_shape():
    """S = 4096 positions x B = 2 sequences, 32 heads of 128, causal (the attention row's shape): the whole
    core forward and backward run, and two (batch, head) pairs (the first head of batch 0 and the last of
    batch 1, so both corners of the grid) are checked in full against the oracle."""
    S, B, H = 4096, 2, 32
    d = H * HD
    w = inputs.small_workload(64, 64, 2, name="attn_bench_shape")
    qkv = inputs.draw(w, "QKV", shape=(S * B, 3 * d), dist=(0.0, 1.0))
    dO = inputs.draw(w, "dO", shape=(S * B, d), dist=(0.0, 1.0))
    QKV = dev(qkv[0])
    O = torch.empty(S * B, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(binding.attention_lse_shape(S, B, H), dtype=torch.float32, device="cuda")
    binding.tpmlp_attention_core(QKV, S, B, H, O, causal=True, LSE=lse)
    dQKV = torch.empty(S * B, 3 * d, dtype=torch.bfloat16, device="cuda")
    binding.tpmlp_attention_core_backward(QKV, O, dev(dO[0]), lse, S, B, H, dQKV, causal=True)
    torch.cuda.synchronize()
    Og, dQKVg = f64(O), f64(dQKV)
    for b, h in ((0, 0), (1, H - 1)):
        rows = slice(b, S * B, B)
        c = [slice(part * d + h * HD, part * d + (h + 1) * HD) for part in range(3)]
        q, k, v = (qkv[1][rows, cc] for cc in c)
        ref_o = oracle.attention_head(q, k, v, True)
        assert_bf16_close(f"O (b={b}, h={h})", Og[rows, h * HD:(h + 1) * HD], ref_o)
        dq, dk, dv = oracle.attention_head_backward(q, k, v, dO[1][rows, h * HD:(h + 1) * HD], True)
        for name, got, ref in (("dQ", dQKVg[rows, c[0]], dq), ("dK", dQKVg[rows, c[1]], dk),
                               ("dV", dQKVg[rows, c[2]], dv)):
            assert_bf16_close(f"{name} (b={b}, h={h})", got, ref)


def _random_attention_shapes(seed, n):
    rng = np.random.default_rng(seed)
    return [(int(rng.integers(1, 600)), int(rng.integers(1, 4)), int(rng.integers(1, 4)), bool(rng.integers(0, 2)))
            for _ in range(n)]


@pytest.mark.parametrize("S,B,H,causal", _random_attention_shapes(20261204, 10))
def test_attention_core_random_shape(S, B, H, causal):
    """A seeded sweep of sequence lengths (ragged against the 128-row tiles, down to one position), batch
    sizes and head counts: the forward output, then dQ, dK, dV from its saved statistics."""
    w = inputs.small_workload(64, 64, 2, name=f"attnrand_{S}_{B}_{H}")
    qkv = inputs.draw(w, "QKV", shape=(S * B, 3 * H * HD), dist=(0.0, 1.0))
    dO = inputs.draw(w, "dO", shape=(S * B, H * HD), dist=(0.0, 1.0))
    QKV = dev(qkv[0])
    O = torch.empty(S * B, H * HD, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(binding.attention_lse_shape(S, B, H), dtype=torch.float32, device="cuda")
    binding.tpmlp_attention_core(QKV, S, B, H, O, causal=causal, LSE=lse)
    dQKV = Guarded((S * B, 3 * H * HD))
    binding.tpmlp_attention_core_backward(QKV, O, dev(dO[0]), lse, S, B, H, dQKV.t, causal=causal)
    torch.cuda.synchronize()
    assert_bf16_close("O", f64(O), _core_reference(qkv[1], S, B, H, causal))
    ref = _core_backward_reference(qkv[1], dO[1], S, B, H, causal)
    got = f64(dQKV.t)
    d = H * HD
    for part, name in enumerate(("dQ", "dK", "dV")):
        assert_bf16_close(name, got[:, part * d:(part + 1) * d], ref[:, part * d:(part + 1) * d])
    assert dQKV.intact()
