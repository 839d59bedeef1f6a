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
