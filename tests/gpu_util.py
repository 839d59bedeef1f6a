"""Helpers of the GPU parity tests: device upload/download of bf16 bit arrays and the tolerance check."""
import numpy as np
import torch

from tensor_transformer_mlp_tp_gb300 import inputs

# Tolerance for bf16 inputs with fp32 accumulation: max|err| <= 2e-2 max|ref| and
# ||err||_F <= 5e-3 ||ref||_F; for the fp32 path 1e-5 relative.
BF16_MAXREL = 2e-2
BF16_FROB = 5e-3
FP32_REL = 1e-5


def dev(bits):
    """bf16 bit array (uint16) -> CUDA bf16 tensor."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def f64(t):
    """CUDA bf16 or fp32 tensor -> float64 numpy array of its exact values."""
    if t.dtype == torch.bfloat16:
        return inputs.bf16_bits_to_f64(t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)).reshape(
            tuple(t.shape))
    return t.double().cpu().numpy()


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = got - ref
    maxrel = float(np.max(np.abs(err)) / max(np.max(np.abs(ref)), 1e-30)) if ref.size else 0.0
    frob = float(np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-30)) if ref.size else 0.0
    return maxrel, frob


def assert_bf16_close(name, got, ref):
    assert np.all(np.isfinite(got)), f"{name}: non-finite output"
    maxrel, frob = errors(got, ref)
    assert maxrel <= BF16_MAXREL and frob <= BF16_FROB, f"{name}: max|err|/max|ref|={maxrel:.3e} frob={frob:.3e}"


def assert_fp32_close(name, got, ref):
    maxrel, frob = errors(got, ref)
    assert maxrel <= FP32_REL and frob <= FP32_REL, f"{name}: max|err|/max|ref|={maxrel:.3e} frob={frob:.3e}"


GUARD = 4096  # elements of guard band on each side of an output buffer


# guard pattern per element size (one byte for E4M3 buffers)
_PATTERN = {1: 0x3B, 2: 0x7F3B, 4: 0x7F3B}


def _bits_dtype(dtype):
    return {1: torch.uint8, 2: torch.int16, 4: torch.int32}[dtype.itemsize]


class Guarded:
    """An output buffer with guard bands before and after it, filled with a pattern that no kernel writes."""

    def __init__(self, shape, dtype=torch.bfloat16):
        n = int(np.prod(shape))
        self.raw = torch.empty(n + 2 * GUARD, dtype=dtype, device="cuda")
        self.raw.view(_bits_dtype(dtype)).fill_(_PATTERN[dtype.itemsize])
        self.t = self.raw[GUARD:GUARD + n].view(*shape)

    def intact(self):
        bits = self.raw.view(_bits_dtype(self.raw.dtype))
        n = self.raw.numel()
        pat = _PATTERN[self.raw.dtype.itemsize]
        return bool((bits[:GUARD] == pat).all()) and bool((bits[n - GUARD:] == pat).all())
