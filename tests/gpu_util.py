"""Helpers shared by the GPU parity tests: conversions and tolerance checks.

No layer arithmetic lives here: expected values always come from the oracle."""
import numpy as np
import torch

import oracle

# the benchmark spec tolerance on bf16 expert / layer outputs versus the fp64 oracle
BF16_ATOL, BF16_RTOL = 2e-2, 1e-2
# float32 CUDA-core path: fp32 accumulation over <= a few thousand terms
F32_ATOL, F32_RTOL = 1e-4, 1e-4
# route weights: float32 softmax (expf, one division) against the fp64 oracle
W_ATOL, W_RTOL = 1e-6, 2e-6


def to_np(t: torch.Tensor) -> np.ndarray:
    """Host copy; bf16 tensors come back as their uint16 bit patterns."""
    t = t.detach().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def as_f32(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bits (uint16) or identity for float arrays."""
    if a.dtype == np.uint16:
        return oracle.bf16_bits_to_f32(a)
    return np.asarray(a, dtype=np.float32)


def assert_close(got, ref, atol, rtol, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    if bad.any():
        i = np.unravel_index(np.argmax(err - (atol + rtol * np.abs(ref))), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; "
                             f"max |err| {err.max():.3e}; worst at {i}: got {got[i]} ref {ref[i]}")
    return float(err.max()) if err.size else 0.0


def rel_fro(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    n = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / n) if n > 0 else float(np.linalg.norm(got))
