"""Helpers shared by the GPU parity tests: conversions and tolerance checks.

No layer arithmetic lives here: expected values always come from the oracle."""
import numpy as np
import torch

import oracle

# tolerance on bf16 expert / layer outputs versus the fp64 oracle: 2e-2 absolute + 1e-2 relative
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


def graph_replay_matches_eager(layer, x_loc, lg_loc, out):
    """The launch configuration the benchmark times: the layer step captured as a CUDA
    graph and replayed writes the same output bits as the eager step that produced
    `out` (already checked against the oracle)."""
    eager = [t.clone() for t in out]
    out2 = [torch.empty_like(t) for t in out]
    g = layer.capture(x_loc, lg_loc, out2)
    for t in out2:                               # the capture's warm-up step wrote them
        t.fill_(7.0)
    g.replay()
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    for a, b in zip(out2, eager):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b)
