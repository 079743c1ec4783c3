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


# ------------------------------------------------------------------ hard rows
def ffn_kernel_of(layer):
    """Which grouped-FFN kernel the library runs for this layer: FP8 -> 'fp8' (weights
    as M, units of up to 64 tokens), or with >= 192 sorted rows per slot on average and
    H, I multiples of 512 'pair8' (the pair kernel's units on FP8, the first MMA up to
    224 tokens); bf16 with >= 192 sorted rows per slot on average
    -> 'pair' (weights as M on SM pairs, units of up to 320 tokens); else 'tc' (tokens
    as M, 128-row m-tiles).  With the split FFN, a function of the slot's rows: 'pair'
    from the hot threshold, else 'tc'."""
    if getattr(layer, "fp8", False):
        # many rows per slot (and H, I multiples of 512): the FP8 pair kernel; 32-191
        # rows per slot on average: the pair kernel for slots of 192 or more rows
        per = layer.cap // max(layer.P, 1)
        if layer.H % 512 == 0 and layer.I % 512 == 0:
            if per >= 192:
                return "pair8"
            if per >= 32 and layer.cap >= 192:
                return lambda rows: "pair8" if rows >= 192 else "fp8"
        return "fp8"
    split = getattr(layer, "ffn_split", None)
    if split:
        return lambda rows: "pair" if rows >= split[0] else "tc"
    return "pair" if layer.cap // max(layer.P, 1) >= 192 else "tc"


def _slot_positions(rows: int, kernel: str):
    """Positions within a slot of `rows` sorted rows where the kernel's tiling changes."""
    pos = set()
    if kernel in ("pair", "pair8"):
        # unit = up to 320 tokens; N = tokens rounded up to 16, CTA c of the pair holds
        # tokens [c*N/2, (c+1)*N/2); the first MMA reads the first N0/2 of each CTA's
        # rows, the tail MMA the rest: bf16 N0 = N up to 256, else N - 64 (the tail
        # takes the last 64 columns); FP8 N0 = min(N, 224)
        for g0 in range(0, rows, 320):
            nt = min(320, rows - g0)
            N = (nt + 15) & ~15
            if kernel == "pair":
                n0 = N if N <= 256 else N - 64
            else:
                n0 = min(N, 224)
            h = N // 2
            for p in (0, 31, 32, n0 // 2 - 1, n0 // 2, h - 1, h, h + 31, h + 32,
                      h + n0 // 2 - 1, h + n0 // 2, N - 1, nt - 1):
                if 0 <= p < nt:
                    pos.add(g0 + p)
    elif kernel == "tc":
        # 128-row m-tiles; epilogue warps own 32-row lane quarters
        tiles = list(range(0, rows, 128))
        for t0 in tiles[:1] + tiles[-1:]:
            for p in (0, 31, 32, 63, 64, 95, 96, 127):
                if t0 + p < rows:
                    pos.add(t0 + p)
        pos.add(rows - 1)
    else:  # fp8: units of up to 64 tokens, two epilogue warps of 32 token columns
        groups = list(range(0, rows, 64))
        for g0 in groups[:2] + groups[-1:]:
            for p in (0, 31, 32, 63):
                if g0 + p < rows:
                    pos.add(g0 + p)
        pos.add(rows - 1)
    return sorted(pos)


def hard_rows(offsets, kernel: str, min_rows: int = 64, seed: int = 0, keep=None):
    """Sorted-buffer rows d at the grouped-FFN kernel's tiling boundaries: the first and
    last token of every unit, lane-quarter and 32-column chunk edges, and (pair kernel)
    both sides of the split between the N <= 256 MMA and the tail MMA of columns
    256-319.  Slots are taken largest first, then the smallest non-empty one, a slot
    whose last unit has a tail MMA, then seeded random slots, until at least min_rows
    rows are chosen; keep (a mask over sorted rows) drops rows such as alignment pads."""
    offsets = np.asarray(offsets, np.int64)
    counts = np.diff(offsets)
    nz = np.nonzero(counts > 0)[0]
    if len(nz) == 0:
        return []
    order = [int(nz[np.argmax(counts[nz])]), int(nz[np.argmin(counts[nz])])]
    if callable(kernel):   # the hottest and coldest slot of each kernel first
        for kern in ("pair", "tc"):
            mine = [int(x) for x in nz if kernel(int(counts[x])) == kern]
            if mine:
                order += [max(mine, key=lambda x: counts[x]), min(mine, key=lambda x: counts[x])]
    tail = [int(s) for s in nz if 256 < (counts[s] - 1) % 320 + 1 <= 320]
    order += tail[:2]
    rng = np.random.default_rng(seed)
    order += [int(s) for s in rng.permutation(nz)]
    out, seen = [], set()
    for s in order:
        if s in seen:
            continue
        seen.add(s)
        kern = kernel(int(counts[s])) if callable(kernel) else kernel
        out += [d for d in (int(offsets[s]) + p for p in _slot_positions(int(counts[s]), kern))
                if keep is None or keep[d]]
        if len(set(out)) >= min_rows and len(seen) >= 4:
            break
    return sorted(set(out))


def pairs_to_check(layer, o_o, p_o, i_o, real, kk: int, sample):
    """(token, j) pairs whose expert outputs a layer test compares with the oracle, and
    the tokens whose combined rows it compares.  sample None: every real token and
    all its pairs.  Otherwise the pairs at the kernel's hard rows (at least 64; see
    hard_rows), plus the first two and last two real tokens and `sample` tokens
    spread over the hard pairs, each with all of its kk pairs."""
    if sample is None:
        return [(int(g), j) for g in real for j in range(kk)], real
    kernel = ffn_kernel_of(layer)
    real_d = p_o >= 0                    # sorted rows that hold a token (not an alignment pad)
    hard = hard_rows(o_o, kernel, keep=real_d)
    hard_pairs = [(int(p_o[d]), int(np.nonzero(i_o[p_o[d]] == d)[0][0])) for d in hard]
    # at least 64, unless the layer has fewer boundary rows in all its slots together
    every = hard_rows(o_o, kernel, min_rows=1 << 30, keep=real_d)
    assert len(hard_pairs) >= min(64, len(every)), (len(hard_pairs), len(every))
    picked = np.unique([g for g, _ in hard_pairs])
    spread = picked[np.linspace(0, len(picked) - 1, min(sample, len(picked))).astype(int)]
    toks = np.unique(np.concatenate([real[:2], real[-2:], spread])).astype(np.int64)
    pairs = set(hard_pairs) | {(int(g), j) for g in toks for j in range(kk)}
    return sorted(pairs), toks
