"""Seeded synthetic inputs for the MoE layer between DP attention and EP.

This module holds workload recipes only: replica token counts, hidden states,
router logits, expert weights and the EPLB expert map used by the
EPLB-remapped workload.  It contains none of the layer's arithmetic (no
layout, routing, sorting, FFN or combine), imports neither the CUDA library
nor the oracle, and serves both sides with identical values.

Large tensors are drawn with torch generators on the requested device (the
expert weights of a DeepSeek-V3-shaped layer are 22.5 GB); small integer
choices use numpy's PCG64.  Draws are reproducible for a given (seed, device).

Workloads (hidden 7168, 256 experts, top-8 and expert intermediate 2048 are the
DeepSeek-V3 expert shapes quoted in "SGLang 源码完全拆解(十七)", section
"EP 下专家权重切不均匀的问题"):
  tiny_fp32     4 replicas, counts [16, 0, 40, 8], SUM padding, H=256, 8 experts,
                top-2, I=128, fp32.
  dsv3_decode   8 replicas, counts uniform in [0, 64] with at least one idle
                replica, MAX padding, bf16, logits N(0,1) + Zipf(1.1) bias.
  dsv3_prefill  one replica with 8192 tokens, bf16, uniform popularity.
  pad_sweep     16 replicas with 0/4/8/24 requests of 1 or 4 tokens each,
                SUM, MAX or static bound B=24, bf16.
  eplb          2048 tokens, 256 logical experts on 288 slots (the 32 hottest
                replicated), 16 ranges of 18 slots, Zipf(1.3) bias, bf16.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np
import torch

PAD_SUM, PAD_MAX, PAD_STATIC = 0, 1, 2
MODE_NAMES = {PAD_SUM: "sum", PAD_MAX: "max", PAD_STATIC: "static"}


@dataclasses.dataclass
class LayerSpec:
    name: str
    counts: List[int]          # tokens per replica (already times tokens_per_req)
    mode: int                  # PAD_SUM / PAD_MAX / PAD_STATIC
    H: int
    E: int                     # logical experts
    k: int
    I: int
    dtype: str                 # "f32" or "bf16"
    static_bound: int = 0      # requests per replica under PAD_STATIC
    tokens_per_req: int = 1
    P: Optional[int] = None    # physical slots (E when no map)
    zipf_s: Optional[float] = None
    eplb_extra: int = 0        # redundant slots (EPLB workload)
    n_ranges: int = 1          # contiguous slot ranges standing in for EP ranks
    renormalize: bool = True
    align: int = 1
    seed: int = 0
    w_std: float = 0.02
    n_shared: int = 0          # shared experts (logical ids E .. E + n_shared - 1)

    @property
    def R(self) -> int:
        return len(self.counts)

    @property
    def T(self) -> int:
        return int(sum(self.counts))

    @property
    def slots(self) -> int:
        """Physical slots, shared experts included (they are the last slots)."""
        return (self.P if self.P is not None else self.E) + self.n_shared


# ------------------------------------------------------------------ specs
def spec_tiny() -> LayerSpec:
    return LayerSpec("tiny_fp32", [16, 0, 40, 8], PAD_SUM, H=256, E=8, k=2, I=128, dtype="f32")


def decode_counts(seed: int = 0, R: int = 8, hi: int = 64) -> List[int]:
    rng = np.random.Generator(np.random.PCG64(seed))
    c = rng.integers(0, hi + 1, size=R)
    if not (c == 0).any():
        c[int(rng.integers(0, R))] = 0
    return [int(v) for v in c]


def spec_decode(seed: int = 0, H=7168, E=256, k=8, I=2048) -> LayerSpec:
    return LayerSpec("dsv3_decode", decode_counts(seed), PAD_MAX, H=H, E=E, k=k, I=I,
                     dtype="bf16", zipf_s=1.1, seed=seed)


def spec_prefill(T: int = 8192, H=7168, E=256, k=8, I=2048, seed: int = 0) -> LayerSpec:
    return LayerSpec("dsv3_prefill", [T], PAD_SUM, H=H, E=E, k=k, I=I, dtype="bf16",
                     seed=seed)


SWEEP_MIXES = ("mix0", "mix1", "mix2", "all4", "all8", "all24")


def sweep_requests(mix: str, R: int = 16) -> List[int]:
    if mix.startswith("all"):
        return [int(mix[3:])] * R
    rng = np.random.Generator(np.random.PCG64(100 + int(mix[3:])))
    return [int(v) for v in rng.choice(np.array([0, 4, 8, 24]), size=R)]


def spec_pad_sweep(mix: str = "mix0", tokens_per_req: int = 1, mode: int = PAD_MAX,
                   H=7168, E=256, k=8, I=2048) -> LayerSpec:
    reqs = sweep_requests(mix)
    counts = [r * tokens_per_req for r in reqs]
    return LayerSpec(f"pad_sweep_{mix}_tpr{tokens_per_req}_{MODE_NAMES[mode]}", counts, mode,
                     H=H, E=E, k=k, I=I, dtype="bf16", static_bound=24,
                     tokens_per_req=tokens_per_req, seed=7)


def spec_eplb(T: int = 2048, H=7168, E=256, k=8, I=2048, extra=32, n_ranges=16) -> LayerSpec:
    return LayerSpec("eplb_288", [T], PAD_SUM, H=H, E=E, k=k, I=I, dtype="bf16",
                     P=E + extra, zipf_s=1.3, eplb_extra=extra, n_ranges=n_ranges, seed=3)


# ------------------------------------------------------------------ draws
def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def popularity_rank(E: int, seed: int) -> np.ndarray:
    """A seeded permutation: rank[e] = popularity rank of expert e (0 = hottest)."""
    rng = np.random.Generator(np.random.PCG64(10_000 + seed))
    return rng.permutation(E)


def zipf_bias(E: int, s: float, seed: int) -> np.ndarray:
    """Per-expert additive logit bias -s*ln(rank+1): softmax probabilities then scale
    as (rank+1)**-s, a Zipf(s) popularity over a seeded ranking."""
    rank = popularity_rank(E, seed)
    return (-s * np.log(rank.astype(np.float64) + 1.0)).astype(np.float32)


def hidden_states(spec: LayerSpec, device="cpu") -> List[torch.Tensor]:
    """Per-replica hidden states [c_r, H], N(0,1), in the layer's dtype."""
    g = _gen(device, spec.seed * 1000 + 1)
    x = torch.randn(spec.T, spec.H, generator=g, device=device, dtype=torch.float32)
    x = x.to(torch_dtype(spec.dtype))
    return list(torch.split(x, spec.counts, dim=0))


def router_logits(spec: LayerSpec, device="cpu") -> List[torch.Tensor]:
    """Per-replica router logits [c_r, E] fp32: N(0,1) plus the optional Zipf bias."""
    g = _gen(device, spec.seed * 1000 + 2)
    lg = torch.randn(spec.T, spec.E, generator=g, device=device, dtype=torch.float32)
    if spec.zipf_s is not None:
        lg = lg + torch.from_numpy(zipf_bias(spec.E, spec.zipf_s, spec.seed)).to(device)
    return list(torch.split(lg, spec.counts, dim=0))


def router_gate(spec: LayerSpec, device="cpu"):
    """Gate weights [E, H] bf16, N(0, 1/H), and the optional Zipf bias [E] fp32: the
    gate of hidden states N(0,1) then gives logits N(0,1) plus the same popularity
    bias as router_logits."""
    g = _gen(device, spec.seed * 1000 + 7)
    w = torch.randn(spec.E, spec.H, generator=g, device=device, dtype=torch.float32)
    w = (w / spec.H ** 0.5).to(torch.bfloat16)
    b = None
    if spec.zipf_s is not None:
        b = torch.from_numpy(zipf_bias(spec.E, spec.zipf_s, spec.seed)).to(device)
    return w, b


def expert_weights_logical(spec: LayerSpec, e: int, device="cpu"):
    """Weights of logical expert e: (wgu [2I, H], wd [H, I]) in the layer dtype.
    Gate rows 0..I-1, up rows I..2I-1; each expert has its own seed so any
    subset can be regenerated alone."""
    g = _gen(device, spec.seed * 100_003 + 17 + e)
    dt = torch_dtype(spec.dtype)
    wgu = torch.randn(2 * spec.I, spec.H, generator=g, device=device, dtype=torch.float32)
    wgu = wgu.mul_(spec.w_std).to(dt)
    wd = torch.randn(spec.H, spec.I, generator=g, device=device, dtype=torch.float32)
    wd = wd.mul_(spec.w_std).to(dt)
    return wgu, wd


def expert_weights(spec: LayerSpec, slot_to_logical: Optional[np.ndarray] = None,
                   device="cpu"):
    """Slot weights wgu [P, 2I, H] and wd [P, H, I]; slot s holds the weights of
    logical expert slot_to_logical[s] (identity without a map)."""
    P = spec.slots
    if slot_to_logical is None:
        s2l = np.arange(P) % spec.E
    else:
        s2l = np.asarray(slot_to_logical)
    if spec.n_shared:  # shared expert s sits in slot P - n_shared + s
        s2l = np.concatenate([s2l[: P - spec.n_shared],
                              spec.E + np.arange(spec.n_shared)])
    dt = torch_dtype(spec.dtype)
    wgu = torch.empty(P, 2 * spec.I, spec.H, device=device, dtype=dt)
    wd = torch.empty(P, spec.H, spec.I, device=device, dtype=dt)
    for e in range(spec.E + spec.n_shared):
        slots = np.nonzero(s2l == e)[0]
        if len(slots) == 0:
            continue
        a, b = expert_weights_logical(spec, e, device)
        for s in slots:
            wgu[int(s)].copy_(a)
            wd[int(s)].copy_(b)
    return wgu, wd


# ------------------------------------------------------------------ expert maps
def trivial_map(E: int, P: int):
    """Slot i holds logical expert i mod E ("init_trivial" in the EPLB section of
    the SGLang chapter).  Returns (l2p [E, X], nrep [E], p2l [P])."""
    p2l = np.arange(P) % E
    return _maps_from_p2l(p2l, E)


def _maps_from_p2l(p2l: np.ndarray, E: int):
    nrep = np.bincount(p2l, minlength=E).astype(np.int32)
    X = max(1, int(nrep.max()))
    l2p = np.full((E, X), -1, np.int32)
    fill = np.zeros(E, np.int64)
    for s, e in enumerate(p2l):
        l2p[e, fill[e]] = s
        fill[e] += 1
    return l2p, nrep, p2l.astype(np.int32)


def eplb_expected_counts(spec: LayerSpec) -> np.ndarray:
    """Logical expert token counts the EPLB map is planned from: T*k routings drawn
    multinomially from the Zipf(s) popularity of the workload's logit bias."""
    rank = popularity_rank(spec.E, spec.seed)
    p = (rank + 1.0) ** (-spec.zipf_s)
    p = p / p.sum()
    rng = np.random.Generator(np.random.PCG64(20_000 + spec.seed))
    return rng.multinomial(spec.T * spec.k, p).astype(np.int64)


def eplb_map(counts: np.ndarray, extra: int, n_ranges: int):
    """Host planning step that builds the EPLB-remapped workload's expert map.

    Replicate: the `extra` hottest logical experts (count descending, id
    ascending) get one redundant slot each.  Pack: the replicas, each carrying
    count / replicas, are placed heaviest first into the range with the least
    load that still has room and does not yet hold a replica of the same
    expert (ties: lowest range).  Slots are numbered range by range.
    Returns (l2p [E, X], nrep [E], p2l [P])."""
    E = len(counts)
    P = E + extra
    assert P % n_ranges == 0
    per = P // n_ranges
    order = sorted(range(E), key=lambda e: (-int(counts[e]), e))
    nrep = np.ones(E, np.int64)
    for e in order[:extra]:
        nrep[e] += 1
    reps = [(counts[e] / nrep[e], e, x) for e in range(E) for x in range(nrep[e])]
    reps.sort(key=lambda t: (-t[0], t[1], t[2]))
    load = [0.0] * n_ranges
    members: List[List[int]] = [[] for _ in range(n_ranges)]
    for w, e, _ in reps:
        best = None
        for r in range(n_ranges):
            if len(members[r]) >= per or e in members[r]:
                continue
            if best is None or load[r] < load[best]:
                best = r
        if best is None:  # only ranges holding e have room left
            best = min((r for r in range(n_ranges) if len(members[r]) < per),
                       key=lambda r: (load[r], r))
        members[best].append(e)
        load[best] += w
    p2l = np.array([e for r in range(n_ranges) for e in members[r]], np.int64)
    return _maps_from_p2l(p2l, E)


def slot_ranges(P: int, n_ranges: int):
    per = P // n_ranges
    return [(r * per, (r + 1) * per) for r in range(n_ranges)]


def make_map(spec: LayerSpec):
    """(l2p, nrep, p2l) for the spec, or (None, None, None) without a map."""
    if spec.P is None or spec.P == spec.E:
        return None, None, None
    if spec.eplb_extra:
        return eplb_map(eplb_expected_counts(spec), spec.eplb_extra, spec.n_ranges)
    return trivial_map(spec.E, spec.P)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a bf16 tensor (copied to host)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def flops_ffn(T: int, k: int, H: int, I: int) -> float:
    """Algorithmic FLOPs of the routed SwiGLU FFN: 3 GEMMs of 2*H*I per routed row."""
    return 6.0 * T * k * H * I


def describe(spec: LayerSpec) -> dict:
    return dict(workload=spec.name, replicas=spec.R, tokens=spec.T, padding=MODE_NAMES[spec.mode],
                hidden=spec.H, experts=spec.E, slots=spec.slots, topk=spec.k,
                intermediate=spec.I, dtype=spec.dtype,
                static_bound=spec.static_bound if spec.mode == PAD_STATIC else None,
                tokens_per_req=spec.tokens_per_req,
                zipf_s=spec.zipf_s)


