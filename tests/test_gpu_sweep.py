"""Seeded sweep of small whole-layer configurations against the oracle.

Each case draws the replica count and token counts (idle replicas included),
the padding mode (SUM, MAX, or a static bound at or above the largest count),
the expert count, top-k, hidden and intermediate widths, expert alignment,
shared experts and the softmax variant.  A few cases have many tokens per expert,
so the grouped FFN takes the two-SM kernel with the weights as M.  The checks
are those of the layer tests: layouts, ids, counts, offsets, permutations and
copied rows bit for bit, route weights and expert / layer outputs within
tolerance (on sampled tokens for the FFN), replica outputs equal to the combined
rows.  FP8 cases run the quantising dispatch and the FP8 grouped FFN."""
import gc

import numpy as np
import pytest
import torch

from combine_dp_gather_gb300 import synth
from test_gpu_fp8 import _layer_fp8_check
from test_gpu_parity import _check_layer, _layer_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def md():
    from combine_dp_gather_gb300 import build, moe_dp
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    moe_dp.lib()
    return moe_dp


@pytest.fixture(autouse=True)
def _free_gpu():
    yield
    gc.collect()
    torch.cuda.empty_cache()


def _spec(seed: int, fp8: bool) -> synth.LayerSpec:
    rng = np.random.default_rng(1000 + seed + (500 if fp8 else 0))
    many = seed % 5 == 4            # many tokens per expert: the weights-as-M kernel
    R = int(rng.integers(1, 4 if many else 13))
    counts = [int(c) for c in (rng.integers(150, 500, size=R) if many else
                               rng.integers(0, 60, size=R))]
    if R > 1:
        counts[int(rng.integers(0, R))] = 0           # an idle replica
    if sum(counts) == 0:
        counts[-1] = 7
    mode = int(rng.integers(0, 2 if fp8 else 3))
    static_bound = max(counts) + int(rng.integers(0, 4)) if mode == synth.PAD_STATIC else 0
    E = int(rng.choice([4, 8])) if many else int(rng.choice([8, 16, 40, 64, 96, 256]))
    k = int(rng.integers(1, min(4 if many else 8, E) + 1))
    return synth.LayerSpec(
        f"sweep{'_fp8' if fp8 else ''}{seed}", counts, mode,
        H=int(rng.choice([256, 512, 768])), E=E, k=k, I=int(rng.choice([128, 256, 384])),
        dtype="bf16", static_bound=static_bound, renormalize=bool(rng.integers(0, 2)),
        align=1 if fp8 else int(rng.choice([1, 1, 8, 128])),
        n_shared=int(rng.choice([0, 0, 1])), zipf_s=1.1 if rng.integers(0, 2) else None,
        w_std=0.05, seed=seed)


@pytest.mark.parametrize("seed", range(15))
def test_layer_sweep(md, orc, seed):
    spec = _spec(seed, fp8=False)
    res = _layer_gpu(md, spec)
    _check_layer(md, orc, spec, *res, sample=8)


@pytest.mark.parametrize("seed", range(6))
def test_layer_sweep_fp8(md, orc, seed):
    _layer_fp8_check(md, orc, _spec(seed, fp8=True), sample=8)
