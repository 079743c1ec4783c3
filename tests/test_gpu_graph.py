"""CUDA-graph replay of a layer step: bit-identical to eager steps, counts may change
between replays as long as the global row count does not."""
import gc

import numpy as np
import pytest
import torch

from gpu_util import to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


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


@pytest.mark.parametrize("fp8", [False, True])
def test_graph_replay_matches_eager(md, fp8):
    from combine_dp_gather_gb300 import synth
    spec = synth.LayerSpec("tiny_graph", [16, 0, 140, 8, 1], 1, H=512, E=16, k=4, I=256,
                           dtype="bf16", w_std=0.05, zipf_s=1.1)
    x = synth.hidden_states(spec, DEV)
    lg = synth.router_logits(spec, DEV)
    wgu, wd = synth.expert_weights(spec, None, DEV)
    _, rows = md.moe_dp_layout(spec.counts, spec.mode)
    layer = md.MoeLayer(R=spec.R, H=spec.H, E=spec.E, k=spec.k, I=spec.I, w_gate_up=wgu,
                        w_down=wd, max_rows=rows, mode=spec.mode, fp8=fp8)
    # replica buffers sized for the largest count, views used per step
    bx = [torch.zeros(140, spec.H, device=DEV, dtype=torch.bfloat16) for _ in spec.counts]
    bl = [torch.zeros(140, spec.E, device=DEV, dtype=torch.float32) for _ in spec.counts]
    bo = [torch.zeros(140, spec.H, device=DEV, dtype=torch.bfloat16) for _ in spec.counts]
    for b, t in zip(bx, x):
        b[: len(t)] = t
    for b, t in zip(bl, lg):
        b[: len(t)] = t
    layer.set_counts(spec.counts)
    g = layer.capture(bx, bl, bo)
    # same counts: replay equals an eager step
    eager = [torch.zeros_like(o) for o in bo]
    layer.forward(bx, bl, eager, counts=spec.counts)
    for o in bo:
        o.zero_()
    g.replay(spec.counts)
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    for a, b, c in zip(bo, eager, spec.counts):
        assert np.array_equal(to_np(a[:c]), to_np(b[:c]))
    # different counts, same max (same global rows under MAX padding)
    counts2 = [20, 3, 140, 0, 7]
    layer.forward(bx, bl, eager, counts=counts2)
    g.replay(counts2)
    torch.cuda.synchronize()
    for a, b, c in zip(bo, eager, counts2):
        assert np.array_equal(to_np(a[:c]), to_np(b[:c]))
    with pytest.raises(md.MoeError):
        g.replay([20, 3, 139, 0, 7])      # 5 x 139 rows: another layout
    # counts staged on another stream, the replay ordered after it
    counts3 = [140, 0, 0, 1, 99]
    layer.forward(bx, bl, eager, counts=counts3)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g.stage(counts3, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    g.replay()
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    for a, b, c in zip(bo, eager, counts3):
        assert np.array_equal(to_np(a[:c]), to_np(b[:c]))


def test_short_replica_tensors_are_rejected_on_the_host(md):
    """The kernels only see pointers: a replica tensor with fewer rows than its count
    (or the wrong width or dtype) is refused before anything is launched, in forward
    and when a graph stages new counts."""
    from combine_dp_gather_gb300 import synth
    spec = synth.LayerSpec("tiny_check", [16, 0, 40], 1, H=512, E=16, k=4, I=256,
                           dtype="bf16", w_std=0.05)
    x = synth.hidden_states(spec, DEV)
    lg = synth.router_logits(spec, DEV)
    wgu, wd = synth.expert_weights(spec, None, DEV)
    layer = md.MoeLayer(R=spec.R, H=spec.H, E=spec.E, k=spec.k, I=spec.I, w_gate_up=wgu,
                        w_down=wd, max_rows=3 * 40, mode=spec.mode)
    out = [torch.empty(c, spec.H, device=DEV, dtype=torch.bfloat16) for c in spec.counts]
    short = [x[0], x[1], x[2][:39]]
    with pytest.raises(md.MoeError):
        layer.forward(short, lg, out, counts=spec.counts)
    with pytest.raises(md.MoeError):
        layer.forward(x, [t.to(torch.bfloat16) for t in lg], out, counts=spec.counts)
    with pytest.raises(md.MoeError):
        layer.forward(x, lg, out[:2], counts=spec.counts)
    layer.forward(x, lg, out, counts=spec.counts)        # the right tensors pass
    g = layer.capture(x, lg, out)
    with pytest.raises(md.MoeError):
        g.replay([40, 0, 16])                            # replica 0 holds 16 rows only
    g.replay([16, 0, 40])
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
