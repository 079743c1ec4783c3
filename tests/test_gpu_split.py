"""GPU tests of moe_grouped_ffn_split: the grouped FFN of a skewed layer split by
slot over two streams (hot slots on the pair kernel, cold slots on the single-SM
kernel beside it, each on its own SM budget).

Each part must equal what its kernel computes alone: the cold slots' rows bit for
bit those of moe_grouped_ffn on the single-SM kernel, the hot slots' rows bit for
bit those of a split in which every slot is hot (the pair kernel alone).  The
layer output is checked against the oracle on the kernels' hard rows, and a CUDA
graph of the split layer replays to the same bits."""
import gc

import numpy as np
import pytest
import torch

from combine_dp_gather_gb300 import synth
from gpu_util import graph_replay_matches_eager

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


def _bits(t):
    return t.view(torch.int16)


def _split_parts_exact(md, layer, hot_rows, hot_sms):
    """Re-run the layer's grouped FFN three ways on its sorted rows: the split, the
    single-SM kernel alone and the pair kernel alone; compare slot by slot."""
    P = layer.P
    n = int(layer.offsets_P[-1].item())
    offs = layer.offsets_P.cpu().numpy()
    counts = np.diff(offs)
    ys_split = torch.full_like(layer.ys, 3.0)
    md.moe_grouped_ffn_split(layer.xs, layer.offsets_P, layer.wgu, layer.wd, ys_split,
                             layer.ws_ffn, hot_rows, hot_sms, layer.stream_hot,
                             d_status=layer.status)
    ys_pair = torch.full_like(layer.ys, 4.0)       # every slot hot: the pair kernel alone
    md.moe_grouped_ffn_split(layer.xs, layer.offsets_P, layer.wgu, layer.wd, ys_pair,
                             layer.ws_ffn, 1, hot_sms, layer.stream_hot, d_status=layer.status)
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    ys_tc = None
    if layer.cap // P < 192:                        # moe_grouped_ffn takes the single-SM kernel
        ys_tc = torch.full_like(layer.ys, 5.0)
        md.moe_grouped_ffn(layer.xs, layer.offsets_P, layer.wgu, layer.wd, ys_tc, layer.ws_ffn,
                           d_status=layer.status)
        torch.cuda.synchronize()
    hot = cold = 0
    for s in range(P):
        a, b = int(offs[s]), int(offs[s + 1])
        if b == a:
            continue
        if counts[s] >= hot_rows:
            hot += 1
            assert torch.equal(_bits(ys_split[a:b]), _bits(ys_pair[a:b])), f"hot slot {s}"
        else:
            cold += 1
            if ys_tc is not None:
                assert torch.equal(_bits(ys_split[a:b]), _bits(ys_tc[a:b])), f"cold slot {s}"
    assert torch.equal(_bits(ys_split[:n]), _bits(layer.ys[:n]))   # the layer's own step
    return hot, cold


def _skewed_spec():
    # 32 experts with a steep Zipf popularity: six slots above 192 rows (up to ~1200),
    # the rest below, and 150 sorted rows per slot on average, so moe_grouped_ffn
    # alone takes the single-SM kernel (the cold slots' reference)
    return synth.LayerSpec("skewed", [700, 0, 500], 0, H=512, E=32, k=4, I=256, dtype="bf16",
                           w_std=0.05, zipf_s=1.6)


def test_split_small_skewed_layer(md, orc):
    from test_gpu_parity import _check_layer
    spec = _skewed_spec()
    hot_rows, hot_sms = 192, 32
    x_loc = synth.hidden_states(spec, DEV)
    lg_loc = synth.router_logits(spec, DEV)
    wgu, wd = synth.expert_weights(spec, None, DEV)
    offs, rows = md.moe_dp_layout(spec.counts, spec.mode)
    layer = md.MoeLayer(R=spec.R, H=spec.H, E=spec.E, k=spec.k, I=spec.I, w_gate_up=wgu,
                        w_down=wd, max_rows=rows, mode=spec.mode, keep_global=True,
                        ffn_split=(hot_rows, hot_sms))
    out = [torch.empty(c, spec.H, device=DEV, dtype=torch.bfloat16) for c in spec.counts]
    layer.forward(x_loc, lg_loc, out, counts=spec.counts)
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    hot, cold = _split_parts_exact(md, layer, hot_rows, hot_sms)
    assert hot >= 4 and cold >= 10, (hot, cold)
    _check_layer(md, orc, spec, layer, out, x_loc, lg_loc, wgu, wd, offs, rows)
    graph_replay_matches_eager(layer, x_loc, lg_loc, out)


def test_split_one_stream_equals_two(md):
    """stream_hot None: the two parts run one after the other on one stream, same bits."""
    spec = _skewed_spec()
    x_loc = synth.hidden_states(spec, DEV)
    lg_loc = synth.router_logits(spec, DEV)
    wgu, wd = synth.expert_weights(spec, None, DEV)
    offs, rows = md.moe_dp_layout(spec.counts, spec.mode)
    layer = md.MoeLayer(R=spec.R, H=spec.H, E=spec.E, k=spec.k, I=spec.I, w_gate_up=wgu,
                        w_down=wd, max_rows=rows, mode=spec.mode, ffn_split=(192, 40))
    out = [torch.empty(c, spec.H, device=DEV, dtype=torch.bfloat16) for c in spec.counts]
    layer.forward(x_loc, lg_loc, out, counts=spec.counts)
    ys1 = torch.full_like(layer.ys, 6.0)
    md.moe_grouped_ffn_split(layer.xs, layer.offsets_P, wgu, wd, ys1, layer.ws_ffn, 192, 40,
                             None, d_status=layer.status)
    torch.cuda.synchronize()
    n = int(layer.offsets_P[-1].item())
    assert int(layer.status.item()) == 0
    assert torch.equal(_bits(ys1[:n]), _bits(layer.ys[:n]))


def test_split_eplb_full_size(md, orc):
    """The EPLB workload (288 slots, a dozen with 500-1000 rows) with the split the
    benchmark runs: parts exact against each kernel alone, layer against the oracle."""
    from test_gpu_parity import _check_layer
    spec = synth.spec_eplb()
    l2p_np, nrep_np, p2l = synth.make_map(spec)
    x_loc = synth.hidden_states(spec, DEV)
    lg_loc = synth.router_logits(spec, DEV)
    wgu, wd = synth.expert_weights(spec, p2l, DEV)
    offs, rows = md.moe_dp_layout(spec.counts, spec.mode)
    layer = md.MoeLayer(R=spec.R, H=spec.H, E=spec.E, k=spec.k, I=spec.I, w_gate_up=wgu,
                        w_down=wd, max_rows=rows, mode=spec.mode, keep_global=True,
                        l2p=torch.from_numpy(l2p_np).to(DEV),
                        nrep=torch.from_numpy(nrep_np).to(DEV), ffn_split=(192, 48))
    out = [torch.empty(c, spec.H, device=DEV, dtype=torch.bfloat16) for c in spec.counts]
    layer.forward(x_loc, lg_loc, out, counts=spec.counts)
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    hot, cold = _split_parts_exact(md, layer, 192, 48)
    assert hot >= 4 and cold >= 50, (hot, cold)
    _check_layer(md, orc, spec, layer, out, x_loc, lg_loc, wgu, wd, offs, rows, sample=6,
                 l2p=l2p_np, nrep=nrep_np)
    graph_replay_matches_eager(layer, x_loc, lg_loc, out)
