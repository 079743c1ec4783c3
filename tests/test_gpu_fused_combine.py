"""GPU tests of moe_grouped_ffn_combine: the grouped FFN with the combine and
DP scatter, in the down projection's epilogue on the tokens-as-M kernel (few
rows per slot) and as its own launch after the pair kernel (many rows per
slot).

The call must give, bit for bit, what the grouped FFN followed by
moe_combine_scatter gives (the same float32 sum in j order, one rounding),
whichever MM2 unit ends up owning a token's tile; the separate path is itself
checked against the oracle in test_gpu_parity.py, and the last test here checks
the fused call's replica rows against the oracle's combine directly.  The
arrival counters must be back at zero after every call."""
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


def _layers(md, spec, keep_global=True):
    x_loc = synth.hidden_states(spec, DEV)
    lg_loc = synth.router_logits(spec, DEV)
    wgu, wd = synth.expert_weights(spec, None, DEV)
    offs, rows = md.moe_dp_layout(spec.counts, spec.mode, spec.static_bound, spec.tokens_per_req)
    common = dict(R=spec.R, H=spec.H, E=spec.E, k=spec.k, I=spec.I, w_gate_up=wgu, w_down=wd,
                  max_rows=max(rows, 1), mode=spec.mode, static_bound=spec.static_bound,
                  tokens_per_req=spec.tokens_per_req, renormalize=spec.renormalize,
                  align=spec.align, n_shared=spec.n_shared, keep_global=keep_global)
    fused = md.MoeLayer(fused_combine=True, **common)
    sep = md.MoeLayer(fused_combine=False, **common)
    return fused, sep, x_loc, lg_loc, rows


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t


def _counters(md, layer):
    h = (layer.cap * layer.I * layer.wgu.element_size() + 255) // 256 * 256
    return layer.ws_ffn[h:].view(torch.int32)     # rows x H/256 arrival counters


def _run_both(md, spec, keep_global=True, repeats=2):
    fused, sep, x_loc, lg_loc, rows = _layers(md, spec, keep_global)
    out_s = [torch.full((c, spec.H), 7.0, device=DEV, dtype=torch.bfloat16) for c in spec.counts]
    sep.forward(x_loc, lg_loc, out_s, counts=spec.counts)
    for _ in range(repeats):              # the second call starts from the counters the first left
        out_f = [torch.full_like(t, 9.0) for t in out_s]
        if keep_global:
            fused.yg.fill_(5.0)           # pad rows must come back zero
        fused.forward(x_loc, lg_loc, out_f, counts=spec.counts)
        torch.cuda.synchronize()
        assert int(fused.status.item()) == 0 and int(sep.status.item()) == 0
        for a, b in zip(out_f, out_s):
            assert torch.equal(_bits(a), _bits(b))
        if keep_global:
            assert torch.equal(_bits(fused.yg[:rows]), _bits(sep.yg[:rows]))
        n = int(sep.offsets_P[-1].item())
        assert torch.equal(_bits(fused.ys[:n]), _bits(sep.ys[:n]))
        assert not _counters(md, fused).any(), "arrival counters left non-zero"
    return fused, sep, x_loc, lg_loc, out_f


@pytest.mark.parametrize("kernel,counts,mode,H,E,k,I,align,shared", [
    ("tc", [16, 0, 140, 8, 1], 1, 512, 16, 4, 256, 1, 0),        # tokens as M
    ("tc", [300, 0, 77], 0, 512, 32, 8, 256, 16, 0),             # alignment pad rows
    ("tc", [16, 0, 140, 8, 1], 0, 512, 16, 4, 256, 1, 1),        # shared expert slot
    ("pair", [2048], 0, 512, 8, 2, 256, 1, 0),                   # weights as M, SM pairs
    ("pair", [700, 0, 913, 5], 0, 768, 8, 3, 256, 1, 0),         # >320 tokens per slot
    ("pair", [300, 0, 77], 1, 512, 32, 8, 256, 128, 0),          # alignment pad rows
])
def test_fused_combine_equals_separate_bitexact(md, kernel, counts, mode, H, E, k, I, align,
                                                shared):
    spec = synth.LayerSpec("fused", counts, mode, H=H, E=E, k=k, I=I, dtype="bf16",
                           w_std=0.05, zipf_s=1.1, align=align, n_shared=shared)
    fused, sep = _run_both(md, spec)[:2]
    # which grouped-FFN kernel ran (>= 192 sorted rows per slot: the pair kernel, whose
    # combine is its own launch; else the tokens-as-M kernel's epilogue combined)
    assert ("pair" if fused.cap // fused.P >= 192 else "tc") == kernel


def test_fused_combine_without_global_buffer(md):
    spec = synth.LayerSpec("lean", [33, 0, 250, 7], 1, H=512, E=16, k=4, I=256, dtype="bf16",
                           w_std=0.05)
    _run_both(md, spec, keep_global=False)


def test_fused_combine_dsv3_decode_and_graph(md):
    spec = synth.spec_decode(seed=0)
    fused, sep, x_loc, lg_loc, out_f = _run_both(md, spec, repeats=1)
    graph_replay_matches_eager(fused, x_loc, lg_loc, out_f)
    assert not _counters(md, fused).any()


def test_fused_combine_dsv3_prefill_and_graph(md):
    spec = synth.spec_prefill()
    fused, sep, x_loc, lg_loc, out_f = _run_both(md, spec, repeats=1)
    assert fused.cap // fused.P >= 192          # the pair kernel, then the combine launch
    graph_replay_matches_eager(fused, x_loc, lg_loc, out_f)
    assert not _counters(md, fused).any()


def test_fused_combine_stale_counter_flagged(md):
    """A workspace whose counters were not zeroed: the arrival that finds its counter
    above the token's target sets MOE_DEV_BAD_WORKSPACE (no wait, no fault); with the
    counters zeroed again the next call is exact."""
    spec = synth.LayerSpec("stale", [40, 0, 90], 1, H=512, E=16, k=4, I=256, dtype="bf16",
                           w_std=0.05)
    fused, sep, x_loc, lg_loc, rows = _layers(md, spec)
    out_s = [torch.empty(c, spec.H, device=DEV, dtype=torch.bfloat16) for c in spec.counts]
    sep.forward(x_loc, lg_loc, out_s, counts=spec.counts)
    cnt = _counters(md, fused)
    cnt[::7] = 1000                      # planted on the host side of the contract
    out_f = [torch.empty_like(t) for t in out_s]
    fused.forward(x_loc, lg_loc, out_f, counts=spec.counts)
    torch.cuda.synchronize()
    assert int(fused.status.item()) & md.MOE_DEV_BAD_WORKSPACE
    cnt.zero_()
    fused.status.zero_()
    fused.forward(x_loc, lg_loc, out_f, counts=spec.counts)
    torch.cuda.synchronize()
    assert int(fused.status.item()) == 0
    for a, b in zip(out_f, out_s):
        assert torch.equal(_bits(a), _bits(b))
    assert not cnt.any()


def test_fused_combine_call_matches_oracle_combine(md, orc):
    """Through the C ABI directly (no MoeLayer): dispatch, then the fused call, then
    the replica rows against the oracle's combine of the GPU's own expert rows."""
    from gpu_util import as_f32, to_np
    spec = synth.LayerSpec("direct", [120, 0, 64], 1, H=512, E=8, k=2, I=256, dtype="bf16",
                           w_std=0.05)
    fused, sep, x_loc, lg_loc, rows = _layers(md, spec, keep_global=True)
    out = [torch.empty(c, spec.H, device=DEV, dtype=torch.bfloat16) for c in spec.counts]
    fused.forward(x_loc, lg_loc, out, counts=spec.counts)
    torch.cuda.synchronize()
    assert int(fused.status.item()) == 0
    ys = as_f32(to_np(fused.ys)).astype(np.float64)
    yg_o = orc.combine(ys, to_np(fused.inv[:rows]), to_np(fused.w[:rows]).astype(np.float64))
    offs_o, _ = orc.dp_layout(spec.counts, spec.mode, 0, 1)
    loc_o = orc.dp_scatter(yg_o, spec.counts, offs_o)
    for a, b in zip(out, loc_o):
        # one bf16 rounding of the float32 sum against the fp64 sum of the same rows
        np.testing.assert_allclose(as_f32(to_np(a)), b, rtol=8e-3, atol=1e-6)
