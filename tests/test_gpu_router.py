"""GPU parity of the router gate GEMM fused ahead of top-k.

The logits are checked against the oracle's fp64 gate projection; the selection
against the oracle's top-k run on the GPU's own fp32 logits (the decision taken in
the same precision on both sides, so ids are bit-exact); and where the fp64 top-k
picks a different set, the swapped experts must be a near-tie in fp64."""
import gc

import numpy as np
import pytest
import torch

from gpu_util import W_ATOL, W_RTOL, as_f32, assert_close, to_np

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


@pytest.mark.parametrize("counts,mode,H,E,k,renorm,n_shared,bias", [
    ([8192], 0, 7168, 256, 8, 1, 0, False),             # fused: 64 row tiles
    ([8192], 0, 7168, 256, 8, 1, 0, True),              # fused, Zipf-like expert bias
    ([55, 0, 33, 17, 20, 2, 4, 1], 1, 7168, 256, 8, 1, 0, True),   # MAX padding, split K
    ([100, 200], 0, 512, 64, 10, 0, 1, False),          # k > 8: split, full softmax, shared
    ([5000], 0, 1024, 128, 4, 0, 0, False),             # fused, full softmax
    ([1], 0, 256, 32, 1, 1, 0, False)])
def test_route_gemm_topk(md, orc, counts, mode, H, E, k, renorm, n_shared, bias):
    offs, rows = md.moe_dp_layout(counts, mode)
    g = torch.Generator(device=DEV).manual_seed(rows + H + E)
    x = torch.randn(rows, H, generator=g, device=DEV).to(torch.bfloat16)
    wr = (torch.randn(E, H, generator=g, device=DEV) / H ** 0.5).to(torch.bfloat16)
    b = (-1.1 * torch.log(torch.randperm(E, generator=g, device=DEV).float() + 1.0)
         if bias else None)
    d_counts = torch.tensor(counts, dtype=torch.int32, device=DEV)
    d_offs = torch.tensor(offs, dtype=torch.int32, device=DEV)
    kk = k + n_shared
    ids = torch.full((rows, kk), -7, dtype=torch.int32, device=DEV)
    w = torch.full((rows, kk), 9.0, dtype=torch.float32, device=DEV)
    logits = torch.empty(rows, E, dtype=torch.float32, device=DEV)
    ws = torch.empty(max(md.moe_route_gemm_ws_bytes(rows, H, E, k), 16), dtype=torch.uint8,
                     device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    md.moe_route_gemm_topk(x, wr, k, bool(renorm), d_counts, d_offs, ids, w, ws, logits, st,
                           n_shared=n_shared, bias=b)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    valid = orc.valid_rows(counts, np.array(offs), rows)
    ref = orc.router_logits(as_f32(to_np(x)), as_f32(to_np(wr)), None if b is None else to_np(b))
    got_l = to_np(logits)
    # fp32 sums of H bf16 products (logits ~ N(0, 1)): each addition rounds by about
    # 2^-24 x |partial sum| (~1e-7 here), ~1e-5 over 7168 terms as a random walk and
    # ~1e-3 in the linear worst case; 2e-4 sits between, with the observed max 4.4e-5
    assert_close(got_l, ref, 2e-4, 1e-5, "router logits")
    # the selection on the GPU's own logits is exact
    ids_o, w_o = orc.route_topk(got_l, k, bool(renorm), valid, n_shared)
    assert np.array_equal(to_np(ids), ids_o)
    assert_close(to_np(w), w_o, W_ATOL, W_RTOL, "route weights")
    # against the fp64 logits: the same set except at near-ties
    ids_64, _ = orc.route_topk(ref.astype(np.float32), k, bool(renorm), valid, n_shared)
    for r in np.nonzero(valid)[0]:
        a, b = set(to_np(ids)[r, :k].tolist()), set(ids_64[r, :k].tolist())
        if a != b:
            kth = np.sort(ref[r])[::-1]
            assert kth[k - 1] - kth[k] < 5e-4, (r, a ^ b)   # twice the logit tolerance


def test_layer_with_router_gate(md, orc):
    """MoeLayer(router_weight=...): the gathered rows go through the gate GEMM (with
    the Zipf bias) instead of given logits; routing and the layer output match the
    oracle (selection up to fp64 near-ties, output on rows with the oracle's set)."""
    from combine_dp_gather_gb300 import synth
    spec = synth.LayerSpec("tiny_gate", [16, 0, 140, 8, 1], 1, H=512, E=32, k=4, I=256,
                           dtype="bf16", w_std=0.05, zipf_s=1.1)
    x_loc = synth.hidden_states(spec, DEV)
    lg_loc = synth.router_logits(spec, DEV)          # ignored by the gate path
    wgu, wd = synth.expert_weights(spec, None, DEV)
    gw, gb = synth.router_gate(spec, DEV)
    offs, rows = md.moe_dp_layout(spec.counts, spec.mode)
    layer = md.MoeLayer(R=spec.R, H=spec.H, E=spec.E, k=spec.k, I=spec.I, w_gate_up=wgu,
                        w_down=wd, max_rows=rows, mode=spec.mode, router_weight=gw,
                        router_bias=gb, keep_global=True)
    out = [torch.empty(c, spec.H, device=DEV, dtype=torch.bfloat16) for c in spec.counts]
    layer.forward(x_loc, lg_loc, out, counts=spec.counts)
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    offs_o, rows_o = orc.dp_layout(spec.counts, spec.mode, 0, 1)
    valid = orc.valid_rows(spec.counts, offs_o, rows_o)
    xg_o = orc.dp_gather([to_np(t) for t in x_loc], spec.counts, offs_o, rows_o)
    assert np.array_equal(to_np(layer.xg[:rows]), xg_o)
    lg64 = orc.router_logits(as_f32(xg_o), as_f32(to_np(gw)), to_np(gb))
    ids_o, w_o = orc.route_topk(lg64.astype(np.float32), spec.k, True, valid)
    ids_g, w_g = to_np(layer.ids[:rows]), to_np(layer.w[:rows])
    same = np.array([set(ids_g[r]) == set(ids_o[r]) for r in range(rows)])
    for r in np.nonzero(valid & ~same)[0]:
        kth = np.sort(lg64[r])[::-1]
        assert kth[spec.k - 1] - kth[spec.k] < 5e-4, r
    assert same[valid == 1].mean() > 0.95
    assert np.array_equal(ids_g[same], ids_o[same])
    assert_close(w_g[same], w_o[same], 1e-5, 1e-4, "gate route weights")
    # layer output on the rows routed as the oracle routes them
    x_f = as_f32(xg_o)
    yg = as_f32(to_np(layer.yg[:rows]))
    for r in np.nonzero(valid & same)[0][::7]:
        ref = np.zeros(spec.H)
        for j in range(spec.k):
            e = int(ids_o[r, j])
            y = orc.expert_ffn(x_f[r:r + 1], as_f32(to_np(wgu[e])), as_f32(to_np(wd[e])))[0]
            ref += w_o[r, j] * y
        assert_close(yg[r], ref, 2e-2, 1e-2, f"gate layer row {r}")


@pytest.mark.parametrize("fp8", [False, True])
def test_layer_all_options_together(md, fp8):
    """The fused boundary (residual add + RMSNorm), the router gate GEMM with its bias
    and (optionally) the FP8 experts in one layer: the step equals, bit for bit, a
    layer with the gate GEMM (and FP8) fed the rows the fused boundary normed; the
    residual holds the exact sum; a graph replay repeats the step."""
    from combine_dp_gather_gb300 import synth
    spec = synth.LayerSpec("all_opts", [16, 0, 140, 8, 1], 1, H=512, E=32, k=4, I=256,
                           dtype="bf16", w_std=0.05, zipf_s=1.1)
    x_loc = synth.hidden_states(spec, DEV)
    lg_loc = synth.router_logits(spec, DEV)          # ignored by the gate path
    wgu, wd = synth.expert_weights(spec, None, DEV)
    gw, gb = synth.router_gate(spec, DEV)
    g = torch.Generator(device=DEV).manual_seed(5)
    res = [torch.randn(c, spec.H, generator=g, device=DEV).to(torch.bfloat16)
           for c in spec.counts]
    res0 = [t.clone() for t in res]
    gamma = (1 + 0.1 * torch.randn(spec.H, generator=g, device=DEV)).to(torch.bfloat16)
    offs, rows = md.moe_dp_layout(spec.counts, spec.mode)
    common = dict(R=spec.R, H=spec.H, E=spec.E, k=spec.k, I=spec.I, w_gate_up=wgu, w_down=wd,
                  max_rows=rows, mode=spec.mode, router_weight=gw, router_bias=gb, fp8=fp8)
    layer = md.MoeLayer(norm_gamma=gamma, norm_eps=1e-6, **common)
    out = [torch.empty(c, spec.H, device=DEV, dtype=torch.bfloat16) for c in spec.counts]
    layer.forward(x_loc, lg_loc, out, counts=spec.counts, local_residual=res)
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    for a, b, h in zip(res, res0, x_loc):
        assert torch.equal(a, (b.float() + h.float()).to(torch.bfloat16))
    normed = [layer.xg[offs[r]: offs[r] + c].clone() for r, c in enumerate(spec.counts)]
    plain = md.MoeLayer(**common)
    out2 = [torch.full_like(t, 7.0) for t in out]
    plain.forward(normed, lg_loc, out2, counts=spec.counts)
    torch.cuda.synchronize()
    assert int(plain.status.item()) == 0
    for a, b in zip(out2, out):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    for t, t0 in zip(res, res0):
        t.copy_(t0)
    graph = layer.capture(x_loc, lg_loc, out, local_residual=res)
    for t, t0 in zip(res, res0):      # the capture's warm-up ran the step once
        t.copy_(t0)
    first = [t.clone() for t in out]
    for t in out:
        t.fill_(7.0)
    graph.replay()
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    for a, b in zip(first, out):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
