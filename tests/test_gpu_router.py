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


@pytest.mark.parametrize("counts,mode,H,E,k,renorm,n_shared", [
    ([8192], 0, 7168, 256, 8, 1, 0),             # fused: 64 row tiles
    ([55, 0, 33, 17, 20, 2, 4, 1], 1, 7168, 256, 8, 1, 0),   # MAX padding, split K
    ([100, 200], 0, 512, 64, 10, 0, 1),          # k > 8: split path, full softmax, shared
    ([5000], 0, 1024, 128, 4, 0, 0),             # fused, full softmax
    ([1], 0, 256, 32, 1, 1, 0)])
def test_route_gemm_topk(md, orc, counts, mode, H, E, k, renorm, n_shared):
    offs, rows = md.moe_dp_layout(counts, mode)
    g = torch.Generator(device=DEV).manual_seed(rows + H + E)
    x = torch.randn(rows, H, generator=g, device=DEV).to(torch.bfloat16)
    wr = (torch.randn(E, H, generator=g, device=DEV) / H ** 0.5).to(torch.bfloat16)
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
                           n_shared=n_shared)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    valid = orc.valid_rows(counts, np.array(offs), rows)
    ref = orc.router_logits(as_f32(to_np(x)), as_f32(to_np(wr)))
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
