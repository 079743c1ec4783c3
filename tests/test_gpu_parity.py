"""GPU parity: every step of the CUDA path against the CPU oracle, called through
the C ABI (ctypes binding), on seeded inputs.

Integer work (layouts, ids, counts, offsets, permutations, inverse maps) and
row copies must match bit for bit; float outputs must lie within the stated
tolerances (bf16: |gpu - oracle| <= 2e-2 + 1e-2 |oracle|).  Small cases span
several tiles and ragged tails and are compared element by element; the
full-size workloads are compared in full on everything integer or copied and
on sampled tokens for the expert FFN and combine."""
import gc

import numpy as np
import pytest
import torch

import oracle as orc_mod
from combine_dp_gather_gb300 import synth
from gpu_util import (BF16_ATOL, BF16_RTOL, F32_ATOL, F32_RTOL, W_ATOL, W_RTOL, as_f32,
                      assert_close, graph_replay_matches_eager, pairs_to_check, rel_fro,
                      to_np)

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


def dev_i32(values):
    return torch.tensor(list(values), dtype=torch.int32, device=DEV)


def status_of(st):
    torch.cuda.synchronize()
    return int(st.item())


# ------------------------------------------------------------------ gather / scatter
@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_gather_scatter_bitexact(md, orc, mode, dtype):
    rng = np.random.default_rng(mode + (10 if dtype == torch.float32 else 0))
    R, B, tpr = 16, 24, 2
    counts = [int(v) for v in rng.choice([0, 1, 4, 8, 24, 33, 48], size=R)]
    counts[3] = 0
    H = 7168 if dtype == torch.bfloat16 else 256
    g = torch.Generator(device=DEV).manual_seed(5)
    local = [torch.randn(c, H, generator=g, device=DEV).to(dtype) for c in counts]
    offs, rows = md.moe_dp_layout(counts, mode, B, tpr)
    offs_o, rows_o = orc.dp_layout(counts, mode, B, tpr)
    assert offs == offs_o.tolist() and rows == rows_o
    d_c, d_o = dev_i32(counts), dev_i32(offs)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.full((rows, H), 3.0, device=DEV, dtype=dtype)   # pad rows must be zeroed
    md.moe_dp_gather(local, d_c, d_o, out, st)
    back = [torch.full_like(t, 5.0) for t in local]
    md.moe_dp_scatter(out, d_c, d_o, back, st)
    assert status_of(st) == 0
    ref = orc.dp_gather([to_np(t) for t in local], counts, offs_o, rows_o)
    assert np.array_equal(to_np(out), ref)
    for a, b in zip(local, back):
        assert torch.equal(a.view(torch.int16) if dtype == torch.bfloat16 else a,
                           b.view(torch.int16) if dtype == torch.bfloat16 else b)


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_gather2_bitexact(md, orc, mode):
    """Hidden states (bf16) and router logits (fp32) of the same replicas in one
    launch: each output is the oracle's gather, bit for bit."""
    rng = np.random.default_rng(30 + mode)
    R, B, tpr, H, E = 12, 24, 1, 7168, 256
    counts = [int(v) for v in rng.choice([0, 1, 5, 17, 24], size=R)]
    counts[0] = 0
    g = torch.Generator(device=DEV).manual_seed(31)
    xs = [torch.randn(c, H, generator=g, device=DEV).to(torch.bfloat16) for c in counts]
    ls = [torch.randn(c, E, generator=g, device=DEV) for c in counts]
    offs, rows = md.moe_dp_layout(counts, mode, B, tpr)
    offs_o, rows_o = orc.dp_layout(counts, mode, B, tpr)
    d_c, d_o = dev_i32(counts), dev_i32(offs)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    xg = torch.full((rows, H), 3.0, device=DEV, dtype=torch.bfloat16)
    lg = torch.full((rows, E), 3.0, device=DEV)
    md.moe_dp_gather2(xs, ls, d_c, d_o, xg, lg, st)
    assert status_of(st) == 0
    assert np.array_equal(to_np(xg), orc.dp_gather([to_np(t) for t in xs], counts, offs_o, rows_o))
    assert np.array_equal(to_np(lg), orc.dp_gather([to_np(t) for t in ls], counts, offs_o, rows_o))


def test_gather_all_idle_and_bad_counts(md):
    counts = [0, 0, 0]
    offs, rows = md.moe_dp_layout(counts, 1)
    assert rows == 0
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.empty(0, 64, device=DEV, dtype=torch.bfloat16)
    md.moe_dp_gather([out[:0]] * 3, dev_i32(counts), dev_i32(offs), out, st)  # no launch
    # device counts larger than their segment: flagged, copies clipped, no fault
    local = [torch.ones(10, 64, device=DEV, dtype=torch.bfloat16) for _ in range(2)]
    d_c = dev_i32([10, 10])
    d_o = dev_i32([0, 4, 8])
    g = torch.full((8, 64), 7.0, device=DEV, dtype=torch.bfloat16)
    md.moe_dp_gather(local, d_c, d_o, g, st)
    assert status_of(st) & md.MOE_DEV_BAD_COUNTS
    assert torch.equal(g.float(), torch.ones(8, 64, device=DEV))


def test_fused_gather_and_combine_scatter_bad_counts_flag_without_fault(md):
    """Device counts larger than their segment: both fused kernels set
    MOE_DEV_BAD_COUNTS, copy or write only the rows that fit, and touch nothing
    outside the buffers."""
    local = [torch.ones(10, 64, device=DEV, dtype=torch.bfloat16) for _ in range(2)]
    lgl = [torch.full((10, 32), 2.0, device=DEV) for _ in range(2)]
    d_c, d_o = dev_i32([10, 10]), dev_i32([0, 4, 8])
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    xg = torch.full((8, 64), 7.0, device=DEV, dtype=torch.bfloat16)
    lg = torch.full((8, 32), 7.0, device=DEV)
    md.moe_dp_gather2(local, lgl, d_c, d_o, xg, lg, st)
    assert status_of(st) & md.MOE_DEV_BAD_COUNTS
    assert torch.equal(xg.float(), torch.ones(8, 64, device=DEV))
    assert torch.equal(lg, torch.full((8, 32), 2.0, device=DEV))
    # combine + scatter into replicas whose counts overflow their segments
    ys = torch.ones(16, 64, device=DEV, dtype=torch.bfloat16)
    inv = torch.arange(16, dtype=torch.int32, device=DEV).view(8, 2)
    w = torch.full((8, 2), 0.5, device=DEV)
    outs = [torch.full((10, 64), 3.0, device=DEV, dtype=torch.bfloat16) for _ in range(2)]
    st.zero_()
    md.moe_combine_scatter(ys, inv, w, d_c, d_o, outs, None, st)
    assert status_of(st) & md.MOE_DEV_BAD_COUNTS
    for o in outs:                      # the 4 rows of each segment, the rest untouched
        assert torch.equal(o[:4].float(), torch.ones(4, 64, device=DEV))
        assert torch.equal(o[4:].float(), torch.full((6, 64), 3.0, device=DEV))


@pytest.mark.parametrize("dtype,H,mode,E,route", [(torch.bfloat16, 7168, 1, 0, False),
                                                  (torch.bfloat16, 7168, 1, 256, False),
                                                  (torch.bfloat16, 7168, 1, 256, True),
                                                  (torch.bfloat16, 512, 0, 0, False),
                                                  (torch.float32, 1024, 2, 36, True)])
def test_gather_add_rmsnorm(md, orc, dtype, H, mode, E, route):
    """E > 0: the router logits [count, E] float32 ride in the same launch and must
    equal the plain gather's output bit for bit (zero pad rows); with route the rows
    are also routed (top-6 of E, one shared expert) as the oracle routes them."""
    counts = [5, 0, 33, 1, 17]
    offs, rows = md.moe_dp_layout(counts, mode, 40, 1)
    g = torch.Generator(device=DEV).manual_seed(H + mode)
    hid = [torch.randn(c, H, generator=g, device=DEV).to(dtype) for c in counts]
    res = [torch.randn(c, H, generator=g, device=DEV).to(dtype) for c in counts]
    gamma = (1 + 0.1 * torch.randn(H, generator=g, device=DEV)).to(dtype)
    res0 = [t.clone() for t in res]
    out = torch.full((rows, H), 3.0, device=DEV, dtype=dtype)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    if E:
        lg = [torch.randn(c, E, generator=g, device=DEV) for c in counts]
        lg_out = torch.full((rows, E), 3.0, device=DEV)
        if route:
            ids = torch.full((rows, 7), -7, dtype=torch.int32, device=DEV)
            w = torch.full((rows, 7), 9.0, device=DEV)
            md.moe_dp_gather_add_rmsnorm_route(hid, res, gamma, 1e-6, lg, dev_i32(counts),
                                               dev_i32(offs), out, 6, True, ids, w, lg_out, 1,
                                               st)
        else:
            md.moe_dp_gather_add_rmsnorm(hid, res, gamma, 1e-6, dev_i32(counts), dev_i32(offs),
                                         out, st, local_b=lg, out_b=lg_out)
        lg_o = orc.dp_gather([to_np(t) for t in lg], counts, np.array(offs, np.int32), rows)
        assert np.array_equal(to_np(lg_out), lg_o)
        if route:
            valid_r = orc.valid_rows(counts, np.array(offs, np.int32), rows)
            ids_o, w_o = orc.route_topk(lg_o, 6, True, valid_r, 1)
            assert np.array_equal(to_np(ids), ids_o)
            assert_close(to_np(w), w_o, W_ATOL, W_RTOL, "route weights")
    else:
        md.moe_dp_gather_add_rmsnorm(hid, res, gamma, 1e-6, dev_i32(counts), dev_i32(offs), out,
                                     st)
    assert status_of(st) == 0
    bf = dtype == torch.bfloat16
    f32 = lambda t: as_f32(to_np(t))
    y = np.zeros((rows, H))
    for r, c in enumerate(counts):
        r_new, y_r = orc.add_rmsnorm(f32(hid[r]), f32(res0[r]), f32(gamma), 1e-6, bf)
        assert np.array_equal(f32(res[r]), r_new)                   # stored residual: exact
        y[offs[r]: offs[r] + c] = y_r
    valid = orc.valid_rows(counts, np.array(offs, np.int32), rows)
    got = f32(out).astype(np.float64)
    tol = (1e-6, 8e-3) if bf else (1e-6, 1e-5)   # one bf16 rounding (<= 1 ulp apart)
    assert_close(got[valid == 1], y[valid == 1], *tol, what="normed rows")
    assert not got[valid == 0].any()


# ------------------------------------------------------------------ routing
@pytest.mark.parametrize("E,k", [(8, 2), (256, 8), (300, 6), (64, 1), (32, 32), (1024, 4)])
@pytest.mark.parametrize("renorm", [True, False])
def test_route_topk(md, orc, E, k, renorm):
    counts = [37, 0, 100, 5]
    offs, rows = md.moe_dp_layout(counts, 1)             # MAX: pad rows inside segments
    g = torch.Generator(device=DEV).manual_seed(E * 7 + k)
    logits = torch.randn(rows, E, generator=g, device=DEV)
    logits[::3] = torch.round(logits[::3] * 2) / 2       # many exact ties
    ids = torch.empty(rows, k, dtype=torch.int32, device=DEV)
    w = torch.empty(rows, k, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    md.moe_route_topk(logits, k, renorm, dev_i32(counts), dev_i32(offs), ids, w, st)
    assert status_of(st) == 0
    valid = orc.valid_rows(counts, np.array(offs, np.int32), rows)
    ids_o, w_o = orc.route_topk(to_np(logits), k, renorm, valid)
    assert np.array_equal(to_np(ids), ids_o)
    assert_close(to_np(w), w_o, W_ATOL, W_RTOL, "route weights")


@pytest.mark.parametrize("E,k,n_shared,mode", [(256, 8, 0, 1), (256, 8, 1, 0), (8, 2, 0, 2),
                                                (300, 6, 0, 1), (32, 32, 0, 0), (1024, 4, 2, 1),
                                                (30, 3, 0, 1)])
@pytest.mark.parametrize("renorm", [True, False])
def test_gather_route_bitexact(md, orc, E, k, n_shared, mode, renorm):
    """The gather that routes its rows in the same launch equals moe_dp_gather2 +
    moe_route_topk_shared bit for bit (hidden states, logits when gathered, ids and
    weights), and the oracle's gather and top-k; E = 30 cannot gather its 120-byte
    logit rows and routes without them."""
    rng = np.random.default_rng(E + k + mode)
    R, B, H = 9, 40, 512
    counts = [int(v) for v in rng.choice([0, 1, 7, 33, 40], size=R)]
    counts[1] = 0
    g = torch.Generator(device=DEV).manual_seed(E * 3 + k)
    xs = [torch.randn(c, H, generator=g, device=DEV).to(torch.bfloat16) for c in counts]
    ls = [torch.randn(c, E, generator=g, device=DEV) for c in counts]
    for t in ls:
        t[::3] = torch.round(t[::3] * 2) / 2               # many exact ties
    offs, rows = md.moe_dp_layout(counts, mode, B, 1)
    offs_o, rows_o = orc.dp_layout(counts, mode, B, 1)
    d_c, d_o = dev_i32(counts), dev_i32(offs)
    kk = k + n_shared
    gather_logits = E * 4 % 16 == 0
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    xg = torch.full((rows, H), 3.0, device=DEV, dtype=torch.bfloat16)
    lg = torch.full((rows, E), 3.0, device=DEV) if gather_logits else None
    ids = torch.full((rows, kk), -7, dtype=torch.int32, device=DEV)
    w = torch.full((rows, kk), 9.0, device=DEV)
    md.moe_dp_gather_route(xs, ls, d_c, d_o, xg, k, renorm, ids, w, lg, n_shared, st)
    assert status_of(st) == 0
    assert np.array_equal(to_np(xg), orc.dp_gather([to_np(t) for t in xs], counts, offs_o, rows_o))
    lg_o = orc.dp_gather([to_np(t) for t in ls], counts, offs_o, rows_o)
    if gather_logits:
        assert np.array_equal(to_np(lg), lg_o)
    valid = orc.valid_rows(counts, offs_o, rows_o)
    ids_o, w_o = orc.route_topk(lg_o, k, renorm, valid, n_shared)
    assert np.array_equal(to_np(ids), ids_o)
    assert_close(to_np(w), w_o, W_ATOL, W_RTOL, "route weights")
    # the same bits as the two separate kernels
    ids2, w2 = torch.empty_like(ids), torch.empty_like(w)
    md.moe_route_topk(torch.from_numpy(lg_o).to(DEV), k, renorm, d_c, d_o, ids2, w2, st,
                      n_shared=n_shared)
    assert status_of(st) == 0
    assert torch.equal(ids, ids2) and torch.equal(w.view(torch.int32), w2.view(torch.int32))


# ------------------------------------------------------------------ dispatch
def _distinct_ids(rows, k, E, seed, pad_every=7):
    g = torch.Generator(device=DEV).manual_seed(seed)
    ids = torch.rand(rows, E, generator=g, device=DEV).argsort(dim=1)[:, :k].to(torch.int32)
    ids[::pad_every] = -1
    return ids.contiguous()


@pytest.mark.parametrize("rows,E,use_map,align", [
    (3001, 64, False, 1), (3001, 64, False, 128), (3001, 64, True, 1), (3001, 64, True, 4),
    (500, 64, False, 1), (500, 64, True, 4), (1900, 256, True, 1), (1024, 256, False, 1),
    (2048, 256, False, 1),
    (8192, 256, False, 1), (9001, 64, True, 4), (2047, 300, False, 1), (2047, 400, False, 1),
    (1, 64, False, 1)])
def test_dispatch_bitexact(md, orc, rows, E, use_map, align):
    """rows x 8 pairs: <= 8192 whose per-warp tables fit 48 KB (E <= ~340) runs the
    one-CTA path (1024 rows is exactly the pair limit); more pairs (1900 rows: 15 chunks
    of 1024 + a ragged tail) or E = 400 run the chunked histogram / scan / rank path
    (four warps per chunk)."""
    k, H = 8, 512
    l2p = nrep = None
    P = E
    if use_map:
        cnt = np.random.default_rng(1).zipf(1.5, size=E).astype(np.int64)
        l2p_np, nrep_np, p2l = synth.eplb_map(cnt, 16, 8)
        P = len(p2l)
        l2p, nrep = torch.from_numpy(l2p_np).to(DEV), torch.from_numpy(nrep_np).to(DEV)
    ids = _distinct_ids(rows, k, E, seed=11 + align)
    x = torch.randn(rows, H, device=DEV).to(torch.bfloat16)
    cap = md.moe_dispatch_cap_bound(rows, k, P, align)
    counts_P = torch.empty(P, dtype=torch.int32, device=DEV)
    offsets_P = torch.empty(P + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(cap, dtype=torch.int32, device=DEV)
    inv = torch.empty(rows, k, dtype=torch.int32, device=DEV)
    xs = torch.full((cap, H), 9.0, device=DEV, dtype=torch.bfloat16)
    ws = torch.empty(md.moe_dispatch_ws_bytes(rows, k, E), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    md.moe_dispatch(x, ids, E, P, counts_P, offsets_P, perm, inv, xs, ws, l2p, nrep, align, st)
    assert status_of(st) == 0
    c_o, o_o, p_o, i_o = orc.dispatch(to_np(ids), E, P, None if l2p is None else to_np(l2p),
                                      None if nrep is None else to_np(nrep), align, cap)
    n = int(o_o[-1])
    assert np.array_equal(to_np(counts_P), c_o)
    assert np.array_equal(to_np(offsets_P), o_o)
    assert np.array_equal(to_np(perm)[:n], p_o[:n])
    assert np.array_equal(to_np(inv), i_o)
    assert np.array_equal(to_np(xs)[:n], orc.permute_rows(to_np(x), p_o[:n]))


def test_dispatch_zero_rows(md):
    E, k, H = 16, 4, 64
    counts_P = torch.full((E,), 7, dtype=torch.int32, device=DEV)
    offsets_P = torch.full((E + 1,), 7, dtype=torch.int32, device=DEV)
    ws = torch.empty(max(md.moe_dispatch_ws_bytes(0, k, E), 16), dtype=torch.uint8, device=DEV)
    empty_i = torch.empty(0, k, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    md.moe_dispatch(None, empty_i, E, E, counts_P, offsets_P, torch.empty(0, dtype=torch.int32,
                    device=DEV), empty_i, None, ws, d_status=st)
    assert status_of(st) == 0
    assert not counts_P.any() and not offsets_P.any()


@pytest.mark.parametrize("E", [16, 400])                 # one-CTA path, chunked path
def test_dispatch_device_errors_flag_without_fault(md, E):
    rows, k, H = 200, 4, 64
    ids = _distinct_ids(rows, k, E, seed=3, pad_every=1000)
    ids[5, 1] = E            # out of range
    ids[9, 0] = -7           # negative, not the pad marker
    x = torch.randn(rows, H, device=DEV).to(torch.bfloat16)
    need = rows * k
    cap = need - 50          # capacity too small
    guard = 64
    perm_buf = torch.full((cap + guard,), -123, dtype=torch.int32, device=DEV)
    xs_buf = torch.full((cap + guard, H), 4.0, device=DEV, dtype=torch.bfloat16)
    counts_P = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets_P = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    inv = torch.empty(rows, k, dtype=torch.int32, device=DEV)
    ws = torch.empty(md.moe_dispatch_ws_bytes(rows, k, E), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    md.moe_dispatch(x, ids, E, E, counts_P, offsets_P, perm_buf[:cap], inv, xs_buf[:cap], ws,
                    d_status=st)
    s = status_of(st)
    assert s & md.MOE_DEV_BAD_EXPERT_ID and s & md.MOE_DEV_CAPACITY
    assert (to_np(perm_buf)[cap:] == -123).all()
    assert (to_np(xs_buf[cap:]).view(np.uint16) == to_np(torch.tensor([4.0]).to(torch.bfloat16))[0]).all()
    assert (to_np(inv) < cap).all()


# ------------------------------------------------------------------ grouped FFN
def _ffn_inputs(counts, H, I, dtype, seed, extra_rows=64, w_std=0.05):
    P = len(counts)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    cap = int(offsets[-1]) + extra_rows
    g = torch.Generator(device=DEV).manual_seed(seed)
    xs = torch.randn(cap, H, generator=g, device=DEV).to(dtype)
    wgu = (torch.randn(P, 2 * I, H, generator=g, device=DEV) * w_std).to(dtype)
    wd = (torch.randn(P, H, I, generator=g, device=DEV) * w_std).to(dtype)
    return offsets, cap, xs, wgu, wd


@pytest.mark.parametrize("counts", [[0, 1, 127, 128, 129, 300, 5, 0], [256] * 4 + [0] * 3 + [17],
                                    [1] * 8, [0] * 7 + [700]])
def test_grouped_ffn_bf16_tcgen05(md, orc, counts):
    H, I = 512, 256
    offsets, cap, xs, wgu, wd = _ffn_inputs(counts, H, I, torch.bfloat16, seed=sum(counts))
    sentinel = 1232.0                                   # exactly representable in bf16
    ys = torch.full((cap, H), sentinel, device=DEV, dtype=torch.bfloat16)
    ws = torch.empty(md.moe_grouped_ffn_ws_bytes(cap, I, torch.bfloat16), dtype=torch.uint8,
                     device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    md.moe_grouped_ffn(xs, dev_i32(offsets), wgu, wd, ys, ws, d_status=st)
    assert status_of(st) == 0
    n = int(offsets[-1])
    ref = orc.grouped_ffn(as_f32(to_np(xs)), offsets, as_f32(to_np(wgu)), as_f32(to_np(wd)))
    got = as_f32(to_np(ys)).astype(np.float64)
    err = assert_close(got[:n], ref[:n], BF16_ATOL, BF16_RTOL, "grouped FFN bf16")
    assert rel_fro(got[:n], ref[:n]) < 8e-3, err
    assert (got[n:] == sentinel).all()                  # rows past the last slot untouched


@pytest.mark.parametrize("counts,lo,hi", [([300, 0, 257, 129, 512, 1], 0, 6),
                                           ([256, 255, 0, 385, 200, 640], 1, 5),
                                           ([1000, 0, 0, 3], 0, 4),
                                           ([15, 33, 255, 321, 641, 240, 48, 272], 0, 8)])
def test_grouped_ffn_bf16_pair_kernel(md, orc, counts, lo, hi):
    """>= 192 rows per slot on average selects the two-SM (cta_group::2) kernel with the
    weights as M and a slot's tokens as N: token groups of up to 320 (one MMA of N <= 256,
    or 256 plus 16..64), ragged widths rounded up to 16, several groups per slot, empty
    slots and slot ranges."""
    H, I = 512, 256
    offsets, cap, xs, wgu, wd = _ffn_inputs(counts, H, I, torch.bfloat16, seed=len(counts) + lo,
                                            extra_rows=40)
    assert cap // len(counts) >= 192
    sentinel = 1232.0
    ys = torch.full((cap, H), sentinel, device=DEV, dtype=torch.bfloat16)
    ws = torch.empty(md.moe_grouped_ffn_ws_bytes(cap, I, torch.bfloat16), dtype=torch.uint8,
                     device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    md.moe_grouped_ffn(xs, dev_i32(offsets), wgu, wd, ys, ws, lo, hi, d_status=st)
    assert status_of(st) == 0
    a, b = int(offsets[lo]), int(offsets[hi])
    ref = orc.grouped_ffn(as_f32(to_np(xs)), offsets, as_f32(to_np(wgu)), as_f32(to_np(wd)),
                          lo, hi)
    got = as_f32(to_np(ys)).astype(np.float64)
    assert_close(got[a:b], ref[a:b], BF16_ATOL, BF16_RTOL, "pair kernel")
    assert rel_fro(got[a:b], ref[a:b]) < 8e-3
    assert (got[:a] == sentinel).all() and (got[b:] == sentinel).all()


def test_grouped_ffn_slot_range_and_dsv3_width(md, orc):
    counts = [40, 0, 130, 7, 256, 1]
    H, I = 7168, 2048
    offsets, cap, xs, wgu, wd = _ffn_inputs(counts, H, I, torch.bfloat16, seed=77, extra_rows=8,
                                            w_std=0.02)
    sentinel = -77.0
    ys = torch.full((cap, H), sentinel, device=DEV, dtype=torch.bfloat16)
    ws = torch.empty(md.moe_grouped_ffn_ws_bytes(cap, I, torch.bfloat16), dtype=torch.uint8,
                     device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    lo, hi = 1, 4
    md.moe_grouped_ffn(xs, dev_i32(offsets), wgu, wd, ys, ws, lo, hi, d_status=st)
    assert status_of(st) == 0
    got = as_f32(to_np(ys)).astype(np.float64)
    a, b = int(offsets[lo]), int(offsets[hi])
    assert (got[:a] == sentinel).all() and (got[b:] == sentinel).all()
    xs_f = as_f32(to_np(xs))
    for s in range(lo, hi):
        r0, r1 = int(offsets[s]), int(offsets[s + 1])
        if r1 == r0:
            continue
        rows = sorted({r0, r1 - 1, (r0 + r1) // 2, min(r0 + 128, r1 - 1)})
        ref = orc.expert_ffn(xs_f[rows], as_f32(to_np(wgu[s])), as_f32(to_np(wd[s])))
        assert_close(got[rows], ref, BF16_ATOL, BF16_RTOL, f"slot {s}")


def test_grouped_ffn_f32(md, orc):
    counts = [16, 0, 40, 8, 33, 1]
    H, I = 256, 128
    offsets, cap, xs, wgu, wd = _ffn_inputs(counts, H, I, torch.float32, seed=5, w_std=0.05)
    ys = torch.full((cap, H), 11.0, device=DEV)
    ws = torch.empty(md.moe_grouped_ffn_ws_bytes(cap, I, torch.float32), dtype=torch.uint8,
                     device=DEV)
    md.moe_grouped_ffn(xs, dev_i32(offsets), wgu, wd, ys, ws)
    torch.cuda.synchronize()
    n = int(offsets[-1])
    ref = orc.grouped_ffn(to_np(xs), offsets, to_np(wgu), to_np(wd))
    assert_close(to_np(ys)[:n], ref[:n], F32_ATOL, F32_RTOL, "grouped FFN f32")
    assert (to_np(ys)[n:] == 11.0).all()


# ------------------------------------------------------------------ combine
def test_combine_identity_experts_bitexact(md, orc):
    rows, k, E, H = 500, 8, 64, 7168
    ids = _distinct_ids(rows, k, E, seed=21, pad_every=9)
    logits = torch.randn(rows, E, device=DEV)
    counts = [rows]
    w = torch.empty(rows, k, device=DEV)
    ids2 = torch.empty_like(ids)
    md.moe_route_topk(logits, k, True, dev_i32(counts), dev_i32([0, rows]), ids2, w)
    ids2[::9] = -1
    w[::9] = 0
    x = torch.randn(rows, H, device=DEV).to(torch.bfloat16)
    cap = md.moe_dispatch_cap_bound(rows, k, E, 1)
    counts_P = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets_P = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(cap, dtype=torch.int32, device=DEV)
    inv = torch.empty(rows, k, dtype=torch.int32, device=DEV)
    xs = torch.empty(cap, H, device=DEV, dtype=torch.bfloat16)
    ws = torch.empty(md.moe_dispatch_ws_bytes(rows, k, E), dtype=torch.uint8, device=DEV)
    md.moe_dispatch(x, ids2, E, E, counts_P, offsets_P, perm, inv, xs, ws)
    out = torch.full((rows, H), 2.0, device=DEV, dtype=torch.bfloat16)
    md.moe_combine(xs, inv, w, out)                      # identity experts: ys = xs
    torch.cuda.synchronize()
    got, xb = to_np(out), to_np(x)
    valid = np.ones(rows, bool)
    valid[::9] = False
    assert np.array_equal(got[valid], xb[valid])
    assert not got[~valid].any()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_combine_random(md, orc, dtype):
    rows, k, H, cap = 300, 6, 1024, 2000
    g = torch.Generator(device=DEV).manual_seed(8)
    ys = torch.randn(cap, H, generator=g, device=DEV).to(dtype)
    inv = torch.stack([torch.randperm(cap, generator=g, device=DEV)[:k] for _ in range(rows)])
    inv = inv.to(torch.int32)
    inv[::5] = -1
    inv[1::7, 2] = -1
    w = torch.rand(rows, k, generator=g, device=DEV)
    out = torch.empty(rows, H, device=DEV, dtype=dtype)
    md.moe_combine(ys, inv, w, out)
    torch.cuda.synchronize()
    ref = orc.combine(as_f32(to_np(ys)).astype(np.float64), to_np(inv), to_np(w).astype(np.float64))
    tol = (4e-3, 4e-3) if dtype == torch.bfloat16 else (1e-5, 1e-5)
    assert_close(as_f32(to_np(out)), ref, *tol, what="combine")


@pytest.mark.parametrize("dtype,mode", [(torch.bfloat16, 1), (torch.bfloat16, 0),
                                        (torch.float32, 2)])
def test_combine_scatter(md, orc, dtype, mode):
    """Combine fused with the DP scatter: the replicas' outputs are bit for bit those
    of moe_combine followed by moe_dp_scatter (and within tolerance of the oracle's
    combine + scatter); the optional global buffer equals moe_combine's."""
    rng = np.random.default_rng(40 + mode)
    counts = [int(v) for v in rng.choice([0, 3, 9, 24], size=10)]
    counts[2] = 0
    offs, rows = md.moe_dp_layout(counts, mode, 24, 1)
    offs_o, rows_o = orc.dp_layout(counts, mode, 24, 1)
    valid = orc.valid_rows(counts, offs_o, rows_o)
    k, H, cap = 6, 1024 if dtype == torch.bfloat16 else 512, 1500
    g = torch.Generator(device=DEV).manual_seed(41)
    ys = torch.randn(cap, H, generator=g, device=DEV).to(dtype)
    inv = torch.stack([torch.randperm(cap, generator=g, device=DEV)[:k] for _ in range(rows)])
    inv = inv.to(torch.int32)
    inv[torch.from_numpy(valid == 0).to(DEV)] = -1          # pad rows are not routed
    w = torch.rand(rows, k, generator=g, device=DEV)
    d_c, d_o = dev_i32(counts), dev_i32(offs)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ref_g = torch.empty(rows, H, device=DEV, dtype=dtype)
    md.moe_combine(ys, inv, w, ref_g, st)
    ref_l = [torch.full((c, H), 5.0, device=DEV, dtype=dtype) for c in counts]
    md.moe_dp_scatter(ref_g, d_c, d_o, ref_l, st)
    for keep in (False, True):
        out = [torch.full((c, H), 7.0, device=DEV, dtype=dtype) for c in counts]
        glob = torch.full((rows, H), 9.0, device=DEV, dtype=dtype) if keep else None
        md.moe_combine_scatter(ys, inv, w, d_c, d_o, out, glob, st)
        assert status_of(st) == 0
        for a, b in zip(out, ref_l):
            assert torch.equal(a.view(torch.int16) if dtype == torch.bfloat16 else a,
                               b.view(torch.int16) if dtype == torch.bfloat16 else b)
        if keep:
            assert torch.equal(glob, ref_g)
    yg_o = orc.combine(as_f32(to_np(ys)).astype(np.float64), to_np(inv),
                       to_np(w).astype(np.float64))
    loc_o = orc.dp_scatter(yg_o, counts, offs_o)
    tol = (4e-3, 4e-3) if dtype == torch.bfloat16 else (1e-5, 1e-5)
    for a, b in zip(out, loc_o):
        assert_close(as_f32(to_np(a)), b, *tol, what="combine_scatter")


# ------------------------------------------------------------------ whole layer
def _layer_gpu(md, spec, l2p_np=None, nrep_np=None, p2l=None, ranges=None):
    x_loc = synth.hidden_states(spec, DEV)
    lg_loc = synth.router_logits(spec, DEV)
    wgu, wd = synth.expert_weights(spec, p2l, DEV)
    offs, rows = md.moe_dp_layout(spec.counts, spec.mode, spec.static_bound, spec.tokens_per_req)
    l2p = None if l2p_np is None else torch.from_numpy(l2p_np).to(DEV)
    nrep = None if nrep_np is None else torch.from_numpy(nrep_np).to(DEV)
    layer = md.MoeLayer(R=spec.R, H=spec.H, E=spec.E, k=spec.k, I=spec.I, w_gate_up=wgu,
                        w_down=wd, max_rows=max(rows, 1), mode=spec.mode,
                        static_bound=spec.static_bound, tokens_per_req=spec.tokens_per_req,
                        renormalize=spec.renormalize, align=spec.align, l2p=l2p, nrep=nrep,
                        n_shared=spec.n_shared, keep_global=True)
    out = [torch.empty(c, spec.H, device=DEV, dtype=wgu.dtype) for c in spec.counts]
    layer.forward(x_loc, lg_loc, out, counts=spec.counts)
    if ranges is not None:          # re-run the FFN as one call per simulated EP rank
        ys_one = layer.ys.clone()
        layer.ys.fill_(0)
        for lo, hi in ranges:
            md.moe_grouped_ffn(layer.xs, layer.offsets_P, wgu, wd, layer.ys, layer.ws_ffn, lo, hi,
                               layer.status)
        torch.cuda.synchronize()
        n = int(layer.offsets_P[-1].item())
        assert torch.equal(layer.ys[:n].view(torch.int16), ys_one[:n].view(torch.int16))
    assert status_of(layer.status) == 0
    return layer, out, x_loc, lg_loc, wgu, wd, offs, rows


def _check_layer(md, orc, spec, layer, out, x_loc, lg_loc, wgu, wd, offs, rows, sample=None,
                 l2p=None, nrep=None, atol=BF16_ATOL, rtol=BF16_RTOL):
    offs_o, rows_o = orc.dp_layout(spec.counts, spec.mode, spec.static_bound, spec.tokens_per_req)
    assert offs == offs_o.tolist() and rows == rows_o
    valid = orc.valid_rows(spec.counts, offs_o, rows_o)
    x_bits = [to_np(t) for t in x_loc]
    xg_o = orc.dp_gather(x_bits, spec.counts, offs_o, rows_o)
    assert np.array_equal(to_np(layer.xg[:rows]), xg_o)
    lg_o = orc.dp_gather([to_np(t) for t in lg_loc], spec.counts, offs_o, rows_o)
    ids_o, w_o = orc.route_topk(lg_o, spec.k, spec.renormalize, valid, spec.n_shared)
    kk = spec.k + spec.n_shared
    assert np.array_equal(to_np(layer.ids[:rows]), ids_o)
    assert_close(to_np(layer.w[:rows]), w_o, W_ATOL, W_RTOL, "route weights")
    P = layer.P
    c_o, o_o, p_o, i_o = orc.dispatch(ids_o, spec.E + spec.n_shared, P, l2p, nrep, spec.align,
                                      layer.cap)
    n = int(o_o[-1])
    assert int(c_o.sum()) == spec.T * kk
    assert n == int(sum((int(c) + spec.align - 1) // spec.align * spec.align for c in c_o))
    assert np.array_equal(to_np(layer.counts_P), c_o)
    assert np.array_equal(to_np(layer.offsets_P), o_o)
    assert np.array_equal(to_np(layer.perm)[:n], p_o[:n])
    assert np.array_equal(to_np(layer.inv[:rows]), i_o)
    assert np.array_equal(to_np(layer.xs[:n]), orc.permute_rows(xg_o, p_o[:n]))
    if spec.align > 1:                                   # alignment rows compute zeros
        pad = np.nonzero(p_o[:n] < 0)[0]
        assert not as_f32(to_np(layer.ys[:n]))[pad].any()
    x_f = as_f32(xg_o)
    real = np.nonzero(valid)[0]
    # every pair of small layers; at full size the kernel's hard rows and a few
    # tokens' combined rows
    check, toks = pairs_to_check(layer, o_o, p_o, i_o, real, kk, sample)
    slot_of = np.searchsorted(o_o, np.arange(n), side="right") - 1
    need = {}
    for g, j in check:
        need.setdefault(int(slot_of[i_o[g, j]]), []).append((g, j))
    y_ref = {}
    for s, pairs in need.items():
        wg_s, wd_s = as_f32(to_np(wgu[s])), as_f32(to_np(wd[s]))
        ys_s = orc.expert_ffn(x_f[[g for g, _ in pairs]], wg_s, wd_s)
        for (g, j), y in zip(pairs, ys_s):
            y_ref[(g, j)] = y
    ys_gpu = {d: as_f32(to_np(layer.ys[d])) for d in {int(i_o[g, j]) for g, j in y_ref}}
    yg_gpu = as_f32(to_np(layer.yg[:rows]))
    worst = 0.0
    for (g, j), y in y_ref.items():
        worst = max(worst, assert_close(ys_gpu[int(i_o[g, j])], y, atol, rtol,
                                        f"expert out row {g} j {j} (sorted row {i_o[g, j]})"))
    for g in toks:
        ref = np.zeros(spec.H)
        for j in range(kk):
            ref += w_o[g, j] * y_ref[(int(g), j)]
        assert_close(yg_gpu[g], ref, atol, rtol, f"combined row {g}")
    assert not yg_gpu[valid == 0].any()                                   # pad rows zero
    # scatter returns exactly the valid rows of the combined buffer (any size)
    got = np.concatenate([as_f32(to_np(t)) for t in out]) if spec.T else np.zeros((0, spec.H))
    assert np.array_equal(got, yg_gpu[valid == 1])
    return worst


def test_layer_tiny_fp32_full(md, orc):
    spec = synth.spec_tiny()
    res = _layer_gpu(md, spec)
    _check_layer(md, orc, spec, *res, atol=F32_ATOL, rtol=F32_RTOL)


@pytest.mark.parametrize("mode", [0, 1])
def test_layer_tiny_bf16_all_rows(md, orc, mode):
    spec = synth.LayerSpec("tiny_bf16", [16, 0, 140, 8, 1], mode, H=512, E=16, k=4, I=256,
                           dtype="bf16", w_std=0.05, zipf_s=1.1)
    res = _layer_gpu(md, spec)
    _check_layer(md, orc, spec, *res)
    # without the global output buffer (the default) the replicas get the same bits
    layer, out, x_loc, lg_loc, wgu, wd, offs, rows = res
    lean = md.MoeLayer(R=spec.R, H=spec.H, E=spec.E, k=spec.k, I=spec.I, w_gate_up=wgu,
                       w_down=wd, max_rows=rows, mode=spec.mode)
    out2 = [torch.full_like(t, 7.0) for t in out]
    lean.forward(x_loc, lg_loc, out2, counts=spec.counts)
    torch.cuda.synchronize()
    assert int(lean.status.item()) == 0
    for a, b in zip(out2, out):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("mode", [0, 1])
def test_layer_shared_expert_all_rows(md, orc, mode):
    spec = synth.LayerSpec("tiny_shared", [16, 0, 140, 8, 1], mode, H=512, E=16, k=4, I=256,
                           dtype="bf16", w_std=0.05, zipf_s=1.1, n_shared=1)
    res = _layer_gpu(md, spec)
    _check_layer(md, orc, spec, *res)


def test_layer_dsv3_decode_with_shared_expert(md, orc):
    spec = synth.spec_decode(seed=1)
    spec.n_shared = 1
    res = _layer_gpu(md, spec)
    _check_layer(md, orc, spec, *res, sample=6)


def test_layer_dsv3_decode_full_size(md, orc):
    spec = synth.spec_decode(seed=0)
    res = _layer_gpu(md, spec)
    _check_layer(md, orc, spec, *res, sample=10)
    layer, out, x_loc, lg_loc = res[:4]
    graph_replay_matches_eager(layer, x_loc, lg_loc, out)


def test_layer_dsv3_prefill_full_size(md, orc):
    spec = synth.spec_prefill()
    res = _layer_gpu(md, spec)
    _check_layer(md, orc, spec, *res, sample=6)
    layer, out, x_loc, lg_loc = res[:4]
    graph_replay_matches_eager(layer, x_loc, lg_loc, out)


@pytest.mark.parametrize("mix,tpr,mode", [("mix0", 1, 0), ("mix1", 4, 1), ("mix2", 4, 2),
                                          ("all4", 1, 2), ("all24", 1, 1)])
def test_layer_pad_sweep_full_size(md, orc, mix, tpr, mode):
    spec = synth.spec_pad_sweep(mix, tpr, mode)
    res = _layer_gpu(md, spec)
    _check_layer(md, orc, spec, *res, sample=3)


def test_layer_eplb_full_size_with_ep_ranges(md, orc):
    spec = synth.spec_eplb()
    l2p, nrep, p2l = synth.make_map(spec)
    ranges = synth.slot_ranges(spec.slots, spec.n_ranges)
    res = _layer_gpu(md, spec, l2p, nrep, p2l, ranges=ranges)
    _check_layer(md, orc, spec, *res, sample=6, l2p=l2p, nrep=nrep)


def test_layer_align128_and_determinism(md, orc):
    spec = synth.LayerSpec("align128", [300, 0, 77], 1, H=512, E=32, k=8, I=256, dtype="bf16",
                           w_std=0.05, align=128)
    layer, out, *rest = _layer_gpu(md, spec)
    _check_layer(md, orc, spec, layer, out, *rest)
    first = [t.clone() for t in out]
    layer.forward(rest[0], rest[1], out)
    torch.cuda.synchronize()
    for a, b in zip(first, out):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("mode", [0, 1])
def test_layer_addnorm_boundary(md, orc, mode):
    """The residual add + RMSNorm boundary (the rows routed in the same launch):
    residuals are updated exactly as the oracle's add, the normed rows are within one
    rounding of the oracle's norm, the routing equals the oracle's, and the rest of the
    step equals a plain layer fed the normed rows (checked against the oracle), bit
    for bit, in eager mode and under graph replay."""
    spec = synth.LayerSpec("addnorm", [16, 0, 140, 8, 1], mode, H=512, E=16, k=4, I=256,
                           dtype="bf16", w_std=0.05, zipf_s=1.1)
    x_loc = synth.hidden_states(spec, DEV)
    lg_loc = synth.router_logits(spec, DEV)
    wgu, wd = synth.expert_weights(spec, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(77 + mode)
    res = [torch.randn(c, spec.H, generator=g, device=DEV).to(torch.bfloat16)
           for c in spec.counts]
    res0 = [t.clone() for t in res]
    gamma = (1 + 0.1 * torch.randn(spec.H, generator=g, device=DEV)).to(torch.bfloat16)
    offs, rows = md.moe_dp_layout(spec.counts, spec.mode)
    layer = md.MoeLayer(R=spec.R, H=spec.H, E=spec.E, k=spec.k, I=spec.I, w_gate_up=wgu,
                        w_down=wd, max_rows=rows, mode=spec.mode, keep_global=True,
                        norm_gamma=gamma, norm_eps=1e-6)
    out = [torch.empty(c, spec.H, device=DEV, dtype=torch.bfloat16) for c in spec.counts]
    layer.forward(x_loc, lg_loc, out, counts=spec.counts, local_residual=res)
    assert status_of(layer.status) == 0
    f32 = lambda t: as_f32(to_np(t))
    xg = layer.xg[:rows].clone()
    for r, c in enumerate(spec.counts):
        r_new, y_r = orc.add_rmsnorm(f32(x_loc[r]), f32(res0[r]), f32(gamma), 1e-6, True)
        assert np.array_equal(f32(res[r]), r_new)
        assert_close(f32(xg[offs[r]: offs[r] + c]).astype(np.float64), y_r, 1e-6, 8e-3,
                     "normed rows")
    valid = orc.valid_rows(spec.counts, np.array(offs, np.int32), rows)
    lg_o = orc.dp_gather([to_np(t) for t in lg_loc], spec.counts, np.array(offs, np.int32), rows)
    ids_o, w_o = orc.route_topk(lg_o, spec.k, True, valid)
    assert np.array_equal(to_np(layer.ids[:rows]), ids_o)     # routed in the same launch
    assert_close(to_np(layer.w[:rows]), w_o, W_ATOL, W_RTOL, "route weights")
    # the rest of the step: a plain layer on the normed rows gives the same bits
    normed = [xg[offs[r]: offs[r] + c].clone() for r, c in enumerate(spec.counts)]
    plain = md.MoeLayer(R=spec.R, H=spec.H, E=spec.E, k=spec.k, I=spec.I, w_gate_up=wgu,
                        w_down=wd, max_rows=rows, mode=spec.mode, keep_global=True)
    out2 = [torch.full_like(t, 7.0) for t in out]
    plain.forward(normed, lg_loc, out2, counts=spec.counts)
    assert status_of(plain.status) == 0
    for a, b in zip(out2, out):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    _check_layer(md, orc, spec, plain, out2, normed, lg_loc, wgu, wd, offs, rows)
    # a graph replay from the same residuals repeats the step bit for bit
    for t, t0 in zip(res, res0):
        t.copy_(t0)
    graph = layer.capture(x_loc, lg_loc, out, local_residual=res)
    for t, t0 in zip(res, res0):     # capture's warm-up ran the step once
        t.copy_(t0)
    first = [t.clone() for t in out]
    for t in out:
        t.fill_(7.0)
    graph.replay()
    torch.cuda.synchronize()
    assert status_of(layer.status) == 0
    for a, b in zip(first, out):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
