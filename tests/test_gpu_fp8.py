"""GPU parity of the FP8 path against the oracle: quantisation and dispatch codes
bit-exact, the FP8 grouped FFN within the bf16 output tolerance.

Expected values come from the oracle only; the FP8 operands fed to the FFN are
the oracle's quantisation of the seeded inputs."""
import gc

import numpy as np
import pytest
import torch

from gpu_util import (BF16_ATOL, BF16_RTOL, as_f32, assert_close, graph_replay_matches_eager,
                      pairs_to_check, rel_fro, to_np)

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


def _status(st):
    torch.cuda.synchronize()
    return int(st.item())


def _rows(n, K, seed, dtype=torch.bfloat16):
    """Rows with per-group magnitudes from 2^-20 to 2^12, zero groups and exact ties."""
    g = torch.Generator(device=DEV).manual_seed(seed)
    x = torch.randn(n, K, generator=g, device=DEV)
    mag = 2.0 ** torch.randint(-20, 13, (n, K // 128), generator=g, device=DEV).float()
    x = x * mag.repeat_interleave(128, dim=1)
    if n > 2:
        x[1, :128] = 0.0                              # an all-zero group
        x[2, :4] = torch.tensor([448.0, 464.0, -0.5, 3.25])  # codes at and near the top
    return x.to(dtype).contiguous()


@pytest.mark.parametrize("n,K,dtype", [(37, 256, torch.bfloat16), (1, 7168, torch.bfloat16),
                                       (129, 1152, torch.float32), (0, 128, torch.bfloat16)])
def test_quantize_groups_bitexact(md, orc, n, K, dtype):
    x = _rows(n, K, seed=n + K, dtype=dtype) if n else torch.empty(0, K, device=DEV, dtype=dtype)
    q = torch.full((n, K), 0x55, dtype=torch.uint8, device=DEV)
    s = torch.full((n, K // 128), 0x55, dtype=torch.uint8, device=DEV)
    md.moe_quantize_fp8_groups(x, q, s)
    torch.cuda.synchronize()
    if n == 0:
        return
    xq_o, xs_o = orc.quant_groups(as_f32(to_np(x)))
    assert np.array_equal(to_np(q), xq_o)
    assert np.array_equal(to_np(s), xs_o)


@pytest.mark.parametrize("R,K,dtype", [(256, 384, torch.bfloat16), (128, 7168, torch.float32)])
def test_quantize_blocks_bitexact(md, orc, R, K, dtype):
    g = torch.Generator(device=DEV).manual_seed(R + K)
    w = torch.randn(R, K, generator=g, device=DEV) * 0.02
    mag = 2.0 ** torch.randint(-6, 7, (R // 128, K // 128), generator=g, device=DEV).float()
    w = (w * mag.repeat_interleave(128, 0).repeat_interleave(128, 1)).to(dtype).contiguous()
    q = torch.empty(R, K, dtype=torch.uint8, device=DEV)
    s = torch.empty(R // 128, K // 128, dtype=torch.uint8, device=DEV)
    md.moe_quantize_fp8_blocks(w, q, s)
    torch.cuda.synchronize()
    wq_o, ws_o = orc.quant_blocks(as_f32(to_np(w)))
    assert np.array_equal(to_np(q), wq_o)
    assert np.array_equal(to_np(s), ws_o)


@pytest.mark.parametrize("rows,E,align", [(300, 16, 1), (3001, 64, 128), (700, 64, 1)])
def test_dispatch_fp8_bitexact(md, orc, rows, E, align):
    k, H = 8, 1152          # 9 groups: one 1024-value segment plus a 128-value tail
    g = torch.Generator(device=DEV).manual_seed(rows)
    ids = torch.rand(rows, E, generator=g, device=DEV).argsort(dim=1)[:, :k].to(torch.int32)
    ids[::7] = -1
    ids = ids.contiguous()
    x = _rows(rows, H, seed=rows + 1)
    cap = md.moe_dispatch_cap_bound(rows, k, E, align)
    counts_P = torch.empty(E, dtype=torch.int32, device=DEV)
    offsets_P = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(cap, dtype=torch.int32, device=DEV)
    inv = torch.empty(rows, k, dtype=torch.int32, device=DEV)
    xq = torch.full((cap, H), 0x55, dtype=torch.uint8, device=DEV)
    xs = torch.full((cap, H // 128), 0x55, dtype=torch.uint8, device=DEV)
    ws = torch.empty(md.moe_dispatch_ws_bytes(rows, k, E), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    md.moe_dispatch_fp8(x, ids, E, E, counts_P, offsets_P, perm, inv, xq, xs, ws, align=align,
                        d_status=st)
    assert _status(st) == 0
    c_o, o_o, p_o, i_o = orc.dispatch(to_np(ids), E, E, None, None, align, cap)
    n = int(o_o[-1])
    assert np.array_equal(to_np(counts_P), c_o)
    assert np.array_equal(to_np(offsets_P), o_o)
    assert np.array_equal(to_np(perm)[:n], p_o[:n])
    assert np.array_equal(to_np(inv), i_o)
    q_o, s_o = orc.quant_groups(as_f32(to_np(x)))
    real = p_o[:n] >= 0
    got_q, got_s = to_np(xq)[:n], to_np(xs)[:n]
    assert np.array_equal(got_q[real], q_o[p_o[:n][real]])
    assert np.array_equal(got_s[real], s_o[p_o[:n][real]])
    assert (got_q[~real] == 0).all() and (got_s[~real] == 127).all()   # alignment padding
    assert (to_np(xq)[n:] == 0x55).all()                                  # past the last slot


def _fp8_inputs(orc, counts, H, I, seed, extra_rows=40, w_std=0.05):
    P = len(counts)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    cap = int(offsets[-1]) + extra_rows
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((cap, H)).astype(np.float32)
    xq, xe = orc.quant_groups(x)
    # per-block weight magnitudes differ, so a misread block scale shows
    def blocks(R, K):
        m = 2.0 ** rng.integers(-3, 4, (R // 128, K // 128))
        return (rng.standard_normal((R, K)) * w_std * m.repeat(128, 0).repeat(128, 1))
    wgu = [orc.quant_blocks(blocks(2 * I, H)) for _ in range(P)]
    wd = [orc.quant_blocks(blocks(H, I)) for _ in range(P)]
    return offsets, cap, xq, xe, wgu, wd


def _dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


@pytest.mark.parametrize("counts,lo,hi,H,I", [
    ([0, 1, 15, 16, 17, 31, 32, 33, 64, 100], 0, 10, 512, 256),
    ([5, 0, 40, 3], 1, 3, 512, 256),
    ([1] * 6, 0, 6, 512, 256),
    ([7, 70, 0, 33], 0, 4, 768, 640)])   # 6 and 5 k-blocks per unit
def test_grouped_ffn_fp8(md, orc, counts, lo, hi, H, I):
    """Token groups of up to 64 per unit: N = 16 .. 64, ragged groups, several groups per
    slot, empty slots, slot ranges; rows outside the range untouched; K / 128 = 2, 4, 5
    and 6 k-blocks per unit."""
    offsets, cap, xq, xe, wgu, wd = _fp8_inputs(orc, counts, H, I, seed=sum(counts) + lo)
    P = len(counts)
    w_fp8 = (_dev_u8(np.stack([w[0] for w in wgu])), _dev_u8(np.stack([w[1] for w in wgu])),
             _dev_u8(np.stack([w[0] for w in wd])), _dev_u8(np.stack([w[1] for w in wd])))
    sentinel = 1232.0
    ys = torch.full((cap, H), sentinel, device=DEV, dtype=torch.bfloat16)
    ws = md.fp8_ffn_workspace(cap, I, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    md.moe_grouped_ffn_fp8(_dev_u8(xq), _dev_u8(xe), torch.from_numpy(offsets).to(DEV), w_fp8, ys,
                           ws, lo, hi, d_status=st)
    assert _status(st) == 0
    a, b = int(offsets[lo]), int(offsets[hi])
    ref = orc.grouped_ffn_fp8(xq, xe, offsets, lambda s: (*wgu[s], *wd[s]), lo, hi)
    got = as_f32(to_np(ys)).astype(np.float64)
    assert_close(got[a:b], ref[a:b], BF16_ATOL, BF16_RTOL, "grouped FFN fp8")
    assert rel_fro(got[a:b], ref[a:b]) < 1e-2
    assert (got[:a] == sentinel).all() and (got[b:] == sentinel).all()


@pytest.mark.parametrize("counts,lo,hi,H,I", [
    ([0, 1, 15, 16, 17, 100, 223, 224, 225, 240, 256, 300, 320, 321, 700, 1000], 0, 16,
     1024, 512),
    ([250, 0, 333, 96, 260, 640, 5, 255], 1, 7, 1536, 1024),
    # 87 rows per slot on average: slots of 192 or more rows on the pair kernel, the
    # rest on the one-launch kernel after it
    ([0, 3, 500, 10, 17, 64, 191, 192, 5, 0, 250, 1, 30, 80, 2, 7], 0, 16, 1024, 512),
    ([0, 3, 500, 10, 17, 64, 191, 192, 5, 0, 250, 1, 30, 80, 2, 7], 2, 11, 1024, 512)])
def test_grouped_ffn_fp8_pair(md, orc, counts, lo, hi, H, I):
    """Many rows per slot: the FP8 pair kernel (weights as M on SM pairs, scales applied
    by the block-scaled MMA, units of up to 320 tokens split 224 + 96).  Ragged groups,
    tails of 1-96 tokens, several groups per slot, empty slots, slot ranges; rows
    outside the range untouched; K / 128 = 8 and 4 (first case), 12 and 8 k-blocks.
    The weights are small enough that every gate value goes through a sigmoid that is
    not 1 in fp32: with large gates the activation is an exact product of e4m3 values
    and lands on e4m3 rounding ties, where the kernel's fp32 and the oracle's fp64 round
    to neighbouring codes (both correct)."""
    offsets, cap, xq, xe, wgu, wd = _fp8_inputs(orc, counts, H, I, seed=sum(counts) + lo,
                                                w_std=0.01)
    P = len(counts)
    assert cap // P >= 32 and max(counts) >= 192     # the pair kernel serves some slots
    w_fp8 = (_dev_u8(np.stack([w[0] for w in wgu])), _dev_u8(np.stack([w[1] for w in wgu])),
             _dev_u8(np.stack([w[0] for w in wd])), _dev_u8(np.stack([w[1] for w in wd])))
    sentinel = 1232.0
    ys = torch.full((cap, H), sentinel, device=DEV, dtype=torch.bfloat16)
    ws = md.fp8_ffn_workspace(cap, I, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    md.moe_grouped_ffn_fp8(_dev_u8(xq), _dev_u8(xe), torch.from_numpy(offsets).to(DEV), w_fp8, ys,
                           ws, lo, hi, d_status=st)
    assert _status(st) == 0
    a, b = int(offsets[lo]), int(offsets[hi])
    ref = orc.grouped_ffn_fp8(xq, xe, offsets, lambda s: (*wgu[s], *wd[s]), lo, hi)
    got = as_f32(to_np(ys)).astype(np.float64)
    assert_close(got[a:b], ref[a:b], BF16_ATOL, BF16_RTOL, "grouped FFN fp8, pair kernel")
    assert rel_fro(got[a:b], ref[a:b]) < 1e-2
    assert (got[:a] == sentinel).all() and (got[b:] == sentinel).all()
    # a second call on the same workspace gives the same bits
    ys2 = torch.full((cap, H), sentinel, device=DEV, dtype=torch.bfloat16)
    md.moe_grouped_ffn_fp8(_dev_u8(xq), _dev_u8(xe), torch.from_numpy(offsets).to(DEV), w_fp8,
                           ys2, ws, lo, hi, d_status=st)
    assert _status(st) == 0
    assert torch.equal(ys.view(torch.int16), ys2.view(torch.int16))


def test_grouped_ffn_fp8_dsv3_width(md, orc):
    """DeepSeek-V3 expert shapes (H=7168, I=2048): 56 and 16 k-blocks per unit."""
    counts = [3, 20, 0, 9]
    H, I = 7168, 2048
    offsets, cap, xq, xe, wgu, wd = _fp8_inputs(orc, counts, H, I, seed=3, extra_rows=8)
    w_fp8 = (_dev_u8(np.stack([w[0] for w in wgu])), _dev_u8(np.stack([w[1] for w in wgu])),
             _dev_u8(np.stack([w[0] for w in wd])), _dev_u8(np.stack([w[1] for w in wd])))
    ys = torch.zeros((cap, H), device=DEV, dtype=torch.bfloat16)
    ws = md.fp8_ffn_workspace(cap, I, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    md.moe_grouped_ffn_fp8(_dev_u8(xq), _dev_u8(xe), torch.from_numpy(offsets).to(DEV), w_fp8, ys,
                           ws, d_status=st)
    assert _status(st) == 0
    n = int(offsets[-1])
    ref = orc.grouped_ffn_fp8(xq, xe, offsets, lambda s: (*wgu[s], *wd[s]))
    got = as_f32(to_np(ys)).astype(np.float64)
    assert_close(got[:n], ref[:n], BF16_ATOL, BF16_RTOL, "grouped FFN fp8, DSV3 width")
    assert rel_fro(got[:n], ref[:n]) < 1e-2


def test_grouped_ffn_fp8_max_slots_and_ep_ranges(md, orc):
    """MOE_MAX_SLOTS (1024) slots, tokens in a scattered few (the first and last
    included, one with two token groups): one call over all slots matches the oracle,
    and sixteen calls over 64-slot ranges (as EP ranks would) on the same workspace
    give the same bits."""
    P, H, I = 1024, 256, 128
    rng = np.random.default_rng(21)
    counts = [0] * P
    for s_ in [0, 1, 77, 300, 511, 512, 640, 1000, 1023]:
        counts[s_] = int(rng.integers(1, 40))
    counts[512] = 90
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    cap = int(offsets[-1]) + 24
    x = rng.standard_normal((cap, H)).astype(np.float32)
    xq, xe = orc.quant_groups(x)
    wgu1 = orc.quant_blocks(rng.standard_normal((2 * I, H)) * 0.05)
    wd1 = orc.quant_blocks(rng.standard_normal((H, I)) * 0.05)
    wgu2 = orc.quant_blocks(rng.standard_normal((2 * I, H)) * 0.05)
    wd2 = orc.quant_blocks(rng.standard_normal((H, I)) * 0.05)
    pick = lambda s_: (wgu1, wd1) if s_ % 2 == 0 else (wgu2, wd2)     # two weight sets
    w_fp8 = tuple(_dev_u8(np.stack([pick(s_)[j][i] for s_ in range(P)]))
                  for j, i in [(0, 0), (0, 1), (1, 0), (1, 1)])
    ws = md.fp8_ffn_workspace(cap, I, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    args = (_dev_u8(xq), _dev_u8(xe), torch.from_numpy(offsets).to(DEV), w_fp8)
    ys_a = torch.zeros((cap, H), device=DEV, dtype=torch.bfloat16)
    md.moe_grouped_ffn_fp8(*args, ys_a, ws, d_status=st)
    assert _status(st) == 0
    ys_b = torch.zeros((cap, H), device=DEV, dtype=torch.bfloat16)
    for lo in range(0, P, 64):
        md.moe_grouped_ffn_fp8(*args, ys_b, ws, lo, lo + 64, d_status=st)
    assert _status(st) == 0
    n = int(offsets[-1])
    assert torch.equal(ys_a[:n].view(torch.int16), ys_b[:n].view(torch.int16))
    ref = orc.grouped_ffn_fp8(xq, xe, offsets, lambda s_: (*pick(s_)[0], *pick(s_)[1]))
    got = as_f32(to_np(ys_a)).astype(np.float64)
    assert_close(got[:n], ref[:n], BF16_ATOL, BF16_RTOL, "grouped FFN fp8, 1024 slots")


def test_grouped_ffn_fp8_stale_workspace_flagged_and_cleared(md, orc):
    """The scheduler words at the end of the workspace start at zero and every call
    leaves them zero.  A call that finds a stale unit ticket claims no unit, sets
    MOE_DEV_BAD_WORKSPACE and clears the words; the next call on the same workspace
    is correct."""
    counts = [7, 70, 0, 33]
    H, I = 512, 256
    offsets, cap, xq, xe, wgu, wd = _fp8_inputs(orc, counts, H, I, seed=11)
    w_fp8 = (_dev_u8(np.stack([w[0] for w in wgu])), _dev_u8(np.stack([w[1] for w in wgu])),
             _dev_u8(np.stack([w[0] for w in wd])), _dev_u8(np.stack([w[1] for w in wd])))
    ws = md.fp8_ffn_workspace(cap, I, DEV)
    words = ws[-4 * (3 + 1024):].view(torch.int32)        # ticket, done, reserved, per slot
    words[0] = 1 << 30
    ys = torch.zeros((cap, H), device=DEV, dtype=torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    args = (_dev_u8(xq), _dev_u8(xe), torch.from_numpy(offsets).to(DEV), w_fp8, ys, ws)
    md.moe_grouped_ffn_fp8(*args, d_status=st)
    assert _status(st) == md.MOE_DEV_BAD_WORKSPACE
    assert not words.any()
    st.zero_()
    md.moe_grouped_ffn_fp8(*args, d_status=st)
    assert _status(st) == 0
    assert not words.any()
    n = int(offsets[-1])
    ref = orc.grouped_ffn_fp8(xq, xe, offsets, lambda s: (*wgu[s], *wd[s]))
    got = as_f32(to_np(ys)).astype(np.float64)
    assert_close(got[:n], ref[:n], BF16_ATOL, BF16_RTOL, "grouped FFN fp8 after clearing")


def test_grouped_ffn_fp8_slot_wait_times_out_and_recovers(md, orc):
    """An MM2 unit waits, with a time limit, until its slot's MM1 units are counted.
    A slot count planted far below zero never reaches its target: the waiting CTAs
    give up after the limit (about 2 s), the call sets MOE_DEV_TIMEOUT (not
    MOE_DEV_BAD_WORKSPACE), the device stays usable, the scheduler words are
    cleared, and the next call on the same workspace is correct."""
    counts = [7, 70, 0, 33]
    H, I = 512, 256
    offsets, cap, xq, xe, wgu, wd = _fp8_inputs(orc, counts, H, I, seed=12)
    w_fp8 = (_dev_u8(np.stack([w[0] for w in wgu])), _dev_u8(np.stack([w[1] for w in wgu])),
             _dev_u8(np.stack([w[0] for w in wd])), _dev_u8(np.stack([w[1] for w in wd])))
    ws = md.fp8_ffn_workspace(cap, I, DEV)
    words = ws[-4 * (3 + 1024):].view(torch.int32)        # ticket, done, reserved, per slot
    words[3 + 1] = -(1 << 20)                              # slot 1 (70 tokens)
    ys = torch.zeros((cap, H), device=DEV, dtype=torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    args = (_dev_u8(xq), _dev_u8(xe), torch.from_numpy(offsets).to(DEV), w_fp8, ys, ws)
    md.moe_grouped_ffn_fp8(*args, d_status=st)
    code = _status(st)
    assert code & md.MOE_DEV_TIMEOUT and not code & md.MOE_DEV_BAD_WORKSPACE
    assert not words.any()
    st.zero_()
    md.moe_grouped_ffn_fp8(*args, d_status=st)
    assert _status(st) == 0
    n = int(offsets[-1])
    ref = orc.grouped_ffn_fp8(xq, xe, offsets, lambda s: (*wgu[s], *wd[s]))
    got = as_f32(to_np(ys)).astype(np.float64)
    assert_close(got[:n], ref[:n], BF16_ATOL, BF16_RTOL, "grouped FFN fp8 after the timeout")


# ------------------------------------------------------------------ whole layer
def _layer_fp8_check(md, orc, spec, sample=None, l2p_np=None, nrep_np=None, p2l=None):
    from combine_dp_gather_gb300 import synth
    x_loc = synth.hidden_states(spec, DEV)
    lg_loc = synth.router_logits(spec, DEV)
    wgu, wd = synth.expert_weights(spec, p2l, DEV)
    offs, rows = md.moe_dp_layout(spec.counts, spec.mode, spec.static_bound, spec.tokens_per_req)
    l2p = None if l2p_np is None else torch.from_numpy(l2p_np).to(DEV)
    nrep = None if nrep_np is None else torch.from_numpy(nrep_np).to(DEV)
    layer = md.MoeLayer(R=spec.R, H=spec.H, E=spec.E, k=spec.k, I=spec.I, w_gate_up=wgu,
                        w_down=wd, max_rows=max(rows, 1), mode=spec.mode,
                        renormalize=spec.renormalize, n_shared=spec.n_shared, fp8=True,
                        keep_global=True, l2p=l2p, nrep=nrep)
    out = [torch.empty(c, spec.H, device=DEV, dtype=wgu.dtype) for c in spec.counts]
    layer.forward(x_loc, lg_loc, out, counts=spec.counts)
    assert _status(layer.status) == 0
    offs_o, rows_o = orc.dp_layout(spec.counts, spec.mode, 0, 1)
    valid = orc.valid_rows(spec.counts, offs_o, rows_o)
    xg_o = orc.dp_gather([to_np(t) for t in x_loc], spec.counts, offs_o, rows_o)
    lg_o = orc.dp_gather([to_np(t) for t in lg_loc], spec.counts, offs_o, rows_o)
    ids_o, w_o = orc.route_topk(lg_o, spec.k, spec.renormalize, valid, spec.n_shared)
    kk = spec.k + spec.n_shared
    assert np.array_equal(to_np(layer.ids[:rows]), ids_o)
    c_o, o_o, p_o, i_o = orc.dispatch(ids_o, spec.E + spec.n_shared, layer.P, l2p_np, nrep_np,
                                      1, layer.cap)
    n = int(o_o[-1])
    assert np.array_equal(to_np(layer.offsets_P), o_o)
    assert np.array_equal(to_np(layer.inv[:rows]), i_o)
    x_f = as_f32(xg_o)
    q_o, s_o = orc.quant_groups(x_f)                     # every global row, then permuted
    assert np.array_equal(to_np(layer.xq[:n]), q_o[p_o[:n]])
    assert np.array_equal(to_np(layer.xq_scales[:n]), s_o[p_o[:n]])
    real = np.nonzero(valid)[0]
    # every pair of small layers; at full size the kernel's hard rows and a few
    # tokens' combined rows
    check, toks = pairs_to_check(layer, o_o, p_o, i_o, real, kk, sample)
    slot_of = np.searchsorted(o_o, np.arange(n), side="right") - 1
    need = {}
    for g, j in check:
        need.setdefault(int(slot_of[i_o[g, j]]), []).append((g, j))
    guq, gus, dq, ds = layer.w_fp8
    y_ref = {}
    for s, pairs in need.items():
        wq = orc.quant_blocks(as_f32(to_np(wgu[s])))
        dq_o = orc.quant_blocks(as_f32(to_np(wd[s])))
        assert np.array_equal(to_np(guq[s]), wq[0]) and np.array_equal(to_np(gus[s]), wq[1])
        assert np.array_equal(to_np(dq[s]), dq_o[0]) and np.array_equal(to_np(ds[s]), dq_o[1])
        rows_s = [g for g, _ in pairs]
        ys_s = orc.expert_ffn_fp8(q_o[rows_s], s_o[rows_s], *wq, *dq_o)
        for (g, j), y in zip(pairs, ys_s):
            y_ref[(g, j)] = y
    yg = as_f32(to_np(layer.yg[:rows]))
    for (g, j), y in y_ref.items():
        assert_close(as_f32(to_np(layer.ys[int(i_o[g, j])])), y, BF16_ATOL, BF16_RTOL,
                     f"fp8 expert out row {g} j {j} (sorted row {i_o[g, j]})")
    for g in toks:
        ref = np.zeros(spec.H)
        for j in range(kk):
            ref += w_o[g, j] * y_ref[(int(g), j)]
        assert_close(yg[g], ref, BF16_ATOL, BF16_RTOL, f"fp8 combined row {g}")
    assert not yg[valid == 0].any()
    got = np.concatenate([as_f32(to_np(t)) for t in out])
    assert np.array_equal(got, yg[valid == 1])
    graph_replay_matches_eager(layer, x_loc, lg_loc, out)


@pytest.mark.parametrize("mode", [0, 1])
def test_layer_fp8_tiny_all_rows(md, orc, mode):
    from combine_dp_gather_gb300 import synth
    spec = synth.LayerSpec("tiny_fp8", [16, 0, 140, 8, 1], mode, H=512, E=16, k=4, I=256,
                           dtype="bf16", w_std=0.05, zipf_s=1.1)
    _layer_fp8_check(md, orc, spec)


def test_layer_fp8_dsv3_decode(md, orc):
    from combine_dp_gather_gb300 import synth
    _layer_fp8_check(md, orc, synth.spec_decode(seed=0), sample=6)


def test_layer_fp8_eplb_full_size(md, orc):
    """The EPLB workload on the FP8 path: 256 logical experts on 288 slots through the
    map, hot slots with up to ~1000 rows (16 token groups per weight tile)."""
    from combine_dp_gather_gb300 import synth
    spec = synth.spec_eplb()
    l2p, nrep, p2l = synth.make_map(spec)
    _layer_fp8_check(md, orc, spec, sample=6, l2p_np=l2p, nrep_np=nrep, p2l=p2l)


def test_layer_fp8_prefill_full_size(md, orc):
    """The prefill workload (8192 tokens, ~256 rows per slot: four token groups per
    weight tile) on the FP8 path."""
    from combine_dp_gather_gb300 import synth
    _layer_fp8_check(md, orc, synth.spec_prefill(), sample=4)


def test_layer_fp8_with_shared_expert(md, orc):
    from combine_dp_gather_gb300 import synth
    spec = synth.LayerSpec("tiny_fp8_shared", [16, 0, 140, 8, 1], 1, H=512, E=16, k=4, I=256,
                           dtype="bf16", w_std=0.05, zipf_s=1.1, n_shared=1)
    _layer_fp8_check(md, orc, spec)
