"""Pins of the CPU oracle against what the pages and the mathematics fix.

Every check here is independent of the oracle's own code path: numpy
concatenation / padding, Python's sort with a tuple key, brute force over all
k-subsets, scipy's softmax, numpy float64 matmul, a dense per-token
formulation of the layer, and golden values cited from the pages.  The
"mutant" tests feed deliberately wrong variants to the same checks to show
that each check catches the mistake it is meant to catch.
"""
import itertools

import numpy as np
import pytest
import scipy.special
import torch

from conftest import ints, read_golden

MODES = {"sum": 0, "max": 1, "static": 2}


# ----------------------------------------------------------------- layout
@pytest.mark.parametrize("row", read_golden("dp_layout.txt"))
def test_layout_golden(orc, row):
    counts, mode, B, tpr, offs, rows = row
    o, n = orc.dp_layout(ints(counts), MODES[mode], int(B), int(tpr))
    assert o.tolist() == ints(offs)
    assert n == int(rows)


@pytest.mark.parametrize("row", read_golden("dp_layout_errors.txt"))
def test_layout_errors_golden(orc, row):
    counts, mode, B, tpr, err = row
    with pytest.raises(orc.OracleError) as ei:
        orc.dp_layout(ints(counts), MODES[mode], int(B), int(tpr))
    assert ei.value.code == {"bound": 3, "arg": 1}[err]


@pytest.mark.parametrize("row", read_golden("dp_padding_mode.txt"))
def test_padding_mode_golden(orc, row):
    counts, width, ext, idle, mode = row
    assert orc.dp_padding_mode(ints(counts), int(width), int(ext), int(idle)) == MODES[mode]


def _segments(rng, counts, H, dtype=np.float32):
    return [rng.standard_normal((c, H)).astype(dtype) for c in counts]


def check_sum_is_concatenation(gather, layout, counts, H=5, seed=0):
    rng = np.random.default_rng(seed)
    segs = _segments(rng, counts, H)
    offs, rows = layout(counts, 0)
    g = gather(segs, counts, offs, rows)
    return rows == sum(counts) and np.array_equal(g, np.concatenate(segs, axis=0))


def check_max_is_padded_stack(gather, layout, counts, H=3, seed=1):
    rng = np.random.default_rng(seed)
    segs = _segments(rng, counts, H)
    offs, rows = layout(counts, 1)
    mx = max(counts)
    g = gather(segs, counts, offs, rows)
    ref = np.stack([np.pad(s, ((0, mx - len(s)), (0, 0))) for s in segs])
    return rows == len(counts) * mx and np.array_equal(g.reshape(len(counts), mx, H), ref)


def test_layout_sum_exhaustive_small(orc):
    for R in range(1, 4):
        for counts in itertools.product(range(0, 4), repeat=R):
            assert check_sum_is_concatenation(orc.dp_gather, orc.dp_layout, list(counts))
            if max(counts) > 0:
                assert check_max_is_padded_stack(orc.dp_gather, orc.dp_layout, list(counts))


def test_layout_static_blocks(orc):
    rng = np.random.default_rng(3)
    for tpr in (1, 4):
        counts = [int(v) * tpr for v in rng.choice([0, 4, 8, 24], size=16)]
        offs, rows = orc.dp_layout(counts, 2, 24, tpr)
        seg = 24 * tpr
        assert rows == 16 * seg
        segs = _segments(rng, counts, 4)
        g = orc.dp_gather(segs, counts, offs, rows).reshape(16, seg, 4)
        for r in range(16):
            assert np.array_equal(g[r, : counts[r]], segs[r])
            assert not g[r, counts[r]:].any()


def test_gather_scatter_identity(orc):
    rng = np.random.default_rng(4)
    for mode in (0, 1):
        counts = [int(v) for v in rng.integers(0, 9, size=6)]
        segs = [rng.integers(0, 2**16, size=(c, 7), dtype=np.uint16) for c in counts]
        offs, rows = orc.dp_layout(counts, mode)
        g = orc.dp_gather(segs, counts, offs, rows)
        back = orc.dp_scatter(g, counts, offs)
        assert all(np.array_equal(a, b) for a, b in zip(segs, back))
        valid = orc.valid_rows(counts, offs, rows)
        assert int(valid.sum()) == sum(counts)
        assert not g[valid == 0].any()  # pad rows are zero


def test_mutant_inclusive_prefix_is_caught(orc):
    def bad_layout(counts, mode, *a):
        o, n = orc.dp_layout(counts, mode, *a)
        o = o.copy()
        o[:-1] = np.cumsum(counts)  # inclusive instead of exclusive
        return o, n

    def tolerant_gather(segs, counts, offs, rows):
        out = np.zeros((rows + max(counts, default=0),) + segs[0].shape[1:], segs[0].dtype)
        for r, s in enumerate(segs):
            out[offs[r]: offs[r] + len(s)] = s
        return out[:rows]

    assert not check_sum_is_concatenation(tolerant_gather, bad_layout, [2, 3, 1])


# ----------------------------------------------------------------- top-k routing
def brute_force_topk(lrow, k):
    """Best k-subset by total logit; ties by the lexicographically smallest ids."""
    E = len(lrow)
    best = None
    for sub in itertools.combinations(range(E), k):
        key = (sum(float(lrow[e]) for e in sub), tuple(-e for e in sub))
        if best is None or key > best[0]:
            best = (key, sub)
    sub = best[1]
    return sorted(sub, key=lambda e: (-float(lrow[e]), e))


def check_topk(route, E, k, seed, renorm=True):
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((12, E)).astype(np.float32)
    valid = np.ones(12, np.uint8)
    valid[[3, 7]] = 0
    ids, w = route(logits, k, renorm, valid)
    for g in range(12):
        if not valid[g]:
            if not ((ids[g] == -1).all() and (w[g] == 0).all()):
                return False
            continue
        ref = brute_force_topk(logits[g], k)
        if ids[g].tolist() != ref:
            return False
        sel = logits[g].astype(np.float64)[ref]
        wref = (scipy.special.softmax(sel) if renorm
                else scipy.special.softmax(logits[g].astype(np.float64))[ref])
        if not np.allclose(w[g], wref, rtol=1e-12, atol=0):
            return False
    return True


@pytest.mark.parametrize("E,k", [(8, 2), (6, 3), (5, 1), (5, 5), (9, 4)])
@pytest.mark.parametrize("renorm", [True, False])
def test_topk_brute_force(orc, E, k, renorm):
    assert check_topk(orc.route_topk, E, k, seed=E * 10 + k, renorm=renorm)


def test_topk_ties_lower_id_and_special_cases(orc):
    E = 8
    logits = np.zeros((3, E), np.float32)
    logits[1, [2, 5, 6]] = 1.5          # a 3-way tie for the top
    logits[2] = np.arange(E)[::-1]      # strictly decreasing
    ids, w = orc.route_topk(logits, 4, True, np.ones(3, np.uint8))
    assert ids[0].tolist() == [0, 1, 2, 3] and np.all(w[0] == 0.25)
    assert ids[1].tolist() == [2, 5, 6, 0]
    assert ids[2].tolist() == [0, 1, 2, 3]
    ids1, w1 = orc.route_topk(logits, 1, True, np.ones(3, np.uint8))
    assert np.all(w1 == 1.0)
    idsE, wE = orc.route_topk(logits, E, True, np.ones(3, np.uint8))
    assert np.allclose(wE.sum(1), 1.0, rtol=0, atol=1e-15)


def test_mutant_tie_to_higher_id_is_caught(orc):
    def bad_route(logits, k, renorm, valid):
        # picks among equal logits the higher id
        rev = np.ascontiguousarray(logits[:, ::-1])
        ids, w = orc.route_topk(rev, k, renorm, valid)
        E = logits.shape[1]
        return np.where(ids >= 0, E - 1 - ids, ids), w

    rng_logits = np.round(np.random.default_rng(5).standard_normal((12, 6)), 0)

    def tied_route(logits, k, renorm, valid):
        return bad_route(rng_logits.astype(np.float32), k, renorm, valid)

    ok = True
    valid = np.ones(12, np.uint8)
    ids, _ = tied_route(None, 3, True, valid)
    for g in range(12):
        if ids[g].tolist() != brute_force_topk(rng_logits[g].astype(np.float32), 3):
            ok = False
    assert not ok


# ----------------------------------------------------------------- dispatch
def sort_reference(ids, E, P, l2p=None, nrep=None, align=1):
    """Dispatch by definition: slot choice by round-robin occurrence count, then
    Python's sort of (slot, row, j) tuples."""
    rows, k = ids.shape
    seen = {}
    keys = []
    for g in range(rows):
        for j in range(k):
            l = int(ids[g, j])
            if l < 0:
                continue
            if l2p is None:
                slot = l
            else:
                p = seen.get(l, 0)
                seen[l] = p + 1
                slot = int(l2p[l, p % int(nrep[l])])
            keys.append((slot, g, j))
    keys.sort()
    counts = np.zeros(P, np.int64)
    for s, _, _ in keys:
        counts[s] += 1
    padded = (counts + align - 1) // align * align
    offsets = np.concatenate([[0], np.cumsum(padded)])
    perm = np.full(offsets[-1], -1, np.int64)
    inv = np.full((rows, k), -1, np.int64)
    i = 0
    for s in range(P):
        for c in range(counts[s]):
            _, g, j = keys[i]
            perm[offsets[s] + c] = g
            inv[g, j] = offsets[s] + c
            i += 1
    return counts, offsets, perm, inv


def _random_ids(rng, rows, k, E, pad_rows=()):
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(rows)]).astype(np.int32)
    ids[list(pad_rows)] = -1
    return ids


@pytest.mark.parametrize("align", [1, 4, 128])
def test_dispatch_matches_tuple_sort(orc, align):
    rng = np.random.default_rng(6)
    E, k, rows = 8, 3, 37
    ids = _random_ids(rng, rows, k, E, pad_rows=(0, 5, 36))
    c, o, perm, inv = orc.dispatch(ids, E, E, align=align)
    rc, ro, rp, ri = sort_reference(ids, E, E, align=align)
    assert np.array_equal(c, rc) and np.array_equal(o, ro)
    assert np.array_equal(perm[: o[-1]], rp) and np.array_equal(inv, ri)
    assert (perm[o[-1]:] == -1).all()
    assert int(c.sum()) == (rows - 3) * k
    assert all(v % align == 0 for v in o)


def test_dispatch_with_map_matches_tuple_sort(orc):
    from combine_dp_gather_gb300 import synth
    rng = np.random.default_rng(7)
    E, P, k, rows = 6, 10, 2, 50
    l2p, nrep, p2l = synth.trivial_map(E, P)
    ids = _random_ids(rng, rows, k, E, pad_rows=(3,))
    c, o, perm, inv = orc.dispatch(ids, E, P, l2p, nrep)
    rc, ro, rp, ri = sort_reference(ids, E, P, l2p, nrep)
    assert np.array_equal(c, rc) and np.array_equal(perm[: o[-1]], rp)
    assert np.array_equal(inv, ri)
    # physical -> logical counts by scatter-add conserve the logical histogram
    logical = np.zeros(E, np.int64)
    np.add.at(logical, p2l, c)
    assert np.array_equal(logical, np.bincount(ids[ids >= 0], minlength=E))
    # round robin: replicas of one expert differ by at most one, earlier replicas first
    for e in range(E):
        rc_e = [int(c[l2p[e, x]]) for x in range(nrep[e])]
        assert max(rc_e) - min(rc_e) <= 1 and rc_e == sorted(rc_e, reverse=True)


def test_dispatch_bijection_and_errors(orc):
    rng = np.random.default_rng(8)
    E, k, rows = 16, 4, 200
    ids = _random_ids(rng, rows, k, E)
    c, o, perm, inv = orc.dispatch(ids, E, E)
    flat = inv.reshape(-1)
    assert sorted(flat.tolist()) == list(range(rows * k))
    for g in range(rows):
        for j in range(k):
            assert perm[inv[g, j]] == g
    with pytest.raises(orc.OracleError) as ei:
        orc.dispatch(ids, E, E, cap=rows * k - 1)
    assert ei.value.code == 2
    bad = ids.copy()
    bad[5, 1] = E
    with pytest.raises(orc.OracleError) as ei:
        orc.dispatch(bad, E, E)
    assert ei.value.code == 4


def test_mutant_reversed_order_is_caught(orc):
    rng = np.random.default_rng(9)
    ids = _random_ids(rng, 20, 2, 4)
    c, o, perm, inv = orc.dispatch(ids, 4, 4)
    bad_perm = perm.copy()
    for s in range(4):
        bad_perm[o[s]: o[s + 1]] = perm[o[s]: o[s + 1]][::-1]
    _, _, rp, _ = sort_reference(ids, 4, 4)
    assert not np.array_equal(bad_perm[: o[-1]], rp)


def test_permute_rows(orc):
    rng = np.random.default_rng(10)
    xg = rng.integers(0, 2**16, size=(9, 6), dtype=np.uint16)
    perm = np.array([3, -1, 0, 8, 8, -1], np.int32)
    xs = orc.permute_rows(xg, perm)
    for d, p in enumerate(perm):
        assert np.array_equal(xs[d], xg[p] if p >= 0 else np.zeros(6, np.uint16))


# ----------------------------------------------------------------- FFN
def numpy_swiglu(x, wgu, wd):
    I = wd.shape[1]
    x = x.astype(np.float64)
    g = x @ wgu[:I].astype(np.float64).T
    u = x @ wgu[I:].astype(np.float64).T
    a = g * scipy.special.expit(g) * u
    return a @ wd.astype(np.float64).T


@pytest.mark.parametrize("n,H,I", [(5, 16, 8), (3, 64, 32), (1, 7, 3)])
def test_ffn_matches_numpy(orc, n, H, I):
    rng = np.random.default_rng(n * H + I)
    x = rng.standard_normal((n, H)).astype(np.float32)
    wgu = (0.2 * rng.standard_normal((2 * I, H))).astype(np.float32)
    wd = (0.2 * rng.standard_normal((H, I))).astype(np.float32)
    y = orc.expert_ffn(x, wgu, wd)
    ref = numpy_swiglu(x, wgu, wd)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-13)


def test_grouped_ffn_runs_each_slot_through_its_own_expert(orc):
    """Slot s's rows [offsets[s], offsets[s+1]) go through expert s (against the numpy
    SwiGLU), an empty slot is skipped, and rows of slots outside [lo, hi) are left NaN."""
    rng = np.random.default_rng(21)
    H, I = 24, 8
    counts = [3, 0, 5, 2, 4]
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    xs = rng.standard_normal((int(offsets[-1]), H)).astype(np.float32)
    wgu = (0.3 * rng.standard_normal((5, 2 * I, H))).astype(np.float32)
    wd = (0.3 * rng.standard_normal((5, H, I))).astype(np.float32)
    ys = orc.grouped_ffn(xs, offsets, wgu, wd, 1, 4)
    for s in range(5):
        a, b = int(offsets[s]), int(offsets[s + 1])
        if 1 <= s < 4:
            assert np.allclose(ys[a:b], numpy_swiglu(xs[a:b], wgu[s], wd[s]), rtol=1e-12,
                               atol=1e-13)
        else:
            assert np.isnan(ys[a:b]).all()
    # a slot read with another slot's weights would show: experts differ
    assert not np.allclose(ys[3:8], numpy_swiglu(xs[3:8], wgu[3], wd[3]))


def test_ffn_special_cases(orc):
    rng = np.random.default_rng(11)
    x = rng.standard_normal((4, 16)).astype(np.float32)
    wgu = rng.standard_normal((16, 16)).astype(np.float32)
    wd = rng.standard_normal((16, 8)).astype(np.float32)
    assert not orc.expert_ffn(x, np.zeros_like(wgu), wd).any()
    up0 = wgu.copy()
    up0[8:] = 0
    assert not orc.expert_ffn(x, up0, wd).any()
    assert not orc.expert_ffn(np.zeros_like(x), wgu, wd).any()
    # gate and up swapped must change the result: silu is not symmetric
    swapped = np.concatenate([wgu[8:], wgu[:8]])
    assert not np.allclose(orc.expert_ffn(x, swapped, wd), orc.expert_ffn(x, wgu, wd))


# ----------------------------------------------------------------- combine
def test_combine_identity_experts_return_input(orc):
    rng = np.random.default_rng(12)
    rows, k, E, H = 30, 4, 8, 64
    xb = orc.f64_to_bf16_bits(rng.standard_normal((rows, H)))
    x = orc.bf16_bits_to_f32(xb).astype(np.float64)
    logits = rng.standard_normal((rows, E)).astype(np.float32)
    valid = np.ones(rows, np.uint8)
    valid[[2, 9]] = 0
    ids, w = orc.route_topk(logits, k, True, valid)
    c, o, perm, inv = orc.dispatch(ids, E, E)
    xs = orc.permute_rows(x, perm[: o[-1]])
    out = orc.combine(xs, inv, w)          # identity experts: ys = xs
    assert np.array_equal(orc.f64_to_bf16_bits(out[valid == 1]), xb[valid == 1])
    assert not out[valid == 0].any()


def test_combine_matches_einsum(orc):
    rng = np.random.default_rng(13)
    rows, k, H, cap = 10, 3, 5, 40
    ys = rng.standard_normal((cap, H))
    inv = np.stack([rng.choice(cap, size=k, replace=False) for _ in range(rows)]).astype(np.int32)
    inv[4] = -1
    w = rng.random((rows, k))
    out = orc.combine(ys, inv, w)
    g = np.where(inv[..., None] >= 0, ys[np.maximum(inv, 0)], 0.0)
    assert np.allclose(out, np.einsum("rk,rkh->rh", w, g), rtol=1e-14, atol=1e-14)


def test_mutant_dropped_term_is_caught(orc):
    rng = np.random.default_rng(14)
    xb = orc.f64_to_bf16_bits(rng.standard_normal((6, 8)))
    x = orc.bf16_bits_to_f32(xb).astype(np.float64)
    ids, w = orc.route_topk(rng.standard_normal((6, 4)).astype(np.float32), 2, True,
                            np.ones(6, np.uint8))
    c, o, perm, inv = orc.dispatch(ids, 4, 4)
    xs = orc.permute_rows(x, perm[: o[-1]])
    inv_bad = inv.copy()
    inv_bad[:, -1] = -1                     # last expert's term dropped
    out = orc.combine(xs, inv_bad, w)
    assert not np.array_equal(orc.f64_to_bf16_bits(out), xb)


# ----------------------------------------------------------------- bf16 helpers
def test_bf16_rounding_matches_torch_cast(orc):
    rng = np.random.default_rng(15)
    x = (rng.standard_normal(100_000) * np.exp(rng.uniform(-20, 20, 100_000))).astype(np.float32)
    mine = orc.f64_to_bf16_bits(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)
    assert np.array_equal(orc.bf16_bits_to_f32(ref),
                          torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())


# ----------------------------------------------------------------- whole layer
def dense_layer(x_tokens, logits_tokens, k, wgu, wd):
    """Per-token definition with no dispatch: out_t = sum_j w_tj FFN_{e_tj}(x_t)."""
    out = np.zeros((len(x_tokens), x_tokens.shape[1]))
    for t in range(len(x_tokens)):
        lr = logits_tokens[t]
        sel = brute_force_topk(lr, k) if len(lr) <= 10 else list(
            np.lexsort((np.arange(len(lr)), -lr.astype(np.float64)))[:k])
        wts = scipy.special.softmax(lr.astype(np.float64)[sel])
        for j, e in enumerate(sel):
            out[t] += wts[j] * numpy_swiglu(x_tokens[t: t + 1], wgu[e], wd[e])[0]
    return out


@pytest.mark.parametrize("mode", [0, 1])
def test_layer_tiny_matches_dense_definition(orc, mode):
    from combine_dp_gather_gb300 import synth
    spec = synth.spec_tiny()
    xs = [t.numpy() for t in synth.hidden_states(spec)]
    lg = [t.numpy() for t in synth.router_logits(spec)]
    wgu, wd = synth.expert_weights(spec)
    wgu, wd = wgu.numpy(), wd.numpy()
    offs, rows = orc.dp_layout(spec.counts, mode)
    logits = orc.dp_gather(lg, spec.counts, offs, rows)
    res = orc.layer(xs, logits, spec.counts, mode, spec.k, True, wgu, wd, spec.E)
    dense = dense_layer(np.concatenate(xs), np.concatenate(lg), spec.k, wgu, wd)
    got = np.concatenate([o for o in res["outs"]])
    assert np.allclose(got, dense, rtol=1e-10, atol=1e-12)


def test_layer_with_replicated_map_equals_without(orc):
    """rank_invariant reading: replicas hold identical weights, so routing a
    logical expert to any of its replicas must not change the layer output."""
    from combine_dp_gather_gb300 import synth
    spec = synth.spec_tiny()
    xs = [t.numpy() for t in synth.hidden_states(spec)]
    lg = [t.numpy() for t in synth.router_logits(spec)]
    offs, rows = orc.dp_layout(spec.counts, 0)
    logits = orc.dp_gather(lg, spec.counts, offs, rows)
    wgu, wd = synth.expert_weights(spec)
    base = orc.layer(xs, logits, spec.counts, 0, spec.k, True, wgu.numpy(), wd.numpy(), spec.E)
    P = 12
    l2p, nrep, p2l = synth.trivial_map(spec.E, P)
    wgu_p, wd_p = wgu.numpy()[p2l], wd.numpy()[p2l]
    mapped = orc.layer(xs, logits, spec.counts, 0, spec.k, True, wgu_p, wd_p, spec.E, P=P,
                       l2p=l2p, nrep=nrep)
    assert (mapped["counts"][spec.E:] > 0).any()   # replicas really used
    for a, b in zip(base["outs"], mapped["outs"]):
        assert np.array_equal(a, b)


# ----------------------------------------------------------------- add + RMSNorm
def test_add_rmsnorm_matches_numpy_and_special_cases(orc):
    rng = np.random.default_rng(21)
    n, H = 7, 96
    h = rng.standard_normal((n, H)).astype(np.float32)
    r = rng.standard_normal((n, H)).astype(np.float32)
    g = (1 + 0.1 * rng.standard_normal(H)).astype(np.float32)
    r_new, y = orc.add_rmsnorm(h, r, g, 1e-6, False)
    s = h.astype(np.float32) + r.astype(np.float32)          # float32 add, no rounding
    assert np.array_equal(r_new, s)
    ref = s.astype(np.float64) / np.sqrt(np.mean(s.astype(np.float64) ** 2, axis=1,
                                                 keepdims=True) + 1e-6) * g
    assert np.allclose(y, ref, rtol=1e-13, atol=0)
    # unit gamma, zero hidden: the norm of a row has root-mean-square 1
    _, y1 = orc.add_rmsnorm(np.zeros_like(h), r, np.ones(H, np.float32), 0.0, False)
    assert np.allclose(np.sqrt(np.mean(y1 ** 2, axis=1)), 1.0, rtol=1e-13)
    # scale invariance: scaling the residual leaves the normed rows unchanged (eps = 0)
    _, y2 = orc.add_rmsnorm(np.zeros_like(h), 4 * r, np.ones(H, np.float32), 0.0, False)
    assert np.allclose(y1, y2, rtol=1e-13, atol=1e-15)


def test_add_rmsnorm_bf16_rounding_matches_torch(orc):
    rng = np.random.default_rng(22)
    h = torch.randn(5, 64, dtype=torch.float32).to(torch.bfloat16)
    r = torch.randn(5, 64, dtype=torch.float32).to(torch.bfloat16)
    r_new, _ = orc.add_rmsnorm(h.float().numpy(), r.float().numpy(), np.ones(64, np.float32),
                               1e-6, True)
    ref = (h.float() + r.float()).to(torch.bfloat16).float().numpy()   # fp32 add, RNE to bf16
    assert np.array_equal(r_new, ref)
    del rng


# ----------------------------------------------------------------- shared experts
def test_shared_experts_follow_routed_ids(orc):
    rng = np.random.default_rng(23)
    logits = rng.standard_normal((9, 8)).astype(np.float32)
    valid = np.ones(9, np.uint8)
    valid[4] = 0
    ids, w = orc.route_topk(logits, 2, True, valid, n_shared=2)
    ids0, w0 = orc.route_topk(logits, 2, True, valid)
    assert np.array_equal(ids[:, :2], ids0) and np.array_equal(w[:, :2], w0)
    assert ids[valid == 1][:, 2:].tolist() == [[8, 9]] * 8
    assert (w[valid == 1][:, 2:] == 1.0).all()
    assert (ids[4] == -1).all() and (w[4] == 0).all()


def test_layer_with_shared_expert_matches_dense_definition(orc):
    from combine_dp_gather_gb300 import synth
    spec = synth.spec_tiny()
    xs = [t.numpy() for t in synth.hidden_states(spec)]
    lg = [t.numpy() for t in synth.router_logits(spec)]
    rng = np.random.default_rng(24)
    wgu = (0.02 * rng.standard_normal((9, 2 * spec.I, spec.H))).astype(np.float32)
    wd = (0.02 * rng.standard_normal((9, spec.H, spec.I))).astype(np.float32)
    offs, rows = orc.dp_layout(spec.counts, 0)
    logits = orc.dp_gather(lg, spec.counts, offs, rows)
    res = orc.layer(xs, logits, spec.counts, 0, spec.k, True, wgu, wd, spec.E, n_shared=1)
    x = np.concatenate(xs)
    dense = dense_layer(x, np.concatenate(lg), spec.k, wgu[:8], wd[:8])
    dense += numpy_swiglu(x, wgu[8], wd[8])           # the shared expert, weight 1
    got = np.concatenate(res["outs"])
    assert np.allclose(got, dense, rtol=1e-10, atol=1e-12)


# ----------------------------------------------------------------- FP8 path
# Independent e4m3 rounding: the values of the 127 non-negative finite codes come
# from torch's float8_e4m3fn decoding (a library routine), ascending with the code;
# a value goes to the nearest of them, ties to the even code, |x| >= 448 saturates.
_E4M3_POS = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def _nearest_e4m3(v):
    v = np.asarray(v, np.float64)
    a = np.minimum(np.abs(v), 448.0)
    idx = np.searchsorted(_E4M3_POS, a)
    lo = np.clip(idx - 1, 0, 126)
    hi = np.clip(idx, 0, 126)
    dlo, dhi = a - _E4M3_POS[lo], _E4M3_POS[hi] - a
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    return (pick | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)


def _scale_exp_by_search(amax):
    """Smallest integer e with amax <= 448 * 2**e, found by stepping (0 for amax 0)."""
    out = []
    for a in np.ravel(amax):
        if a == 0:
            out.append(0)
            continue
        e = 0
        while a > 448.0 * 2.0 ** e:
            e += 1
        while a <= 448.0 * 2.0 ** (e - 1):
            e -= 1
        out.append(max(-127, min(127, e)))
    return np.array(out, np.int64).reshape(np.shape(amax))


def test_e4m3_encode_matches_nearest_and_torch(orc):
    rng = np.random.default_rng(5)
    mags = (2.0 ** rng.uniform(-12, 9, 20000)).astype(np.float32).astype(np.float64)
    x = np.where(rng.random(20000) < 0.5, -mags, mags)
    mids = (_E4M3_POS[1:] + _E4M3_POS[:-1]) / 2          # every tie between neighbours
    x = np.concatenate([x, mids, -mids, _E4M3_POS, [0.0, -0.0, 447.875, 463.9921875, 464.0]])
    got = orc.e4m3_encode(x)
    assert (got == _nearest_e4m3(x)).all()
    ok = np.abs(x) <= 464.0                              # torch overflows to NaN above 464
    x32 = x[ok].astype(np.float32)
    assert (x32.astype(np.float64) == x[ok]).all()       # exact in float32
    via_torch = torch.from_numpy(x32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (got[ok] == via_torch).all()


def test_e4m3_saturation_and_decode(orc):
    assert orc.e4m3_encode(np.array([448.0, 500.0, 1e30, -1e30, -449.0])).tolist() == \
        [0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    assert orc.e4m3_encode(np.array([np.nan]))[0] & 0x7F == 0x7F
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    via_torch = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert (orc.e4m3_decode(codes) == via_torch).all()
    assert (orc.e4m3_encode(orc.e4m3_decode(codes)) == codes).all()   # round trip


def test_ue8m0_scale_rule(orc):
    rng = np.random.default_rng(6)
    amax = np.concatenate([2.0 ** rng.uniform(-40, 40, 5000), 448.0 * 2.0 ** np.arange(-20, 21),
                           [0.0, 448.0, 448.0000001, 224.0, 1.0]])
    e = orc.ue8m0_exp(amax).astype(np.int64)
    assert (e == _scale_exp_by_search(amax)).all()
    pos = amax > 0
    assert (amax[pos] <= 448.0 * 2.0 ** e[pos]).all()
    assert (amax[pos] > 448.0 * 2.0 ** (e[pos] - 1)).all()


def test_quant_groups_scales_codes_and_indexing(orc):
    rng = np.random.default_rng(7)
    n, K = 5, 512
    x = rng.standard_normal((n, K)) * (2.0 ** np.repeat(np.arange(K // 128) * 3, 128))[None, :]
    x[2, 128:256] = 0.0                                  # an all-zero group
    q, e = orc.quant_groups(x)
    amax = np.abs(x).reshape(n, K // 128, 128).max(-1)
    ee = _scale_exp_by_search(amax)
    assert (e.astype(np.int64) - 127 == ee).all()
    assert e[2, 1] == 127
    assert (np.diff(ee[[0, 1, 3, 4]], axis=1) >= 2).all()   # group g scaled by 8**g
    scaled = x / 2.0 ** np.repeat(ee, 128, axis=1)
    assert (q == _nearest_e4m3(scaled)).all()
    assert np.abs(orc.e4m3_decode(q)).max() <= 448.0
    # the largest element of each non-zero group lands in (224, 448]
    top = np.abs(orc.e4m3_decode(q)).reshape(n, K // 128, 128).max(-1)
    assert ((top > 224.0) | (amax == 0)).all()


def test_quant_blocks_indexing(orc):
    rng = np.random.default_rng(8)
    R, K = 256, 384
    bi = np.repeat(np.arange(R // 128), 128)[:, None]
    bj = np.repeat(np.arange(K // 128), 128)[None, :]
    w = rng.uniform(-1, 1, (R, K)) * 2.0 ** (3 * bi + bj)
    q, e = orc.quant_blocks(w)
    amax = np.abs(w).reshape(R // 128, 128, K // 128, 128).max(axis=(1, 3))
    ee = _scale_exp_by_search(amax)
    assert (e.astype(np.int64) - 127 == ee).all()
    assert (q == _nearest_e4m3(w / 2.0 ** ee[bi[:, 0]][:, bj[0]])).all()


def _deq_groups(q, e):
    return _E4M3_SIGNED(q) * 2.0 ** np.repeat(e.astype(np.int64) - 127, 128, axis=1)


def _deq_blocks(q, e):
    s = 2.0 ** (e.astype(np.int64) - 127)
    return _E4M3_SIGNED(q) * np.repeat(np.repeat(s, 128, axis=0), 128, axis=1)


def _E4M3_SIGNED(q):
    return torch.from_numpy(np.ascontiguousarray(q)).view(torch.float8_e4m3fn).double().numpy()


def _fp8_ffn_numpy(xq, xe, wguq, wgue, wdq, wde, up_block_shift=True):
    """Dense numpy evaluation on dequantised operands; h re-quantised per token in
    groups of 128 with the independent rounding above.  up_block_shift=False is a
    mutant that reads the up rows' scales from the gate rows' blocks."""
    I = wdq.shape[1]
    wgu = _deq_blocks(wguq, wgue)
    if not up_block_shift:
        wgu[I:] = _E4M3_SIGNED(wguq[I:]) * np.repeat(np.repeat(
            2.0 ** (wgue[: I // 128].astype(np.int64) - 127), 128, axis=0), 128, axis=1)
    x = _deq_groups(xq, xe)
    g, u = x @ wgu[:I].T, x @ wgu[I:].T
    h = g / (1.0 + np.exp(-g)) * u
    he = _scale_exp_by_search(np.abs(h).reshape(len(h), I // 128, 128).max(-1))
    hq = _nearest_e4m3(h / 2.0 ** np.repeat(he, 128, axis=1))
    return _deq_groups(hq, (he + 127).astype(np.uint8)) @ _deq_blocks(wdq, wde).T


def test_ffn_fp8_matches_numpy_on_dequantised_operands(orc):
    rng = np.random.default_rng(9)
    n, H, I = 4, 256, 256
    x = rng.standard_normal((n, H))
    # every weight block gets its own magnitude, gate and up blocks differ
    wgu = rng.standard_normal((2 * I, H)) * 0.05 * \
        2.0 ** rng.integers(-3, 4, (2 * I // 128, H // 128)).repeat(128, 0).repeat(128, 1)
    wd = rng.standard_normal((H, I)) * 0.05 * \
        2.0 ** rng.integers(-3, 4, (H // 128, I // 128)).repeat(128, 0).repeat(128, 1)
    xq, xe = orc.quant_groups(x)
    wguq, wgue = orc.quant_blocks(wgu)
    wdq, wde = orc.quant_blocks(wd)
    y = orc.expert_ffn_fp8(xq, xe, wguq, wgue, wdq, wde)
    ref = _fp8_ffn_numpy(xq, xe, wguq, wgue, wdq, wde)
    np.testing.assert_allclose(y, ref, rtol=1e-9, atol=1e-12)
    mutant = _fp8_ffn_numpy(xq, xe, wguq, wgue, wdq, wde, up_block_shift=False)
    assert not np.allclose(y, mutant, rtol=1e-3, atol=1e-6)
    # FP8 stays close to the unquantised FFN (3 mantissa bits: a few % error)
    dense = orc.expert_ffn(x.astype(np.float32), wgu.astype(np.float32), wd.astype(np.float32))
    rel = np.linalg.norm(y - dense) / np.linalg.norm(dense)
    assert rel < 0.1, rel


def test_grouped_ffn_fp8_runs_each_slot_through_its_own_expert(orc):
    """FP8 grouped FFN: every slot against the dense numpy evaluation on its own
    dequantised operands; rows outside the slot range stay NaN."""
    rng = np.random.default_rng(22)
    H, I = 256, 128
    counts = [2, 3, 0, 1]
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    xq, xe = orc.quant_groups(rng.standard_normal((int(offsets[-1]), H)))
    ws = [(*orc.quant_blocks(0.05 * rng.standard_normal((2 * I, H))),
           *orc.quant_blocks(0.05 * rng.standard_normal((H, I)))) for _ in counts]
    ys = orc.grouped_ffn_fp8(xq, xe, offsets, lambda s: ws[s], 0, 3)
    for s in range(4):
        a, b = int(offsets[s]), int(offsets[s + 1])
        if s < 3 and b > a:
            ref = _fp8_ffn_numpy(xq[a:b], xe[a:b], *ws[s])
            np.testing.assert_allclose(ys[a:b], ref, rtol=1e-9, atol=1e-12)
        elif b > a:
            assert np.isnan(ys[a:b]).all()


# ----------------------------------------------------------------- router GEMM
def test_router_logits_match_numpy_and_feed_topk(orc):
    rng = np.random.default_rng(10)
    x = rng.standard_normal((7, 96)).astype(np.float32)
    w = rng.standard_normal((12, 96)).astype(np.float32)
    lg = orc.router_logits(x, w)
    np.testing.assert_allclose(lg, x.astype(np.float64) @ w.astype(np.float64).T, rtol=1e-12,
                               atol=1e-12)
    # a one-hot gate row selects its expert: logits = x . w_e, so w_e = x's own row wins
    w2 = np.zeros((5, 96), np.float32)
    w2[3] = x[0]
    ids, _ = orc.route_topk(orc.router_logits(x[:1], w2), 1, True, np.ones(1, np.uint8))
    assert ids.tolist() == [[3]]


def test_router_logits_bias(orc):
    """The optional per-expert bias is added once to every row's logits."""
    rng = np.random.default_rng(11)
    x = rng.standard_normal((6, 40)).astype(np.float32)
    w = rng.standard_normal((9, 40)).astype(np.float32)
    b = rng.standard_normal(9).astype(np.float32)
    lg = orc.router_logits(x, w, b)
    np.testing.assert_allclose(lg, x.astype(np.float64) @ w.astype(np.float64).T
                               + b.astype(np.float64)[None, :], rtol=1e-12, atol=1e-12)
    # without a bias it is the plain gate
    np.testing.assert_array_equal(orc.router_logits(x, w, None), orc.router_logits(x, w))
    # a zero gate returns the bias itself in every row, exactly
    z = orc.router_logits(x, np.zeros_like(w), b)
    np.testing.assert_array_equal(z, np.tile(b.astype(np.float64), (6, 1)))
    # a bias that lifts expert 2 above expert 3 moves the top-1 there: the gate's row
    # for expert 3 is the token itself (x . x > 0), expert 2's row is zero
    w3 = np.zeros((5, 40), np.float32)
    w3[3] = x[0]
    gap = float(np.dot(x[0].astype(np.float64), x[0].astype(np.float64)))
    b3 = np.zeros(5, np.float32)
    b3[2] = np.float32(gap + 1.0)
    one = np.ones(1, np.uint8)
    assert orc.route_topk(orc.router_logits(x[:1], w3), 1, True, one)[0].tolist() == [[3]]
    assert orc.route_topk(orc.router_logits(x[:1], w3, b3), 1, True, one)[0].tolist() == [[2]]
