"""C-ABI checks that need no GPU: the library builds and loads, exports every
symbol include/moe_dp.h declares, its host helpers agree with the oracle, and
every device entry point rejects invalid arguments before launching anything
(host-side fault injection)."""
import ctypes
import itertools
import os
import re

import numpy as np
import pytest

from conftest import ROOT, ints, read_golden

HEADER = os.path.join(ROOT, "include", "moe_dp.h")


@pytest.fixture(scope="module")
def md():
    from combine_dp_gather_gb300 import build, moe_dp
    build.build()
    moe_dp.lib()
    return moe_dp


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(
        r"^\s*(?:moe_status|int|int64_t|size_t|double|const char\*)\s+(moe_\w+)\s*\(", text, re.M)))


def test_header_declarations_are_exported(md):
    names = declared_symbols()
    assert len(names) >= 12
    lib = ctypes.CDLL(md.lib_path())
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(md.exported_symbols()) == names


@pytest.mark.parametrize("row", read_golden("dp_layout.txt"))
def test_layout_golden(md, row):
    counts, mode, B, tpr, offs, rows = row
    o, n = md.moe_dp_layout(ints(counts), {"sum": 0, "max": 1, "static": 2}[mode], int(B),
                            int(tpr))
    assert o == ints(offs) and n == int(rows)


@pytest.mark.parametrize("row", read_golden("dp_layout_errors.txt"))
def test_layout_errors_golden(md, row):
    counts, mode, B, tpr, err = row
    with pytest.raises(md.MoeError) as ei:
        md.moe_dp_layout(ints(counts), {"sum": 0, "max": 1, "static": 2}[mode], int(B), int(tpr))
    assert ei.value.code == {"bound": md.MOE_ERR_BOUND_EXCEEDED, "arg": md.MOE_ERR_INVALID_ARG}[err]


@pytest.mark.parametrize("row", read_golden("dp_padding_mode.txt"))
def test_padding_mode_golden(md, row):
    counts, width, ext, idle, mode = row
    assert md.moe_dp_padding_mode(ints(counts), int(width), bool(int(ext)), bool(int(idle))) == \
        {"sum": 0, "max": 1}[mode]


def test_layout_and_mode_agree_with_oracle_exhaustively(md, orc):
    for R in (1, 2, 3):
        for counts in itertools.product([0, 1, 3, 24, 25], repeat=R):
            counts = list(counts)
            for mode in (0, 1):
                assert md.moe_dp_layout(counts, mode)[0] == orc.dp_layout(counts, mode)[0].tolist()
            for B, tpr in ((24, 1), (6, 4)):
                try:
                    ref = orc.dp_layout(counts, 2, B, tpr)
                except orc.OracleError as e:
                    with pytest.raises(md.MoeError) as ei:
                        md.moe_dp_layout(counts, 2, B, tpr)
                    assert ei.value.code == e.code
                else:
                    assert md.moe_dp_layout(counts, 2, B, tpr) == (ref[0].tolist(), ref[1])
            for w, ext, idle in itertools.product((1, R, 4), (0, 1), (0, 1)):
                assert md.moe_dp_padding_mode(counts, w, ext, idle) == \
                    orc.dp_padding_mode(counts, w, ext, idle)


@pytest.mark.parametrize("row", read_golden("balancedness.txt"))
def test_balancedness_golden(md, row):
    assert md.moe_balancedness(ints(row[0])) == pytest.approx(float(row[1]), rel=1e-15)


def test_balancedness_rejects_bad_loads(md):
    for bad in ([], [3, -1]):
        with pytest.raises(md.MoeError):
            md.moe_balancedness(bad)


def test_range_loads_and_logical_counts(md):
    counts = [3, 0, 5, 7, 1, 1, 0, 2, 9]
    # three ranges of three slots each: closed-form sums
    assert md.moe_range_loads(counts, 3) == [8, 9, 11]
    assert md.moe_range_loads(counts, 1) == [sum(counts)]
    assert md.moe_range_loads(counts, 9) == counts
    for bad_n in (2, 4, 0):            # 9 slots do not split into equal ranges of these
        with pytest.raises(md.MoeError):
            md.moe_range_loads(counts, bad_n)
    with pytest.raises(md.MoeError):
        md.moe_range_loads([1, -2], 1)
    # slots 0, 4 and 8 replicate logical expert 0; the rest map one to one
    p2l = [0, 1, 2, 3, 0, 4, 5, 6, 0]
    got = md.moe_logical_counts(counts, p2l, 7)
    assert got == [3 + 1 + 9, 0, 5, 7, 1, 0, 2]
    assert sum(got) == sum(counts)
    # the identity map returns the counts themselves
    assert md.moe_logical_counts(counts, list(range(9)), 9) == counts
    for bad_map in ([0] * 8 + [7], [0] * 8 + [-1]):
        with pytest.raises(md.MoeError):
            md.moe_logical_counts(counts, bad_map, 7)


def test_sizes(md):
    assert md.moe_dispatch_cap_bound(8192, 8, 256, 1) == 65536
    assert md.moe_dispatch_cap_bound(10, 2, 4, 128) == 20 + 4 * 127
    assert md.moe_dispatch_ws_bytes(8192, 8, 256) == 64 * 256 * 4
    assert md.moe_grouped_ffn_ws_bytes(100, 2048, __import__("torch").bfloat16) == 100 * 2048 * 2


# ---------------------------------------------------------------- fault injection
NULL = None
FAKE = ctypes.c_void_p(0x1000)      # aligned, never dereferenced: calls must fail first
MISAL = ctypes.c_void_p(0x1008)     # not 16-byte aligned


def _ptrs(*p):
    return ctypes.cast((ctypes.c_void_p * len(p))(*p), ctypes.c_void_p)


def test_gather_scatter_reject_bad_args(md):
    L = md.lib()
    two = _ptrs(0x2000, 0x3000)
    E_ARG, E_UNS = md.MOE_ERR_INVALID_ARG, md.MOE_ERR_UNSUPPORTED
    assert L.moe_dp_gather(two, NULL, FAKE, 2, 8, 64, 1, FAKE, NULL, NULL) == E_ARG
    assert L.moe_dp_gather(two, FAKE, FAKE, 0, 8, 64, 1, FAKE, NULL, NULL) == E_ARG
    assert L.moe_dp_gather(two, FAKE, FAKE, 300, 8, 64, 1, FAKE, NULL, NULL) == E_ARG
    assert L.moe_dp_gather(two, FAKE, FAKE, 2, -1, 64, 1, FAKE, NULL, NULL) == E_ARG
    assert L.moe_dp_gather(two, FAKE, FAKE, 2, 8, 7, 1, FAKE, NULL, NULL) == E_ARG  # 14 B rows
    assert L.moe_dp_gather(two, FAKE, FAKE, 2, 8, 64, 9, FAKE, NULL, NULL) == E_UNS
    assert L.moe_dp_gather(two, FAKE, FAKE, 2, 8, 64, 1, MISAL, NULL, NULL) == E_ARG
    assert L.moe_dp_gather(_ptrs(0x2008, 0x3000), FAKE, FAKE, 2, 8, 64, 1, FAKE, NULL, NULL) == E_ARG
    assert L.moe_dp_gather(NULL, FAKE, FAKE, 2, 8, 64, 1, FAKE, NULL, NULL) == E_ARG
    assert L.moe_dp_scatter(FAKE, FAKE, FAKE, 2, 8, 64, 1, NULL, NULL, NULL) == E_ARG
    assert L.moe_dp_scatter(FAKE, NULL, FAKE, 2, 8, 64, 1, two, NULL, NULL) == E_ARG


def test_gather2_and_combine_scatter_reject_bad_args(md):
    L = md.lib()
    two = _ptrs(0x2000, 0x3000)
    E_ARG, E_UNS = md.MOE_ERR_INVALID_ARG, md.MOE_ERR_UNSUPPORTED
    ok = (two, 64, 1, FAKE, two, 256, 0, FAKE, FAKE, FAKE, 2, 8, NULL, NULL)

    def g2(**kw):
        a = list(ok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return L.moe_dp_gather2(*a)
    assert g2(a0=NULL) == E_ARG                      # no replica table for tensor a
    assert g2(a4=NULL) == E_ARG                      # ... or for tensor b
    assert g2(a4=_ptrs(0x2008, 0x3000)) == E_ARG     # misaligned replica row
    assert g2(a1=7) == E_ARG                         # 14-byte rows
    assert g2(a6=9) == E_UNS                         # unknown dtype of b
    assert g2(a7=NULL) == E_ARG                      # no global buffer for b
    assert g2(a3=MISAL) == E_ARG
    assert g2(a8=NULL) == E_ARG                      # no counts
    assert g2(a10=0) == E_ARG and g2(a10=300) == E_ARG
    assert g2(a11=-1) == E_ARG
    assert g2(a11=0) == md.MOE_OK                    # nothing to move, no launch

    cs = (FAKE, FAKE, FAKE, 8, 2, 64, 1, 64, FAKE, FAKE, 2, two, NULL, NULL, NULL)

    def c(**kw):
        a = list(cs)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return L.moe_combine_scatter(*a)
    assert c(a4=0) == E_ARG                          # k = 0
    assert c(a5=4) == E_ARG                          # 8-byte rows
    assert c(a6=3) == E_UNS
    assert c(a1=NULL) == E_ARG and c(a2=NULL) == E_ARG
    assert c(a8=NULL) == E_ARG and c(a9=NULL) == E_ARG
    assert c(a10=0) == E_ARG and c(a10=300) == E_ARG
    assert c(a11=NULL) == E_ARG                      # no replica table
    assert c(a11=_ptrs(0x2008, 0x3000)) == E_ARG
    assert c(a12=MISAL) == E_ARG                     # misaligned optional global buffer
    assert c(a3=0) == md.MOE_OK


def test_grouped_ffn_combine_rejects_bad_args(md):
    """moe_grouped_ffn_combine refuses bad sizes, pointers and workspaces before any
    launch (and before looking for a device)."""
    L = md.lib()
    two = _ptrs(0x2000, 0x3000)
    E_ARG, E_UNS, E_CAP = md.MOE_ERR_INVALID_ARG, md.MOE_ERR_UNSUPPORTED, md.MOE_ERR_CAPACITY
    cap, rows, H, I, k = 64, 16, 256, 128, 4
    import torch
    ws = md.moe_grouped_ffn_combine_ws_bytes(cap, rows, H, I, torch.bfloat16)
    assert ws == cap * I * 2 + rows * (H // 256) * 4     # h, then one counter per 256 features
    assert md.moe_grouped_ffn_combine_ws_bytes(cap, rows, 384, I, torch.bfloat16) == 0
    assert md.moe_grouped_ffn_combine_ws_bytes(cap, rows, 96, I, torch.float32) == cap * I * 4
    ok = (FAKE, FAKE, 8, 0, 8, cap, FAKE, FAKE, H, I, 1, FAKE, FAKE, FAKE, FAKE, rows, k,
          FAKE, FAKE, 2, two, NULL, FAKE, ws, NULL, NULL)

    def f(**kw):
        a = list(ok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return L.moe_grouped_ffn_combine(*a)
    assert f(a2=0) == E_ARG                          # P = 0
    assert f(a3=5, a4=2) == E_ARG                    # slot_lo > slot_hi
    assert f(a4=9) == E_ARG                          # slot_hi > P
    assert f(a16=0) == E_ARG and f(a16=33) == E_ARG  # k outside 1..32
    assert f(a19=0) == E_ARG and f(a19=300) == E_ARG
    assert f(a8=4) == E_ARG                          # 8-byte rows
    assert f(a8=384) == E_UNS                        # bf16 tensor cores need H % 256 == 0
    assert f(a10=3) == E_UNS
    assert f(a12=NULL) == E_ARG                      # no perm
    assert f(a13=NULL) == E_ARG and f(a14=NULL) == E_ARG
    assert f(a17=NULL) == E_ARG and f(a18=NULL) == E_ARG
    assert f(a20=NULL) == E_ARG                      # no replica table
    assert f(a20=_ptrs(0x2008, 0x3000)) == E_ARG     # misaligned replica row
    assert f(a21=MISAL) == E_ARG                     # misaligned optional global buffer
    assert f(a22=NULL) == E_ARG                      # no workspace
    assert f(a23=ws - 1) == E_CAP                    # workspace one byte short
    assert f(a0=MISAL) == E_ARG
    assert f(a15=0) == md.MOE_OK                     # no rows: nothing to do


def test_grouped_ffn_split_rejects_bad_args(md):
    L = md.lib()
    E_ARG, E_UNS, E_CAP = md.MOE_ERR_INVALID_ARG, md.MOE_ERR_UNSUPPORTED, md.MOE_ERR_CAPACITY
    cap, H, I = 64, 256, 128
    ws = cap * I * 2
    ok = (FAKE, FAKE, 8, 0, 8, cap, FAKE, FAKE, H, I, 1, FAKE, FAKE, ws, 192, 32, NULL, NULL,
          NULL)

    def f(**kw):
        a = list(ok)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return L.moe_grouped_ffn_split(*a)
    assert f(a14=0) == E_ARG                         # hot_rows < 1
    assert f(a10=0) == E_UNS                         # float32: the split is bf16 only
    assert f(a8=384) == E_UNS                        # H % 256 != 0
    assert f(a2=0) == E_ARG and f(a4=9) == E_ARG
    assert f(a0=NULL) == E_ARG and f(a12=NULL) == E_ARG
    assert f(a13=ws - 1) == E_CAP
    assert f(a11=MISAL) == E_ARG
    assert f(a5=0) == md.MOE_OK                      # nothing to compute


def test_routing_gather_bindings_check_output_shapes(md):
    """The bindings refuse ids / w / gathered-logit tensors the kernels would write past."""
    import torch
    xs = [torch.zeros(3, 64, dtype=torch.bfloat16), torch.zeros(0, 64, dtype=torch.bfloat16)]
    ls = [torch.zeros(3, 32), torch.zeros(0, 32)]
    out = torch.zeros(3, 64, dtype=torch.bfloat16)
    good_ids, good_w = torch.zeros(3, 4, dtype=torch.int32), torch.zeros(3, 4)
    bad = [(torch.zeros(3, 3, dtype=torch.int32), good_w, None),      # too few columns
           (good_ids, torch.zeros(2, 4), None),                       # too few rows
           (torch.zeros(3, 4, dtype=torch.int64), good_w, None),      # wrong dtype
           (good_ids, good_w, torch.zeros(3, 16))]                    # logits narrower than E
    for ids, w, lg in bad:
        with pytest.raises(md.MoeError):
            md.moe_dp_gather_route(xs, ls, None, None, out, 4, True, ids, w, lg)
        with pytest.raises(md.MoeError):
            md.moe_dp_gather_add_rmsnorm_route(xs, xs, torch.zeros(64), 1e-6, ls, None, None,
                                               out, 4, True, ids, w, lg)


def test_gather_route_rejects_bad_args(md):
    L = md.lib()
    two = _ptrs(0x2000, 0x3000)
    E_ARG, E_UNS = md.MOE_ERR_INVALID_ARG, md.MOE_ERR_UNSUPPORTED

    def call(**kw):
        a = dict(lx=two, H=64, dt=1, gx=FAKE, ll=two, E=256, gl=NULL, k=8, rn=1, ns=0,
                 cnt=FAKE, off=FAKE, R=2, rows=8, ids=FAKE, w=FAKE)
        a.update(kw)
        return L.moe_dp_gather_route(a["lx"], a["H"], a["dt"], a["gx"], a["ll"], a["E"],
                                     a["gl"], a["k"], a["rn"], a["ns"], a["cnt"], a["off"],
                                     a["R"], a["rows"], a["ids"], a["w"], NULL, NULL)

    assert call(k=0) == E_ARG
    assert call(k=300) == E_ARG                          # k > E
    assert call(E=2000) == E_ARG                         # E > MOE_MAX_EXPERTS
    assert call(ns=-1) == E_ARG
    assert call(k=30, ns=3) == E_ARG                     # k + n_shared > MOE_MAX_TOPK
    assert call(ll=NULL) == E_ARG
    assert call(ids=NULL) == E_ARG
    assert call(w=NULL) == E_ARG
    assert call(ll=_ptrs(0x2000, 0x3002)) == E_ARG      # logits not float-aligned
    assert call(gl=MISAL) == E_ARG                       # misaligned gathered logits
    assert call(E=30, gl=FAKE) == E_ARG                  # 120-byte rows cannot be gathered
    assert call(gx=MISAL) == E_ARG
    assert call(H=3) == E_ARG                            # 6-byte rows
    assert call(dt=7) == E_UNS
    assert call(rows=0) == md.MOE_OK                     # nothing to do


def test_gather_add_rmsnorm_route_rejects_bad_args(md):
    L = md.lib()
    two = _ptrs(0x2000, 0x3000)
    E_ARG = md.MOE_ERR_INVALID_ARG
    f = ctypes.c_float

    def call(**kw):
        a = dict(gm=FAKE, eps=f(1e-6), ll=two, E=256, gl=NULL, k=8, rn=1, ns=0, ids=FAKE,
                 w=FAKE, rows=8, H=64, dt=1, gx=FAKE)
        a.update(kw)
        return L.moe_dp_gather_add_rmsnorm_route(two, two, a["gm"], a["eps"], a["ll"], a["E"],
                                                 a["gl"], a["k"], a["rn"], a["ns"], a["ids"],
                                                 a["w"], FAKE, FAKE, 2, a["rows"], a["H"],
                                                 a["dt"], a["gx"], NULL, NULL)

    assert call(gm=NULL) == E_ARG                        # no gamma
    assert call(eps=f(-1.0)) == E_ARG
    assert call(k=0) == E_ARG
    assert call(k=30, ns=3) == E_ARG                     # k + n_shared > MOE_MAX_TOPK
    assert call(ll=NULL) == E_ARG
    assert call(ids=NULL) == E_ARG
    assert call(ll=_ptrs(0x2000, 0x3002)) == E_ARG      # logits not float-aligned
    assert call(E=30, gl=FAKE) == E_ARG                  # 120-byte rows cannot be gathered
    assert call(H=16384) == md.MOE_ERR_UNSUPPORTED       # 32 KB rows
    assert call(rows=0) == md.MOE_OK


def test_gather_add_rmsnorm_rejects_bad_args(md):
    L = md.lib()
    two = _ptrs(0x2000, 0x3000)
    E_ARG, E_UNS = md.MOE_ERR_INVALID_ARG, md.MOE_ERR_UNSUPPORTED
    f = ctypes.c_float
    assert L.moe_dp_gather_add_rmsnorm(two, two, NULL, f(1e-6), FAKE, FAKE, 2, 8, 64, 1, FAKE,
                                       NULL, NULL) == E_ARG               # no gamma
    assert L.moe_dp_gather_add_rmsnorm(two, two, FAKE, f(-1.0), FAKE, FAKE, 2, 8, 64, 1, FAKE,
                                       NULL, NULL) == E_ARG               # negative eps
    assert L.moe_dp_gather_add_rmsnorm(NULL, two, FAKE, f(1e-6), FAKE, FAKE, 2, 8, 64, 1, FAKE,
                                       NULL, NULL) == E_ARG
    assert L.moe_dp_gather_add_rmsnorm(two, two, FAKE, f(1e-6), FAKE, FAKE, 2, 8, 16384, 1,
                                       FAKE, NULL, NULL) == E_UNS          # 32 KB rows
    assert L.moe_dp_gather_add_rmsnorm(two, two, MISAL, f(1e-6), FAKE, FAKE, 2, 8, 64, 1, FAKE,
                                       NULL, NULL) == E_ARG
    g2 = L.moe_dp_gather_add_rmsnorm2
    # the side plane: rows of whole 16-byte vectors, aligned pointers, a known dtype
    assert g2(two, two, FAKE, f(1e-6), two, 6, 0, FAKE, FAKE, FAKE, 2, 8, 64, 1, FAKE, NULL,
              NULL) == E_ARG                                              # 24-byte rows
    assert g2(two, two, FAKE, f(1e-6), _ptrs(0x2000, 0x3008), 8, 0, FAKE, FAKE, FAKE, 2, 8, 64,
              1, FAKE, NULL, NULL) == E_ARG                               # misaligned replica
    assert g2(two, two, FAKE, f(1e-6), NULL, 8, 0, FAKE, FAKE, FAKE, 2, 8, 64, 1, FAKE, NULL,
              NULL) == E_ARG                                              # no pointer array
    assert g2(two, two, FAKE, f(1e-6), two, 8, 0, MISAL, FAKE, FAKE, 2, 8, 64, 1, FAKE, NULL,
              NULL) == E_ARG                                              # misaligned output
    assert g2(two, two, FAKE, f(1e-6), two, 8, 9, FAKE, FAKE, FAKE, 2, 8, 64, 1, FAKE, NULL,
              NULL) == E_UNS                                              # unknown dtype
    assert g2(two, two, NULL, f(1e-6), two, 8, 0, FAKE, FAKE, FAKE, 2, 8, 64, 1, FAKE, NULL,
              NULL) == E_ARG                                              # no gamma
    assert g2(two, two, FAKE, f(1e-6), two, 8, 0, FAKE, FAKE, FAKE, 2, 0, 64, 1, FAKE, NULL,
              NULL) == md.MOE_OK                                          # no rows: no-op


def test_route_rejects_bad_args(md):
    L = md.lib()
    E_ARG = md.MOE_ERR_INVALID_ARG
    ok = dict(rows=8, E=256, k=8)
    assert L.moe_route_topk(FAKE, 8, 256, 0, 1, FAKE, FAKE, 2, FAKE, FAKE, NULL, NULL) == E_ARG
    assert L.moe_route_topk(FAKE, 8, 4, 5, 1, FAKE, FAKE, 2, FAKE, FAKE, NULL, NULL) == E_ARG
    assert L.moe_route_topk(FAKE, 8, 2048, 8, 1, FAKE, FAKE, 2, FAKE, FAKE, NULL, NULL) == E_ARG
    assert L.moe_route_topk(FAKE, 8, 256, 33, 1, FAKE, FAKE, 2, FAKE, FAKE, NULL, NULL) == E_ARG
    assert L.moe_route_topk(NULL, 8, 256, 8, 1, FAKE, FAKE, 2, FAKE, FAKE, NULL, NULL) == E_ARG
    assert L.moe_route_topk(FAKE, 8, 256, 8, 1, FAKE, FAKE, 0, FAKE, FAKE, NULL, NULL) == E_ARG
    del ok


def test_dispatch_rejects_bad_args(md):
    L = md.lib()
    E_ARG, E_CAP = md.MOE_ERR_INVALID_ARG, md.MOE_ERR_CAPACITY

    def call(**kw):
        a = dict(g=FAKE, ids=FAKE, rows=16, k=2, H=64, dt=1, E=8, P=8, l2p=NULL, nrep=NULL, X=0,
                 align=1, cap=32, cnt=FAKE, off=FAKE, perm=FAKE, inv=FAKE, xs=FAKE, ws=FAKE,
                 wsb=1 << 20)
        a.update(kw)
        return L.moe_dispatch(a["g"], a["ids"], a["rows"], a["k"], a["H"], a["dt"], a["E"],
                              a["P"], a["l2p"], a["nrep"], a["X"], a["align"], a["cap"], a["cnt"],
                              a["off"], a["perm"], a["inv"], a["xs"], a["ws"], a["wsb"], NULL,
                              NULL)

    assert call(P=9) == E_ARG                  # P != E without a map
    assert call(l2p=FAKE) == E_ARG             # map without num_valid
    assert call(l2p=FAKE, nrep=FAKE, X=0, P=9) == E_ARG
    assert call(align=0) == E_ARG
    assert call(k=0) == E_ARG
    assert call(P=2000, E=2000) == E_ARG
    assert call(ids=NULL) == E_ARG
    assert call(xs=NULL) == E_ARG              # rows without a destination
    assert call(xs=MISAL) == E_ARG
    assert call(H=7) == E_ARG
    assert call(wsb=0) == E_CAP


def test_ffn_and_combine_reject_bad_args(md):
    L = md.lib()
    E_ARG, E_UNS, E_CAP = md.MOE_ERR_INVALID_ARG, md.MOE_ERR_UNSUPPORTED, md.MOE_ERR_CAPACITY

    def ffn(**kw):
        a = dict(xs=FAKE, off=FAKE, P=8, lo=0, hi=8, cap=64, wgu=FAKE, wd=FAKE, H=512, I=256, dt=1,
                 ys=FAKE, ws=FAKE, wsb=1 << 30)
        a.update(kw)
        return L.moe_grouped_ffn(a["xs"], a["off"], a["P"], a["lo"], a["hi"], a["cap"], a["wgu"],
                                 a["wd"], a["H"], a["I"], a["dt"], a["ys"], a["ws"], a["wsb"],
                                 NULL, NULL)

    assert ffn(hi=9) == E_ARG
    assert ffn(lo=5, hi=4) == E_ARG
    assert ffn(wsb=10) == E_CAP
    assert ffn(H=384) == E_UNS                 # bf16 path needs H % 256 == 0
    assert ffn(I=192) == E_UNS                 # and I % 128 == 0
    assert ffn(P=2000, hi=2000) == E_UNS
    assert ffn(dt=5) == E_UNS
    assert ffn(wgu=MISAL) == E_ARG
    assert ffn(off=NULL) == E_ARG
    assert L.moe_combine(FAKE, FAKE, FAKE, 8, 0, 64, 1, 64, FAKE, NULL, NULL) == E_ARG
    assert L.moe_combine(FAKE, FAKE, FAKE, 8, 2, 4, 1, 64, FAKE, NULL, NULL) == E_ARG
    assert L.moe_combine(FAKE, NULL, FAKE, 8, 2, 64, 1, 64, FAKE, NULL, NULL) == E_ARG
    assert L.moe_combine(FAKE, FAKE, FAKE, 8, 2, 64, 3, 64, FAKE, NULL, NULL) == E_UNS


def test_status_strings(md):
    for code in range(8):
        assert md.lib().moe_status_string(code).decode() != "unknown status"
    assert md.lib().moe_status_string(99).decode() == "unknown status"


def test_fp8_entries_reject_bad_args(md):
    L = md.lib()
    E_ARG, E_UNS, E_CAP = md.MOE_ERR_INVALID_ARG, md.MOE_ERR_UNSUPPORTED, md.MOE_ERR_CAPACITY
    assert L.moe_quantize_fp8_groups(FAKE, 4, 100, 1, FAKE, FAKE, NULL) == E_ARG   # K % 128
    assert L.moe_quantize_fp8_groups(FAKE, 4, 256, 7, FAKE, FAKE, NULL) == E_UNS   # dtype
    assert L.moe_quantize_fp8_groups(MISAL, 4, 256, 1, FAKE, FAKE, NULL) == E_ARG
    assert L.moe_quantize_fp8_groups(FAKE, 4, 256, 1, FAKE, NULL, NULL) == E_ARG
    assert L.moe_quantize_fp8_groups(NULL, 0, 256, 1, NULL, NULL, NULL) == md.MOE_OK
    assert L.moe_quantize_fp8_blocks(FAKE, 100, 256, 1, FAKE, FAKE, NULL) == E_ARG  # R % 128
    assert L.moe_quantize_fp8_blocks(FAKE, 128, 64, 1, FAKE, FAKE, NULL) == E_ARG
    assert L.moe_quantize_fp8_blocks(FAKE, 128, 256, 1, MISAL, FAKE, NULL) == E_ARG

    def disp(**kw):
        a = dict(g=FAKE, ids=FAKE, rows=16, k=2, H=256, dt=1, E=8, P=8, l2p=NULL, nrep=NULL,
                 X=0, align=1, cap=32, cnt=FAKE, off=FAKE, perm=FAKE, inv=FAKE, q=FAKE, s=FAKE,
                 ws=FAKE, wsb=1 << 20)
        a.update(kw)
        return L.moe_dispatch_fp8(a["g"], a["ids"], a["rows"], a["k"], a["H"], a["dt"], a["E"],
                                  a["P"], a["l2p"], a["nrep"], a["X"], a["align"], a["cap"],
                                  a["cnt"], a["off"], a["perm"], a["inv"], a["q"], a["s"],
                                  a["ws"], a["wsb"], NULL, NULL)

    assert disp(H=192) == E_ARG                # H % 128
    assert disp(q=NULL) == E_ARG
    assert disp(q=MISAL) == E_ARG
    assert disp(g=NULL) == E_ARG
    assert disp(dt=5) == E_UNS
    assert disp(P=9) == E_ARG                  # the index checks of moe_dispatch apply
    assert disp(wsb=0) == E_CAP

    def ffn(**kw):
        a = dict(xq=FAKE, xs=FAKE, off=FAKE, P=8, lo=0, hi=8, cap=64, gq=FAKE, gs=FAKE, dq=FAKE,
                 ds=FAKE, H=512, I=256, ys=FAKE, ws=FAKE, wsb=1 << 30)
        a.update(kw)
        return L.moe_grouped_ffn_fp8(a["xq"], a["xs"], a["off"], a["P"], a["lo"], a["hi"],
                                     a["cap"], a["gq"], a["gs"], a["dq"], a["ds"], a["H"], a["I"],
                                     a["ys"], a["ws"], a["wsb"], NULL, NULL)

    assert ffn(H=384) == E_ARG                 # H % 256
    assert ffn(I=192) == E_ARG                 # I % 128
    assert ffn(hi=9) == E_ARG
    assert ffn(gs=NULL) == E_ARG
    assert ffn(gq=MISAL) == E_ARG
    assert ffn(wsb=16) == E_CAP
    assert ffn(cap=0) == md.MOE_OK             # nothing to do
    assert L.moe_grouped_ffn_fp8_ws_bytes(64, 100) == 0
    # layout: h codes [cap, I], scale bytes [cap, I/128], h in fp32 [cap, I] (the pair
    # kernel's path; each from a 256-byte boundary), then the scheduler's
    # 3 + MOE_MAX_SLOTS int32 words, last
    up = lambda n: (n + 255) // 256 * 256
    for cap, I in [(64, 256), (1, 128), (1000, 2048), (65600, 2048)]:
        words = up(up(up(cap * I) + cap * (I // 128)) + 4 * cap * I)
        assert L.moe_grouped_ffn_fp8_ws_bytes(cap, I) == words + 4 * (3 + 1024)
        assert md.fp8_ffn_workspace(cap, I, "cpu").numel() == words + 4 * (3 + 1024)
    assert not md.fp8_ffn_workspace(64, 256, "cpu").any()      # zero-filled


def test_router_gemm_rejects_bad_args(md):
    L = md.lib()
    E_ARG = md.MOE_ERR_INVALID_ARG

    def call(**kw):
        a = dict(x=FAKE, wr=FAKE, b=NULL, rows=16, H=512, E=64, k=4, rn=1, ns=0, cnt=FAKE,
                 off=FAKE, R=2, ids=FAKE, w=FAKE, lg=NULL, ws=FAKE, wsb=1 << 30)
        a.update(kw)
        return L.moe_route_gemm_topk(a["x"], a["wr"], a["b"], a["rows"], a["H"], a["E"], a["k"],
                                     a["rn"], a["ns"], a["cnt"], a["off"], a["R"], a["ids"],
                                     a["w"], a["lg"], a["ws"], a["wsb"], NULL, NULL)

    assert call(E=48) == E_ARG                 # E a multiple of 32
    assert call(E=512) == E_ARG                # at most 256
    assert call(H=100) == E_ARG                # H a multiple of 64
    assert call(k=65) == E_ARG                 # k <= E
    assert call(k=30, ns=3) == E_ARG           # k + n_shared <= 32
    assert call(x=MISAL) == E_ARG
    assert call(lg=MISAL) == E_ARG
    assert call(wr=NULL) == E_ARG
    assert call(R=0) == E_ARG
    assert call(rows=0) == md.MOE_OK
    assert L.moe_route_gemm_ws_bytes(16, 512, 48, 4) == 0
