"""Plain CPU oracle of the MoE layer between DP attention and expert parallelism.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product library never loads it and shares no code with it.

The arithmetic lives in ``moe_oracle.c`` (plain C, double precision, every
reduction in index order); this module compiles it with gcc, loads it with
ctypes and converts numpy arrays.  bf16 tensors arrive as their uint16 bit
patterns and are widened exactly to float32 here.

Parity status per function (pins in ``tests/test_oracle_pins.py``):
  dp_layout, dp_padding_mode, dp_gather, dp_scatter ..... pinned
  route_topk ............................................ pinned
  dispatch, permute_rows ................................ pinned
  expert_ffn / grouped_ffn .............................. pinned
  combine ............................................... pinned
  add_rmsnorm ........................................... pinned
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "liborc.so")
_lock = threading.Lock()
_lib = None

PAD_SUM, PAD_MAX, PAD_STATIC = 0, 1, 2
_STATUS = {0: "ok", 1: "invalid argument", 2: "capacity exceeded", 3: "static bound exceeded",
           4: "invalid device input"}


class OracleError(RuntimeError):
    def __init__(self, code: int):
        super().__init__(f"oracle status {code}: {_STATUS.get(code, '?')}")
        self.code = code


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into liborc.so (gcc, no fast-math, no FMA contraction)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int32, ctypes.c_int64
        sig = {
            "orc_dp_layout": (ctypes.c_int, [P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, P, P]),
            "orc_dp_padding_mode": (ctypes.c_int, [P, ctypes.c_int, ctypes.c_int,
                                                   ctypes.c_int, ctypes.c_int]),
            "orc_valid_rows": (None, [P, P, ctypes.c_int, i64, P]),
            "orc_set_threads": (None, [ctypes.c_int]),
            "orc_dp_gather": (None, [P, P, P, ctypes.c_int, i64, i64, P]),
            "orc_dp_scatter": (None, [P, P, P, ctypes.c_int, i64, P]),
            "orc_route_topk": (ctypes.c_int, [P, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                              P, P, P]),
            "orc_route_topk_shared": (ctypes.c_int, [P, i64, ctypes.c_int, ctypes.c_int,
                                                     ctypes.c_int, ctypes.c_int, P, P, P]),
            "orc_dispatch": (ctypes.c_int, [P, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            P, P, ctypes.c_int, ctypes.c_int, i64, P, P, P, P]),
            "orc_permute_rows": (None, [P, P, i64, i64, P]),
            "orc_expert_ffn": (None, [P, i64, ctypes.c_int, ctypes.c_int, P, P, P]),
            "orc_combine": (None, [P, P, P, i64, ctypes.c_int, ctypes.c_int, P]),
            "orc_add_rmsnorm": (None, [P, P, P, i64, ctypes.c_int, ctypes.c_double,
                                       ctypes.c_int, P]),
            "orc_e4m3_encode_array": (None, [P, i64, P]),
            "orc_e4m3_decode_array": (None, [P, i64, P]),
            "orc_ue8m0_exp_array": (None, [P, i64, P]),
            "orc_quant_groups": (None, [P, i64, ctypes.c_int, P, P]),
            "orc_quant_blocks": (None, [P, i64, ctypes.c_int, P, P]),
            "orc_expert_ffn_fp8": (None, [P, P, i64, ctypes.c_int, ctypes.c_int, P, P, P, P,
                                          P]),
            "orc_router_logits": (None, [P, i64, ctypes.c_int, P, ctypes.c_int, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        del i32
        _lib = lib
        return lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- bf16 bits
def bf16_bits_to_f32(u16: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float32."""
    u16 = np.ascontiguousarray(u16).view(np.uint16)
    return (u16.astype(np.uint32) << 16).view(np.float32)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round real values to the nearest bf16 value, ties to even, returned as float64.

    bf16 keeps 8 significant bits: with x = m * 2**e, 0.5 <= |m| < 1, the
    result is rint(m * 2**8) * 2**(e - 8) (numpy's rint rounds half to even).
    Normal range only; the layer's values are far from bf16 overflow/underflow.
    """
    m, e = np.frexp(np.asarray(x, dtype=np.float64))
    return np.ldexp(np.rint(m * 256.0), e - 8)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    return (round_to_bf16(x).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


# ---------------------------------------------------------------- steps
def dp_layout(counts, mode: int, static_bound: int = 0, tokens_per_req: int = 1):
    lib = _load()
    counts = _c(counts, np.int32)
    offsets = np.zeros(len(counts) + 1, np.int32)
    rows = np.zeros(1, np.int64)
    st = lib.orc_dp_layout(_p(counts), len(counts), mode, static_bound, tokens_per_req,
                           _p(offsets), _p(rows))
    if st:
        raise OracleError(st)
    return offsets, int(rows[0])


def dp_padding_mode(counts, gather_width: int, is_extend_in_batch: bool,
                    max_len_with_idle: bool) -> int:
    counts = _c(counts, np.int32)
    return _load().orc_dp_padding_mode(_p(counts), len(counts), gather_width,
                                       int(is_extend_in_batch), int(max_len_with_idle))


def set_threads(n: int) -> None:
    """Threads of the oracle's parallel loops (OpenMP); n < 1 keeps the default."""
    _load().orc_set_threads(int(n))


def valid_rows(counts, offsets, rows: int) -> np.ndarray:
    counts, offsets = _c(counts, np.int32), _c(offsets, np.int32)
    out = np.zeros(rows, np.uint8)
    _load().orc_valid_rows(_p(counts), _p(offsets), len(counts), rows, _p(out))
    return out


def dp_gather(locals_, counts, offsets, rows: int) -> np.ndarray:
    """locals_: list of R arrays [c_r, ...] of one dtype; returns [rows, ...]."""
    counts, offsets = _c(counts, np.int32), _c(offsets, np.int32)
    arrs = [np.ascontiguousarray(a) for a in locals_]
    row_shape = arrs[0].shape[1:]
    dtype = arrs[0].dtype
    out = np.empty((rows,) + row_shape, dtype)
    row_bytes = int(np.prod(row_shape, dtype=np.int64)) * dtype.itemsize
    ptrs = (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])
    _load().orc_dp_gather(ctypes.cast(ptrs, ctypes.c_void_p), _p(counts), _p(offsets),
                          len(arrs), rows, row_bytes, _p(out))
    return out


def dp_scatter(global_arr, counts, offsets):
    counts, offsets = _c(counts, np.int32), _c(offsets, np.int32)
    g = np.ascontiguousarray(global_arr)
    outs = [np.empty((int(c),) + g.shape[1:], g.dtype) for c in counts]
    row_bytes = int(np.prod(g.shape[1:], dtype=np.int64)) * g.dtype.itemsize
    ptrs = (ctypes.c_void_p * len(outs))(*[o.ctypes.data for o in outs])
    _load().orc_dp_scatter(_p(g), _p(counts), _p(offsets), len(outs), row_bytes,
                           ctypes.cast(ptrs, ctypes.c_void_p))
    return outs


def route_topk(logits, k: int, renormalize: bool, valid, n_shared: int = 0):
    """Top-k routing; with n_shared > 0 every real row also lists the shared experts
    E .. E + n_shared - 1 (weight 1) after its k routed ids."""
    logits = _c(logits, np.float32)
    rows, E = logits.shape
    valid = _c(valid, np.uint8)
    ids = np.empty((rows, k + n_shared), np.int32)
    w = np.empty((rows, k + n_shared), np.float64)
    st = _load().orc_route_topk_shared(_p(logits), rows, E, k, int(renormalize), n_shared,
                                       _p(valid), _p(ids), _p(w))
    if st:
        raise OracleError(st)
    return ids, w


def dispatch_cap_bound(rows: int, k: int, P: int, align: int) -> int:
    return rows * k + P * (align - 1)


def dispatch(ids, E: int, P: int, l2p=None, nrep=None, align: int = 1, cap: int | None = None):
    ids = _c(ids, np.int32)
    rows, k = ids.shape
    if cap is None:
        cap = dispatch_cap_bound(rows, k, P, align)
    X = 0
    if l2p is not None:
        l2p = _c(l2p, np.int32)
        nrep = _c(nrep, np.int32)
        X = l2p.shape[1]
    counts = np.zeros(P, np.int32)
    offsets = np.zeros(P + 1, np.int32)
    perm = np.empty(cap, np.int32)
    inv = np.empty((rows, k), np.int32)
    st = _load().orc_dispatch(_p(ids), rows, k, E, P, _p(l2p), _p(nrep), X, align, cap,
                              _p(counts), _p(offsets), _p(perm), _p(inv))
    if st:
        raise OracleError(st)
    return counts, offsets, perm, inv


def permute_rows(xg, perm) -> np.ndarray:
    xg = np.ascontiguousarray(xg)
    perm = _c(perm, np.int32)
    out = np.empty((len(perm),) + xg.shape[1:], xg.dtype)
    row_bytes = int(np.prod(xg.shape[1:], dtype=np.int64)) * xg.dtype.itemsize
    _load().orc_permute_rows(_p(xg), _p(perm), len(perm), row_bytes, _p(out))
    return out


def expert_ffn(x, wgu, wd) -> np.ndarray:
    """SwiGLU FFN of one expert: x [n,H] f32, wgu [2I,H] f32, wd [H,I] f32 -> [n,H] f64."""
    x, wgu, wd = _c(x, np.float32), _c(wgu, np.float32), _c(wd, np.float32)
    n, H = x.shape
    I = wd.shape[1]
    assert wgu.shape == (2 * I, H) and wd.shape == (H, I)
    y = np.empty((n, H), np.float64)
    if n:
        _load().orc_expert_ffn(_p(x), n, H, I, _p(wgu), _p(wd), _p(y))
    return y


def grouped_ffn(xs, offsets, wgu, wd, slot_lo: int = 0, slot_hi: int | None = None):
    """Per slot s in [slot_lo, slot_hi): rows [offsets[s], offsets[s+1]) of xs through
    expert s.  wgu [P,2I,H], wd [P,H,I] (f32 arrays or callables slot -> array).
    Rows of other slots are NaN in the result."""
    xs = _c(xs, np.float32)
    P = len(offsets) - 1
    slot_hi = P if slot_hi is None else slot_hi
    ys = np.full(xs.shape, np.nan, np.float64)
    for s in range(slot_lo, slot_hi):
        a, b = int(offsets[s]), int(offsets[s + 1])
        if b > a:
            ws = wgu(s) if callable(wgu) else wgu[s]
            wds = wd(s) if callable(wd) else wd[s]
            ys[a:b] = expert_ffn(xs[a:b], ws, wds)
    return ys


def combine(ys, inv, w) -> np.ndarray:
    ys = _c(ys, np.float64)
    inv = _c(inv, np.int32)
    w = _c(w, np.float64)
    rows, k = inv.shape
    H = ys.shape[1]
    out = np.empty((rows, H), np.float64)
    _load().orc_combine(_p(ys), _p(inv), _p(w), rows, k, H, _p(out))
    return out


def add_rmsnorm(hidden, residual, gamma, eps: float, round_bf16: bool):
    """Residual add + RMSNorm of one replica's rows (float32 inputs; bf16 values widened).
    Returns (updated residual float32 [n, H], normed rows float64 [n, H])."""
    h = _c(hidden, np.float32)
    r = _c(residual, np.float32).copy()
    g = _c(gamma, np.float32)
    n, H = h.shape
    y = np.empty((n, H), np.float64)
    if n:
        _load().orc_add_rmsnorm(_p(h), _p(r), _p(g), n, H, float(eps), int(round_bf16), _p(y))
    return r, y


def layer(locals_f32, logits, counts, mode, k, renormalize, wgu, wd, E, P=None,
          l2p=None, nrep=None, align=1, static_bound=0, tokens_per_req=1, n_shared=0):
    """Whole layer, step by step: layout, gather, route, dispatch, FFN, combine,
    scatter.  locals_f32: per-replica float32 hidden states (bf16 already
    widened).  Returns a dict of every intermediate."""
    P = E + n_shared if P is None else P
    offsets, rows = dp_layout(counts, mode, static_bound, tokens_per_req)
    valid = valid_rows(counts, offsets, rows)
    xg = dp_gather(locals_f32, counts, offsets, rows)
    ids, w = route_topk(logits, k, renormalize, valid, n_shared)
    cnt, offs, perm, inv = dispatch(ids, E + n_shared, P, l2p, nrep, align)
    xs = permute_rows(xg, perm[: offs[-1]])
    ys = grouped_ffn(xs, offs, wgu, wd)
    yg = combine(ys, inv, w)
    outs = dp_scatter(yg, counts, offsets)
    return dict(offsets=offsets, rows=rows, valid=valid, xg=xg, ids=ids, w=w, counts=cnt,
                slot_offsets=offs, perm=perm, inv=inv, xs=xs, ys=ys, yg=yg, outs=outs)


# ---------------------------------------------------------------- FP8 path
def e4m3_encode(x) -> np.ndarray:
    """Real values -> e4m3 codes (uint8): nearest, ties to even, saturating at +-448."""
    x = _c(x, np.float64)
    out = np.empty(x.shape, np.uint8)
    if x.size:
        _load().orc_e4m3_encode_array(_p(x), x.size, _p(out))
    return out


def e4m3_decode(codes) -> np.ndarray:
    codes = _c(codes, np.uint8)
    out = np.empty(codes.shape, np.float64)
    if codes.size:
        _load().orc_e4m3_decode_array(_p(codes), codes.size, _p(out))
    return out


def ue8m0_exp(amax) -> np.ndarray:
    """Smallest e with amax <= 448 * 2**e (0 for amax == 0), clamped to [-127, 127]."""
    amax = _c(amax, np.float64)
    out = np.empty(amax.shape, np.int32)
    if amax.size:
        _load().orc_ue8m0_exp_array(_p(amax), amax.size, _p(out))
    return out


def quant_groups(x):
    """Per-token groups of 128 along the last axis: (codes [n, K] u8, scale bytes [n, K/128])."""
    x = _c(x, np.float64)
    n, K = x.shape
    assert K % 128 == 0
    q = np.empty((n, K), np.uint8)
    e = np.empty((n, K // 128), np.uint8)
    if n:
        _load().orc_quant_groups(_p(x), n, K, _p(q), _p(e))
    return q, e


def quant_blocks(w):
    """128 x 128 blocks of w [R, K]: (codes [R, K] u8, scale bytes [R/128, K/128])."""
    w = _c(w, np.float64)
    R, K = w.shape
    assert R % 128 == 0 and K % 128 == 0
    q = np.empty((R, K), np.uint8)
    e = np.empty((R // 128, K // 128), np.uint8)
    _load().orc_quant_blocks(_p(w), R, K, _p(q), _p(e))
    return q, e


def expert_ffn_fp8(xq, xe, wguq, wgue, wdq, wde) -> np.ndarray:
    """SwiGLU FFN of one expert on FP8 operands (codes + scale bytes) -> [n, H] f64."""
    xq, xe = _c(xq, np.uint8), _c(xe, np.uint8)
    wguq, wgue, wdq, wde = (_c(a, np.uint8) for a in (wguq, wgue, wdq, wde))
    n, H = xq.shape
    I = wdq.shape[1]
    assert wguq.shape == (2 * I, H) and wdq.shape == (H, I)
    assert xe.shape == (n, H // 128) and wgue.shape == (2 * I // 128, H // 128)
    assert wde.shape == (H // 128, I // 128)
    y = np.empty((n, H), np.float64)
    if n:
        _load().orc_expert_ffn_fp8(_p(xq), _p(xe), n, H, I, _p(wguq), _p(wgue), _p(wdq),
                                   _p(wde), _p(y))
    return y


def grouped_ffn_fp8(xq, xe, offsets, wq, slot_lo: int = 0, slot_hi: int | None = None):
    """Per slot s: rows [offsets[s], offsets[s+1]) of (xq, xe) through expert s;
    wq(s) -> (wguq, wgue, wdq, wde).  Rows of other slots are NaN."""
    P = len(offsets) - 1
    slot_hi = P if slot_hi is None else slot_hi
    ys = np.full(xq.shape, np.nan, np.float64)
    for s in range(slot_lo, slot_hi):
        a, b = int(offsets[s]), int(offsets[s + 1])
        if b > a:
            ys[a:b] = expert_ffn_fp8(xq[a:b], xe[a:b], *wq(s))
    return ys


# ---------------------------------------------------------------- router GEMM
def router_logits(x, w, bias=None) -> np.ndarray:
    """Gate projection: x [rows, H] f32, w [E, H] f32, optional bias [E] f32
    -> logits [rows, E] f64 (x . w^T, plus the bias)."""
    x, w = _c(x, np.float32), _c(w, np.float32)
    rows, H = x.shape
    E = w.shape[0]
    assert w.shape == (E, H)
    b = None
    if bias is not None:
        b = _c(bias, np.float32)
        assert b.shape == (E,)
    out = np.empty((rows, E), np.float64)
    if rows:
        _load().orc_router_logits(_p(x), rows, H, _p(w), E, None if b is None else _p(b),
                                  _p(out))
    return out
