"""Python binding of libmoe_dp (C ABI in include/moe_dp.h).

Argument marshalling only: every function here forwards torch tensors' device
pointers, sizes and the current CUDA stream to the C entry point of the same
name and raises MoeError on a non-zero status.  No arithmetic of the layer
happens in Python, and nothing falls back to the CPU: if the shared library
is missing the call raises.

``MoeLayer`` strings the six device calls into one MoE layer step with
buffers allocated once (PyTorch is the allocator).
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import List, Optional, Sequence

import torch

from . import build as _build

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_CAPACITY, MOE_ERR_BOUND_EXCEEDED = 0, 1, 2, 3
MOE_ERR_DEVICE_INPUT, MOE_ERR_TIMEOUT, MOE_ERR_CUDA, MOE_ERR_UNSUPPORTED = 4, 5, 6, 7
MOE_PAD_SUM, MOE_PAD_MAX, MOE_PAD_STATIC = 0, 1, 2
MOE_F32, MOE_BF16 = 0, 1
MOE_DEV_BAD_EXPERT_ID, MOE_DEV_BAD_MAP, MOE_DEV_CAPACITY = 0x1, 0x2, 0x4
MOE_DEV_TIMEOUT, MOE_DEV_BAD_COUNTS, MOE_DEV_BAD_WORKSPACE = 0x8, 0x10, 0x20

_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t

_SIGS = {
    "moe_dp_layout": (_I, [_P, _I, _I, _I, _I, _P, _P]),
    "moe_dp_padding_mode": (_I, [_P, _I, _I, _I, _I]),
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_dispatch_cap_bound": (_I64, [_I64, _I, _I, _I]),
    "moe_balancedness": (ctypes.c_double, [_P, _I]),
    "moe_range_loads": (_I, [_P, _I, _I, _P]),
    "moe_logical_counts": (_I, [_P, _P, _I, _I, _P]),
    "moe_dispatch_ws_bytes": (_SZ, [_I64, _I, _I]),
    "moe_grouped_ffn_ws_bytes": (_SZ, [_I64, _I, _I]),
    "moe_dp_gather": (_I, [_P, _P, _P, _I, _I64, _I, _I, _P, _P, _P]),
    "moe_route_topk": (_I, [_P, _I64, _I, _I, _I, _P, _P, _I, _P, _P, _P, _P]),
    "moe_dispatch": (_I, [_P, _P, _I64, _I, _I, _I, _I, _I, _P, _P, _I, _I, _I64, _P, _P, _P,
                          _P, _P, _P, _SZ, _P, _P]),
    "moe_grouped_ffn": (_I, [_P, _P, _I, _I, _I, _I64, _P, _P, _I, _I, _I, _P, _P, _SZ, _P,
                             _P]),
    "moe_combine": (_I, [_P, _P, _P, _I64, _I, _I, _I, _I64, _P, _P, _P]),
    "moe_dp_scatter": (_I, [_P, _P, _P, _I, _I64, _I, _I, _P, _P, _P]),
    "moe_dp_gather2": (_I, [_P, _I, _I, _P, _P, _I, _I, _P, _P, _P, _I, _I64, _P, _P]),
    "moe_combine_scatter": (_I, [_P, _P, _P, _I64, _I, _I, _I, _I64, _P, _P, _I, _P, _P, _P,
                                 _P]),
    "moe_route_topk_shared": (_I, [_P, _I64, _I, _I, _I, _I, _P, _P, _I, _P, _P, _P, _P]),
    "moe_dp_gather_add_rmsnorm": (_I, [_P, _P, _P, ctypes.c_float, _P, _P, _I, _I64, _I, _I, _P,
                                       _P, _P]),
    "moe_dp_gather_route": (_I, [_P, _I, _I, _P, _P, _I, _P, _I, _I, _I, _P, _P, _I, _I64, _P,
                                 _P, _P, _P]),
    "moe_dp_gather_add_rmsnorm_route": (_I, [_P, _P, _P, ctypes.c_float, _P, _I, _P, _I, _I, _I,
                                             _P, _P, _P, _P, _I, _I64, _I, _I, _P, _P, _P]),
    "moe_dp_gather_add_rmsnorm2": (_I, [_P, _P, _P, ctypes.c_float, _P, _I, _I, _P, _P, _P, _I,
                                        _I64, _I, _I, _P, _P, _P]),
    "moe_dispatch_noalloc": (_I, [_P, _P, _I64, _I, _I, _I, _I, _I, _P, _P, _I, _I, _I64, _P,
                                  _P, _P, _P, _P, _P, _P]),
    "moe_quantize_fp8_groups": (_I, [_P, _I64, _I, _I, _P, _P, _P]),
    "moe_quantize_fp8_blocks": (_I, [_P, _I64, _I, _I, _P, _P, _P]),
    "moe_dispatch_fp8": (_I, [_P, _P, _I64, _I, _I, _I, _I, _I, _P, _P, _I, _I, _I64, _P, _P,
                              _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "moe_grouped_ffn_fp8_ws_bytes": (_SZ, [_I64, _I]),
    "moe_route_gemm_ws_bytes": (_SZ, [_I64, _I, _I, _I]),
    "moe_route_gemm_topk": (_I, [_P, _P, _P, _I64, _I, _I, _I, _I, _I, _P, _P, _I, _P, _P, _P,
                                 _P, _SZ, _P, _P]),
    "moe_grouped_ffn_fp8": (_I, [_P, _P, _P, _I, _I, _I, _I64, _P, _P, _P, _P, _I, _I, _P, _P,
                                 _SZ, _P, _P]),
    "moe_grouped_ffn_split": (_I, [_P, _P, _I, _I, _I, _I64, _P, _P, _I, _I, _I, _P, _P, _SZ,
                                   _I, _I, _P, _P, _P]),
    "moe_grouped_ffn_combine_ws_bytes": (_SZ, [_I64, _I64, _I, _I, _I]),
    "moe_grouped_ffn_combine_in_epilogue": (_I, [_I64, _I, _I]),
    "moe_grouped_ffn_combine": (_I, [_P, _P, _I, _I, _I, _I64, _P, _P, _I, _I, _I, _P, _P, _P, _P,
                                     _I64, _I, _P, _P, _I, _P, _P, _P, _SZ, _P, _P]),
}
MOE_NOALLOC_SCRATCH_BYTES = 256 * 1024


class MoeError(RuntimeError):
    def __init__(self, fn: str, code: int):
        name = lib().moe_status_string(code).decode() if _lib is not None else str(code)
        super().__init__(f"{fn} failed: status {code} ({name})")
        self.code = code


def lib_path() -> str:
    return _build.LIB


def lib():
    """Load libmoe_dp.so (built in-tree by combine_dp_gather_gb300.build)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_build.LIB):
                raise RuntimeError(
                    f"{_build.LIB} is missing: build it with "
                    "`python -m combine_dp_gather_gb300.build` (there is no CPU fallback)")
            handle = ctypes.CDLL(_build.LIB)
            for name, (res, args) in _SIGS.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
        return _lib


def exported_symbols() -> List[str]:
    return list(_SIGS)


def _check(fn: str, code: int):
    if code != MOE_OK:
        raise MoeError(fn, code)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return MOE_BF16
    if dt == torch.float32:
        return MOE_F32
    raise ValueError(f"unsupported dtype {dt}")


def _host_i32(values: Sequence[int]):
    arr = (ctypes.c_int32 * len(values))(*[int(v) for v in values])
    return arr


# ---------------------------------------------------------------- host helpers
def moe_dp_layout(counts: Sequence[int], mode: int, static_bound: int = 0,
                  tokens_per_req: int = 1):
    """Host layout: returns (offsets list of R+1 ints, rows)."""
    c = _host_i32(counts)
    offs = (ctypes.c_int32 * (len(counts) + 1))()
    rows = ctypes.c_int64(0)
    _check("moe_dp_layout", lib().moe_dp_layout(ctypes.cast(c, _P), len(counts), mode,
                                                 static_bound, tokens_per_req,
                                                 ctypes.cast(offs, _P), ctypes.byref(rows)))
    return list(offs), int(rows.value)


def moe_dp_padding_mode(counts: Sequence[int], gather_width: int, is_extend_in_batch: bool,
                        max_len_with_idle: bool) -> int:
    c = _host_i32(counts)
    m = lib().moe_dp_padding_mode(ctypes.cast(c, _P), len(counts), gather_width,
                                  int(is_extend_in_batch), int(max_len_with_idle))
    if m < 0:
        raise MoeError("moe_dp_padding_mode", MOE_ERR_INVALID_ARG)
    return m


def moe_dispatch_cap_bound(rows: int, k: int, P: int, align: int) -> int:
    return int(lib().moe_dispatch_cap_bound(rows, k, P, align))


def moe_dispatch_ws_bytes(rows: int, k: int, E: int) -> int:
    return int(lib().moe_dispatch_ws_bytes(rows, k, E))


def moe_grouped_ffn_ws_bytes(cap: int, I: int, dtype: torch.dtype) -> int:
    return int(lib().moe_grouped_ffn_ws_bytes(cap, I, dtype_code(dtype)))


def moe_balancedness(loads: Sequence[int]) -> float:
    """Balancedness of per-rank token loads (host helper of the C ABI)."""
    arr = (ctypes.c_int64 * len(loads))(*[int(v) for v in loads])
    v = float(lib().moe_balancedness(ctypes.cast(arr, _P), len(loads)))
    if v < 0:
        raise MoeError("moe_balancedness", MOE_ERR_INVALID_ARG)
    return v


def moe_range_loads(counts: Sequence[int], n_ranges: int) -> List[int]:
    """Token loads of n_ranges contiguous equal slot ranges (host helper of the C ABI)."""
    c = _host_i32(counts)
    out = (ctypes.c_int64 * n_ranges)()
    _check("moe_range_loads", lib().moe_range_loads(ctypes.cast(c, _P), len(counts), n_ranges,
                                                    ctypes.cast(out, _P)))
    return [int(v) for v in out]


def moe_logical_counts(counts_P: Sequence[int], p2l: Sequence[int], E: int) -> List[int]:
    """Tokens per logical expert from tokens per physical slot (host helper of the C ABI)."""
    if len(p2l) != len(counts_P):
        raise MoeError("moe_logical_counts", MOE_ERR_INVALID_ARG)
    c, m = _host_i32(counts_P), _host_i32(p2l)
    out = (ctypes.c_int64 * E)()
    _check("moe_logical_counts", lib().moe_logical_counts(ctypes.cast(c, _P), ctypes.cast(m, _P),
                                                          len(counts_P), E, ctypes.cast(out, _P)))
    return [int(v) for v in out]


# ---------------------------------------------------------------- device calls
def moe_dp_gather(local: Sequence[torch.Tensor], d_counts, d_offsets, out: torch.Tensor,
                  d_status=None, stream=None):
    R = len(local)
    ptrs = (ctypes.c_void_p * R)(*[t.data_ptr() if t.numel() else None for t in local])
    _check("moe_dp_gather", lib().moe_dp_gather(
        ctypes.cast(ptrs, _P), _ptr(d_counts), _ptr(d_offsets), R, out.shape[0], out.shape[1],
        dtype_code(out.dtype), _ptr(out), _ptr(d_status), _stream(stream)))


def moe_dp_gather2(local_a: Sequence[torch.Tensor], local_b: Sequence[torch.Tensor], d_counts,
                   d_offsets, out_a: torch.Tensor, out_b: torch.Tensor, d_status=None,
                   stream=None):
    """DP gather of two row tensors of the same replicas in one launch."""
    R = len(local_a)
    if len(local_b) != R or out_a.shape[0] != out_b.shape[0]:
        raise MoeError("moe_dp_gather2", MOE_ERR_INVALID_ARG)
    pa = (ctypes.c_void_p * R)(*[t.data_ptr() if t.numel() else None for t in local_a])
    pb = (ctypes.c_void_p * R)(*[t.data_ptr() if t.numel() else None for t in local_b])
    _check("moe_dp_gather2", lib().moe_dp_gather2(
        ctypes.cast(pa, _P), out_a.shape[1], dtype_code(out_a.dtype), _ptr(out_a),
        ctypes.cast(pb, _P), out_b.shape[1], dtype_code(out_b.dtype), _ptr(out_b),
        _ptr(d_counts), _ptr(d_offsets), R, out_a.shape[0], _ptr(d_status), _stream(stream)))


def _check_route_outputs(fn: str, rows: int, kk: int, ids, w, out_logits, E: int):
    """The kernels write ids / w [rows, kk] (and the gathered logits [rows, E]): refuse
    tensors of another shape or dtype before any launch."""
    ok = (tuple(ids.shape) == (rows, kk) and ids.dtype == torch.int32 and ids.is_contiguous()
          and tuple(w.shape) == (rows, kk) and w.dtype == torch.float32 and w.is_contiguous())
    if out_logits is not None:
        ok = ok and (tuple(out_logits.shape) == (rows, E) and out_logits.dtype == torch.float32
                     and out_logits.is_contiguous())
    if not ok:
        raise MoeError(fn, MOE_ERR_INVALID_ARG)


def moe_dp_gather_route(local_x: Sequence[torch.Tensor], local_logits: Sequence[torch.Tensor],
                        d_counts, d_offsets, out_x: torch.Tensor, k: int, renormalize: bool,
                        ids: torch.Tensor, w: torch.Tensor, out_logits=None, n_shared: int = 0,
                        d_status=None, stream=None):
    """DP gather of the hidden states and top-k routing of the gathered rows (from
    the replicas' float32 logits) in one launch; out_logits optionally receives the
    gathered logits."""
    R = len(local_x)
    if len(local_logits) != R:
        raise MoeError("moe_dp_gather_route", MOE_ERR_INVALID_ARG)
    E = int(local_logits[0].shape[1]) if local_logits[0].dim() == 2 else 0
    _check_route_outputs("moe_dp_gather_route", out_x.shape[0], k + n_shared, ids, w,
                         out_logits, E)
    px = (ctypes.c_void_p * R)(*[t.data_ptr() if t.numel() else None for t in local_x])
    pl = (ctypes.c_void_p * R)(*[t.data_ptr() if t.numel() else None for t in local_logits])
    _check("moe_dp_gather_route", lib().moe_dp_gather_route(
        ctypes.cast(px, _P), out_x.shape[1], dtype_code(out_x.dtype), _ptr(out_x),
        ctypes.cast(pl, _P), E, _ptr(out_logits), k, int(renormalize), n_shared,
        _ptr(d_counts), _ptr(d_offsets), R, out_x.shape[0], _ptr(ids), _ptr(w), _ptr(d_status),
        _stream(stream)))


def moe_dp_gather_add_rmsnorm(local_hidden: Sequence[torch.Tensor],
                              local_residual: Sequence[torch.Tensor], gamma: torch.Tensor,
                              eps: float, d_counts, d_offsets, out: torch.Tensor, d_status=None,
                              stream=None, local_b: Optional[Sequence[torch.Tensor]] = None,
                              out_b: Optional[torch.Tensor] = None):
    """Residual add (in place) + RMSNorm + DP gather of the normed rows; with
    local_b / out_b a second row tensor (the router logits) is gathered plainly in
    the same launch."""
    R = len(local_hidden)
    hp = (ctypes.c_void_p * R)(*[t.data_ptr() if t.numel() else None for t in local_hidden])
    rp = (ctypes.c_void_p * R)(*[t.data_ptr() if t.numel() else None for t in local_residual])
    if local_b is None:
        _check("moe_dp_gather_add_rmsnorm", lib().moe_dp_gather_add_rmsnorm(
            ctypes.cast(hp, _P), ctypes.cast(rp, _P), _ptr(gamma), float(eps), _ptr(d_counts),
            _ptr(d_offsets), R, out.shape[0], out.shape[1], dtype_code(out.dtype), _ptr(out),
            _ptr(d_status), _stream(stream)))
        return
    if out_b is None or len(local_b) != R or out_b.shape[0] != out.shape[0]:
        raise MoeError("moe_dp_gather_add_rmsnorm2", MOE_ERR_INVALID_ARG)
    bp = (ctypes.c_void_p * R)(*[t.data_ptr() if t.numel() else None for t in local_b])
    _check("moe_dp_gather_add_rmsnorm2", lib().moe_dp_gather_add_rmsnorm2(
        ctypes.cast(hp, _P), ctypes.cast(rp, _P), _ptr(gamma), float(eps), ctypes.cast(bp, _P),
        out_b.shape[1], dtype_code(out_b.dtype), _ptr(out_b), _ptr(d_counts), _ptr(d_offsets),
        R, out.shape[0], out.shape[1], dtype_code(out.dtype), _ptr(out), _ptr(d_status),
        _stream(stream)))


def moe_dp_gather_add_rmsnorm_route(local_hidden: Sequence[torch.Tensor],
                                    local_residual: Sequence[torch.Tensor], gamma: torch.Tensor,
                                    eps: float, local_logits: Sequence[torch.Tensor], d_counts,
                                    d_offsets, out: torch.Tensor, k: int, renormalize: bool,
                                    ids: torch.Tensor, w: torch.Tensor, out_logits=None,
                                    n_shared: int = 0, d_status=None, stream=None):
    """Residual add (in place) + RMSNorm + DP gather of the normed rows, with the top-k
    routing of every row from the replicas' float32 logits in the same launch."""
    R = len(local_hidden)
    if len(local_residual) != R or len(local_logits) != R:
        raise MoeError("moe_dp_gather_add_rmsnorm_route", MOE_ERR_INVALID_ARG)
    E = int(local_logits[0].shape[1]) if local_logits[0].dim() == 2 else 0
    _check_route_outputs("moe_dp_gather_add_rmsnorm_route", out.shape[0], k + n_shared, ids, w,
                         out_logits, E)
    hp = (ctypes.c_void_p * R)(*[t.data_ptr() if t.numel() else None for t in local_hidden])
    rp = (ctypes.c_void_p * R)(*[t.data_ptr() if t.numel() else None for t in local_residual])
    lp = (ctypes.c_void_p * R)(*[t.data_ptr() if t.numel() else None for t in local_logits])
    _check("moe_dp_gather_add_rmsnorm_route", lib().moe_dp_gather_add_rmsnorm_route(
        ctypes.cast(hp, _P), ctypes.cast(rp, _P), _ptr(gamma), float(eps), ctypes.cast(lp, _P), E,
        _ptr(out_logits), k, int(renormalize), n_shared, _ptr(ids), _ptr(w), _ptr(d_counts),
        _ptr(d_offsets), R, out.shape[0], out.shape[1], dtype_code(out.dtype), _ptr(out),
        _ptr(d_status), _stream(stream)))


def moe_route_topk(logits: torch.Tensor, k: int, renormalize: bool, d_counts, d_offsets,
                   ids: torch.Tensor, w: torch.Tensor, d_status=None, stream=None,
                   n_shared: int = 0):
    """Top-k routing; n_shared > 0 appends the shared experts (weight 1) to every
    real row (ids / w then have k + n_shared columns)."""
    rows, E = logits.shape
    if n_shared:
        _check("moe_route_topk_shared", lib().moe_route_topk_shared(
            _ptr(logits), rows, E, k, int(renormalize), n_shared, _ptr(d_counts),
            _ptr(d_offsets), d_counts.numel(), _ptr(ids), _ptr(w), _ptr(d_status),
            _stream(stream)))
        return
    _check("moe_route_topk", lib().moe_route_topk(
        _ptr(logits), rows, E, k, int(renormalize), _ptr(d_counts), _ptr(d_offsets),
        d_counts.numel(), _ptr(ids), _ptr(w), _ptr(d_status), _stream(stream)))


def moe_dispatch(x: Optional[torch.Tensor], ids: torch.Tensor, E: int, P: int, counts_P, offsets_P,
                 perm, inv, sorted_out: Optional[torch.Tensor], ws: torch.Tensor, l2p=None,
                 nrep=None, align: int = 1, d_status=None, stream=None):
    rows, k = ids.shape
    H = x.shape[1] if x is not None else 0
    dt = dtype_code(x.dtype) if x is not None else MOE_BF16
    X = l2p.shape[1] if l2p is not None else 0
    _check("moe_dispatch", lib().moe_dispatch(
        _ptr(x), _ptr(ids), rows, k, H, dt, E, P, _ptr(l2p), _ptr(nrep), X, align,
        perm.numel(), _ptr(counts_P), _ptr(offsets_P), _ptr(perm), _ptr(inv), _ptr(sorted_out),
        _ptr(ws), ws.numel() * ws.element_size(), _ptr(d_status), _stream(stream)))


def moe_dispatch_noalloc(x: Optional[torch.Tensor], ids: torch.Tensor, E: int, P: int,
                         counts_P, offsets_P, perm, inv, sorted_out: Optional[torch.Tensor],
                         l2p=None, nrep=None, align: int = 1, d_status=None, stream=None):
    """moe_dispatch without a workspace argument: the library's fixed device
    scratch holds the histograms (for callers that cannot allocate)."""
    rows, k = ids.shape
    H = x.shape[1] if x is not None else 0
    dt = dtype_code(x.dtype) if x is not None else MOE_BF16
    # the kernels write these through plain pointers: refuse other shapes before any launch
    i32 = lambda t, shape: (t is not None and tuple(t.shape) == shape  # noqa: E731
                            and t.dtype == torch.int32 and t.is_contiguous())
    ok = (i32(counts_P, (P,)) and i32(offsets_P, (P + 1,)) and i32(inv, (rows, k))
          and perm is not None and perm.dtype == torch.int32 and perm.dim() == 1
          and perm.is_contiguous())
    if sorted_out is not None:
        ok = ok and (x is not None and sorted_out.dtype == x.dtype and sorted_out.dim() == 2
                     and sorted_out.shape[0] == perm.numel() and sorted_out.shape[1] == H
                     and sorted_out.is_contiguous())
    if not ok:
        raise MoeError("moe_dispatch_noalloc", MOE_ERR_INVALID_ARG)
    X = l2p.shape[1] if l2p is not None else 0
    _check("moe_dispatch_noalloc", lib().moe_dispatch_noalloc(
        _ptr(x), _ptr(ids), rows, k, H, dt, E, P, _ptr(l2p), _ptr(nrep), X, align,
        perm.numel(), _ptr(counts_P), _ptr(offsets_P), _ptr(perm), _ptr(inv), _ptr(sorted_out),
        _ptr(d_status), _stream(stream)))


def moe_route_gemm_ws_bytes(rows: int, H: int, E: int, k: int) -> int:
    return int(lib().moe_route_gemm_ws_bytes(rows, H, E, k))


def moe_route_gemm_topk(x: torch.Tensor, w_router: torch.Tensor, k: int, renormalize: bool,
                        d_counts, d_offsets, ids: torch.Tensor, w: torch.Tensor,
                        ws: Optional[torch.Tensor] = None, logits: Optional[torch.Tensor] = None,
                        d_status=None, stream=None, n_shared: int = 0,
                        bias: Optional[torch.Tensor] = None):
    """Gate GEMM (x [rows, H] . w_router [E, H]^T + bias, bf16) fused ahead of top-k."""
    rows, H = x.shape
    E = w_router.shape[0]
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check("moe_route_gemm_topk", lib().moe_route_gemm_topk(
        _ptr(x), _ptr(w_router), _ptr(bias), rows, H, E, k, int(renormalize), n_shared,
        _ptr(d_counts),
        _ptr(d_offsets), d_counts.numel(), _ptr(ids), _ptr(w), _ptr(logits), _ptr(ws), nbytes,
        _ptr(d_status), _stream(stream)))


# ---------------------------------------------------------------- FP8 path
def moe_quantize_fp8_groups(x: torch.Tensor, q: torch.Tensor, scales: torch.Tensor, stream=None):
    """Per-token groups of 128: x [n, K] bf16/f32 -> q uint8 [n, K], scales uint8 [n, K/128]."""
    n, K = x.shape
    _check("moe_quantize_fp8_groups", lib().moe_quantize_fp8_groups(
        _ptr(x), n, K, dtype_code(x.dtype), _ptr(q), _ptr(scales), _stream(stream)))


def moe_quantize_fp8_blocks(w: torch.Tensor, q: torch.Tensor, scales: torch.Tensor, stream=None):
    """128 x 128 blocks: w [R, K] -> q uint8 [R, K], scales uint8 [R/128, K/128]."""
    R, K = w.shape
    _check("moe_quantize_fp8_blocks", lib().moe_quantize_fp8_blocks(
        _ptr(w), R, K, dtype_code(w.dtype), _ptr(q), _ptr(scales), _stream(stream)))


def quantize_expert_weights_fp8(w_gate_up: torch.Tensor, w_down: torch.Tensor, stream=None):
    """[P, 2I, H] and [P, H, I] expert weights -> (gate_up codes, gate_up scales [P, 2I/128,
    H/128], down codes, down scales [P, H/128, I/128]), all uint8 on the weights' device."""
    P, I2, H = w_gate_up.shape
    I = w_down.shape[2]
    u8 = dict(dtype=torch.uint8, device=w_gate_up.device)
    guq = torch.empty(P, I2, H, **u8)
    gus = torch.empty(P, I2 // 128, H // 128, **u8)
    dq = torch.empty(P, H, I, **u8)
    ds = torch.empty(P, H // 128, I // 128, **u8)
    moe_quantize_fp8_blocks(w_gate_up.reshape(P * I2, H), guq.view(P * I2, H),
                            gus.view(P * I2 // 128, H // 128), stream)
    moe_quantize_fp8_blocks(w_down.reshape(P * H, I), dq.view(P * H, I),
                            ds.view(P * H // 128, I // 128), stream)
    return guq, gus, dq, ds


def moe_dispatch_fp8(x: torch.Tensor, ids: torch.Tensor, E: int, P: int, counts_P, offsets_P,
                     perm, inv, sorted_q: torch.Tensor, sorted_scales: torch.Tensor,
                     ws: torch.Tensor, l2p=None, nrep=None, align: int = 1, d_status=None,
                     stream=None):
    rows, k = ids.shape
    H = x.shape[1]
    X = l2p.shape[1] if l2p is not None else 0
    _check("moe_dispatch_fp8", lib().moe_dispatch_fp8(
        _ptr(x), _ptr(ids), rows, k, H, dtype_code(x.dtype), E, P, _ptr(l2p), _ptr(nrep), X,
        align, perm.numel(), _ptr(counts_P), _ptr(offsets_P), _ptr(perm), _ptr(inv),
        _ptr(sorted_q), _ptr(sorted_scales), _ptr(ws), ws.numel() * ws.element_size(),
        _ptr(d_status), _stream(stream)))


def moe_grouped_ffn_fp8_ws_bytes(cap: int, I: int) -> int:
    return int(lib().moe_grouped_ffn_fp8_ws_bytes(cap, I))


def fp8_ffn_workspace(cap: int, I: int, device="cuda") -> torch.Tensor:
    """A workspace for moe_grouped_ffn_fp8: zero-filled, as its scheduler words (the
    last bytes) must be zero before the first call; every call leaves them zero."""
    n = moe_grouped_ffn_fp8_ws_bytes(cap, I)
    if n == 0:
        raise MoeError("moe_grouped_ffn_fp8_ws_bytes", MOE_ERR_INVALID_ARG)
    return torch.zeros(n, device=device, dtype=torch.uint8)


def moe_grouped_ffn_fp8(xq: torch.Tensor, x_scales: torch.Tensor, offsets_P: torch.Tensor,
                        w_fp8, ys: torch.Tensor, ws: torch.Tensor, slot_lo: int = 0,
                        slot_hi: Optional[int] = None, d_status=None, stream=None):
    """w_fp8 = quantize_expert_weights_fp8(...); ys bf16 [cap, H] out; ws from
    fp8_ffn_workspace (zero-filled scheduler words, left zero by every call)."""
    guq, gus, dq, ds = w_fp8
    P, I2, H = guq.shape
    slot_hi = P if slot_hi is None else slot_hi
    _check("moe_grouped_ffn_fp8", lib().moe_grouped_ffn_fp8(
        _ptr(xq), _ptr(x_scales), _ptr(offsets_P), P, slot_lo, slot_hi, xq.shape[0], _ptr(guq),
        _ptr(gus), _ptr(dq), _ptr(ds), H, I2 // 2, _ptr(ys), _ptr(ws),
        ws.numel() * ws.element_size(), _ptr(d_status), _stream(stream)))


def moe_grouped_ffn(xs: torch.Tensor, offsets_P: torch.Tensor, w_gate_up: torch.Tensor,
                    w_down: torch.Tensor, ys: torch.Tensor, ws: torch.Tensor, slot_lo: int = 0,
                    slot_hi: Optional[int] = None, d_status=None, stream=None):
    P = w_gate_up.shape[0]
    slot_hi = P if slot_hi is None else slot_hi
    H = xs.shape[1]
    I = w_down.shape[2]
    _check("moe_grouped_ffn", lib().moe_grouped_ffn(
        _ptr(xs), _ptr(offsets_P), P, slot_lo, slot_hi, xs.shape[0], _ptr(w_gate_up),
        _ptr(w_down), H, I, dtype_code(xs.dtype), _ptr(ys), _ptr(ws),
        ws.numel() * ws.element_size(), _ptr(d_status), _stream(stream)))


def moe_grouped_ffn_split(xs: torch.Tensor, offsets_P: torch.Tensor, w_gate_up: torch.Tensor,
                          w_down: torch.Tensor, ys: torch.Tensor, ws: torch.Tensor,
                          hot_rows: int, hot_sms: int, stream_hot=None, slot_lo: int = 0,
                          slot_hi: Optional[int] = None, d_status=None, stream=None):
    """Grouped FFN split by slot over two streams: slots with >= hot_rows rows on the
    pair kernel (hot_sms SMs, stream_hot), the rest on the single-SM kernel."""
    P = w_gate_up.shape[0]
    slot_hi = P if slot_hi is None else slot_hi
    H = xs.shape[1]
    I = w_down.shape[2]
    sh = None if stream_hot is None else ctypes.c_void_p(stream_hot.cuda_stream)
    _check("moe_grouped_ffn_split", lib().moe_grouped_ffn_split(
        _ptr(xs), _ptr(offsets_P), P, slot_lo, slot_hi, xs.shape[0], _ptr(w_gate_up),
        _ptr(w_down), H, I, dtype_code(xs.dtype), _ptr(ys), _ptr(ws),
        ws.numel() * ws.element_size(), hot_rows, hot_sms, _ptr(d_status), _stream(stream), sh))


def moe_grouped_ffn_combine_ws_bytes(cap: int, rows: int, H: int, I: int,
                                     dtype: torch.dtype) -> int:
    return int(lib().moe_grouped_ffn_combine_ws_bytes(cap, rows, H, I, dtype_code(dtype)))


def moe_grouped_ffn_combine_in_epilogue(cap: int, P: int, dtype: torch.dtype) -> bool:
    """True if moe_grouped_ffn_combine combines in the down projection's epilogue for
    this buffer (few rows per slot), False if it runs the combine as its own launch."""
    return bool(lib().moe_grouped_ffn_combine_in_epilogue(cap, P, dtype_code(dtype)))


def ffn_combine_workspace(cap: int, rows: int, H: int, I: int, dtype: torch.dtype,
                          device="cuda") -> torch.Tensor:
    """A workspace for moe_grouped_ffn_combine: zero-filled, as its arrival counters
    must be zero before the first call; every call that completes leaves them zero."""
    n = moe_grouped_ffn_combine_ws_bytes(cap, rows, H, I, dtype)
    if n == 0:
        raise MoeError("moe_grouped_ffn_combine_ws_bytes", MOE_ERR_INVALID_ARG)
    return torch.zeros(n, device=device, dtype=torch.uint8)


def moe_grouped_ffn_combine(xs: torch.Tensor, offsets_P: torch.Tensor, w_gate_up: torch.Tensor,
                            w_down: torch.Tensor, ys: torch.Tensor, perm: torch.Tensor,
                            inv: torch.Tensor, w: torch.Tensor, d_counts, d_offsets,
                            local: Sequence[torch.Tensor], ws: torch.Tensor,
                            global_out: Optional[torch.Tensor] = None, slot_lo: int = 0,
                            slot_hi: Optional[int] = None, d_status=None, stream=None):
    """Grouped FFN whose down projection also combines each token's rows (top-k
    weights, j order) and writes them to the replicas; ws from ffn_combine_workspace."""
    P = w_gate_up.shape[0]
    slot_hi = P if slot_hi is None else slot_hi
    rows, kk = inv.shape
    H = xs.shape[1]
    I = w_down.shape[2]
    ok = (inv.dtype == torch.int32 and inv.is_contiguous() and tuple(w.shape) == (rows, kk)
          and w.dtype == torch.float32 and w.is_contiguous() and perm.dtype == torch.int32
          and perm.dim() == 1 and perm.numel() >= xs.shape[0] and tuple(ys.shape) == tuple(xs.shape)
          and (global_out is None or tuple(global_out.shape) == (rows, H)))
    if not ok:
        raise MoeError("moe_grouped_ffn_combine", MOE_ERR_INVALID_ARG)
    R = len(local)
    ptrs = (ctypes.c_void_p * R)(*[t.data_ptr() if t.numel() else None for t in local])
    _check("moe_grouped_ffn_combine", lib().moe_grouped_ffn_combine(
        _ptr(xs), _ptr(offsets_P), P, slot_lo, slot_hi, xs.shape[0], _ptr(w_gate_up),
        _ptr(w_down), H, I, dtype_code(xs.dtype), _ptr(ys), _ptr(perm), _ptr(inv), _ptr(w), rows,
        kk, _ptr(d_counts), _ptr(d_offsets), R, ctypes.cast(ptrs, _P), _ptr(global_out),
        _ptr(ws), ws.numel() * ws.element_size(), _ptr(d_status), _stream(stream)))


def moe_combine(ys: torch.Tensor, inv: torch.Tensor, w: torch.Tensor, out: torch.Tensor,
                d_status=None, stream=None):
    rows, k = inv.shape
    _check("moe_combine", lib().moe_combine(
        _ptr(ys), _ptr(inv), _ptr(w), rows, k, out.shape[1], dtype_code(out.dtype),
        ys.shape[0], _ptr(out), _ptr(d_status), _stream(stream)))


def moe_combine_scatter(ys: torch.Tensor, inv: torch.Tensor, w: torch.Tensor, d_counts, d_offsets,
                        local: Sequence[torch.Tensor], global_out: Optional[torch.Tensor] = None,
                        d_status=None, stream=None):
    """moe_combine then moe_dp_scatter in one launch; global_out (optional) also
    receives the combined global buffer."""
    rows, k = inv.shape
    R = len(local)
    ptrs = (ctypes.c_void_p * R)(*[t.data_ptr() if t.numel() else None for t in local])
    _check("moe_combine_scatter", lib().moe_combine_scatter(
        _ptr(ys), _ptr(inv), _ptr(w), rows, k, ys.shape[1], dtype_code(ys.dtype), ys.shape[0],
        _ptr(d_counts), _ptr(d_offsets), R, ctypes.cast(ptrs, _P),
        _ptr(global_out) if global_out is not None else None, _ptr(d_status), _stream(stream)))


def moe_dp_scatter(global_buf: torch.Tensor, d_counts, d_offsets, local: Sequence[torch.Tensor],
                   d_status=None, stream=None):
    R = len(local)
    ptrs = (ctypes.c_void_p * R)(*[t.data_ptr() if t.numel() else None for t in local])
    _check("moe_dp_scatter", lib().moe_dp_scatter(
        _ptr(global_buf), _ptr(d_counts), _ptr(d_offsets), R, global_buf.shape[0],
        global_buf.shape[1], dtype_code(global_buf.dtype), ctypes.cast(ptrs, _P),
        _ptr(d_status), _stream(stream)))


# ---------------------------------------------------------------- one layer
class MoeLayer:
    """One MoE layer between DP attention and EP on one GPU.

    Buffers are sized once for `max_rows` global rows; `forward` runs
    gather -> route -> dispatch -> grouped FFN -> combine -> scatter on the
    current stream without a host synchronisation (the hidden-state gather routes
    every row from its replica's logits in the same launch, with or without the fused
    residual add + RMSNorm; combine and scatter share one launch).  With router_weight
    [E, H] (bf16) the router logits are computed from the gathered hidden states by
    the gate GEMM fused ahead of top-k instead.  With fp8=True (bf16 layer) the expert
    weights are quantised once here (e4m3, 128 x 128 blocks), the dispatch quantises
    the permuted rows per token group and the grouped FFN (one launch for both GEMMs)
    runs on FP8 operands."""

    def __init__(self, *, R: int, H: int, E: int, k: int, I: int, w_gate_up: torch.Tensor,
                 w_down: torch.Tensor, max_rows: int, mode: int = MOE_PAD_SUM,
                 static_bound: int = 0, tokens_per_req: int = 1, renormalize: bool = True,
                 align: int = 1, l2p: Optional[torch.Tensor] = None,
                 nrep: Optional[torch.Tensor] = None, slot_range=None,
                 norm_gamma: Optional[torch.Tensor] = None, norm_eps: float = 1e-6,
                 n_shared: int = 0, fp8: bool = False,
                 router_weight: Optional[torch.Tensor] = None,
                 router_bias: Optional[torch.Tensor] = None, keep_global: bool = False,
                 fused_combine: bool = False, ffn_split=None):
        dev = w_gate_up.device
        # keep_global: also write the combined global buffer (yg, pad rows zero);
        # otherwise the combine writes the replicas' outputs only
        self.keep_global = keep_global
        self.R, self.H, self.E, self.k, self.I = R, H, E, k, I
        self.P = w_gate_up.shape[0]
        self.dtype = w_gate_up.dtype
        self.mode, self.static_bound, self.tpr = mode, static_bound, tokens_per_req
        self.renormalize, self.align = renormalize, align
        self.wgu, self.wd, self.l2p, self.nrep = w_gate_up, w_down, l2p, nrep
        self.slot_range = slot_range or (0, self.P)
        self.norm_gamma, self.norm_eps = norm_gamma, norm_eps
        # shared experts: logical ids E .. E+n_shared-1, the last slots of the weights
        self.n_shared = n_shared
        self.kk = k + n_shared
        self.max_rows = max_rows
        self.cap = moe_dispatch_cap_bound(max_rows, k + n_shared, self.P, align)
        i32 = dict(device=dev, dtype=torch.int32)
        # counts [R] and offsets [R + 1] side by side: one host->device copy per step
        self.d_meta = torch.zeros(2 * R + 1, **i32)
        self.d_counts, self.d_offsets = self.d_meta[:R], self.d_meta[R:]
        self._stage = _MetaStager(R)
        self.status = torch.zeros(1, **i32)
        self.xg = torch.empty(max_rows, H, device=dev, dtype=self.dtype)
        self.ids = torch.empty(max_rows, self.kk, **i32)
        self.w = torch.empty(max_rows, self.kk, device=dev, dtype=torch.float32)
        self.counts_P = torch.empty(self.P, **i32)
        self.offsets_P = torch.empty(self.P + 1, **i32)
        self.perm = torch.empty(self.cap, **i32)
        self.inv = torch.empty(max_rows, self.kk, **i32)
        self.fp8 = fp8
        if fp8:
            if self.dtype != torch.bfloat16:
                raise ValueError("the FP8 path takes a bf16 layer")
            self.w_fp8 = quantize_expert_weights_fp8(w_gate_up, w_down)
            self.xs = None
            self.xq = torch.empty(self.cap, H, device=dev, dtype=torch.uint8)
            self.xq_scales = torch.empty(self.cap, H // 128, device=dev, dtype=torch.uint8)
        else:
            self.xs = torch.empty(self.cap, H, device=dev, dtype=self.dtype)
        self.ys = torch.empty(self.cap, H, device=dev, dtype=self.dtype)
        self.yg = torch.empty(max_rows, H, device=dev, dtype=self.dtype)
        self.ws_dispatch = torch.empty(max(moe_dispatch_ws_bytes(max_rows, self.kk,
                                                                 E + n_shared), 16),
                                       device=dev, dtype=torch.uint8)
        # fused_combine: the grouped FFN and the combine + scatter as one call
        # (moe_grouped_ffn_combine; bf16 layers whose one grouped-FFN call covers every
        # slot).  Off by default: the separate combine launch measured faster at both
        # decode and prefill sizes.
        can_fuse = not fp8 and self.slot_range == (0, self.P)
        self.fused_combine = bool(fused_combine)
        # ffn_split = (hot_rows, hot_sms): the grouped FFN split by slot over two
        # streams (moe_grouped_ffn_split), for skewed layers; bf16 only
        self.ffn_split = tuple(ffn_split) if ffn_split else None
        self.stream_hot = None
        if self.ffn_split:
            if fp8 or self.fused_combine:
                raise ValueError("ffn_split takes a bf16 layer with the separate combine")
            self.stream_hot = torch.cuda.Stream(device=dev)
        if self.fused_combine and not can_fuse:
            raise ValueError("the fused combine needs a non-FP8 layer over all its slots")
        if self.fused_combine:
            self.ws_ffn = ffn_combine_workspace(self.cap, max_rows, H, I, self.dtype, dev)
        else:
            ws_ffn = (moe_grouped_ffn_fp8_ws_bytes(self.cap, I) if fp8
                      else moe_grouped_ffn_ws_bytes(self.cap, I, self.dtype))
            self.ws_ffn = (fp8_ffn_workspace(self.cap, I, dev) if fp8 else
                           torch.empty(max(ws_ffn, 16), device=dev, dtype=torch.uint8))
        self.router_weight, self.router_bias = router_weight, router_bias
        if router_weight is not None:
            if router_weight.shape != (E, H) or router_weight.dtype != torch.bfloat16:
                raise ValueError("router_weight must be bf16 [E, H]")
            self.ws_router = torch.empty(max(moe_route_gemm_ws_bytes(max_rows, H, E, k), 16),
                                         device=dev, dtype=torch.uint8)
        self.rows = 0
        self.counts = [0] * R

    def set_counts(self, counts: Sequence[int]) -> int:
        """Host layout for this step's replica counts; stages counts and offsets on
        the device (one pinned H2D copy on the current stream).  Returns the global
        row count."""
        offsets, rows = moe_dp_layout(counts, self.mode, self.static_bound, self.tpr)
        if rows > self.max_rows:
            raise MoeError("MoeLayer.set_counts", MOE_ERR_CAPACITY)
        self._stage(counts, offsets, self.d_meta, None)
        self.rows = rows
        self.counts = [int(c) for c in counts]
        return rows

    def check_inputs(self, local_x, local_logits, out, local_residual=None,
                     counts: Optional[Sequence[int]] = None):
        """Host-side check of the replica tensors against the counts (the current
        layout's by default): raises MoeError instead of letting a kernel read or write
        past a replica's rows."""
        counts = self.counts if counts is None else counts
        _check_replicas("MoeLayer inputs", counts, local_x, self.H, self.dtype)
        _check_replicas("MoeLayer outputs", counts, out, self.H, self.dtype)
        if self.router_weight is None:
            _check_replicas("MoeLayer logits", counts, local_logits, self.E, torch.float32)
        if local_residual is not None:
            _check_replicas("MoeLayer residual", counts, local_residual, self.H, self.dtype)

    def capture(self, local_x: Sequence[torch.Tensor], local_logits: Sequence[torch.Tensor],
                out: Sequence[torch.Tensor],
                local_residual: Optional[Sequence[torch.Tensor]] = None,
                timings=None) -> "LayerGraph":
        """Capture one step for the current counts layout (set_counts first) as a CUDA
        graph; see LayerGraph."""
        return LayerGraph(self, local_x, local_logits, out, local_residual, timings)

    def forward(self, local_x: Sequence[torch.Tensor], local_logits: Sequence[torch.Tensor],
                out: Sequence[torch.Tensor], counts: Optional[Sequence[int]] = None,
                stream=None, timings=None,
                local_residual: Optional[Sequence[torch.Tensor]] = None):
        """One layer step.  With local_residual (and norm_gamma set at construction)
        the hidden states are first added into the residual in place and the
        RMSNorm of the updated residual is what gets gathered and routed."""
        if counts is not None:
            self.set_counts(counts)
        self.check_inputs(local_x, local_logits, out, local_residual)
        rows = self.rows
        st = self.status
        xg = self.xg[:rows]
        ids, w, inv, yg = self.ids[:rows], self.w[:rows], self.inv[:rows], self.yg[:rows]
        ev = timings.mark if timings is not None else (lambda name: None)
        ev("start")
        if local_residual is not None:
            if self.norm_gamma is None:
                raise ValueError("local_residual needs norm_gamma")
            if self.router_weight is None:  # the rows are routed in the same launch
                moe_dp_gather_add_rmsnorm_route(local_x, local_residual, self.norm_gamma,
                                                self.norm_eps, local_logits, self.d_counts,
                                                self.d_offsets, xg, self.k, self.renormalize,
                                                ids, w, None, self.n_shared, st, stream)
            else:
                moe_dp_gather_add_rmsnorm(local_x, local_residual, self.norm_gamma,
                                          self.norm_eps, self.d_counts, self.d_offsets, xg, st,
                                          stream)
        elif self.router_weight is None:  # the gather routes its rows in the same launch
            moe_dp_gather_route(local_x, local_logits, self.d_counts, self.d_offsets, xg, self.k,
                                self.renormalize, ids, w, None, self.n_shared, st, stream)
        else:
            moe_dp_gather(local_x, self.d_counts, self.d_offsets, xg, st, stream)
        ev("gather")
        if self.router_weight is not None:  # (given logits: routed by the gather)
            moe_route_gemm_topk(xg, self.router_weight, self.k, self.renormalize, self.d_counts,
                                self.d_offsets, ids, w, self.ws_router, None, st, stream,
                                n_shared=self.n_shared, bias=self.router_bias)
        ev("route")
        E_all = self.E + self.n_shared
        if self.fp8:
            moe_dispatch_fp8(xg, ids, E_all, self.P, self.counts_P, self.offsets_P, self.perm,
                             inv, self.xq, self.xq_scales, self.ws_dispatch, self.l2p, self.nrep,
                             self.align, st, stream)
            ev("dispatch")
            moe_grouped_ffn_fp8(self.xq, self.xq_scales, self.offsets_P, self.w_fp8, self.ys,
                                self.ws_ffn, self.slot_range[0], self.slot_range[1], st, stream)
        else:
            moe_dispatch(xg, ids, E_all, self.P, self.counts_P, self.offsets_P, self.perm, inv,
                         self.xs, self.ws_dispatch, self.l2p, self.nrep, self.align, st, stream)
            ev("dispatch")
            if self.fused_combine:  # combine + scatter inside the down projection
                moe_grouped_ffn_combine(self.xs, self.offsets_P, self.wgu, self.wd, self.ys,
                                        self.perm, inv, w, self.d_counts, self.d_offsets, out,
                                        self.ws_ffn, yg if self.keep_global else None,
                                        self.slot_range[0], self.slot_range[1], st, stream)
                ev("ffn")
                return out
            if self.ffn_split:
                moe_grouped_ffn_split(self.xs, self.offsets_P, self.wgu, self.wd, self.ys,
                                      self.ws_ffn, self.ffn_split[0], self.ffn_split[1],
                                      self.stream_hot, self.slot_range[0], self.slot_range[1],
                                      st, stream)
            else:
                moe_grouped_ffn(self.xs, self.offsets_P, self.wgu, self.wd, self.ys, self.ws_ffn,
                                self.slot_range[0], self.slot_range[1], st, stream)
        ev("ffn")
        moe_combine_scatter(self.ys, inv, w, self.d_counts, self.d_offsets, out,
                            yg if self.keep_global else None, st, stream)
        ev("combine_scatter")
        return out


def _check_replicas(what: str, counts: Sequence[int], tensors, width: int, dtype):
    """The kernels see plain pointers: every replica tensor must be a contiguous CUDA
    [>= counts[r], width] array of `dtype`, or rows past its end would be touched."""
    if tensors is None or len(tensors) != len(counts):
        raise MoeError(what, MOE_ERR_INVALID_ARG)
    for c, t in zip(counts, tensors):
        if c == 0:
            continue
        if (not t.is_cuda or t.dtype != dtype or t.dim() != 2 or t.shape[1] != width or
                t.shape[0] < c or not t.is_contiguous()):
            raise MoeError(what, MOE_ERR_INVALID_ARG)


class _MetaStager:
    """Ring of pinned staging buffers for the per-step counts/offsets copy, so the
    host only waits when it laps a copy still in flight."""

    def __init__(self, R: int, depth: int = 4):
        self.R = R
        self.ring = [torch.zeros(2 * R + 1, dtype=torch.int32, pin_memory=True)
                     for _ in range(depth)]
        self.done = [torch.cuda.Event() for _ in range(depth)]
        for ev in self.done:
            ev.record()
        self.i = 0

    def __call__(self, counts, offsets, d_meta: torch.Tensor, stream):
        i = self.i
        self.i = (i + 1) % len(self.ring)
        self.done[i].synchronize()  # the copy that last used this buffer has run
        h = self.ring[i]
        h[: self.R] = torch.tensor(list(counts), dtype=torch.int32)
        h[self.R:] = torch.tensor(offsets, dtype=torch.int32)
        s = stream if stream is not None else torch.cuda.current_stream()
        with torch.cuda.stream(s):
            d_meta.copy_(h, non_blocking=True)
            self.done[i].record(s)


class LayerGraph:
    """One MoeLayer step captured as a CUDA graph: the layer's kernels replay with
    one launch, reading the replica counts and offsets from a device buffer of the
    graph's own.

    A replay uses the tensors given at capture (the same replica inputs, outputs
    and residuals) and the global row count of the layout at capture.  stage(counts,
    stream) copies a step's counts and offsets into the graph's buffer on any stream
    (e.g. the copy stream that brings the step's inputs, so the compute stream sees
    no copy between replays); replay(counts) stages on the current stream and
    replays.  New counts must give the same row count (always true under a static
    bound, where every step has identical kernel grids)."""

    def __init__(self, layer: MoeLayer, local_x, local_logits, out, local_residual=None,
                 timings=None):
        if layer.rows == 0:
            raise MoeError("LayerGraph", MOE_ERR_INVALID_ARG)
        self.layer, self.rows = layer, layer.rows
        self.tensors = (local_x, local_logits, out, local_residual)
        self.d_meta = layer.d_meta.clone()       # the layer's current layout
        self._stage = _MetaStager(layer.R)
        saved = layer.d_meta, layer.d_counts, layer.d_offsets
        layer.d_meta = self.d_meta
        layer.d_counts, layer.d_offsets = self.d_meta[: layer.R], self.d_meta[layer.R:]
        try:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):  # one eager step first: host-side setup runs once
                layer.forward(local_x, local_logits, out, local_residual=local_residual)
            torch.cuda.current_stream().wait_stream(side)
            self.graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.graph):
                layer.forward(local_x, local_logits, out, local_residual=local_residual,
                              timings=timings)
        finally:
            layer.d_meta, layer.d_counts, layer.d_offsets = saved

    def stage(self, counts: Sequence[int], stream=None):
        """Copy this step's counts and offsets into the graph's buffer on `stream`
        (default: the current stream); order the replay after it."""
        L = self.layer
        offsets, rows = moe_dp_layout(counts, L.mode, L.static_bound, L.tpr)
        if rows != self.rows:
            raise MoeError("LayerGraph.stage", MOE_ERR_INVALID_ARG)
        L.check_inputs(*self.tensors, counts=counts)   # the captured tensors hold the rows
        self._stage(counts, offsets, self.d_meta, stream)

    def replay(self, counts: Optional[Sequence[int]] = None):
        if counts is not None:
            self.stage(counts)
        self.graph.replay()
