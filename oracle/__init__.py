"""CPU oracle for MoE dispatch / combine -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package. The product path (the CUDA library and its
Python binding) never imports, links or runs it, and the two share no code.

``oracle.c`` is a plain single-threaded C99 restatement of the method; this
module compiles it with gcc and wraps it with ctypes over numpy arrays.
``brute.py`` is a second, independent NumPy formulation used to pin it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
# A prebuilt library to load instead (tests/test_oracle_mutations.py points
# it at copies of oracle.c with a planted mistake); nothing is compiled then.
_OVERRIDE = os.environ.get("ORACLE_LIBRARY") or None
_LIB = None
_LOCK = threading.Lock()

OK, ERR_ARG, ERR_EXPERT, ERR_CAPACITY = 0, 1, 2, 3


def compile_command(src: str, out: str) -> list[str]:
    """gcc command that builds the oracle library from `src` into `out`."""
    return ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math",
            "-fno-strict-aliasing", "-fPIC", "-shared", "-o", out, src, "-lm"]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (IEEE fp32, no contraction)."""
    if _OVERRIDE:
        return _OVERRIDE
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.run(compile_command(_SRC, tmp), check=True)
        os.replace(tmp, _SO)
    return _SO


def _lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            L = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64, i32 = ctypes.c_int64, ctypes.c_int
            L.orc_layout.argtypes = [P, i64, i32, i32, i32, P, P, P, P, P]
            L.orc_layout.restype = i32
            L.orc_layout_aligned.argtypes = [P, i64, i32, i32, i32, i32, P, P, P, P, P]
            L.orc_layout_aligned.restype = i32
            L.orc_layout_strided.argtypes = [P, i64, i32, i32, i32, i32, P, P, P, P, P]
            L.orc_layout_strided.restype = i32
            L.orc_layout_nonexpand.argtypes = [P, i64, i32, i32, i32, P, P, P, P, P]
            L.orc_layout_nonexpand.restype = i32
            L.orc_nonexpand_recv_topk.argtypes = [P, P, P, i64, i32, i32, i32, P, P]
            L.orc_nonexpand_recv_topk.restype = None
            L.orc_fill_pad_rows.argtypes = [P, P, i32, i64, P, P, i32, P, P]
            L.orc_fill_pad_rows.restype = None
            L.orc_pow2_ceil.argtypes = [ctypes.c_float]
            L.orc_pow2_ceil.restype = ctypes.c_float
            L.orc_quant_row_e4m3_pow2.argtypes = [P, i32, i32, P, P, P]
            L.orc_quant_row_e4m3_pow2.restype = None
            L.orc_dispatch_rows.argtypes = [P, i64, i64, P, i32, P]
            L.orc_dispatch_rows.restype = None
            L.orc_topk_to_routing_map.argtypes = [P, P, i64, i32, i32, P, P]
            L.orc_topk_to_routing_map.restype = i32
            L.orc_routing_map_to_topk.argtypes = [P, P, i64, i32, i32, P, P]
            L.orc_routing_map_to_topk.restype = i32
            L.orc_combine_backward.argtypes = [P, P, i32, P, i64, i32, P, P, P]
            L.orc_combine_backward.restype = None
            L.orc_dispatch_backward.argtypes = [P, P, i32, P, i64, i32, P, P]
            L.orc_dispatch_backward.restype = None
            L.orc_dispatch_bf16.argtypes = [P, i64, i32, P, i32, P, P, P, P]
            L.orc_dispatch_bf16.restype = None
            L.orc_dispatch_e4m3.argtypes = [P, i64, i32, P, i32, P, P, P, P, P]
            L.orc_dispatch_e4m3.restype = None
            L.orc_quant_row_e4m3.argtypes = [P, i32, P, P]
            L.orc_quant_row_e4m3.restype = None
            L.orc_combine_row.argtypes = [P, i32, P, P, i32, P]
            L.orc_combine_row.restype = None
            L.orc_combine.argtypes = [P, i32, P, i64, i32, P, P]
            L.orc_combine.restype = None
            L.orc_f32_to_bf16_array.argtypes = [P, i64, P]
            L.orc_f32_to_e4m3_array.argtypes = [P, i64, P]
            L.orc_e4m3_sweep.argtypes = [ctypes.c_uint32, ctypes.c_uint32, P]
            L.orc_f32_to_e4m3.argtypes = [ctypes.c_float]
            L.orc_f32_to_e4m3.restype = ctypes.c_uint8
            L.orc_e4m3_to_f32.argtypes = [ctypes.c_uint8]
            L.orc_e4m3_to_f32.restype = ctypes.c_float
            L.orc_f32_to_e5m2_array.argtypes = [P, i64, P]
            L.orc_e5m2_sweep.argtypes = [ctypes.c_uint32, ctypes.c_uint32, P]
            L.orc_e5m2_to_f32.argtypes = [ctypes.c_uint8]
            L.orc_e5m2_to_f32.restype = ctypes.c_float
            L.orc_quant_row_e5m2.argtypes = [P, i32, i32, P, P, P]
            L.orc_quant_row_e5m2.restype = None
            _LIB = L
    return _LIB


def _p(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def layout(topk_idx: np.ndarray, E: int, R: int) -> dict:
    """Routing layout (counts, masks, offsets, slot -> row map) of topk_idx [T, K]."""
    idx = _c(topk_idx, np.int64)
    T, K = idx.shape
    out = dict(
        num_tokens_per_expert=np.zeros(E, np.int32),
        num_tokens_per_rank=np.zeros(R, np.int32),
        is_token_in_rank=np.zeros((T, R), np.uint8),
        expert_offsets=np.zeros(E + 1, np.int32),
        row_of_slot=np.zeros((T, K), np.int32),
    )
    st = _lib().orc_layout(_p(idx), T, K, E, R, _p(out["num_tokens_per_expert"]),
                           _p(out["num_tokens_per_rank"]), _p(out["is_token_in_rank"]),
                           _p(out["expert_offsets"]), _p(out["row_of_slot"]))
    out["status"] = int(st)
    return out


def layout_aligned(topk_idx: np.ndarray, E: int, R: int, alignment: int) -> dict:
    """Layout whose expert row ranges start on multiples of `alignment`."""
    idx = _c(topk_idx, np.int64)
    T, K = idx.shape
    out = dict(
        num_tokens_per_expert=np.zeros(E, np.int32),
        num_tokens_per_rank=np.zeros(R, np.int32),
        is_token_in_rank=np.zeros((T, R), np.uint8),
        expert_offsets=np.zeros(E + 1, np.int32),
        row_of_slot=np.zeros((T, K), np.int32),
    )
    st = _lib().orc_layout_aligned(_p(idx), T, K, E, R, alignment, _p(out["num_tokens_per_expert"]),
                                   _p(out["num_tokens_per_rank"]), _p(out["is_token_in_rank"]),
                                   _p(out["expert_offsets"]), _p(out["row_of_slot"]))
    out["status"] = int(st)
    return out


def layout_strided(topk_idx: np.ndarray, E: int, R: int, cap: int) -> dict:
    """Layout with expert e's rows at e * cap + 0, 1, ... (slots past cap dropped)."""
    idx = _c(topk_idx, np.int64)
    T, K = idx.shape
    out = dict(
        num_tokens_per_expert=np.zeros(E, np.int32),
        num_tokens_per_rank=np.zeros(R, np.int32),
        is_token_in_rank=np.zeros((T, R), np.uint8),
        expert_offsets=np.zeros(E + 1, np.int32),
        row_of_slot=np.zeros((T, K), np.int32),
    )
    st = _lib().orc_layout_strided(_p(idx), T, K, E, R, cap, _p(out["num_tokens_per_expert"]),
                                   _p(out["num_tokens_per_rank"]), _p(out["is_token_in_rank"]),
                                   _p(out["expert_offsets"]), _p(out["row_of_slot"]))
    out["status"] = int(st)
    return out


def layout_nonexpand(topk_idx: np.ndarray, E: int, R: int) -> dict:
    """One row per (token, rank); rank_offsets in place of expert_offsets."""
    idx = _c(topk_idx, np.int64)
    T, K = idx.shape
    out = dict(
        num_tokens_per_expert=np.zeros(E, np.int32),
        num_tokens_per_rank=np.zeros(R, np.int32),
        is_token_in_rank=np.zeros((T, R), np.uint8),
        rank_offsets=np.zeros(R + 1, np.int32),
        row_of_slot=np.zeros((T, K), np.int32),
    )
    st = _lib().orc_layout_nonexpand(_p(idx), T, K, E, R, _p(out["num_tokens_per_expert"]),
                                     _p(out["num_tokens_per_rank"]), _p(out["is_token_in_rank"]),
                                     _p(out["rank_offsets"]), _p(out["row_of_slot"]))
    out["status"] = int(st)
    return out


def nonexpand_recv_topk(topk_idx: np.ndarray, topk_weights: np.ndarray | None, row_of_slot: np.ndarray,
                        E: int, R: int, num_rows: int):
    """(recv_topk_idx [rows, K] int64 rank-local ids or -1, recv_topk_weights [rows, K])."""
    idx = _c(topk_idx, np.int64)
    rows = _c(row_of_slot, np.int32)
    T, K = idx.shape
    ri = np.full((num_rows, K), -9, np.int64)
    rw = np.full((num_rows, K), np.nan, np.float32)
    w = _c(topk_weights, np.float32) if topk_weights is not None else None
    _lib().orc_nonexpand_recv_topk(_p(idx), _p(w), _p(rows), T, K, E, R, _p(ri), _p(rw))
    return ri, rw


def fill_pad_rows(layout: dict, recv: np.ndarray, scales=None, src=None, weights=None) -> None:
    """Zero the pad rows of an aligned layout in place (scale 0, source -1, weight 0)."""
    E = len(layout["num_tokens_per_expert"])
    assert recv.flags.c_contiguous
    row_bytes = recv.strides[0]
    nb = 0 if scales is None else scales.shape[1]
    _lib().orc_fill_pad_rows(_p(_c(layout["num_tokens_per_expert"], np.int32)),
                             _p(_c(layout["expert_offsets"], np.int32)), E, row_bytes, _p(recv),
                             _p(scales), nb, _p(src), _p(weights))


def dispatch_bf16(x: np.ndarray, row_of_slot: np.ndarray, num_rows: int,
                  topk_weights: np.ndarray | None = None, fill: int = 0):
    """recv_x [num_rows, H] (uint16 bf16 bits), recv_src_token [num_rows], recv_weights."""
    x = _c(x, np.uint16)
    rows = _c(row_of_slot, np.int32)
    T, H = x.shape
    K = rows.shape[1]
    recv = np.full((num_rows, H), fill, np.uint16)
    src = np.full(num_rows, -1, np.int32)
    rw = np.full(num_rows, np.nan, np.float32) if topk_weights is not None else None
    w = _c(topk_weights, np.float32) if topk_weights is not None else None
    _lib().orc_dispatch_bf16(_p(x), T, H, _p(rows), K, _p(w), _p(recv), _p(src), _p(rw))
    return recv, src, rw


def dispatch_e4m3(x: np.ndarray, row_of_slot: np.ndarray, num_rows: int,
                  topk_weights: np.ndarray | None = None):
    """recv_q [num_rows, H] uint8, recv_scales [num_rows, H/128] fp32, recv_src_token, recv_weights."""
    x = _c(x, np.uint16)
    rows = _c(row_of_slot, np.int32)
    T, H = x.shape
    K = rows.shape[1]
    q = np.zeros((num_rows, H), np.uint8)
    s = np.full((num_rows, H // 128), np.nan, np.float32)
    src = np.full(num_rows, -1, np.int32)
    rw = np.full(num_rows, np.nan, np.float32) if topk_weights is not None else None
    w = _c(topk_weights, np.float32) if topk_weights is not None else None
    _lib().orc_dispatch_e4m3(_p(x), T, H, _p(rows), K, _p(w), _p(q), _p(s), _p(src), _p(rw))
    return q, s, src, rw


def quant_row_e4m3(xrow: np.ndarray):
    xrow = _c(xrow, np.uint16)
    H = xrow.shape[0]
    q = np.zeros(H, np.uint8)
    s = np.zeros(H // 128, np.float32)
    _lib().orc_quant_row_e4m3(_p(xrow), H, _p(q), _p(s))
    return q, s


def pow2_ceil(s: float) -> float:
    return float(_lib().orc_pow2_ceil(float(s)))


def quant_row_e4m3_pow2(xrow: np.ndarray, ue8m0: bool = False):
    """(codes [H] u8, scales [H/128] fp32 powers of two, or u8 exponent bytes if ue8m0)."""
    xrow = _c(xrow, np.uint16)
    H = xrow.shape[0]
    q = np.zeros(H, np.uint8)
    s = np.zeros(H // 128, np.uint8 if ue8m0 else np.float32)
    if ue8m0:
        _lib().orc_quant_row_e4m3_pow2(_p(xrow), H, 1, _p(q), None, _p(s))
    else:
        _lib().orc_quant_row_e4m3_pow2(_p(xrow), H, 0, _p(q), _p(s), None)
    return q, s


def dispatch_e4m3_pow2(x: np.ndarray, row_of_slot: np.ndarray, num_rows: int, ue8m0: bool = False):
    """Power-of-two-scale quantise-permute: (codes [rows, H], scales [rows, H/128])."""
    x = _c(x, np.uint16)
    T, H = x.shape
    q = np.zeros((T, H), np.uint8)
    s = np.zeros((T, H // 128), np.uint8 if ue8m0 else np.float32)
    for t in range(T):
        q[t], s[t] = quant_row_e4m3_pow2(x[t], ue8m0)
    rq = dispatch_rows(q, row_of_slot, num_rows)
    rs = dispatch_rows(s, row_of_slot, num_rows)
    return rq, rs


def quant_row_e5m2(xrow: np.ndarray, scale_mode: int = 0):
    """(codes [H] u8, scales [H/128]): fp32 scales for scale_mode 0 (amax/57344)
    and 1 (its power-of-two ceiling), u8 exponent bytes for scale_mode 2."""
    xrow = _c(xrow, np.uint16)
    H = xrow.shape[0]
    q = np.zeros(H, np.uint8)
    s = np.zeros(H // 128, np.uint8 if scale_mode == 2 else np.float32)
    if scale_mode == 2:
        _lib().orc_quant_row_e5m2(_p(xrow), H, 2, _p(q), None, _p(s))
    else:
        _lib().orc_quant_row_e5m2(_p(xrow), H, scale_mode, _p(q), _p(s), None)
    return q, s


def dispatch_e5m2(x: np.ndarray, row_of_slot: np.ndarray, num_rows: int, scale_mode: int = 0):
    """e5m2 quantise-permute: (codes [rows, H], scales [rows, H/128])."""
    x = _c(x, np.uint16)
    T, H = x.shape
    q = np.zeros((T, H), np.uint8)
    s = np.zeros((T, H // 128), np.uint8 if scale_mode == 2 else np.float32)
    for t in range(T):
        q[t], s[t] = quant_row_e5m2(x[t], scale_mode)
    return dispatch_rows(q, row_of_slot, num_rows), dispatch_rows(s, row_of_slot, num_rows)


def dispatch_rows(src: np.ndarray, row_of_slot: np.ndarray, num_rows: int, fill: int = 0) -> np.ndarray:
    """Byte permute of rows of any dtype: out[row_of_slot[t,k]] = src[t]."""
    src = np.ascontiguousarray(src)
    rows = _c(row_of_slot, np.int32)
    T = src.shape[0]
    K = rows.shape[1]
    out = np.full((num_rows,) + src.shape[1:], fill, src.dtype)
    row_bytes = src.strides[0] if T else 0
    _lib().orc_dispatch_rows(_p(src.view(np.uint8).reshape(T, -1)) if T else None, T, row_bytes, _p(rows), K,
                             _p(out))
    return out


def combine(y: np.ndarray, row_of_slot: np.ndarray, topk_weights: np.ndarray | None):
    """out [T, H] (uint16 bf16 bits) = bf16(sum_k w[t,k] * y[row(t,k)])."""
    y = _c(y, np.uint16)
    rows = _c(row_of_slot, np.int32)
    T, K = rows.shape
    H = y.shape[1]
    w = _c(topk_weights, np.float32) if topk_weights is not None else None
    out = np.zeros((T, H), np.uint16)
    _lib().orc_combine(_p(y), H, _p(rows), T, K, _p(w), _p(out))
    return out


def combine_tokens(y: np.ndarray, row_of_slot: np.ndarray, topk_weights: np.ndarray | None,
                   tokens) -> np.ndarray:
    """The combine output rows of the listed tokens only ([len(tokens), H])."""
    y = _c(y, np.uint16)
    rows = _c(row_of_slot, np.int32)
    K = rows.shape[1]
    H = y.shape[1]
    w = _c(topk_weights, np.float32) if topk_weights is not None else None
    out = np.zeros((len(tokens), H), np.uint16)
    L = _lib()
    for i, t in enumerate(tokens):
        r = np.ascontiguousarray(rows[t])
        wt = None if w is None else np.ascontiguousarray(w[t])
        o = out[i]
        L.orc_combine_row(_p(y), H, _p(r), _p(wt), K, o.ctypes.data)
    return out


def combine_backward(grad_out: np.ndarray, y: np.ndarray, row_of_slot: np.ndarray,
                     topk_weights: np.ndarray | None, num_rows: int):
    """(grad_y [num_rows, H] bf16 bits, zero where no slot writes; grad_w [T, K] float64)."""
    g = _c(grad_out, np.uint16)
    y = _c(y, np.uint16)
    rows = _c(row_of_slot, np.int32)
    T, K = rows.shape
    H = g.shape[1]
    w = _c(topk_weights, np.float32) if topk_weights is not None else None
    gy = np.zeros((num_rows, H), np.uint16)
    gw = np.zeros((T, K), np.float64)
    _lib().orc_combine_backward(_p(g), _p(y), H, _p(rows), T, K, _p(w), _p(gy), _p(gw))
    return gy, gw


def dispatch_backward(grad_recv: np.ndarray, grad_recv_weights: np.ndarray | None, row_of_slot: np.ndarray):
    """(grad_x [T, H] bf16 bits, grad_topk_weights [T, K] fp32 or None)."""
    g = _c(grad_recv, np.uint16)
    rows = _c(row_of_slot, np.int32)
    T, K = rows.shape
    H = g.shape[1]
    gx = np.zeros((T, H), np.uint16)
    gw = np.zeros((T, K), np.float32) if grad_recv_weights is not None else None
    rw = _c(grad_recv_weights, np.float32) if grad_recv_weights is not None else None
    _lib().orc_dispatch_backward(_p(g), _p(rw), H, _p(rows), T, K, _p(gx), _p(gw))
    return gx, gw


def topk_to_routing_map(topk_idx: np.ndarray, topk_weights: np.ndarray | None, E: int):
    """(routing_map [T, E] u8, probs [T, E] fp32 or None, status)."""
    idx = _c(topk_idx, np.int64)
    T, K = idx.shape
    rm = np.zeros((T, E), np.uint8)
    pr = np.zeros((T, E), np.float32) if topk_weights is not None else None
    w = _c(topk_weights, np.float32) if topk_weights is not None else None
    st = _lib().orc_topk_to_routing_map(_p(idx), _p(w), T, K, E, _p(rm), _p(pr))
    return rm, pr, int(st)


def routing_map_to_topk(routing_map: np.ndarray, probs: np.ndarray | None, K: int):
    """(topk_idx [T, K] int64, topk_weights [T, K] fp32, status)."""
    rm = _c(routing_map, np.uint8)
    T, E = rm.shape
    idx = np.zeros((T, K), np.int64)
    w = np.zeros((T, K), np.float32)
    pr = _c(probs, np.float32) if probs is not None else None
    st = _lib().orc_routing_map_to_topk(_p(rm), _p(pr), T, E, K, _p(idx), _p(w))
    return idx, w, int(st)


def f32_to_bf16(a: np.ndarray) -> np.ndarray:
    a = _c(a, np.float32)
    out = np.zeros(a.shape, np.uint16)
    _lib().orc_f32_to_bf16_array(_p(a), a.size, _p(out))
    return out


def f32_to_e4m3(a: np.ndarray) -> np.ndarray:
    a = _c(a, np.float32)
    out = np.zeros(a.shape, np.uint8)
    _lib().orc_f32_to_e4m3_array(_p(a), a.size, _p(out))
    return out


def e4m3_sweep(lo: int, hi: int) -> np.ndarray:
    out = np.zeros(hi - lo, np.uint8)
    _lib().orc_e4m3_sweep(lo, hi, _p(out))
    return out


def e4m3_to_f32(q: np.ndarray) -> np.ndarray:
    L = _lib()
    return np.array([L.orc_e4m3_to_f32(int(v)) for v in np.asarray(q).ravel()],
                    np.float32).reshape(np.shape(q))


def f32_to_e5m2(a: np.ndarray) -> np.ndarray:
    a = _c(a, np.float32)
    out = np.zeros(a.shape, np.uint8)
    _lib().orc_f32_to_e5m2_array(_p(a), a.size, _p(out))
    return out


def e5m2_sweep(lo: int, hi: int) -> np.ndarray:
    out = np.zeros(hi - lo, np.uint8)
    _lib().orc_e5m2_sweep(lo, hi, _p(out))
    return out


def e5m2_to_f32(q: np.ndarray) -> np.ndarray:
    L = _lib()
    return np.array([L.orc_e5m2_to_f32(int(v)) for v in np.asarray(q).ravel()],
                    np.float32).reshape(np.shape(q))
