"""GB300 MoE token dispatch / combine: thin Python binding over libep.so.

Each function has the name of the C entry point it wraps (include/ep.h) and
only marshals arguments: torch tensors become device pointers, the current
torch CUDA stream becomes the stream argument, and a non-OK status raises
EPError. All computation runs in the library's CUDA kernels; there is no CPU
path. If libep.so is missing the first call raises, it never falls back.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB as _LIB_PATH, build

EP_OK, EP_ERR_INVALID_ARG, EP_ERR_INVALID_EXPERT, EP_ERR_CAPACITY, EP_ERR_CUDA, EP_ERR_ALLOC = range(6)
EP_DTYPE_BF16, EP_DTYPE_FP8_E4M3, EP_DTYPE_FP8_E5M2 = 0, 1, 2
EP_SCALE_FP32, EP_SCALE_POW2, EP_SCALE_UE8M0 = 0, 1, 2


class DispatchConfig(ctypes.Structure):
    """ep_dispatch_config_t (include/ep.h)."""
    _fields_ = [("in_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int), ("scale_mode", ctypes.c_int),
                ("scales_col_major", ctypes.c_int), ("scales_ld", ctypes.c_int64), ("overlap_layout", ctypes.c_int)]

# Exported symbols declared in include/ep.h.
EXPORTS = ("ep_layout", "ep_layout_aligned", "ep_layout_strided", "ep_layout_nonexpand",
           "ep_nonexpand_recv_topk", "ep_dispatch", "ep_dispatch_ex", "ep_combine", "ep_combine_backward",
           "ep_dispatch_backward", "ep_topk_to_routing_map", "ep_routing_map_to_topk", "ep_handle_query",
           "ep_handle_copy_row_of_slot", "ep_handle_destroy", "ep_handle_layout_kernels", "ep_layout_cluster_ctas",
           "ep_layout_noalloc", "ep_status_string")

_lib = None


class EPError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        super().__init__(f"{call} -> {status_string(status)} ({status})")


def lib() -> ctypes.CDLL:
    """Load libep.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"libep.so is not built ({_LIB_PATH}); run "
                               "combine_get_dispatch_layout_gb300.build.build()")
        L = ctypes.CDLL(_LIB_PATH)
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        L.ep_layout.argtypes = [P, i32, i32, i32, i32, P, P, P, P, P, P, ctypes.POINTER(P), P]
        L.ep_layout_aligned.argtypes = [P, i32, i32, i32, i32, i32, P, P, P, P, P, P, ctypes.POINTER(P), P]
        L.ep_layout_strided.argtypes = [P, i32, i32, i32, i32, i32, P, P, P, P, P, P, ctypes.POINTER(P), P]
        L.ep_layout_nonexpand.argtypes = [P, i32, i32, i32, i32, P, P, P, P, P, P, ctypes.POINTER(P), P]
        L.ep_nonexpand_recv_topk.argtypes = [P, P, P, i32, P, P, i64, P]
        L.ep_dispatch.argtypes = [P, P, i32, i32, P, P, P, P, P, i64, P]
        L.ep_dispatch_ex.argtypes = [P, P, P, i32, ctypes.POINTER(DispatchConfig), P, P, P, P, P, i64, P]
        L.ep_combine.argtypes = [P, P, i64, i32, P, P, P]
        L.ep_topk_to_routing_map.argtypes = [P, P, i32, i32, i32, P, P, P, P]
        L.ep_routing_map_to_topk.argtypes = [P, P, i32, i32, i32, P, P, P, P]
        L.ep_combine_backward.argtypes = [P, P, P, i64, i32, P, P, i64, P, P]
        L.ep_dispatch_backward.argtypes = [P, P, i64, i32, P, P, P, P]
        L.ep_handle_query.argtypes = [P, ctypes.POINTER(i64), ctypes.POINTER(ctypes.c_int32)]
        L.ep_handle_copy_row_of_slot.argtypes = [P, P, P]
        L.ep_handle_destroy.argtypes = [P]
        L.ep_handle_layout_kernels.argtypes = [P]
        L.ep_handle_layout_kernels.restype = i32
        L.ep_layout_cluster_ctas.argtypes = [i32, i32, i32, i32]
        L.ep_layout_cluster_ctas.restype = i32
        L.ep_layout_noalloc.argtypes = [P, i32, i32, i32, i32, P, P, P, P, P, P, P]
        L.ep_status_string.argtypes = [i32]
        L.ep_status_string.restype = ctypes.c_char_p
        for name in EXPORTS:
            if name != "ep_status_string":
                getattr(L, name).restype = i32
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().ep_status_string(int(status)).decode()


def _ptr(t):
    """Address of a tensor argument (an int is taken as a raw address). The
    kernels index rows as dense row-major arrays and dereference the address
    on the GPU, so a non-empty tensor must be contiguous and either on the
    GPU or in pinned host memory; anything else is refused here, before the
    call."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if t.numel() > 0:
        if not t.is_contiguous():
            raise ValueError("tensor arguments must be contiguous")
        if not t.is_cuda and not t.is_pinned():
            raise ValueError("tensor arguments must be CUDA tensors or pinned host tensors")
    return t.data_ptr()


def _need(t, nbytes: int, what: str) -> None:
    """Refuse a tensor that holds fewer bytes than the call will touch (the C
    ABI takes raw addresses and sizes, so only the binding can see this)."""
    if t is None or isinstance(t, int) or nbytes <= 0:
        return
    have = t.numel() * t.element_size()
    if have < nbytes:
        raise ValueError(f"{what}: {have} bytes, the call touches {nbytes}")


def _int64(t, what: str) -> None:
    if t is not None and not isinstance(t, int) and t.dtype != torch.int64:
        raise ValueError(f"{what} must be int64, got {t.dtype}")


def _layout_checks(topk_idx, E: int, R: int, cnt, ntr, itr, off, n_off: int) -> tuple[int, int]:
    T, K = topk_idx.shape
    _int64(topk_idx, "topk_idx")
    _need(cnt, 4 * E, "num_tokens_per_expert")
    _need(ntr, 4 * R, "num_tokens_per_rank")
    _need(itr, T * R, "is_token_in_rank")
    _need(off, 4 * n_off, "offsets")
    return T, K


def _remember(h, T: int, K: int, E: int):
    h.T, h.K, h.E = T, K, E
    return h


def _tk(handle) -> tuple[int, int]:
    """(T, K) of the handle's last layout through this binding (0, 0 if unknown)."""
    return (handle.T or 0, handle.K or 0) if isinstance(handle, Handle) else (0, 0)


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _fnptr(f):
    """A ctypes CFUNCTYPE callback (or None) as a plain function pointer."""
    return None if f is None else ctypes.cast(f, ctypes.c_void_p).value


def _check(st: int, call: str) -> None:
    if st != EP_OK:
        raise EPError(st, call)


class Handle:
    """Owner of an ep_handle_t; destroyed explicitly or when garbage-collected."""

    def __init__(self):
        self.ptr = ctypes.c_void_p(None)
        self.T = self.K = self.E = None   # routing shape of the last layout through this binding

    def __bool__(self):
        return bool(self.ptr.value)

    def destroy(self):
        if self.ptr.value:
            _check(lib().ep_handle_destroy(self.ptr), "ep_handle_destroy")
            self.ptr = ctypes.c_void_p(None)

    def __del__(self):
        try:
            if self.ptr.value and _lib is not None:
                _lib.ep_handle_destroy(self.ptr)
        except Exception:
            pass


def ep_layout(topk_idx, num_experts: int, num_ranks: int, num_tokens_per_expert,
              num_tokens_per_rank, is_token_in_rank, expert_offsets, handle: Handle | None = None,
              stream=None, alloc_fn=None, free_fn=None) -> Handle:
    """Routing layout of topk_idx [T, K] int64 into the given int32/uint8 outputs.

    Reuses `handle` if given (no allocation), else creates one. Returns the handle.
    """
    T, K = _layout_checks(topk_idx, num_experts, num_ranks, num_tokens_per_expert, num_tokens_per_rank,
                          is_token_in_rank, expert_offsets, num_experts + 1)
    h = handle if handle is not None else Handle()
    st = lib().ep_layout(_ptr(topk_idx), T, K, num_experts, num_ranks, _ptr(num_tokens_per_expert),
                         _ptr(num_tokens_per_rank), _ptr(is_token_in_rank), _ptr(expert_offsets),
                         _fnptr(alloc_fn), _fnptr(free_fn), ctypes.byref(h.ptr), _stream(stream))
    _check(st, "ep_layout")
    return _remember(h, T, K, num_experts)


def ep_layout_aligned(topk_idx, num_experts: int, num_ranks: int, expert_alignment: int,
                      num_tokens_per_expert, num_tokens_per_rank, is_token_in_rank, expert_offsets,
                      handle: Handle | None = None, stream=None, alloc_fn=None, free_fn=None) -> Handle:
    """ep_layout with each expert's rows starting on a multiple of expert_alignment."""
    T, K = _layout_checks(topk_idx, num_experts, num_ranks, num_tokens_per_expert, num_tokens_per_rank,
                          is_token_in_rank, expert_offsets, num_experts + 1)
    h = handle if handle is not None else Handle()
    st = lib().ep_layout_aligned(_ptr(topk_idx), T, K, num_experts, num_ranks, int(expert_alignment),
                                 _ptr(num_tokens_per_expert), _ptr(num_tokens_per_rank), _ptr(is_token_in_rank),
                                 _ptr(expert_offsets), _fnptr(alloc_fn), _fnptr(free_fn), ctypes.byref(h.ptr),
                                 _stream(stream))
    _check(st, "ep_layout_aligned")
    return _remember(h, T, K, num_experts)


def ep_layout_strided(topk_idx, num_experts: int, num_ranks: int, expert_capacity: int,
                      num_tokens_per_expert, num_tokens_per_rank, is_token_in_rank, expert_offsets,
                      handle: Handle | None = None, stream=None, alloc_fn=None, free_fn=None) -> Handle:
    """ep_layout into the padded 3-D receive buffer [E, expert_capacity, H]."""
    T, K = _layout_checks(topk_idx, num_experts, num_ranks, num_tokens_per_expert, num_tokens_per_rank,
                          is_token_in_rank, expert_offsets, num_experts + 1)
    h = handle if handle is not None else Handle()
    st = lib().ep_layout_strided(_ptr(topk_idx), T, K, num_experts, num_ranks, int(expert_capacity),
                                 _ptr(num_tokens_per_expert), _ptr(num_tokens_per_rank), _ptr(is_token_in_rank),
                                 _ptr(expert_offsets), _fnptr(alloc_fn), _fnptr(free_fn), ctypes.byref(h.ptr),
                                 _stream(stream))
    _check(st, "ep_layout_strided")
    return _remember(h, T, K, num_experts)


def ep_layout_nonexpand(topk_idx, num_experts: int, num_ranks: int, num_tokens_per_expert,
                        num_tokens_per_rank, is_token_in_rank, rank_offsets, handle: Handle | None = None,
                        stream=None, alloc_fn=None, free_fn=None) -> Handle:
    """Layout with one receive row per (token, rank) pair, grouped by rank."""
    T, K = _layout_checks(topk_idx, num_experts, num_ranks, num_tokens_per_expert, num_tokens_per_rank,
                          is_token_in_rank, rank_offsets, num_ranks + 1)
    h = handle if handle is not None else Handle()
    st = lib().ep_layout_nonexpand(_ptr(topk_idx), T, K, num_experts, num_ranks, _ptr(num_tokens_per_expert),
                                   _ptr(num_tokens_per_rank), _ptr(is_token_in_rank), _ptr(rank_offsets),
                                   _fnptr(alloc_fn), _fnptr(free_fn), ctypes.byref(h.ptr), _stream(stream))
    _check(st, "ep_layout_nonexpand")
    return _remember(h, T, K, num_experts)


def ep_nonexpand_recv_topk(handle: Handle, topk_idx, num_experts: int, recv_topk_idx, recv_topk_weights=None,
                           topk_weights=None, recv_capacity: int | None = None, stream=None) -> None:
    """Per non-expand receive row: rank-local expert ids (or -1) and weights."""
    cap = int(recv_topk_idx.shape[0]) if recv_capacity is None else int(recv_capacity)
    T, K = topk_idx.shape
    _int64(topk_idx, "topk_idx")
    _int64(recv_topk_idx, "recv_topk_idx")
    _need(topk_weights, 4 * T * K, "topk_weights")
    _need(recv_topk_idx, 8 * cap * K, "recv_topk_idx")
    _need(recv_topk_weights, 4 * cap * K, "recv_topk_weights")
    st = lib().ep_nonexpand_recv_topk(handle.ptr, _ptr(topk_idx), _ptr(topk_weights), num_experts,
                                      _ptr(recv_topk_idx), _ptr(recv_topk_weights), cap, _stream(stream))
    _check(st, "ep_nonexpand_recv_topk")


def ep_dispatch(handle: Handle, x, out_dtype: int, recv_x, recv_capacity: int, recv_scales=None,
                recv_src_token=None, recv_weights=None, topk_weights=None, stream=None) -> None:
    """Permute x [T, H] bf16 into recv_x (bf16 [cap, H] or uint8 [cap, H] for fp8)."""
    H = x.shape[-1]
    T, K = _tk(handle)
    cap = int(recv_capacity)
    _need(x, 2 * T * H, "x")
    _need(recv_x, cap * H * (2 if out_dtype == EP_DTYPE_BF16 else 1), "recv_x")
    if out_dtype != EP_DTYPE_BF16:
        _need(recv_scales, 4 * cap * (H // 128), "recv_scales")
    _need(recv_src_token, 4 * cap, "recv_src_token")
    _need(recv_weights, 4 * cap, "recv_weights")
    _need(topk_weights, 4 * T * K, "topk_weights")
    st = lib().ep_dispatch(handle.ptr, _ptr(x), H, out_dtype, _ptr(topk_weights), _ptr(recv_x),
                           _ptr(recv_scales), _ptr(recv_src_token), _ptr(recv_weights),
                           int(recv_capacity), _stream(stream))
    _check(st, "ep_dispatch")


def ep_dispatch_ex(handle: Handle, x, recv_x, recv_capacity: int, out_dtype: int = EP_DTYPE_FP8_E4M3,
                   in_dtype: int = EP_DTYPE_BF16, scale_mode: int = EP_SCALE_FP32, x_scales=None, recv_scales=None,
                   scales_col_major: bool = False, scales_ld: int = 0, recv_src_token=None, recv_weights=None,
                   topk_weights=None, H: int | None = None, overlap_layout: bool = False, stream=None) -> None:
    """ep_dispatch with fp8 scale modes, column-major scales, fp8 input pass-through and
    overlap with the layout that precedes it on the stream."""
    H = int(x.shape[-1]) if H is None else int(H)
    T, K = _tk(handle)
    cap = int(recv_capacity)
    nb = H // 128
    sbytes = 1 if scale_mode == EP_SCALE_UE8M0 else 4
    _need(x, T * H * (2 if in_dtype == EP_DTYPE_BF16 else 1), "x")
    if in_dtype != EP_DTYPE_BF16:
        _need(x_scales, sbytes * T * nb, "x_scales")
    _need(recv_x, cap * H * (2 if out_dtype == EP_DTYPE_BF16 else 1), "recv_x")
    if out_dtype != EP_DTYPE_BF16:
        _need(recv_scales, sbytes * (nb * int(scales_ld) if scales_col_major else cap * nb), "recv_scales")
    _need(recv_src_token, 4 * cap, "recv_src_token")
    _need(recv_weights, 4 * cap, "recv_weights")
    _need(topk_weights, 4 * T * K, "topk_weights")
    cfg = DispatchConfig(in_dtype, out_dtype, scale_mode, 1 if scales_col_major else 0, int(scales_ld),
                         1 if overlap_layout else 0)
    st = lib().ep_dispatch_ex(handle.ptr, _ptr(x), _ptr(x_scales), H, ctypes.byref(cfg), _ptr(topk_weights),
                              _ptr(recv_x), _ptr(recv_scales), _ptr(recv_src_token), _ptr(recv_weights),
                              int(recv_capacity), _stream(stream))
    _check(st, "ep_dispatch_ex")


def ep_combine(handle: Handle, y, out, topk_weights=None, y_rows: int | None = None, stream=None) -> None:
    """out [T, H] bf16 = weighted sum over each token's slots of y [rows, H] bf16."""
    H = y.shape[-1] if y is not None else out.shape[-1]
    rows = int(y.shape[0]) if y_rows is None else int(y_rows)
    T, K = _tk(handle)
    _need(y, 2 * rows * H, "y")
    _need(out, 2 * T * H, "out")
    _need(topk_weights, 4 * T * K, "topk_weights")
    st = lib().ep_combine(handle.ptr, _ptr(y), rows, H, _ptr(topk_weights), _ptr(out), _stream(stream))
    _check(st, "ep_combine")


def ep_combine_backward(handle: Handle, grad_out, y=None, topk_weights=None, grad_y=None,
                        grad_topk_weights=None, y_rows: int | None = None, grad_y_capacity: int | None = None,
                        stream=None) -> None:
    """grad_y[row] = bf16(w * grad_out[t]); grad_topk_weights[t,k] = <grad_out[t], y[row]>."""
    H = grad_out.shape[-1]
    rows = (int(y.shape[0]) if y is not None else 0) if y_rows is None else int(y_rows)
    cap = (int(grad_y.shape[0]) if grad_y is not None else 0) if grad_y_capacity is None else int(grad_y_capacity)
    T, K = _tk(handle)
    _need(grad_out, 2 * T * H, "grad_out")
    _need(y, 2 * rows * H, "y")
    _need(topk_weights, 4 * T * K, "topk_weights")
    _need(grad_y, 2 * cap * H, "grad_y")
    _need(grad_topk_weights, 4 * T * K, "grad_topk_weights")
    st = lib().ep_combine_backward(handle.ptr, _ptr(grad_out), _ptr(y), rows, H, _ptr(topk_weights), _ptr(grad_y),
                                   cap, _ptr(grad_topk_weights), _stream(stream))
    _check(st, "ep_combine_backward")


def ep_dispatch_backward(handle: Handle, grad_recv, grad_x, grad_recv_weights=None, grad_topk_weights=None,
                         grad_rows: int | None = None, stream=None) -> None:
    """grad_x[t] = bf16(sum_k grad_recv[row(t,k)]); grad_topk_weights[t,k] = grad_recv_weights[row]."""
    H = grad_x.shape[-1]
    rows = int(grad_recv.shape[0]) if grad_rows is None else int(grad_rows)
    T, K = _tk(handle)
    _need(grad_recv, 2 * rows * H, "grad_recv")
    _need(grad_recv_weights, 4 * rows, "grad_recv_weights")
    _need(grad_x, 2 * T * H, "grad_x")
    _need(grad_topk_weights, 4 * T * K, "grad_topk_weights")
    st = lib().ep_dispatch_backward(handle.ptr, _ptr(grad_recv), rows, H, _ptr(grad_recv_weights), _ptr(grad_x),
                                    _ptr(grad_topk_weights), _stream(stream))
    _check(st, "ep_dispatch_backward")


def ep_topk_to_routing_map(topk_idx, num_experts: int, routing_map, topk_weights=None, probs=None,
                           device_error=None, stream=None) -> None:
    """routing_map [T, E] u8 (and probs [T, E] fp32) from topk_idx [T, K]."""
    T, K = topk_idx.shape
    _int64(topk_idx, "topk_idx")
    _need(topk_weights, 4 * T * K, "topk_weights")
    _need(routing_map, T * num_experts, "routing_map")
    _need(probs, 4 * T * num_experts, "probs")
    _need(device_error, 4, "device_error")
    st = lib().ep_topk_to_routing_map(_ptr(topk_idx), _ptr(topk_weights), T, K, num_experts, _ptr(routing_map),
                                      _ptr(probs), _ptr(device_error), _stream(stream))
    _check(st, "ep_topk_to_routing_map")


def ep_routing_map_to_topk(routing_map, num_topk: int, topk_idx, probs=None, topk_weights=None,
                           device_error=None, stream=None) -> None:
    """topk_idx [T, K] int64 (and weights) from routing_map [T, E], experts ascending."""
    T, E = routing_map.shape
    _int64(topk_idx, "topk_idx")
    _need(probs, 4 * T * E, "probs")
    _need(topk_idx, 8 * T * num_topk, "topk_idx")
    _need(topk_weights, 4 * T * num_topk, "topk_weights")
    _need(device_error, 4, "device_error")
    st = lib().ep_routing_map_to_topk(_ptr(routing_map), _ptr(probs), T, E, num_topk, _ptr(topk_idx),
                                      _ptr(topk_weights), _ptr(device_error), _stream(stream))
    _check(st, "ep_routing_map_to_topk")


def ep_handle_query(handle: Handle) -> tuple[int, int]:
    """(N, device error word) after the last ep_layout; synchronises its stream."""
    n = ctypes.c_int64(0)
    err = ctypes.c_int32(0)
    st = lib().ep_handle_query(handle.ptr, ctypes.byref(n), ctypes.byref(err))
    if st not in (EP_OK, EP_ERR_INVALID_EXPERT, EP_ERR_CAPACITY):
        _check(st, "ep_handle_query")
    return n.value, err.value


def ep_handle_copy_row_of_slot(handle: Handle, dst, stream=None) -> None:
    T, K = _tk(handle)
    _need(dst, 4 * T * K, "dst")
    _check(lib().ep_handle_copy_row_of_slot(handle.ptr, _ptr(dst), _stream(stream)),
           "ep_handle_copy_row_of_slot")


def ep_layout_noalloc(topk_idx, num_experts: int, num_ranks: int, num_tokens_per_expert,
                      num_tokens_per_rank, is_token_in_rank, expert_offsets, row_of_slot,
                      device_error=None, stream=None) -> None:
    """ep_layout without a handle or any allocation: the slot -> row map goes
    to the caller's row_of_slot [T, K] int32; scratch is the library's fixed
    array (one call at a time per device, ordered on one stream)."""
    T, K = _layout_checks(topk_idx, num_experts, num_ranks, num_tokens_per_expert, num_tokens_per_rank,
                          is_token_in_rank, expert_offsets, num_experts + 1)
    _need(row_of_slot, 4 * T * K, "row_of_slot")
    _need(device_error, 4, "device_error")
    st = lib().ep_layout_noalloc(_ptr(topk_idx), T, K, num_experts, num_ranks, _ptr(num_tokens_per_expert),
                                 _ptr(num_tokens_per_rank), _ptr(is_token_in_rank), _ptr(expert_offsets),
                                 _ptr(row_of_slot), _ptr(device_error), _stream(stream))
    _check(st, "ep_layout_noalloc")


def ep_handle_layout_kernels(handle: Handle) -> int:
    """Kernels the last ep_layout on `handle` enqueued (1 or 3; 0 for T = 0)."""
    return int(lib().ep_handle_layout_kernels(handle.ptr))


def ep_layout_cluster_ctas(T: int, K: int, E: int, R: int) -> int:
    """CTAs per cluster of the single-launch layout of such a routing on the
    current device, 0 for the three-kernel path, -1 for invalid arguments."""
    return int(lib().ep_layout_cluster_ctas(T, K, E, R))


def ep_handle_destroy(handle: Handle) -> None:
    handle.destroy()
