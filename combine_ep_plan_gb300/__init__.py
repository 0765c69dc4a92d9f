"""GB300 (sm_103a) MoE expert-parallel routing plan, dispatch and combine.

A thin ctypes binding over the C ABI declared in ``include/ep_plan.h``
(``libep_gb300.so``, built in-tree by ``combine_ep_plan_gb300.build``).  This
module only checks and marshals arguments and allocates outputs with torch:
every step of the plan, dispatch and combine runs in the library's CUDA
kernels.  There is no CPU or PyTorch fallback: if the library is missing or a
call fails, an exception is raised.

The P logical ranks of the method live on one GPU: source rank s owns global
tokens g = s*S + t, expert e lives on rank e // (E/P).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

__all__ = [
    "EPError", "EPHandle", "plan", "dispatch", "dispatch_fresh", "dispatch_cached", "combine",
    "worst_expanded_rows", "library_path", "load_library", "FIELDS", "set_plan_wait_debug",
    "dispatch_backward", "combine_backward", "dispatch_metadata",
    "Pending", "dispatch_async", "combine_async", "PROFILE_KERNELS", "PROFILE_WORDS", "summarize_profile",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libep_gb300.so")

EP_OK, EP_ERR_INVALID, EP_ERR_CAPACITY, EP_ERR_TIMEOUT, EP_ERR_CUDA, EP_ERR_MISMATCH, EP_ERR_OOM = range(7)
EP_DTYPE_BF16, EP_DTYPE_FP8_E4M3 = 0, 1
EP_DISPATCH_ZERO_PAD, EP_DISPATCH_SCALES_COL_MAJOR = 1, 2

# field name -> (enum value, torch dtype)
FIELDS = {
    "is_token_in_rank": (0, torch.uint8),
    "send_head": (1, torch.int32),
    "num_tokens_per_rank": (2, torch.int32),
    "num_tokens_per_expert": (3, torch.int32),
    "expert_counts": (4, torch.int32),
    "num_recv": (5, torch.int32),
    "rank_prefix": (6, torch.int32),
    "channel_prefix": (7, torch.int32),
    "recv_channel_prefix": (8, torch.int32),
    "recv_offsets": (9, torch.int32),
    "recv_src_idx": (10, torch.int32),
    "expert_offsets": (11, torch.int32),
    "slot": (12, torch.int32),
    "exp_src": (13, torch.int32),
    "pad_rows": (14, torch.int32),
}

_TYPESTR = {torch.uint8: "|u1", torch.int32: "<i4"}


class EPError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        msg = _lib().ep_status_string(code).decode() if _LIB is not None else f"status {code}"
        super().__init__(f"{what}: {msg}" if what else msg)
        self.code = code


_LIB = None


def library_path() -> str:
    return _LIB_PATH


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = path or _LIB_PATH
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with `python -m combine_ep_plan_gb300.build` "
            "(there is no fallback implementation)")
    lib = ctypes.CDLL(path)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    st = ctypes.c_int
    lib.ep_abi_version.restype = i32
    lib.ep_abi_version.argtypes = []
    lib.ep_status_string.restype = ctypes.c_char_p
    lib.ep_status_string.argtypes = [st]
    lib.ep_plan.restype = st
    lib.ep_plan.argtypes = [vp, i64, i32, i32, i32, i32, i32, vp, ctypes.POINTER(vp)]
    lib.ep_replan.restype = st
    lib.ep_replan.argtypes = [vp, vp, vp]
    lib.ep_plan_sizes.restype = st
    lib.ep_plan_sizes.argtypes = [vp, vp, ctypes.POINTER(i64), ctypes.POINTER(i64)]
    lib.ep_worst_expanded_rows.restype = i64
    lib.ep_worst_expanded_rows.argtypes = [i64, i32, i32, i32]
    lib.ep_dispatch.restype = st
    lib.ep_dispatch.argtypes = [vp, vp, i32, vp, i64, i32, i32, vp, vp, i64, vp]
    lib.ep_dispatch_cached.restype = st
    lib.ep_dispatch_cached.argtypes = [vp, i32, i32, i64, vp, i32, vp, i64, i32, i32, vp, vp, i64, vp]
    lib.ep_dispatch_fresh.restype = st
    lib.ep_dispatch_fresh.argtypes = [vp, i64, i32, i32, i32, i32, i32, vp, i32, vp, i64, i32, i32, vp, vp,
                                      i64, vp, ctypes.POINTER(vp)]
    lib.ep_dispatch_metadata.restype = st
    lib.ep_dispatch_metadata.argtypes = [vp, vp, vp, vp, i64, i32, vp]
    lib.ep_combine.restype = st
    lib.ep_combine.argtypes = [vp, vp, i64, vp, vp, i64, vp, vp]
    lib.ep_dispatch_backward.restype = st
    lib.ep_dispatch_backward.argtypes = [vp, vp, i64, i64, vp, vp]
    lib.ep_combine_backward.restype = st
    lib.ep_combine_backward.argtypes = [vp, vp, vp, i64, vp, i64, i32, vp, i64, vp, vp]
    lib.ep_sync_status.restype = st
    lib.ep_sync_status.argtypes = [vp, vp]
    lib.ep_handle_get.restype = st
    lib.ep_handle_get.argtypes = [vp, i32, ctypes.POINTER(vp), ctypes.POINTER(i64), ctypes.POINTER(i32)]
    lib.ep_handle_info.restype = st
    lib.ep_handle_info.argtypes = [vp, ctypes.POINTER(i64)] + [ctypes.POINTER(i32)] * 5
    lib.ep_handle_destroy.restype = st
    lib.ep_handle_destroy.argtypes = [vp, vp]
    lib.ep_debug_set_plan_wait.restype = None
    lib.ep_debug_set_plan_wait.argtypes = [i64, i32]
    lib.ep_set_num_sms.restype = st
    lib.ep_set_num_sms.argtypes = [vp, i32]
    lib.ep_dispatch_async.restype = st
    lib.ep_dispatch_async.argtypes = [vp, vp, vp, i32, vp, i64, i32, i32, vp, vp, i64, vp, vp, i32,
                                      ctypes.POINTER(vp)]
    lib.ep_combine_async.restype = st
    lib.ep_combine_async.argtypes = [vp, vp, i64, vp, vp, i64, vp, vp, vp, i32, ctypes.POINTER(vp)]
    lib.ep_pending_wait.restype = st
    lib.ep_pending_wait.argtypes = [vp, ctypes.POINTER(i64), ctypes.POINTER(i64)]
    lib.ep_profile_begin.restype = st
    lib.ep_profile_begin.argtypes = [vp, vp, i64]
    lib.ep_profile_end.restype = st
    lib.ep_profile_end.argtypes = [vp, ctypes.POINTER(i64), ctypes.POINTER(i64)]
    _LIB = lib
    return lib


def _lib() -> ctypes.CDLL:
    return _LIB if _LIB is not None else load_library()


def _stream_ptr(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _check(code: int, what: str):
    if code != EP_OK:
        raise EPError(code, what)


def _need(t: torch.Tensor, name: str, dtype, ndim: int):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-d tensor")


class _ArrayView:
    """Non-owning device view handed to torch through __cuda_array_interface__."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {
            "shape": tuple(int(s) for s in shape), "typestr": typestr,
            "data": (ptr, False), "version": 3, "strides": None, "stream": None,
        }


class EPHandle:
    """A routing plan: owns the library handle and its device arrays."""

    def __init__(self, ptr: int, stream: Optional[torch.cuda.Stream]):
        self._ptr = ptr
        lib = _lib()
        S = ctypes.c_int64()
        P, K, E, A, C = (ctypes.c_int() for _ in range(5))
        _check(lib.ep_handle_info(ptr, ctypes.byref(S), ctypes.byref(P), ctypes.byref(K),
                                  ctypes.byref(E), ctypes.byref(A), ctypes.byref(C)), "ep_handle_info")
        self.S, self.P, self.K, self.E, self.A, self.C = S.value, P.value, K.value, E.value, A.value, C.value
        self.device = torch.cuda.current_device()
        self._sizes = None

    @property
    def T(self) -> int:
        return self.P * self.S

    @property
    def ptr(self) -> int:
        if not self._ptr:
            raise RuntimeError("handle has been destroyed")
        return self._ptr

    def field(self, name: str) -> torch.Tensor:
        """A torch view (no copy) of one plan array; valid while the handle lives."""
        enum, dtype = FIELDS[name]
        p = ctypes.c_void_p()
        shape = (ctypes.c_int64 * 3)()
        nd = ctypes.c_int()
        _check(_lib().ep_handle_get(self.ptr, enum, ctypes.byref(p), shape, ctypes.byref(nd)), name)
        view = _ArrayView(p.value, list(shape)[: nd.value], _TYPESTR[dtype])
        return torch.as_tensor(view, device=f"cuda:{self.device}")

    def sizes(self, stream: Optional[torch.cuda.Stream] = None, refresh: bool = False) -> Tuple[int, int]:
        """(N_exp, N_recv); synchronises the stream on the first call after a
        plan made through this object.  refresh=True reads them again (after
        plans this object did not see, such as replays of a captured graph)."""
        if self._sizes is None or refresh:
            ne, nr = ctypes.c_int64(), ctypes.c_int64()
            _check(_lib().ep_plan_sizes(self.ptr, _stream_ptr(stream), ctypes.byref(ne), ctypes.byref(nr)),
                   "ep_plan_sizes")
            self._sizes = (ne.value, nr.value)
        return self._sizes

    def replan(self, topk_idx: torch.Tensor, stream: Optional[torch.cuda.Stream] = None):
        _need(topk_idx, "topk_idx", torch.int64, 2)
        _check(_lib().ep_replan(self.ptr, topk_idx.data_ptr(), _stream_ptr(stream)), "ep_replan")
        self._sizes = None

    def sync_status(self, stream: Optional[torch.cuda.Stream] = None) -> int:
        """Synchronise and return (and clear) the device status code."""
        return _lib().ep_sync_status(self.ptr, _stream_ptr(stream))

    def check(self, stream: Optional[torch.cuda.Stream] = None):
        _check(self.sync_status(stream), "device status")

    def set_num_sms(self, num_sms: int):
        """SM budget of this handle's kernels (0 = the whole device)."""
        _check(_lib().ep_set_num_sms(self.ptr, int(num_sms)), "ep_set_num_sms")

    def profile_begin(self, capacity: int = 1 << 16):
        """Start per-CTA profile records (capacity records of PROFILE_WORDS uint64)."""
        self._prof = torch.zeros((capacity, PROFILE_WORDS), dtype=torch.int64, device=f"cuda:{self.device}")
        _check(_lib().ep_profile_begin(self.ptr, self._prof.data_ptr(), capacity), "ep_profile_begin")

    def profile_end(self, stream: Optional[torch.cuda.Stream] = None):
        """Stop recording; synchronise the device (the launches may have run
        on the handle's communication stream) and return (records [n, 8]
        int64 on the host, dropped count)."""
        n, dropped = ctypes.c_int64(), ctypes.c_int64()
        _check(_lib().ep_profile_end(self.ptr, ctypes.byref(n), ctypes.byref(dropped)), "ep_profile_end")
        torch.cuda.synchronize(self.device)
        rec = self._prof[: n.value].cpu()
        self._prof = None
        return rec, dropped.value

    def destroy(self, stream: Optional[torch.cuda.Stream] = None):
        if self._ptr:
            _check(_lib().ep_handle_destroy(self._ptr, _stream_ptr(stream)), "ep_handle_destroy")
            self._ptr = 0

    def __del__(self):
        try:
            if self._ptr and _LIB is not None and torch.cuda.is_initialized():
                self.destroy()
        except Exception:
            pass


def plan(topk_idx: torch.Tensor, num_ranks: int, num_experts: int, expert_alignment: int = 1,
         num_channels: int = 0, stream: Optional[torch.cuda.Stream] = None) -> EPHandle:
    """Build the routing plan from topk_idx [T,K] int64 (T = num_ranks * S)."""
    _need(topk_idx, "topk_idx", torch.int64, 2)
    T, K = topk_idx.shape
    if T % num_ranks:
        raise ValueError("topk_idx rows must be a multiple of num_ranks")
    h = ctypes.c_void_p()
    _check(_lib().ep_plan(topk_idx.data_ptr(), T // num_ranks, num_ranks, K, num_experts,
                          expert_alignment, num_channels, _stream_ptr(stream), ctypes.byref(h)), "ep_plan")
    return EPHandle(h.value, stream)


def worst_expanded_rows(num_tokens: int, num_topk: int, num_experts: int, expert_alignment: int) -> int:
    return int(_lib().ep_worst_expanded_rows(num_tokens, num_topk, num_experts, expert_alignment))


def _dispatch_outputs(H, out_dtype, recv_x, recv_scales, capacity, device, col_major):
    if recv_x is None:
        dt = torch.bfloat16 if out_dtype == "bf16" else torch.float8_e4m3fn
        recv_x = torch.empty((capacity, H), dtype=dt, device=device)
    if out_dtype == "fp8" and recv_scales is None:
        rows = recv_x.shape[0]
        if col_major:  # [rows, H/128] view of a [H/128, rows] buffer: strides (1, rows)
            recv_scales = torch.empty((H // 128, rows), dtype=torch.float32, device=device).t()
        else:
            recv_scales = torch.empty((rows, H // 128), dtype=torch.float32, device=device)
    return recv_x, recv_scales


def _dtype_code(out_dtype: str) -> int:
    if out_dtype == "bf16":
        return EP_DTYPE_BF16
    if out_dtype == "fp8":
        return EP_DTYPE_FP8_E4M3
    raise ValueError("out_dtype must be 'bf16' or 'fp8'")


def _input_code(x: torch.Tensor, x_scales: Optional[torch.Tensor]):
    if x.dtype == torch.bfloat16:
        if x_scales is not None:
            raise ValueError("x_scales only goes with pre-quantised float8_e4m3fn input")
        return EP_DTYPE_BF16
    if x.dtype == torch.float8_e4m3fn:
        if x_scales is None:
            raise ValueError("pre-quantised input needs x_scales [T, H/128] float32")
        _need(x_scales, "x_scales", torch.float32, 2)
        if tuple(x_scales.shape) != (x.shape[0], x.shape[1] // 128):
            raise ValueError("x_scales must be [T, H/128]")
        return EP_DTYPE_FP8_E4M3
    raise TypeError("x must be bfloat16 or float8_e4m3fn")


def _check_dispatch(x, recv_x, recv_scales, out_dtype, col_major):
    if not isinstance(x, torch.Tensor) or not x.is_cuda or x.dim() != 2 or not x.is_contiguous():
        raise ValueError("x must be a contiguous 2-d CUDA tensor")
    want = torch.bfloat16 if out_dtype == "bf16" else torch.float8_e4m3fn
    _need(recv_x, "recv_x", want, 2)
    if recv_x.shape[1] != x.shape[1]:
        raise ValueError("recv_x hidden size differs from x")
    if out_dtype == "fp8":
        if recv_scales is None or recv_scales.dtype != torch.float32 or not recv_scales.is_cuda:
            raise TypeError("recv_scales must be a float32 CUDA tensor")
        if tuple(recv_scales.shape) != (recv_x.shape[0], x.shape[1] // 128):
            raise ValueError("recv_scales must be [rows, H/128]")
        if col_major and not recv_scales.t().is_contiguous():
            raise ValueError("column-major recv_scales must have strides (1, rows)")
        if not col_major and not recv_scales.is_contiguous():
            raise ValueError("row-major recv_scales must be contiguous")
    elif col_major:
        raise ValueError("column-major scales need FP8 output")


def _flags(zero_pad: bool, col_major: bool) -> int:
    return (EP_DISPATCH_ZERO_PAD if zero_pad else 0) | (EP_DISPATCH_SCALES_COL_MAJOR if col_major else 0)


def dispatch(handle: EPHandle, x: torch.Tensor, out_dtype: str = "bf16", zero_pad: bool = True,
             recv_x: Optional[torch.Tensor] = None, recv_scales: Optional[torch.Tensor] = None,
             capacity: Optional[int] = None, stream: Optional[torch.cuda.Stream] = None,
             x_scales: Optional[torch.Tensor] = None, scales_col_major: bool = False):
    """Row scatter of x [T,H] (bf16, or float8_e4m3fn with x_scales) into the
    expanded layout.

    Without recv_x, the output is allocated with the exact row count, which
    synchronises the stream once (ep_plan_sizes); pass recv_x (e.g. sized by
    worst_expanded_rows) to avoid that.  Returns (recv_x, recv_scales|None).
    """
    code = _dtype_code(out_dtype)
    xcode = _input_code(x, x_scales)
    H = x.shape[1]
    if recv_x is None and capacity is None:
        capacity = handle.sizes(stream)[0]
    recv_x, recv_scales = _dispatch_outputs(H, out_dtype, recv_x, recv_scales, capacity, x.device,
                                            scales_col_major)
    _check_dispatch(x, recv_x, recv_scales, out_dtype, scales_col_major)
    _check(_lib().ep_dispatch(handle.ptr, x.data_ptr(), xcode,
                              x_scales.data_ptr() if x_scales is not None else None, H, code,
                              _flags(zero_pad, scales_col_major), recv_x.data_ptr(),
                              recv_scales.data_ptr() if recv_scales is not None else None,
                              recv_x.shape[0], _stream_ptr(stream)), "ep_dispatch")
    return recv_x, recv_scales


def dispatch_cached(handle: EPHandle, x: torch.Tensor, num_experts: int, expert_alignment: int,
                    num_tokens_per_rank: int, out_dtype: str = "bf16", zero_pad: bool = True,
                    recv_x: Optional[torch.Tensor] = None, recv_scales: Optional[torch.Tensor] = None,
                    stream: Optional[torch.cuda.Stream] = None, x_scales: Optional[torch.Tensor] = None,
                    scales_col_major: bool = False):
    """Cached-handle dispatch: checks (E, A, S) against the handle first."""
    code = _dtype_code(out_dtype)
    xcode = _input_code(x, x_scales)
    H = x.shape[1]
    capacity = handle.sizes(stream)[0] if recv_x is None else None
    recv_x, recv_scales = _dispatch_outputs(H, out_dtype, recv_x, recv_scales, capacity, x.device,
                                            scales_col_major)
    _check_dispatch(x, recv_x, recv_scales, out_dtype, scales_col_major)
    _check(_lib().ep_dispatch_cached(handle.ptr, num_experts, expert_alignment, num_tokens_per_rank,
                                     x.data_ptr(), xcode, x_scales.data_ptr() if x_scales is not None else None,
                                     H, code, _flags(zero_pad, scales_col_major), recv_x.data_ptr(),
                                     recv_scales.data_ptr() if recv_scales is not None else None,
                                     recv_x.shape[0], _stream_ptr(stream)), "ep_dispatch_cached")
    return recv_x, recv_scales


def dispatch_fresh(topk_idx: torch.Tensor, x: torch.Tensor, num_ranks: int, num_experts: int,
                   expert_alignment: int = 1, num_channels: int = 0, out_dtype: str = "bf16",
                   zero_pad: bool = True, recv_x: Optional[torch.Tensor] = None,
                   recv_scales: Optional[torch.Tensor] = None,
                   stream: Optional[torch.cuda.Stream] = None, x_scales: Optional[torch.Tensor] = None,
                   scales_col_major: bool = False):
    """Plan + dispatch in one library call; outputs default to the worst-case
    row count (no synchronisation).  Returns (handle, recv_x, recv_scales)."""
    _need(topk_idx, "topk_idx", torch.int64, 2)
    code = _dtype_code(out_dtype)
    xcode = _input_code(x, x_scales)
    T, K = topk_idx.shape
    H = x.shape[1]
    cap = worst_expanded_rows(T, K, num_experts, expert_alignment)
    recv_x, recv_scales = _dispatch_outputs(H, out_dtype, recv_x, recv_scales, cap, x.device, scales_col_major)
    _check_dispatch(x, recv_x, recv_scales, out_dtype, scales_col_major)
    h = ctypes.c_void_p()
    _check(_lib().ep_dispatch_fresh(topk_idx.data_ptr(), T // num_ranks, num_ranks, K, num_experts,
                                    expert_alignment, num_channels, x.data_ptr(), xcode,
                                    x_scales.data_ptr() if x_scales is not None else None, H, code,
                                    _flags(zero_pad, scales_col_major), recv_x.data_ptr(),
                                    recv_scales.data_ptr() if recv_scales is not None else None,
                                    recv_x.shape[0], _stream_ptr(stream), ctypes.byref(h)),
           "ep_dispatch_fresh")
    return EPHandle(h.value, stream), recv_x, recv_scales


def dispatch_metadata(handle: EPHandle, topk_weights: torch.Tensor, capacity: Optional[int] = None,
                      recv_weights: Optional[torch.Tensor] = None, recv_meta: Optional[torch.Tensor] = None,
                      zero_pad: bool = True, stream: Optional[torch.cuda.Stream] = None):
    """Per expanded row: (routing weight [rows] f32, {source token, slot k} [rows,2] i32)."""
    _need(topk_weights, "topk_weights", torch.float32, 2)
    if tuple(topk_weights.shape) != (handle.T, handle.K):
        raise ValueError("topk_weights must be [T,K]")
    if capacity is None:
        capacity = recv_weights.shape[0] if recv_weights is not None else handle.sizes(stream)[0]
    if recv_weights is None:
        recv_weights = torch.empty(capacity, dtype=torch.float32, device=topk_weights.device)
    if recv_meta is None:
        recv_meta = torch.empty((capacity, 2), dtype=torch.int32, device=topk_weights.device)
    _need(recv_weights, "recv_weights", torch.float32, 1)
    _need(recv_meta, "recv_meta", torch.int32, 2)
    if recv_weights.shape[0] < capacity or recv_meta.shape[0] < capacity:
        raise ValueError("output buffers smaller than capacity")
    _check(_lib().ep_dispatch_metadata(handle.ptr, topk_weights.data_ptr(), recv_weights.data_ptr(),
                                       recv_meta.data_ptr(), capacity, int(bool(zero_pad)), _stream_ptr(stream)),
           "ep_dispatch_metadata")
    return recv_weights, recv_meta


def combine(handle: EPHandle, y: torch.Tensor, topk_weights: torch.Tensor,
            out: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None,
            bias: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Weighted combine of y [rows,H] bf16 back to [T,H] bf16, plus an
    optional bias row [T,H] bf16 added before the rounding."""
    _need(y, "y", torch.bfloat16, 2)
    if bias is not None:
        _need(bias, "bias", torch.bfloat16, 2)
        if tuple(bias.shape) != (handle.T, y.shape[1]):
            raise ValueError("bias must be [T,H]")
    _need(topk_weights, "topk_weights", torch.float32, 2)
    if tuple(topk_weights.shape) != (handle.T, handle.K):
        raise ValueError("topk_weights must be [T,K]")
    H = y.shape[1]
    if out is None:
        out = torch.empty((handle.T, H), dtype=torch.bfloat16, device=y.device)
    _need(out, "out", torch.bfloat16, 2)
    if tuple(out.shape) != (handle.T, H):
        raise ValueError("out must be [T,H]")
    _check(_lib().ep_combine(handle.ptr, y.data_ptr(), y.shape[0], topk_weights.data_ptr(),
                             bias.data_ptr() if bias is not None else None, H, out.data_ptr(),
                             _stream_ptr(stream)), "ep_combine")
    return out


def dispatch_backward(handle: EPHandle, grad_recv: torch.Tensor, grad_x: Optional[torch.Tensor] = None,
                      stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Backward of dispatch on the same handle: grad_recv [rows,H] -> grad_x [T,H]."""
    _need(grad_recv, "grad_recv", torch.bfloat16, 2)
    H = grad_recv.shape[1]
    if grad_x is None:
        grad_x = torch.empty((handle.T, H), dtype=torch.bfloat16, device=grad_recv.device)
    _need(grad_x, "grad_x", torch.bfloat16, 2)
    if tuple(grad_x.shape) != (handle.T, H):
        raise ValueError("grad_x must be [T,H]")
    _check(_lib().ep_dispatch_backward(handle.ptr, grad_recv.data_ptr(), grad_recv.shape[0], H, grad_x.data_ptr(),
                                       _stream_ptr(stream)), "ep_dispatch_backward")
    return grad_x


def combine_backward(handle: EPHandle, grad_out: torch.Tensor, y: torch.Tensor, topk_weights: torch.Tensor,
                     zero_pad: bool = True, grad_y: Optional[torch.Tensor] = None,
                     grad_weights: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None):
    """Backward of combine on the same handle -> (grad_y [rows,H] bf16, grad_weights [T,K] f32)."""
    _need(grad_out, "grad_out", torch.bfloat16, 2)
    _need(y, "y", torch.bfloat16, 2)
    _need(topk_weights, "topk_weights", torch.float32, 2)
    H = grad_out.shape[1]
    if tuple(grad_out.shape) != (handle.T, H) or y.shape[1] != H:
        raise ValueError("grad_out must be [T,H] and y [rows,H]")
    if tuple(topk_weights.shape) != (handle.T, handle.K):
        raise ValueError("topk_weights must be [T,K]")
    if grad_y is None:
        grad_y = torch.empty_like(y)
    if grad_weights is None:
        grad_weights = torch.empty((handle.T, handle.K), dtype=torch.float32, device=y.device)
    _need(grad_y, "grad_y", torch.bfloat16, 2)
    _need(grad_weights, "grad_weights", torch.float32, 2)
    _check(_lib().ep_combine_backward(handle.ptr, grad_out.data_ptr(), y.data_ptr(), y.shape[0],
                                      topk_weights.data_ptr(), H, int(bool(zero_pad)), grad_y.data_ptr(),
                                      grad_y.shape[0], grad_weights.data_ptr(), _stream_ptr(stream)),
           "ep_combine_backward")
    return grad_y, grad_weights


class Pending:
    """An issued dispatch_async / combine_async.  wait() must be called once:
    it makes the compute stream wait for the issued work (no host block) and
    returns the results.  The pending object keeps the tensors the work uses
    alive until then."""

    def __init__(self, ptr: int, kind: str, results, keep):
        self._ptr = ptr
        self.kind = kind
        self._results = results
        self._keep = keep

    def wait(self, counts: bool = True):
        """dispatch: (recv_x, recv_scales|None, N_exp, N_recv); combine: out.
        counts=False skips the count readback (no host wait; N_exp and N_recv
        are then returned as 0)."""
        if not self._ptr:
            raise RuntimeError("pending call already waited on")
        ne, nr = ctypes.c_int64(), ctypes.c_int64()
        want = self.kind == "dispatch" and counts
        code = _lib().ep_pending_wait(self._ptr, ctypes.byref(ne) if want else None,
                                      ctypes.byref(nr) if want else None)
        self._ptr = 0
        self._keep = None
        _check(code, "ep_pending_wait")
        if self.kind == "dispatch":
            return self._results[0], self._results[1], ne.value, nr.value
        return self._results

    def __del__(self):
        try:
            if self._ptr and _LIB is not None:
                _LIB.ep_pending_wait(self._ptr, None, None)
        except Exception:
            pass


def _event_ptr(previous) -> Optional[int]:
    if previous is None:
        return None
    ptr = int(previous.cuda_event)
    if not ptr:
        raise ValueError("previous event has never been recorded")
    return ptr


def dispatch_async(handle: EPHandle, x: torch.Tensor, out_dtype: str = "bf16", zero_pad: bool = True,
                   recv_x: Optional[torch.Tensor] = None, recv_scales: Optional[torch.Tensor] = None,
                   topk_idx: Optional[torch.Tensor] = None, previous: Optional[torch.cuda.Event] = None,
                   defer_epilogue: bool = True, stream: Optional[torch.cuda.Stream] = None,
                   x_scales: Optional[torch.Tensor] = None, scales_col_major: bool = False) -> Pending:
    """Issue a dispatch on the handle's communication stream and return at
    once (defer_epilogue=True) or once the plan's counts are known
    (defer_epilogue=False).  topk_idx re-plans first (fresh dispatch); None
    uses the handle's plan (cached dispatch).  Outputs default to the
    worst-case row count.  `stream` is the compute stream the work is ordered
    after (unless `previous` is given) and that wait() joins."""
    code = _dtype_code(out_dtype)
    xcode = _input_code(x, x_scales)
    H = x.shape[1]
    if topk_idx is not None:
        _need(topk_idx, "topk_idx", torch.int64, 2)
        if tuple(topk_idx.shape) != (handle.T, handle.K):
            raise ValueError("topk_idx must be [T,K] of the handle")
        handle._sizes = None
    cap = worst_expanded_rows(handle.T, handle.K, handle.E, handle.A)
    recv_x, recv_scales = _dispatch_outputs(H, out_dtype, recv_x, recv_scales, cap, x.device, scales_col_major)
    _check_dispatch(x, recv_x, recv_scales, out_dtype, scales_col_major)
    p = ctypes.c_void_p()
    _check(_lib().ep_dispatch_async(handle.ptr, topk_idx.data_ptr() if topk_idx is not None else None,
                                    x.data_ptr(), xcode, x_scales.data_ptr() if x_scales is not None else None,
                                    H, code, _flags(zero_pad, scales_col_major), recv_x.data_ptr(),
                                    recv_scales.data_ptr() if recv_scales is not None else None,
                                    recv_x.shape[0], _stream_ptr(stream), _event_ptr(previous),
                                    int(bool(defer_epilogue)), ctypes.byref(p)), "ep_dispatch_async")
    return Pending(p.value, "dispatch", (recv_x, recv_scales), (x, x_scales, topk_idx, previous))


def combine_async(handle: EPHandle, y: torch.Tensor, topk_weights: torch.Tensor,
                  out: Optional[torch.Tensor] = None, bias: Optional[torch.Tensor] = None,
                  previous: Optional[torch.cuda.Event] = None, defer_epilogue: bool = True,
                  stream: Optional[torch.cuda.Stream] = None) -> Pending:
    """Issue a combine on the handle's communication stream; wait() -> out."""
    _need(y, "y", torch.bfloat16, 2)
    if bias is not None:
        _need(bias, "bias", torch.bfloat16, 2)
        if tuple(bias.shape) != (handle.T, y.shape[1]):
            raise ValueError("bias must be [T,H]")
    _need(topk_weights, "topk_weights", torch.float32, 2)
    if tuple(topk_weights.shape) != (handle.T, handle.K):
        raise ValueError("topk_weights must be [T,K]")
    H = y.shape[1]
    if out is None:
        out = torch.empty((handle.T, H), dtype=torch.bfloat16, device=y.device)
    _need(out, "out", torch.bfloat16, 2)
    if tuple(out.shape) != (handle.T, H):
        raise ValueError("out must be [T,H]")
    p = ctypes.c_void_p()
    _check(_lib().ep_combine_async(handle.ptr, y.data_ptr(), y.shape[0], topk_weights.data_ptr(),
                                   bias.data_ptr() if bias is not None else None, H, out.data_ptr(),
                                   _stream_ptr(stream), _event_ptr(previous), int(bool(defer_epilogue)),
                                   ctypes.byref(p)), "ep_combine_async")
    return Pending(p.value, "combine", out, (y, topk_weights, bias, previous))


# Per-CTA profile records (ep_profile_begin): kernel ids and record width.
PROFILE_KERNELS = {1: "plan", 2: "dispatch_bf16", 3: "dispatch_fp8", 4: "dispatch_fp8_input", 5: "combine",
                   6: "dispatch_backward"}
PROFILE_WORDS = 8


def summarize_profile(records) -> list:
    """Aggregate per-CTA records (an [n, 8] int64 array or tensor) per launch,
    in launch order: kernel, CTAs, units, payload bytes, span from the first
    CTA start to the last CTA end (ns), median and max CTA duration (ns),
    payload GB/s over the span, and for the plan the median stage offsets
    from the launch's first start, in ns: route scan over the CTAs that
    scanned a tile, each grid barrier passed over all CTAs (a one-CTA plan:
    route scan, column counts, offsets)."""
    import numpy as np
    r = np.asarray(records.cpu() if isinstance(records, torch.Tensor) else records).astype(np.uint64)
    if r.size == 0:
        return []
    r = r.reshape(-1, PROFILE_WORDS)
    kind = (r[:, 0] >> np.uint64(56)).astype(np.int64)
    seq = ((r[:, 0] >> np.uint64(32)) & np.uint64(0xFFFFFF)).astype(np.int64)
    out = []
    for s in sorted(set(seq.tolist()), key=lambda v: int(np.argmax(seq == v))):
        m = seq == s
        k = int(kind[m][0])
        t0, t1 = r[m, 1].astype(np.int64), r[m, 5].astype(np.int64)
        span = int(t1.max() - t0.min())
        nbytes = int(r[m, 7].sum())
        row = {"seq": int(s), "kernel": PROFILE_KERNELS.get(k, str(k)), "ctas": int(m.sum()),
               "units": int(r[m, 6].sum()), "bytes": nbytes, "span_ns": span,
               "cta_ns_median": float(np.median(t1 - t0)), "cta_ns_max": int((t1 - t0).max()),
               "gbs": nbytes / span if span > 0 else 0.0}
        if k == 1:
            # route scan over the CTAs that scanned a tile (the others have
            # no scan mark); the two grid barriers over all CTAs.  A one-tile
            # plan runs as one CTA without grid barriers: its marks are the
            # column counts and the offsets instead.
            base = t0.min()
            tiles = r[m, 2] > 0
            one = int(m.sum()) == 1
            for name, col, sel in (("scan_ns", 2, tiles),
                                   ("counts_ns" if one else "barrier1_ns", 3, np.ones_like(tiles)),
                                   ("offsets_ns" if one else "barrier2_ns", 4, np.ones_like(tiles))):
                v = r[m, col].astype(np.int64)[sel]
                v = v[v > 0]
                row[name] = float(np.median(v - base)) if len(v) else 0.0
        out.append(row)
    return out


def set_plan_wait_debug(poll_limit: int = 0, suppress_tile: int = -1):
    """Test hook for the plan's bounded grid-barrier waits (see ep_debug_set_plan_wait)."""
    _lib().ep_debug_set_plan_wait(poll_limit, suppress_tile)
