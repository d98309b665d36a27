"""ctypes binding of libmoe.so (C ABI in include/moe.h).

Argument marshalling only: every step of the layer runs in the library's
CUDA kernels.  The functions keep the C names (moe_init, moe_route,
moe_forward, moe_forward_host, moe_check, moe_set_wait_limit, moe_free,
moe_status_string, moe_selftest_wait_timeout) and take torch tensors where
the C functions take pointers; a non-zero status raises MoeError.
``MoeLayer`` bundles a handle with the weight tensors it borrows.

The library must have been built (``__graft_entry__.build()`` or
``python -m expert_routed_ffn_gemm_gb300.build``); loading raises otherwise.
There is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_TOO_MANY_TOKENS = 2
MOE_ERR_UNSUPPORTED = 3
MOE_ERR_CUDA = 4
MOE_ERR_DEVICE = 5
MOE_ERR_NO_DEVICE = 6

EXPORTED = ("moe_init", "moe_route", "moe_forward", "moe_forward_host", "moe_check", "moe_set_wait_limit",
            "moe_profile_enable", "moe_profile_read", "moe_free", "moe_status_string",
            "moe_selftest_wait_timeout", "moe_dispatch_noalloc", "moe_route_ex", "moe_forward_ex",
            "moe_route_stats", "moe_last_kernel_count", "moe_init_fp8", "moe_quantize_fp8", "moe_ep_init",
            "moe_ep_dispatch", "moe_ep_experts", "moe_ep_combine")
PROFILE_STAGES = ("routing", "dispatch", "gather", "gate_up_gemm", "down_gemm", "combine")


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {moe_status_string(status)} (status {status})")


class moe_config(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int), ("n_experts", ctypes.c_int), ("top_k", ctypes.c_int),
                ("ffn_width", ctypes.c_int), ("has_shared", ctypes.c_int), ("max_tokens", ctypes.c_int),
                ("out_fp32", ctypes.c_int)]


class moe_weights(ctypes.Structure):
    _fields_ = [("w_router", ctypes.c_void_p), ("w_gate_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p)]


class moe_weights_fp8(ctypes.Structure):
    _fields_ = [("w_router", ctypes.c_void_p), ("w_gate_up", ctypes.c_void_p), ("s_gate_up", ctypes.c_void_p),
                ("w_down", ctypes.c_void_p), ("s_down", ctypes.c_void_p)]


class moe_ep_config(ctypes.Structure):
    _fields_ = [("layer", moe_config), ("ep_size", ctypes.c_int), ("ep_rank", ctypes.c_int),
                ("max_recv_rows", ctypes.c_int)]


class moe_call_options(ctypes.Structure):
    _fields_ = [("top_k", ctypes.c_int), ("renormalize", ctypes.c_int)]


def _opts(top_k, renormalize):
    if top_k is None and not renormalize:
        return None
    return ctypes.byref(moe_call_options(int(top_k or 0), int(bool(renormalize))))


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    """libmoe.so, or libmoe_debug.so (the build with the kernels' bounds
    checks) when MOE_LIBRARY=debug is set in the environment."""
    return _build.DEBUG_LIB_PATH if os.environ.get("MOE_LIBRARY") == "debug" else _build.LIB_PATH


def load():
    """Load libmoe.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build the CUDA library first (__graft_entry__.build())")
        lib = ctypes.CDLL(path)
        vp, i, ull = ctypes.c_void_p, ctypes.c_int, ctypes.c_ulonglong
        lib.moe_init.argtypes = [ctypes.POINTER(moe_config), ctypes.POINTER(moe_weights), ctypes.POINTER(vp)]
        lib.moe_init_fp8.argtypes = [ctypes.POINTER(moe_config), ctypes.POINTER(moe_weights_fp8),
                                     ctypes.POINTER(vp)]
        lib.moe_quantize_fp8.argtypes = [vp, ctypes.c_longlong, i, vp, vp, vp]
        lib.moe_ep_init.argtypes = [ctypes.POINTER(moe_ep_config), ctypes.POINTER(moe_weights), ctypes.POINTER(vp)]
        lib.moe_ep_dispatch.argtypes = [vp, vp, i, vp, vp, vp, ctypes.POINTER(ctypes.c_int), vp]
        lib.moe_ep_experts.argtypes = [vp, vp, vp, vp, i, vp, vp, ctypes.POINTER(ctypes.c_int), vp]
        lib.moe_ep_combine.argtypes = [vp, vp, vp, vp, vp]
        lib.moe_route.argtypes = [vp, vp, i, vp, vp, vp, vp, vp, vp]
        lib.moe_forward.argtypes = [vp, vp, i, vp, vp]
        lib.moe_forward_host.argtypes = [vp, vp, i, vp, vp]
        lib.moe_check.argtypes = [vp, vp]
        lib.moe_last_kernel_count.argtypes = [vp]
        lib.moe_set_wait_limit.argtypes = [vp, ull]
        lib.moe_profile_enable.argtypes = [vp, i]
        lib.moe_profile_read.argtypes = [vp, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int)]
        lib.moe_free.argtypes = [vp]
        lib.moe_status_string.argtypes = [i]
        lib.moe_status_string.restype = ctypes.c_char_p
        lib.moe_selftest_wait_timeout.argtypes = [ull, vp]
        lib.moe_dispatch_noalloc.argtypes = [vp, i, i, i, i, vp, vp, vp]
        lib.moe_route_ex.argtypes = [vp, vp, i, vp, vp, vp, vp, vp, vp, vp]
        lib.moe_forward_ex.argtypes = [vp, vp, i, vp, vp, vp]
        lib.moe_route_stats.argtypes = [vp, vp, i, i, vp, vp, vp, vp, vp]
        for name in EXPORTED:
            if name != "moe_status_string":
                getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def moe_status_string(status: int) -> str:
    return load().moe_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != MOE_OK:
        raise MoeError(status, where)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_contiguous():
        raise ValueError("tensors passed to libmoe must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def moe_init(cfg: moe_config, w_router: torch.Tensor, w_gate_up: torch.Tensor, w_down: torch.Tensor) -> int:
    w = moe_weights(_ptr(w_router), _ptr(w_gate_up), _ptr(w_down))
    h = ctypes.c_void_p()
    _check(load().moe_init(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)), "moe_init")
    return h.value


def moe_init_fp8(cfg: moe_config, w_router, q_gate_up, s_gate_up, q_down, s_down) -> int:
    w = moe_weights_fp8(_ptr(w_router), _ptr(q_gate_up), _ptr(s_gate_up), _ptr(q_down), _ptr(s_down))
    h = ctypes.c_void_p()
    _check(load().moe_init_fp8(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)), "moe_init_fp8")
    return h.value


def moe_quantize_fp8(w: torch.Tensor, stream=None):
    """Per-row E4M3 codes (uint8, same shape) and fp32 scales (shape[:-1]) of a
    bf16 device tensor, computed on the device (see include/moe.h)."""
    if w.dtype != torch.bfloat16:
        raise TypeError("moe_quantize_fp8 takes bf16 weights")
    cols = w.shape[-1]
    rows = w.numel() // cols
    q = torch.empty(w.shape, dtype=torch.uint8, device=w.device)
    s = torch.empty(w.shape[:-1], dtype=torch.float32, device=w.device)
    _check(load().moe_quantize_fp8(_ptr(w), rows, cols, _ptr(q), _ptr(s), _stream(stream)), "moe_quantize_fp8")
    return q, s


def moe_ep_init(cfg: moe_ep_config, w_router, w_gate_up_local, w_down_local) -> int:
    """Expert-parallel handle (moe_weights layout: the router over all experts,
    this rank's experts then the shared expert)."""
    w = moe_weights(_ptr(w_router), _ptr(w_gate_up_local), _ptr(w_down_local))
    h = ctypes.c_void_p()
    _check(load().moe_ep_init(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)), "moe_ep_init")
    return h.value


def moe_ep_dispatch(h: int, x, T: int, send_rows, send_w, send_counts, ep_size: int, stream=None) -> list[int]:
    rows = (ctypes.c_int * ep_size)()
    _check(load().moe_ep_dispatch(h, _ptr(x), int(T), _ptr(send_rows), _ptr(send_w), _ptr(send_counts), rows,
                                  _stream(stream)), "moe_ep_dispatch")
    return list(rows)


def moe_ep_experts(h: int, recv_rows, recv_counts, recv_w, n_recv: int, out_rows, out_exp, ep_size: int,
                   stream=None) -> list[int]:
    chunks = (ctypes.c_int * ep_size)()
    _check(load().moe_ep_experts(h, _ptr(recv_rows), _ptr(recv_counts), _ptr(recv_w), int(n_recv), _ptr(out_rows),
                                 _ptr(out_exp), chunks, _stream(stream)), "moe_ep_experts")
    return list(chunks)


def moe_ep_combine(h: int, ret_rows, ret_exp, y, stream=None) -> None:
    _check(load().moe_ep_combine(h, _ptr(ret_rows), _ptr(ret_exp), _ptr(y), _stream(stream)), "moe_ep_combine")


def moe_route(h: int, x, T: int, idx, prob, perm, offsets, gap=None, stream=None) -> None:
    _check(load().moe_route(h, _ptr(x), int(T), _ptr(idx), _ptr(prob), _ptr(perm), _ptr(offsets), _ptr(gap),
                            _stream(stream)), "moe_route")


def moe_forward(h: int, x, T: int, y, stream=None) -> None:
    _check(load().moe_forward(h, _ptr(x), int(T), _ptr(y), _stream(stream)), "moe_forward")


def moe_route_ex(h: int, x, T: int, top_k, renormalize, idx, prob, perm, offsets, gap=None, stream=None) -> None:
    _check(load().moe_route_ex(h, _ptr(x), int(T), _opts(top_k, renormalize), _ptr(idx), _ptr(prob), _ptr(perm),
                               _ptr(offsets), _ptr(gap), _stream(stream)), "moe_route_ex")


def moe_forward_ex(h: int, x, T: int, top_k, renormalize, y, stream=None) -> None:
    _check(load().moe_forward_ex(h, _ptr(x), int(T), _opts(top_k, renormalize), _ptr(y), _stream(stream)),
           "moe_forward_ex")


def moe_route_stats(h: int, x, T: int, n_groups: int, counts, group_f, group_p, summary, stream=None) -> None:
    _check(load().moe_route_stats(h, _ptr(x), int(T), int(n_groups), _ptr(counts), _ptr(group_f), _ptr(group_p),
                                  _ptr(summary), _stream(stream)), "moe_route_stats")


def moe_forward_host(h: int, x_host: torch.Tensor, T: int, y_host: torch.Tensor, stream=None) -> None:
    if x_host.is_cuda or y_host.is_cuda:
        raise ValueError("moe_forward_host takes host tensors")
    _check(load().moe_forward_host(h, _ptr(x_host), int(T), _ptr(y_host), _stream(stream)), "moe_forward_host")


def moe_last_kernel_count(h: int) -> int:
    """Kernels the last forward call on the handle enqueued (-1: bad handle)."""
    return int(load().moe_last_kernel_count(h))


def moe_check(h: int, stream=None) -> int:
    """Returns the status (does not raise): MOE_OK or MOE_ERR_DEVICE/CUDA."""
    return int(load().moe_check(h, _stream(stream)))


def moe_set_wait_limit(h: int, ns: int) -> None:
    _check(load().moe_set_wait_limit(h, int(ns)), "moe_set_wait_limit")


def moe_profile_enable(h: int, enable: bool) -> None:
    _check(load().moe_profile_enable(h, int(bool(enable))), "moe_profile_enable")


def moe_profile_read(h: int):
    """Returns ({stage: total ms}, number of recorded calls) and clears the record."""
    ms = (ctypes.c_float * len(PROFILE_STAGES))()
    n = ctypes.c_int()
    _check(load().moe_profile_read(h, ms, ctypes.byref(n)), "moe_profile_read")
    return dict(zip(PROFILE_STAGES, [float(v) for v in ms])), int(n.value)


def moe_free(h: int) -> None:
    _check(load().moe_free(h), "moe_free")


def moe_selftest_wait_timeout(limit_ns: int, stream=None) -> int:
    return int(load().moe_selftest_wait_timeout(int(limit_ns), _stream(stream)))


def moe_dispatch_noalloc(idx, T: int, n_experts: int, top_k: int, has_shared: bool, offsets, perm,
                         stream=None) -> None:
    """Dispatch order from existing routing without any device allocation
    (for callers that must not call cudaMalloc); see include/moe.h."""
    _check(load().moe_dispatch_noalloc(_ptr(idx), int(T), int(n_experts), int(top_k), int(bool(has_shared)),
                                       _ptr(offsets), _ptr(perm), _stream(stream)), "moe_dispatch_noalloc")


class MoeLayer:
    """A handle plus the device weight tensors it borrows.

    w_router fp32 [E, d]; w_gate_up bf16 [E+1, 2F, d] (gate rows, then up
    rows; group E is the shared expert); w_down bf16 [E+1, d, F].
    """

    def __init__(self, w_router, w_gate_up, w_down, top_k: int, max_tokens: int, has_shared: bool = True,
                 out_fp32: bool = False, scales=None):
        E, d = w_router.shape
        G, twoF, d2 = w_gate_up.shape
        F = twoF // 2
        if d2 != d or G != E + int(has_shared) or tuple(w_down.shape) != (G, d, F):
            raise ValueError("weight shapes do not match [E,d], [G,2F,d], [G,d,F]")
        wdt = torch.uint8 if scales is not None else torch.bfloat16
        if w_router.dtype != torch.float32 or w_gate_up.dtype != wdt or w_down.dtype != wdt:
            raise TypeError("w_router must be fp32 and the expert weights bf16 (or uint8 E4M3 codes with scales)")
        self.weights = (w_router, w_gate_up, w_down) + tuple(scales or ())  # borrowed by the handle
        self.d, self.E, self.k, self.F = d, E, top_k, F
        self.has_shared, self.out_fp32, self.max_tokens = has_shared, out_fp32, max_tokens
        self.device = w_gate_up.device
        cfg = moe_config(d, E, top_k, F, int(has_shared), max_tokens, int(out_fp32))
        if scales is None:
            self.handle = moe_init(cfg, w_router, w_gate_up, w_down)
        else:
            s_gu, s_d = scales
            if tuple(s_gu.shape) != (G, 2 * F) or tuple(s_d.shape) != (G, d):
                raise ValueError("scales must be [G, 2F] and [G, d]")
            self.handle = moe_init_fp8(cfg, w_router, w_gate_up, s_gu, w_down, s_d)

    @classmethod
    def fp8(cls, w_router, q_gate_up, s_gate_up, q_down, s_down, top_k: int, max_tokens: int,
            has_shared: bool = True, out_fp32: bool = False) -> "MoeLayer":
        """A layer with E4M3 expert weights (uint8 codes) and fp32 row scales."""
        return cls(w_router, q_gate_up, q_down, top_k, max_tokens, has_shared, out_fp32,
                   scales=(s_gate_up, s_down))

    def route(self, x: torch.Tensor, stream=None, with_gap: bool = True, top_k: int | None = None,
              renormalize: bool = False):
        T = x.shape[0]
        dev = x.device
        k = top_k or self.k
        idx = torch.empty((T, k), dtype=torch.int32, device=dev)
        prob = torch.empty((T, k), dtype=torch.float32, device=dev)
        perm = torch.empty((T * k,), dtype=torch.int32, device=dev)
        offsets = torch.empty((self.E + 2,), dtype=torch.int32, device=dev)
        gap = torch.empty((T,), dtype=torch.float32, device=dev) if with_gap else None
        if top_k is None and not renormalize:
            moe_route(self.handle, x, T, idx, prob, perm, offsets, gap, stream)
        else:
            moe_route_ex(self.handle, x, T, top_k, renormalize, idx, prob, perm, offsets, gap, stream)
        return idx, prob, perm, offsets, gap

    def forward(self, x: torch.Tensor, y: torch.Tensor | None = None, stream=None, top_k: int | None = None,
                renormalize: bool = False) -> torch.Tensor:
        T = x.shape[0]
        if y is None:
            y = torch.empty((T, self.d), dtype=torch.float32 if self.out_fp32 else torch.bfloat16,
                            device=x.device)
        if top_k is None and not renormalize:
            moe_forward(self.handle, x, T, y, stream)
        else:
            moe_forward_ex(self.handle, x, T, top_k, renormalize, y, stream)
        return y

    def route_stats(self, x: torch.Tensor, n_groups: int, stream=None):
        """(counts [E] int32, group_f [G], group_p [G], summary [4]) on the device."""
        T = x.shape[0]
        dev = x.device
        counts = torch.empty((self.E,), dtype=torch.int32, device=dev)
        group_f = torch.empty((n_groups,), dtype=torch.float32, device=dev)
        group_p = torch.empty((n_groups,), dtype=torch.float32, device=dev)
        summary = torch.empty((4,), dtype=torch.float32, device=dev)
        moe_route_stats(self.handle, x, T, n_groups, counts, group_f, group_p, summary, stream)
        return counts, group_f, group_p, summary

    __call__ = forward

    def forward_host(self, x_host: torch.Tensor, y_host: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        T = x_host.shape[0]
        if y_host is None:
            y_host = torch.empty((T, self.d), dtype=torch.float32 if self.out_fp32 else torch.bfloat16,
                                 pin_memory=True)
        moe_forward_host(self.handle, x_host, T, y_host, stream)
        return y_host

    def check(self, stream=None) -> int:
        return moe_check(self.handle, stream)

    def last_kernel_count(self) -> int:
        return moe_last_kernel_count(self.handle)

    def set_wait_limit(self, ns: int) -> None:
        moe_set_wait_limit(self.handle, ns)

    def profile_enable(self, enable: bool = True) -> None:
        moe_profile_enable(self.handle, enable)

    def profile_read(self):
        return moe_profile_read(self.handle)

    def close(self) -> None:
        if getattr(self, "handle", None):
            moe_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
