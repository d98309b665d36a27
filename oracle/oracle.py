"""ctypes front-end of the C oracle in ``moe_oracle.c`` (test infrastructure).

Every function takes and returns numpy arrays.  bf16 tensors travel as their
raw ``uint16`` bit patterns, so the oracle sees exactly the values the GPU
path sees.  See ``moe_oracle.c`` for what each step computes and which
passage of "Step3.5 Flash 大模型技术深度解析" (jsqmd.com, §3.2.1-§3.2.2) it
follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# MOE_ORACLE_SOURCE names another copy of the oracle's C source to compile and
# load instead (beside it): the test that plants one mistake per copy and
# checks that the pins fail on each uses it.  Unset: moe_oracle.c here.
_VARIANT = os.environ.get("MOE_ORACLE_SOURCE")
_SRC = os.path.abspath(_VARIANT) if _VARIANT else os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(os.path.dirname(_SRC), "libmoe_oracle_variant.so") if _VARIANT else os.path.join(
    _HERE, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")


def build(force: bool = False) -> str:
    """Compile ``moe_oracle.c`` into ``libmoe_oracle.so`` (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(
            ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            lib.oracle_route.argtypes = [_u16p, _f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_void_p, _i32p, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_int]
            lib.oracle_dispatch.argtypes = [_i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            _i32p, _i32p, _i32p]
            lib.oracle_forward.argtypes = [_u16p, _f32p, _u16p, _u16p, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           _i32p, ctypes.c_int, ctypes.c_void_p, _f64p, ctypes.c_int]
            lib.oracle_forward_ex.argtypes = [_u16p, _f32p, _u16p, _u16p, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                              _i32p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, _f64p,
                                              ctypes.c_int]
            lib.oracle_route_stats.argtypes = [_u16p, _f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, _i32p, _f64p, _f64p, _f64p,
                                               ctypes.c_int]
            lib.oracle_expert_ffn.argtypes = [_u16p, _u16p, _u16p, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, _i32p, ctypes.c_int, _f64p, ctypes.c_int]
            lib.oracle_forward_fp8.argtypes = [_u16p, _f32p, _u8p, _f32p, _u8p, _f32p, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, _i32p, ctypes.c_int, ctypes.c_void_p,
                                               ctypes.c_int, _f64p, ctypes.c_int]
            lib.oracle_quantize_e4m3.argtypes = [_u16p, ctypes.c_long, ctypes.c_int, _u8p, _f32p]
            lib.oracle_e4m3_decode.argtypes = [_u8p, ctypes.c_long, _f64p]
            lib.oracle_e4m3_encode.argtypes = [_f32p, ctypes.c_long, _u8p]
            lib.oracle_max_threads.argtypes = []
            for f in ("oracle_route", "oracle_dispatch", "oracle_forward", "oracle_forward_ex",
                      "oracle_route_stats", "oracle_expert_ffn", "oracle_max_threads", "oracle_forward_fp8",
                      "oracle_quantize_e4m3", "oracle_e4m3_decode", "oracle_e4m3_encode"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 operands are passed as uint16 bit patterns")
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def route(x_bits, w_router, k: int, *, want_p: bool = False, threads: int = 0):
    """Router, softmax and top-k for every token.

    Returns ``(idx [T,k] int32, w [T,k] f64, gap [T] f64, p [T,E] f64 or None)``;
    ``gap`` is p(k-th) - p((k+1)-th) (inf when k == E).
    """
    x = _u16(x_bits)
    wr = np.ascontiguousarray(w_router, dtype=np.float32)
    T, d = x.shape
    E = wr.shape[0]
    if wr.shape[1] != d:
        raise ValueError("w_router must be [E, d]")
    idx = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float64)
    gap = np.zeros((T,), np.float64)
    p = np.zeros((T, E), np.float64) if want_p else None
    rc = _load().oracle_route(x, wr, T, d, E, k, _ptr(p), idx, _ptr(w), _ptr(gap), threads)
    if rc != 0:
        raise ValueError("oracle_route rejected its arguments")
    return idx, w, gap, p


def dispatch(idx, n_experts: int):
    """Histogram, exclusive offsets (shared group appended) and stable perm."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T, k = idx.shape
    counts = np.zeros((n_experts,), np.int32)
    offsets = np.zeros((n_experts + 2,), np.int32)
    perm = np.zeros((T * k,), np.int32)
    rc = _load().oracle_dispatch(idx, T, n_experts, k, counts, offsets, perm)
    if rc != 0:
        raise ValueError("oracle_dispatch rejected its arguments")
    return counts, offsets, perm


def forward(x_bits, w_router, w_gate_up_bits, w_down_bits, k: int, *, has_shared: bool = True,
            tokens=None, sel=None, renormalize: bool = False, threads: int = 0) -> np.ndarray:
    """Layer output in float64 for ``tokens`` (all tokens by default).

    ``sel`` ([len(tokens), k] int32) replaces the oracle's own top-k choice;
    ``renormalize`` divides the k weights by their sum.
    """
    x = _u16(x_bits)
    wr = np.ascontiguousarray(w_router, dtype=np.float32)
    wgu = _u16(w_gate_up_bits)
    wd = _u16(w_down_bits)
    T, d = x.shape
    E = wr.shape[0]
    G = E + (1 if has_shared else 0)
    F = wgu.shape[1] // 2
    if wgu.shape != (G, 2 * F, d) or wd.shape != (G, d, F):
        raise ValueError("expert weight shapes do not match [G,2F,d] / [G,d,F]")
    if tokens is None:
        tokens = np.arange(T, dtype=np.int32)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    n = tokens.shape[0]
    if sel is not None:
        sel = np.ascontiguousarray(sel, dtype=np.int32)
        if sel.shape != (n, k):
            raise ValueError("sel must be [len(tokens), k]")
    y = np.zeros((n, d), np.float64)
    rc = _load().oracle_forward_ex(x, wr, wgu, wd, T, d, E, k, F, int(has_shared), tokens, n,
                                   _ptr(sel), int(bool(renormalize)), y, threads)
    if rc != 0:
        raise ValueError("oracle_forward rejected its arguments")
    return y


def forward_fp8(x_bits, w_router, q_gate_up, s_gate_up, q_down, s_down, k: int, *, has_shared: bool = True,
                tokens=None, sel=None, renormalize: bool = False, threads: int = 0) -> np.ndarray:
    """``forward`` with E4M3 expert weights: codes ``q_*`` (uint8) and one fp32
    scale per weight row (``s_gate_up`` [G, 2F], ``s_down`` [G, d])."""
    x = _u16(x_bits)
    wr = np.ascontiguousarray(w_router, dtype=np.float32)
    qgu = np.ascontiguousarray(q_gate_up, dtype=np.uint8)
    qd = np.ascontiguousarray(q_down, dtype=np.uint8)
    sgu = np.ascontiguousarray(s_gate_up, dtype=np.float32)
    sd = np.ascontiguousarray(s_down, dtype=np.float32)
    T, d = x.shape
    E = wr.shape[0]
    G = E + (1 if has_shared else 0)
    F = qgu.shape[1] // 2
    if qgu.shape != (G, 2 * F, d) or qd.shape != (G, d, F) or sgu.shape != (G, 2 * F) or sd.shape != (G, d):
        raise ValueError("fp8 weight or scale shapes do not match [G,2F,d] / [G,d,F] / [G,2F] / [G,d]")
    if tokens is None:
        tokens = np.arange(T, dtype=np.int32)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    n = tokens.shape[0]
    if sel is not None:
        sel = np.ascontiguousarray(sel, dtype=np.int32)
        if sel.shape != (n, k):
            raise ValueError("sel must be [len(tokens), k]")
    y = np.zeros((n, d), np.float64)
    rc = _load().oracle_forward_fp8(x, wr, qgu, sgu, qd, sd, T, d, E, k, F, int(has_shared), tokens, n,
                                    _ptr(sel), int(bool(renormalize)), y, threads)
    if rc != 0:
        raise ValueError("oracle_forward_fp8 rejected its arguments")
    return y


def quantize_e4m3(w_bits):
    """Per-row E4M3 quantisation of bf16 weights ``[..., cols]`` (bit patterns):
    returns (codes uint8 of the same shape, scales float32 ``[...]``)."""
    w = _u16(w_bits)
    cols = w.shape[-1]
    rows = w.size // cols
    q = np.zeros(w.shape, np.uint8)
    s = np.zeros(w.shape[:-1], np.float32)
    rc = _load().oracle_quantize_e4m3(w.reshape(rows, cols), rows, cols, q.reshape(rows, cols),
                                      s.reshape(rows))
    if rc != 0:
        raise ValueError("oracle_quantize_e4m3 rejected its arguments")
    return q, s


def e4m3_decode(codes) -> np.ndarray:
    q = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.zeros(q.shape, np.float64)
    _load().oracle_e4m3_decode(q.reshape(-1), q.size, out.reshape(-1))
    return out


def e4m3_encode(values) -> np.ndarray:
    v = np.ascontiguousarray(values, dtype=np.float32)
    q = np.zeros(v.shape, np.uint8)
    _load().oracle_e4m3_encode(v.reshape(-1), v.size, q.reshape(-1))
    return q


def route_stats(x_bits, w_router, k: int, n_groups: int, threads: int = 0):
    """Routing statistics (see moe_oracle.c): (counts [E] int32, f [G], p [G],
    summary [4] = L_EP, max/mean load, mean entropy, empty experts)."""
    x = _u16(x_bits)
    wr = np.ascontiguousarray(w_router, dtype=np.float32)
    T, d = x.shape
    E = wr.shape[0]
    counts = np.zeros((E,), np.int32)
    f = np.zeros((n_groups,), np.float64)
    p = np.zeros((n_groups,), np.float64)
    summary = np.zeros((4,), np.float64)
    rc = _load().oracle_route_stats(x, wr, T, d, E, k, n_groups, counts, f, p, summary, threads)
    if rc != 0:
        raise ValueError("oracle_route_stats rejected its arguments")
    return counts, f, p, summary


def expert_ffn(x_bits, w_gate_up_bits, w_down_bits, group: int, rows=None, threads: int = 0) -> np.ndarray:
    """FFN of one expert group applied to rows of x, float64."""
    x = _u16(x_bits)
    wgu = _u16(w_gate_up_bits)
    wd = _u16(w_down_bits)
    T, d = x.shape
    F = wgu.shape[1] // 2
    if rows is None:
        rows = np.arange(T, dtype=np.int32)
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    out = np.zeros((rows.shape[0], d), np.float64)
    rc = _load().oracle_expert_ffn(x, wgu, wd, d, F, group, rows, rows.shape[0], out, threads)
    if rc != 0:
        raise ValueError("oracle_expert_ffn rejected its arguments")
    return out
