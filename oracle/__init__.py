"""ORACLE (test infrastructure only): ctypes binding of ``oracle.c``.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg use this package.  The library under ``fusion_backend_gb300`` never
imports it, and it imports nothing from the library.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to its source when missing or stale."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-o", tmp, _SRC, "-lm", "-lpthread"]
        )
        os.replace(tmp, _LIB)
    return _LIB


class _Shapes(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("T", "H", "E", "top_k", "I", "Is")]


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        vp, i64 = ctypes.c_void_p, ctypes.c_int64
        _lib.or_moe_ffn.restype = ctypes.c_int
        _lib.or_moe_ffn.argtypes = [ctypes.POINTER(_Shapes), ctypes.c_int, ctypes.c_int] + [vp] * 5 + [ctypes.c_int] + [vp] * 5
        _lib.or_block_step.restype = ctypes.c_int
        _lib.or_block_step.argtypes = [ctypes.POINTER(_Shapes), ctypes.c_int] + [vp] * 5 + [ctypes.c_double, ctypes.c_int, vp, vp]
        _lib.or_router_logits.restype = None
        _lib.or_router_logits.argtypes = [vp, i64, i64, vp, vp]
        _lib.or_topk.restype = None
        _lib.or_topk.argtypes = [vp, i64, i64, vp, vp]
        _lib.or_bucketing.restype = ctypes.c_int32
        _lib.or_bucketing.argtypes = [vp, i64, i64, i64, vp, vp, vp, vp]
        _lib.or_swiglu_ffn.restype = None
        _lib.or_swiglu_ffn.argtypes = [vp, ctypes.c_int, i64, i64, vp, vp]
        _lib.or_decode_row.restype = None
        _lib.or_decode_row.argtypes = [vp, ctypes.c_int, i64, i64, vp]
        _lib.or_rmsnorm_bf16.restype = None
        _lib.or_rmsnorm_bf16.argtypes = [vp, i64, ctypes.c_double, vp]
        _lib.or_f16_to_double.restype = ctypes.c_double
        _lib.or_f16_to_double.argtypes = [ctypes.c_uint16]
        _lib.or_bf16_to_double.restype = ctypes.c_double
        _lib.or_bf16_to_double.argtypes = [ctypes.c_uint16]
        _lib.or_expert_bytes.restype = i64
        _lib.or_expert_bytes.argtypes = [ctypes.c_int, i64, i64]
        _lib.or_threads_used.restype = ctypes.c_int
        _lib.or_threads_used.argtypes = [ctypes.POINTER(_Shapes), ctypes.c_int]
        _lib.or_float_to_bf16.restype = ctypes.c_uint16
        _lib.or_float_to_bf16.argtypes = [ctypes.c_float]
        _lib.or_quantize_i8.restype = None
        _lib.or_quantize_i8.argtypes = [vp, i64, vp, vp]
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


def nthreads() -> int:
    """Host cores this process may run on (sched_getaffinity)."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def threads_used(shapes, threads=None) -> int:
    """Threads a layer call of these shapes starts when offered ``threads`` (default: all cores)."""
    s = _Shapes(shapes.T, shapes.H, shapes.E, shapes.top_k, shapes.I, shapes.Is)
    return int(lib().or_threads_used(ctypes.byref(s), threads or nthreads()))


def quantize_i8(x_f64):
    """The int8 activation of one row (values must be fp32-representable): (q int8 [n], scale fp32)."""
    x, xp = _c(x_f64, np.float64)
    q = np.empty(x.size, np.int8)
    sc = np.empty(1, np.float32)
    lib().or_quantize_i8(xp, x.size, q.ctypes.data, sc.ctypes.data)
    return q, float(sc[0])


def float_to_bf16(v: float) -> int:
    """The oracle's fp32 -> bf16 conversion (round to nearest even) of one value."""
    return int(lib().or_float_to_bf16(ctypes.c_float(v)))


def moe_ffn(shapes, act, wfmt, x, router_w, expert_w, shexp_w, shexp_gate_w, threads=None):
    """Run the oracle layer. Returns dict(out, logits, ids, p, s)."""
    T, H, E, k = shapes.T, shapes.H, shapes.E, shapes.top_k
    s = _Shapes(shapes.T, shapes.H, shapes.E, shapes.top_k, shapes.I, shapes.Is)
    x, xp = _c(x, np.float32 if act == 0 else np.uint16)
    rw, rwp = _c(router_w, np.uint16)
    ew, ewp = _c(expert_w, np.uint8)
    sw, swp = _c(shexp_w, np.uint8)
    gw, gwp = _c(shexp_gate_w, np.uint16)
    out = np.empty((T, H), np.float32)
    logits = np.empty((T, E), np.float32)
    ids = np.empty((T, k), np.int32)
    p = np.empty((T, k), np.float32)
    sg = np.empty(T, np.float32)
    rc = lib().or_moe_ffn(
        ctypes.byref(s), act, wfmt, xp, rwp, ewp, swp, gwp, threads or nthreads(),
        out.ctypes.data, logits.ctypes.data, ids.ctypes.data, p.ctypes.data, sg.ctypes.data,
    )
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return {"out": out, "logits": logits, "ids": ids, "p": p, "s": sg}


def block_step(shapes, wfmt, x_res, router_w, expert_w, shexp_w, shexp_gate_w, eps=1e-6, threads=None):
    """One pre-norm block on a copy of x_res. Returns (x_res_new, ids, xn_bf16)."""
    s = _Shapes(shapes.T, shapes.H, shapes.E, shapes.top_k, shapes.I, shapes.Is)
    xr = np.array(x_res, dtype=np.float32, copy=True, order="C")
    ids = np.empty((shapes.T, shapes.top_k), np.int32)
    xn = np.empty((shapes.T, shapes.H), np.uint16)
    rw, rwp = _c(router_w, np.uint16)
    ew, ewp = _c(expert_w, np.uint8)
    sw, swp = _c(shexp_w, np.uint8)
    gw, gwp = _c(shexp_gate_w, np.uint16)
    rc = lib().or_block_step(ctypes.byref(s), wfmt, xr.ctypes.data, rwp, ewp, swp, gwp, eps, threads or nthreads(),
                             ids.ctypes.data, xn.ctypes.data)
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return xr, ids, xn


def router_logits(router_w, E, H, x_f64):
    rw, rwp = _c(router_w, np.uint16)
    x, xp = _c(x_f64, np.float64)
    out = np.empty(E, np.float32)
    lib().or_router_logits(rwp, E, H, xp, out.ctypes.data)
    return out


def topk(logits, k):
    lg, lp = _c(logits, np.float32)
    ids = np.empty(k, np.int32)
    p = np.empty(k, np.float64)
    lib().or_topk(lp, lg.size, k, ids.ctypes.data, p.ctypes.data)
    return ids, p


def bucketing(ids, E):
    ids, ip = _c(ids, np.int32)
    T, k = ids.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    active = np.empty(E, np.int32)
    U = lib().or_bucketing(ip, T, k, E, counts.ctypes.data, offsets.ctypes.data, perm.ctypes.data, active.ctypes.data)
    return counts, offsets, perm, active[:U].copy()


def swiglu_ffn(block, wfmt, H, inter, x_f64):
    b, bp = _c(block, np.uint8)
    x, xp = _c(x_f64, np.float64)
    y = np.empty(H, np.float64)
    lib().or_swiglu_ffn(bp, wfmt, H, inter, xp, y.ctypes.data)
    return y


def decode_row(matrix_bytes_arr, wfmt, cols, r):
    b, bp = _c(matrix_bytes_arr, np.uint8)
    out = np.empty(cols, np.float64)
    lib().or_decode_row(bp, wfmt, cols, r, out.ctypes.data)
    return out


def rmsnorm_bf16(x_f32, eps=1e-6):
    x, xp = _c(x_f32, np.float32)
    y = np.empty(x.size, np.uint16)
    lib().or_rmsnorm_bf16(xp, x.size, eps, y.ctypes.data)
    return y


def f16_to_double(bits: int) -> float:
    return lib().or_f16_to_double(bits)


def bf16_to_double(bits: int) -> float:
    return lib().or_bf16_to_double(bits)


def expert_bytes(wfmt, H, inter):
    return lib().or_expert_bytes(wfmt, H, inter)
