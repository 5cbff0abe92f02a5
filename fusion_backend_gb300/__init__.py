"""Python binding of libmoe_ffn.so, the fused MoE FFN layer for GB300.

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current CUDA stream.  The
functions carry the names of the C ABI in ``include/moe_ffn.h``.

There is no CPU fallback: if the library has not been built, or the device is
not a GB300 (sm_103), the calls raise.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

from . import _build

LIB_PATH = _build.LIB

OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_WORKSPACE = -3
ERR_MISALIGNED = -4
ERR_CUDA = -5
ERR_TIMEOUT = -6
ERR_DEVICE = -7

ACT_F32 = 0
ACT_BF16 = 1
W_BF16 = 0
W_Q4B32 = 1
W_I8 = 2

QUERY_PATH = 0
QUERY_LAUNCHES_PER_EXECUTE = 1
QUERY_TWO_STREAM_WORKSPACE = 2

EXPORTS = (
    "moe_ffn_prepare",
    "moe_ffn_execute",
    "moe_ffn_execute_ex",
    "moe_ffn_execute_block",
    "moe_ffn_read_status",
    "moe_ffn_read_routing",
    "moe_ffn_probe_timeout",
    "moe_ffn_query",
    "moe_ffn_destroy",
    "moe_ffn_strerror",
    "moe_ffn_execute_static_scratch",
    "moe_ffn_last_cuda_error",
    "moe_ffn_execute_two_stream",
)

STATIC_SCRATCH_BYTES = 1 << 24


class MoeFFNError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {strerror(status)} ({status})")
        self.status = status


class Shapes(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("T", "H", "E", "top_k", "I", "Is")]


class DType(ctypes.Structure):
    _fields_ = [("act", ctypes.c_int32), ("wfmt", ctypes.c_int32)]


_lib = None


def build(force: bool = False) -> str:
    """Compile the library for sm_103a (nvcc) if it is missing or stale."""
    return _build.build(force=force)


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run fusion_backend_gb300.build() first")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        L.moe_ffn_prepare.restype = ctypes.c_int
        L.moe_ffn_prepare.argtypes = [ctypes.POINTER(Shapes), DType, ctypes.POINTER(vp), ctypes.POINTER(sz)]
        L.moe_ffn_execute.restype = ctypes.c_int
        L.moe_ffn_execute.argtypes = [vp, vp, vp, sz, vp, vp, vp, vp, vp, vp]
        L.moe_ffn_execute_ex.restype = ctypes.c_int
        L.moe_ffn_execute_ex.argtypes = [vp, vp, vp, sz, vp, vp, vp, vp, vp, vp, vp, vp]
        L.moe_ffn_execute_block.restype = ctypes.c_int
        L.moe_ffn_execute_block.argtypes = [vp, vp, vp, sz, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp]
        L.moe_ffn_read_status.restype = ctypes.c_int
        L.moe_ffn_read_status.argtypes = [vp, vp, vp, ctypes.POINTER(i32)]
        L.moe_ffn_read_routing.restype = ctypes.c_int
        L.moe_ffn_read_routing.argtypes = [vp, vp, vp, vp, vp, vp, vp, ctypes.POINTER(i32)]
        L.moe_ffn_query.restype = ctypes.c_int
        L.moe_ffn_query.argtypes = [vp, i32, ctypes.POINTER(ctypes.c_int64)]
        L.moe_ffn_destroy.restype = None
        L.moe_ffn_destroy.argtypes = [vp]
        L.moe_ffn_execute_static_scratch.restype = ctypes.c_int
        L.moe_ffn_execute_static_scratch.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp]
        L.moe_ffn_strerror.restype = ctypes.c_char_p
        L.moe_ffn_strerror.argtypes = [ctypes.c_int]
        L.moe_ffn_probe_timeout.restype = ctypes.c_int
        L.moe_ffn_probe_timeout.argtypes = [vp, vp, vp, sz, i32]
        L.moe_ffn_last_cuda_error.restype = ctypes.c_char_p
        L.moe_ffn_last_cuda_error.argtypes = []
        L.moe_ffn_execute_two_stream.restype = ctypes.c_int
        L.moe_ffn_execute_two_stream.argtypes = [vp, vp, vp, vp, vp, vp, sz, vp, vp, vp, vp, vp, vp]
        _lib = L
    return _lib


def strerror(status: int) -> str:
    try:
        return lib().moe_ffn_strerror(status).decode()
    except RuntimeError:
        return f"status {status}"


def _check(status: int, what: str) -> None:
    if status != OK:
        if status == ERR_CUDA:
            what = f"{what} [{lib().moe_ffn_last_cuda_error().decode()}]"
        raise MoeFFNError(status, what)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ----------------------------------------------------------------------------
# Functions with the C ABI names (raise MoeFFNError on a non-zero status)


def moe_ffn_prepare(shapes, act: int, wfmt: int):
    """Return (plan handle, workspace bytes).  Host only."""
    s = Shapes(shapes.T, shapes.H, shapes.E, shapes.top_k, shapes.I, shapes.Is)
    plan = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    _check(lib().moe_ffn_prepare(ctypes.byref(s), DType(act, wfmt), ctypes.byref(plan), ctypes.byref(ws)),
           "moe_ffn_prepare")
    return plan.value, ws.value


def moe_ffn_execute(plan, workspace, x, router_w, expert_w, shexp_w, shexp_gate_w, out, stream=None,
                    workspace_bytes=None):
    nbytes = workspace_bytes if workspace_bytes is not None else workspace.numel() * workspace.element_size()
    _check(lib().moe_ffn_execute(plan, _stream(stream), _ptr(workspace), nbytes, _ptr(x), _ptr(router_w),
                                 _ptr(expert_w), _ptr(shexp_w), _ptr(shexp_gate_w), _ptr(out)), "moe_ffn_execute")


def moe_ffn_execute_ex(plan, workspace, x, router_w, expert_w, shexp_w, shexp_gate_w, out, topk_ids=None,
                       topk_w=None, stream=None, workspace_bytes=None):
    nbytes = workspace_bytes if workspace_bytes is not None else workspace.numel() * workspace.element_size()
    _check(lib().moe_ffn_execute_ex(plan, _stream(stream), _ptr(workspace), nbytes, _ptr(x), _ptr(router_w),
                                    _ptr(expert_w), _ptr(shexp_w), _ptr(shexp_gate_w), _ptr(out), _ptr(topk_ids),
                                    _ptr(topk_w)), "moe_ffn_execute_ex")


def moe_ffn_execute_block(plan, workspace, x_res, router_w, expert_w, shexp_w, shexp_gate_w, eps=1e-6,
                          topk_ids=None, topk_w=None, stream=None, workspace_bytes=None):
    nbytes = workspace_bytes if workspace_bytes is not None else workspace.numel() * workspace.element_size()
    _check(lib().moe_ffn_execute_block(plan, _stream(stream), _ptr(workspace), nbytes, _ptr(x_res), _ptr(router_w),
                                       _ptr(expert_w), _ptr(shexp_w), _ptr(shexp_gate_w), eps, _ptr(topk_ids),
                                       _ptr(topk_w)), "moe_ffn_execute_block")


def moe_ffn_read_status(plan, workspace, stream=None) -> int:
    st = ctypes.c_int32()
    _check(lib().moe_ffn_read_status(plan, _ptr(workspace), _stream(stream), ctypes.byref(st)), "moe_ffn_read_status")
    return st.value


def moe_ffn_read_routing(plan, workspace, E: int, T: int, top_k: int, stream=None):
    import numpy as np

    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    perm = np.zeros(T * top_k, np.int32)
    active = np.zeros(E, np.int32)
    n = ctypes.c_int32()
    _check(lib().moe_ffn_read_routing(plan, _ptr(workspace), _stream(stream), counts.ctypes.data, offsets.ctypes.data,
                                      perm.ctypes.data, active.ctypes.data, ctypes.byref(n)), "moe_ffn_read_routing")
    return counts, offsets, perm, active[: n.value].copy()


def moe_ffn_probe_timeout(plan, workspace, which: int, stream=None, workspace_bytes=None) -> None:
    nbytes = workspace_bytes if workspace_bytes is not None else workspace.numel() * workspace.element_size()
    _check(lib().moe_ffn_probe_timeout(plan, _stream(stream), _ptr(workspace), nbytes, which), "moe_ffn_probe_timeout")


def moe_ffn_query(plan, what: int) -> int:
    v = ctypes.c_int64()
    _check(lib().moe_ffn_query(plan, what, ctypes.byref(v)), "moe_ffn_query")
    return v.value


def moe_ffn_destroy(plan) -> None:
    if plan:
        lib().moe_ffn_destroy(plan)


def moe_ffn_execute_static_scratch(plan, x, router_w, expert_w, shexp_w, shexp_gate_w, out, stream=None):
    """moe_ffn_execute without a workspace: the scratch is the library's own
    device array (STATIC_SCRATCH_BYTES).  Allocates nothing.  Calls that overlap
    on the GPU share that array and race; serialise them."""
    _check(lib().moe_ffn_execute_static_scratch(plan, _stream(stream), _ptr(x), _ptr(router_w), _ptr(expert_w),
                                                _ptr(shexp_w), _ptr(shexp_gate_w), _ptr(out)),
           "moe_ffn_execute_static_scratch")


def moe_ffn_execute_two_stream(plan, workspace, x, router_w, expert_w, shexp_w, shexp_gate_w, out, aux_stream=None,
                               fork_event=None, join_event=None, stream=None, workspace_bytes=None):
    """The layer as two branches on two streams joined by an add (routed on ``stream``, the gated shared expert
    on ``aux_stream``, torch.cuda.Event objects or raw handles as the fork and join events); with no aux stream the
    same kernels run one after the other on ``stream``."""
    nbytes = workspace_bytes if workspace_bytes is not None else workspace.numel() * workspace.element_size()
    ev = lambda e: None if e is None else (e if isinstance(e, int) else e.cuda_event)
    _check(lib().moe_ffn_execute_two_stream(plan, _stream(stream), None if aux_stream is None else _stream(aux_stream),
                                            ev(fork_event), ev(join_event), _ptr(workspace), nbytes, _ptr(x),
                                            _ptr(router_w), _ptr(expert_w), _ptr(shexp_w), _ptr(shexp_gate_w),
                                            _ptr(out)), "moe_ffn_execute_two_stream")


def moe_ffn_strerror(status: int) -> str:
    return strerror(status)


# ----------------------------------------------------------------------------
# Convenience wrapper


@dataclass
class MoeFFN:
    """A prepared layer: owns the plan and a workspace tensor on the current device."""

    shapes: object
    act: int
    wfmt: int

    def __post_init__(self):
        import torch

        self.plan, self.workspace_bytes = moe_ffn_prepare(self.shapes, self.act, self.wfmt)
        self.workspace = torch.empty(max(self.workspace_bytes, 256), dtype=torch.uint8, device="cuda")

    def __call__(self, x, router_w, expert_w, shexp_w, shexp_gate_w, out=None, topk_ids=None, topk_w=None,
                 stream=None):
        import torch

        if out is None:
            out = torch.empty((self.shapes.T, self.shapes.H), dtype=torch.float32, device=x.device)
        moe_ffn_execute_ex(self.plan, self.workspace, x, router_w, expert_w, shexp_w, shexp_gate_w, out, topk_ids,
                           topk_w, stream)
        return out

    def block(self, x_res, router_w, expert_w, shexp_w, shexp_gate_w, eps=1e-6, topk_ids=None, stream=None):
        moe_ffn_execute_block(self.plan, self.workspace, x_res, router_w, expert_w, shexp_w, shexp_gate_w, eps,
                              topk_ids, None, stream)
        return x_res

    def status(self, stream=None) -> int:
        return moe_ffn_read_status(self.plan, self.workspace, stream)

    def routing(self, stream=None):
        s = self.shapes
        return moe_ffn_read_routing(self.plan, self.workspace, s.E, s.T, s.top_k, stream)

    def close(self):
        if getattr(self, "plan", None):
            moe_ffn_destroy(self.plan)
            self.plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
