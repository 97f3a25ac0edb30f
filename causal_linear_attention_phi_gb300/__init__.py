"""Causal linear attention with phi(x) = elu(x) + 1 on GB300 (sm_103a).

A thin ctypes binding over the C ABI of ``libla.so`` (declared in
``include/la.h``).  It only marshals arguments: every step of the computation
runs in the library's CUDA kernels.  PyTorch supplies device memory (outputs
and the workspace come from its caching allocator) and the current stream.
There is no CPU fallback: if the library is not built, importing works but
every call raises ``RuntimeError``.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

__all__ = [
    "LaError", "noncausal_fwd", "noncausal_bwd", "causal_fwd", "causal_bwd", "causal_step_host", "host_step_bytes",
    "recurrent_step", "retention_fwd", "retention_step", "selftest_bounded_wait", "workspace_bytes",
    "last_error", "clear_error", "timing_enable", "timing_reset", "timing_read", "library", "version",
    "OP_NONCAUSAL_FWD", "OP_CAUSAL_FWD", "OP_CAUSAL_BWD", "OP_NONCAUSAL_BWD", "OP_RETENTION_FWD",
]

OP_NONCAUSAL_FWD, OP_CAUSAL_FWD, OP_CAUSAL_BWD, OP_NONCAUSAL_BWD, OP_RETENTION_FWD = 0, 1, 2, 3, 4
LA_F32, LA_BF16 = 0, 1
_STATUS = {0: "LA_OK", 1: "LA_ERR_INVALID_ARG", 2: "LA_ERR_UNSUPPORTED", 3: "LA_ERR_WORKSPACE",
           4: "LA_ERR_CUDA", 5: "LA_ERR_TIMEOUT", 6: "LA_ERR_BOUNDS"}


class LaError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        super().__init__("%s failed: %s%s" % (where, _STATUS.get(status, str(status)),
                                               (" (%s)" % detail) if detail else ""))


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("N", ctypes.c_int), ("Dk", ctypes.c_int),
                ("Dv", ctypes.c_int), ("dtype", ctypes.c_int)]


class KernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("launches", ctypes.c_int), ("total_ms", ctypes.c_double)]


_lib = None
_lock = threading.Lock()
_vp = ctypes.c_void_p


def _declare(lib):
    lib.la_workspace_bytes.argtypes = [ctypes.c_int, Shape]
    lib.la_workspace_bytes.restype = ctypes.c_size_t
    lib.la_noncausal_fwd.argtypes = [_vp, _vp, _vp, _vp, Shape, _vp, ctypes.c_size_t, _vp]
    lib.la_causal_fwd.argtypes = [_vp, _vp, _vp, _vp, Shape, _vp, ctypes.c_size_t, _vp]
    lib.la_causal_fwd_fused.argtypes = [_vp, _vp, _vp, _vp, Shape, _vp, ctypes.c_size_t, _vp]
    lib.la_causal_bwd.argtypes = [_vp] * 7 + [Shape, _vp, ctypes.c_size_t, _vp]
    lib.la_host_step_bytes.argtypes = [Shape, ctypes.c_int]
    lib.la_host_step_bytes.restype = ctypes.c_size_t
    lib.la_causal_step_host.argtypes = [_vp] * 8 + [Shape, ctypes.c_int, _vp, ctypes.c_size_t, _vp]
    lib.la_noncausal_bwd.argtypes = [_vp] * 7 + [Shape, _vp, ctypes.c_size_t, _vp]
    lib.la_causal_fwd_with_state.argtypes = [_vp] * 6 + [Shape, _vp, ctypes.c_size_t, _vp]
    lib.la_causal_bwd_after_fwd.argtypes = [_vp] * 7 + [Shape, _vp, ctypes.c_size_t, _vp, ctypes.c_size_t, _vp]
    lib.la_recurrent_step.argtypes = [_vp] * 6 + [Shape, _vp]
    lib.la_retention_fwd.argtypes = [_vp] * 6 + [Shape, _vp, ctypes.c_size_t, _vp]
    lib.la_retention_step.argtypes = [_vp] * 6 + [Shape, _vp]
    lib.la_selftest_bounded_wait.argtypes = [_vp]
    lib.la_selftest_lookback_timeout.argtypes = [_vp] * 4 + [Shape, _vp, ctypes.c_size_t, _vp]
    for f in ("la_causal_step_host", "la_noncausal_fwd", "la_noncausal_bwd", "la_causal_fwd",
              "la_causal_fwd_with_state", "la_causal_bwd", "la_causal_bwd_after_fwd", "la_recurrent_step",
              "la_retention_fwd", "la_retention_step", "la_selftest_bounded_wait", "la_selftest_lookback_timeout",
              "la_last_error", "la_causal_fwd_fused",
              "la_clear_error", "la_timing_enable", "la_timing_reset"):
        getattr(lib, f).restype = ctypes.c_int
    lib.la_last_error.argtypes = []
    lib.la_clear_error.argtypes = []
    lib.la_status_string.argtypes = [ctypes.c_int]
    lib.la_status_string.restype = ctypes.c_char_p
    lib.la_error_detail.argtypes = []
    lib.la_error_detail.restype = ctypes.c_char_p
    lib.la_version.argtypes = []
    lib.la_version.restype = ctypes.c_char_p
    lib.la_timing_enable.argtypes = [ctypes.c_int]
    lib.la_timing_reset.argtypes = []
    lib.la_timing_read.argtypes = [ctypes.POINTER(KernelTime), ctypes.c_int]
    lib.la_timing_read.restype = ctypes.c_int
    return lib


def library(path: str | None = None):
    """The loaded libla (ctypes.CDLL).  Raises RuntimeError if it is not built.

    With LA_DEBUG=1 in the environment the debug build (device-side index checks,
    _lib/libla_debug.so) is loaded instead of the regular one."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or _build.lib_path(os.environ.get("LA_DEBUG", "0") == "1")
            if not os.path.exists(p):
                raise RuntimeError("libla.so is not built (%s); run causal_linear_attention_phi_gb300.build."
                                   "build_library() or __graft_entry__.build()" % p)
            _lib = _declare(ctypes.CDLL(p))
    return _lib


def version() -> str:
    return library().la_version().decode()


def _check(st: int, where: str):
    if st != 0:
        raise LaError(st, where, library().la_error_detail().decode(errors="replace"))


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return LA_F32
    if t.dtype == torch.bfloat16:
        return LA_BF16
    raise TypeError("unsupported dtype %s (float32 or bfloat16)" % t.dtype)


def _need_cuda(*ts):
    for t in ts:
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError("expected CUDA tensors")
        if not t.is_contiguous():
            raise ValueError("expected contiguous tensors")


def _stream_ptr(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None and t.numel() > 0 else ctypes.c_void_p(0)


def _shape4(q, k, v):
    if q.dim() != 4 or k.shape != q.shape or v.dim() != 4 or v.shape[:3] != q.shape[:3]:
        raise ValueError("expected q, k [B,H,N,Dk] and v [B,H,N,Dv]; got %s %s %s" %
                         (tuple(q.shape), tuple(k.shape), tuple(v.shape)))
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share a dtype")
    B, H, N, Dk = q.shape
    return Shape(B, H, N, Dk, v.shape[3], _dtype_code(q))


def workspace_bytes(op: int, B: int, H: int, N: int, Dk: int, Dv: int, dtype: torch.dtype) -> int:
    if dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("unsupported dtype %s (float32 or bfloat16)" % dtype)
    code = LA_BF16 if dtype == torch.bfloat16 else LA_F32
    return int(library().la_workspace_bytes(op, Shape(B, H, N, Dk, Dv, code)))


def _workspace(op, s: Shape, device, workspace):
    need = int(library().la_workspace_bytes(op, s))
    if workspace is not None:
        if not workspace.is_cuda:
            raise ValueError("workspace must be a device tensor")
        return workspace, workspace.numel() * workspace.element_size()  # its real size: the library checks it
    if need == 0:
        return None, 0
    return torch.empty(need, dtype=torch.uint8, device=device), need


def noncausal_fwd(q, k, v, out=None, workspace=None, stream=None):
    """o_i = phi(q_i)^T S / phi(q_i)^T z with S = phi(K)^T V, z = phi(K)^T 1 over all positions."""
    _need_cuda(q, k, v)
    s = _shape4(q, k, v)
    if out is None:
        out = torch.empty_like(v)
    ws, nb = _workspace(OP_NONCAUSAL_FWD, s, q.device, workspace)
    _check(library().la_noncausal_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), s, _ptr(ws), nb, _stream_ptr(stream)),
           "la_noncausal_fwd")
    return out


def causal_fwd(q, k, v, out=None, workspace=None, stream=None, return_state=False, one_launch=False):
    """Causal linear attention (j <= i) in the chunked form; returns o [B,H,N,Dv].

    With return_state, returns (o, S, z): the fp32 state after the last position
    (S [B,H,Dk,Dv], z [B,H,Dk]), from which recurrent_step continues.  With
    one_launch, runs la_causal_fwd_fused (the same results from one kernel launch
    with a chained scan; bf16 heads of 64 or 128).
    """
    _need_cuda(q, k, v)
    s = _shape4(q, k, v)
    if out is None:
        out = torch.empty_like(v)
    ws, nb = _workspace(OP_CAUSAL_FWD, s, q.device, workspace)
    if not return_state:
        fn = library().la_causal_fwd_fused if one_launch else library().la_causal_fwd
        _check(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(out), s, _ptr(ws), nb, _stream_ptr(stream)),
               "la_causal_fwd_fused" if one_launch else "la_causal_fwd")
        return out
    B, H, _, Dk = q.shape
    S = torch.empty(B, H, Dk, v.shape[-1], dtype=torch.float32, device=q.device)
    z = torch.empty(B, H, Dk, dtype=torch.float32, device=q.device)
    _check(library().la_causal_fwd_with_state(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(S), _ptr(z), s, _ptr(ws),
                                              nb, _stream_ptr(stream)), "la_causal_fwd_with_state")
    return out, S, z


def causal_bwd(q, k, v, dout, dq=None, dk=None, dv=None, workspace=None, stream=None, fwd_workspace=None):
    """Gradients (dq, dk, dv) of the causal form for upstream gradient dout.

    With fwd_workspace (the workspace of the causal_fwd call on the same q, k,
    v, unchanged since), the per-segment forward states are read from it
    (la_causal_bwd_after_fwd); otherwise they are recomputed (la_causal_bwd).
    """
    _need_cuda(q, k, v, dout)
    s = _shape4(q, k, v)
    if dout.shape != v.shape or dout.dtype != v.dtype:
        raise ValueError("dout must match v in shape and dtype")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws, nb = _workspace(OP_CAUSAL_BWD, s, q.device, workspace)
    if fwd_workspace is None:
        _check(library().la_causal_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), s,
                                       _ptr(ws), nb, _stream_ptr(stream)), "la_causal_bwd")
    else:
        if not fwd_workspace.is_cuda:
            raise ValueError("fwd_workspace must be the device workspace of the forward call")
        fnb = fwd_workspace.numel() * fwd_workspace.element_size()
        _check(library().la_causal_bwd_after_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                                                 s, _ptr(fwd_workspace), fnb, _ptr(ws), nb, _stream_ptr(stream)),
               "la_causal_bwd_after_fwd")
    return dq, dk, dv


def noncausal_bwd(q, k, v, dout, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Gradients (dq, dk, dv) of the non-causal form for upstream gradient dout."""
    _need_cuda(q, k, v, dout)
    s = _shape4(q, k, v)
    if dout.shape != v.shape or dout.dtype != v.dtype:
        raise ValueError("dout must match v in shape and dtype")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws, nb = _workspace(OP_NONCAUSAL_BWD, s, q.device, workspace)
    _check(library().la_noncausal_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), s,
                                      _ptr(ws), nb, _stream_ptr(stream)), "la_noncausal_bwd")
    return dq, dk, dv


def host_step_bytes(B: int, H: int, N: int, Dk: int, Dv: int, dtype: torch.dtype, group_heads: int) -> int:
    code = LA_BF16 if dtype == torch.bfloat16 else LA_F32
    return int(library().la_host_step_bytes(Shape(B, H, N, Dk, Dv, code), group_heads))


def causal_step_host(q, k, v, dout, o, dq, dk, dv, group_heads=2, dev_buf=None, stream=None):
    """One causal forward + backward on pinned host tensors (la_causal_step_host).

    q, k, v, dout are read and o, dq, dk, dv written, all pinned CPU tensors of
    the [B,H,N,D] shapes; transfers and kernels are pipelined over groups of
    `group_heads` heads.  Returns after queueing: synchronise the stream before
    reading the outputs.
    """
    for t in (q, k, v, dout, o, dq, dk, dv):
        if t.is_cuda or not t.is_pinned():
            raise ValueError("causal_step_host takes pinned host tensors")
    s = _shape4(q, k, v)
    if dout.shape != v.shape or o.shape != v.shape or dv.shape != v.shape or dq.shape != q.shape or \
            dk.shape != k.shape:
        raise ValueError("output and gradient shapes must match the inputs")
    need = int(library().la_host_step_bytes(s, group_heads))
    if dev_buf is None:
        dev_buf = torch.empty(need, dtype=torch.uint8, device=torch.device("cuda", torch.cuda.current_device()))
    nb = dev_buf.numel() * dev_buf.element_size()
    _check(library().la_causal_step_host(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(o), _ptr(dq), _ptr(dk), _ptr(dv),
                                         s, group_heads, _ptr(dev_buf), nb, _stream_ptr(stream)),
           "la_causal_step_host")
    return o, dq, dk, dv


def recurrent_step(q, k, v, S, z, out=None, stream=None):
    """One decode step: S += phi(k) v^T, z += phi(k) (in place), out = phi(q)^T S / phi(q)^T z."""
    _need_cuda(q, k, v, S, z)
    if q.dim() != 3 or k.shape != q.shape or v.shape[:2] != q.shape[:2]:
        raise ValueError("expected q, k [B,H,Dk] and v [B,H,Dv]")
    B, H, Dk = q.shape
    Dv = v.shape[2]
    if S.dtype != torch.float32 or z.dtype != torch.float32 or S.shape != (B, H, Dk, Dv) or z.shape != (B, H, Dk):
        raise ValueError("S must be fp32 [B,H,Dk,Dv] and z fp32 [B,H,Dk]")
    if out is None:
        out = torch.empty_like(v)
    s = Shape(B, H, 1, Dk, Dv, _dtype_code(q))
    _check(library().la_recurrent_step(_ptr(q), _ptr(k), _ptr(v), _ptr(S), _ptr(z), _ptr(out), s, _stream_ptr(stream)),
           "la_recurrent_step")
    return out


def _gamma(gamma, H):
    _need_cuda(gamma)
    if gamma.dtype != torch.float32 or gamma.shape != (H,):
        raise ValueError("gamma must be an fp32 CUDA tensor of shape [H] (one decay per head)")
    return gamma


def retention_fwd(q, k, v, gamma, out=None, workspace=None, stream=None, return_state=False):
    """Retention with a constant decay per head: o_t = sum_{j<=t} gamma^(t-j) (q_t . k_j) v_j.

    No feature map and no normaliser; gamma is fp32 [H] on the device.  With
    return_state, returns (o, S): S [B,H,Dk,Dv] fp32 is the state after the
    last position, from which retention_step continues.
    """
    _need_cuda(q, k, v)
    s = _shape4(q, k, v)
    _gamma(gamma, q.shape[1])
    if out is None:
        out = torch.empty_like(v)
    S = None
    if return_state:
        B, H, _, Dk = q.shape
        S = torch.empty(B, H, Dk, v.shape[-1], dtype=torch.float32, device=q.device)
    ws, nb = _workspace(OP_RETENTION_FWD, s, q.device, workspace)
    _check(library().la_retention_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(gamma), _ptr(out), _ptr(S), s, _ptr(ws), nb,
                                      _stream_ptr(stream)), "la_retention_fwd")
    return (out, S) if return_state else out


def retention_step(q, k, v, gamma, S, out=None, stream=None):
    """One retention decode step: S <- gamma S + k v^T (in place), out = S^T q."""
    _need_cuda(q, k, v, S)
    if q.dim() != 3 or k.shape != q.shape or v.shape[:2] != q.shape[:2]:
        raise ValueError("expected q, k [B,H,Dk] and v [B,H,Dv]")
    B, H, Dk = q.shape
    Dv = v.shape[2]
    _gamma(gamma, H)
    if S.dtype != torch.float32 or S.shape != (B, H, Dk, Dv):
        raise ValueError("S must be fp32 [B,H,Dk,Dv]")
    if out is None:
        out = torch.empty_like(v)
    s = Shape(B, H, 1, Dk, Dv, _dtype_code(q))
    _check(library().la_retention_step(_ptr(q), _ptr(k), _ptr(v), _ptr(gamma), _ptr(S), _ptr(out), s,
                                       _stream_ptr(stream)), "la_retention_step")
    return out


def selftest_bounded_wait(stream=None):
    """Launch the bounded-wait self-test (a wait that runs out after about a second and
    records LA_ERR_TIMEOUT in the sticky status word); read it with last_error()."""
    _check(library().la_selftest_bounded_wait(_stream_ptr(stream)), "la_selftest_bounded_wait")


def selftest_lookback_timeout(q, k, v, out=None, workspace=None, stream=None):
    """The one-launch causal forward with segment 0 of head 0 withholding its sums: the
    later segments of that head time out (about a second) and record LA_ERR_TIMEOUT; read
    it with last_error().  Other heads' outputs are complete."""
    _need_cuda(q, k, v)
    s = _shape4(q, k, v)
    if out is None:
        out = torch.empty_like(v)
    ws, nb = _workspace(OP_CAUSAL_FWD, s, q.device, workspace)
    _check(library().la_selftest_lookback_timeout(_ptr(q), _ptr(k), _ptr(v), _ptr(out), s, _ptr(ws), nb,
                                                  _stream_ptr(stream)), "la_selftest_lookback_timeout")
    return out


def last_error() -> int:
    """Sticky device-side status (0 = LA_OK); synchronises the device."""
    return int(library().la_last_error())


def clear_error():
    _check(library().la_clear_error(), "la_clear_error")


def timing_enable(on: bool = True):
    _check(library().la_timing_enable(1 if on else 0), "la_timing_enable")


def timing_reset():
    _check(library().la_timing_reset(), "la_timing_reset")


def timing_read() -> dict:
    """{kernel name: (launches, total_ms)} since the last reset."""
    lib = library()
    n = lib.la_timing_read(None, 0)
    buf = (KernelTime * max(n, 1))()
    n = lib.la_timing_read(buf, n)
    return {buf[i].name.decode(): (buf[i].launches, buf[i].total_ms) for i in range(n)}
