"""GB300 (sm_103a) fused attention forward: Python binding of the C ABI.

The binding only marshals arguments: every step of the computation runs in the
CUDA kernels of ``libfa_fwd.so`` (built in-tree by ``build()``), called through
the C ABI declared in ``include/fa_fwd.h``.  PyTorch provides device memory and
the current stream.  There is no fallback: if the library is missing, or a call
returns an error status, the call raises.

    >>> o, lse = fa_fwd(q, k, v, causal=True)      # q, k, v: CUDA [B, H, S, D]
"""
from __future__ import annotations

import contextlib
import ctypes
import math
import os
import re

import torch

from . import _build

__all__ = ["fa_fwd", "fa_fwd_splitkv", "fa_fwd_splitkv_static", "splitkv_workspace_bytes", "fa_fwd_hostio", "launch_info", "plan", "schedule_table", "device_status",
           "selftest_wait_timeout", "selftest_exp2_poly", "strerror", "build", "lib", "header_functions",
           "set_layout", "layout", "LAYOUT_AUTO", "LAYOUT_TWO_TILE", "LAYOUT_ONE_TILE", "debug_stats",
           "FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED", "FA_ERR_MISALIGNED",
           "FA_ERR_CUDA", "FA_ERR_TIMEOUT", "FA_ERR_SCRATCH", "FA_ERR_RANGE", "FaError"]

(FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_MISALIGNED, FA_ERR_CUDA, FA_ERR_TIMEOUT,
 FA_ERR_SCRATCH, FA_ERR_RANGE) = range(8)
_DTYPE = {torch.float16: 0, torch.bfloat16: 1}
HEADER = os.path.join(_build.ROOT, "include", "fa_fwd.h")

_lib = None


class FaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {strerror(status)} (status {status})")
        self.status = status


class LaunchInfo(ctypes.Structure):
    _fields_ = [("grid", ctypes.c_int), ("block", ctypes.c_int), ("smem_bytes", ctypes.c_int),
                ("tiles_per_unit", ctypes.c_int), ("units", ctypes.c_int),
                ("head_group", ctypes.c_int), ("num_sms", ctypes.c_int), ("schedule", ctypes.c_int),
                ("layout", ctypes.c_int), ("key_step", ctypes.c_int)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


def build(force: bool = False) -> str:
    """Compile the CUDA library for sm_103a (nvcc) if it is missing or stale."""
    return _build.build(force=force)


def lib() -> ctypes.CDLL:
    """The loaded C library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"{_build.LIB} is missing: build it with attention_fa_fwd_gb300.build()")
        L = ctypes.CDLL(_build.LIB)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        dims = [i, i, i, i, i, f, i, vp]
        L.fa_fwd.argtypes = [vp, vp, vp, vp, vp] + dims
        L.fa_fwd_hostio.argtypes = [vp] * 10 + dims
        L.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, ctypes.c_size_t, vp]
        L.fa_fwd_splitkv_workspace.argtypes = [i, i, i, i, i, i, ctypes.POINTER(ctypes.c_size_t)]
        L.fa_fwd_splitkv_static.argtypes = [vp, vp, vp, vp, vp] + dims
        L.fa_fwd_launch_info.argtypes = [i, i, i, i, i, i, ctypes.POINTER(LaunchInfo)]
        L.fa_fwd_plan.argtypes = [i, i, i, i, i, i, i, ctypes.POINTER(LaunchInfo)]
        us = ctypes.POINTER(ctypes.c_ushort)
        L.fa_fwd_schedule_table.argtypes = [i, i, i, i, i, i, i, us, i, us, i, ctypes.POINTER(i),
                                            ctypes.POINTER(i)]
        L.fa_device_status.argtypes = [vp, i, ctypes.POINTER(ctypes.c_uint)]
        L.fa_selftest_wait_timeout.argtypes = [ctypes.c_uint, vp]
        L.fa_selftest_exp2_poly.argtypes = [vp, vp, i, vp]
        L.fa_fwd_set_layout.argtypes = [i]
        L.fa_fwd_set_layout.restype = i
        L.fa_strerror.argtypes = [i]
        L.fa_strerror.restype = ctypes.c_char_p
        for name in ("fa_fwd", "fa_fwd_hostio", "fa_fwd_launch_info", "fa_fwd_plan", "fa_fwd_schedule_table",
                     "fa_device_status", "fa_selftest_wait_timeout", "fa_selftest_exp2_poly", "fa_fwd_splitkv",
                     "fa_fwd_splitkv_workspace", "fa_fwd_splitkv_static"):
            getattr(L, name).restype = i
        _lib = L
    return _lib


def header_functions() -> list[str]:
    """Names of the functions include/fa_fwd.h declares."""
    with open(HEADER, encoding="utf-8") as fh:
        text = fh.read()
    return sorted(set(re.findall(r"^(?:int|const char\*|size_t)\s+(fa_\w+)\s*\(", text, re.M)))


LAYOUT_AUTO, LAYOUT_TWO_TILE, LAYOUT_ONE_TILE = 0, 1, 2


def set_layout(layout: int) -> int:
    """Process-wide kernel layout of one-pass launches (0 automatic, 1 two query
    tiles per unit, 2 one query tile per unit); returns the previous one."""
    prev = lib().fa_fwd_set_layout(int(layout))
    if prev < 0:
        raise ValueError(f"layout must be 0, 1 or 2, got {layout}")
    return prev


@contextlib.contextmanager
def layout(value: int):
    """Context in which one-pass launches use kernel layout `value`."""
    prev = set_layout(value)
    try:
        yield
    finally:
        set_layout(prev)


def strerror(status: int) -> str:
    return lib().fa_strerror(int(status)).decode()


def _stream_ptr(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _on_device(device):
    """Context that makes `device` current; a no-op when it already is (the
    switch costs microseconds, comparable to a small problem's kernel)."""
    if device.index is None or device.index == torch.cuda.current_device():
        return contextlib.nullcontext()
    return torch.cuda.device(device)


def _check_qkv(q, k, v):
    # The valid case in one expression (a small problem's kernel takes less
    # time than the call's host work); otherwise the failing check's message.
    try:
        shp, dt, dev = q.shape, q.dtype, q.device
        if (q.is_cuda and len(shp) == 4 and k.shape == shp and v.shape == shp and k.dtype == dt
                and v.dtype == dt and dt in _DTYPE and k.device == dev and v.device == dev
                and q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
            return
    except AttributeError:
        pass
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dim() != 4:
            raise ValueError(f"{name} must be [B, H, S, D]")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if not (q.shape == k.shape == v.shape):
        raise ValueError("q, k, v must share one [B, H, S, D] shape")
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in _DTYPE:
        raise ValueError("q, k, v must all be float16 or all bfloat16")
    if not (q.device == k.device == v.device):
        raise ValueError("q, k, v must be on one device")


def _prepare(q, k, v, scale, out, lse):
    """Checks q, k, v and the output buffers (allocating those not given):
    every buffer the kernels touch is exactly the size they assume."""
    _check_qkv(q, k, v)
    B, H, S, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, S), device=q.device, dtype=torch.float32)
    if not isinstance(out, torch.Tensor) or out.shape != q.shape or out.dtype != q.dtype \
            or not out.is_contiguous() or out.device != q.device:
        raise ValueError("out must be a contiguous tensor like q")
    if not isinstance(lse, torch.Tensor) or lse.shape != (B, H, S) or lse.dtype != torch.float32 \
            or not lse.is_contiguous() or lse.device != q.device:
        raise ValueError("lse must be a contiguous float32 [B, H, S] tensor on q's device")
    return B, H, S, D, scale, out, lse


def fa_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
           scale: float | None = None, out: torch.Tensor | None = None,
           lse: torch.Tensor | None = None, stream=None):
    """O, LSE of softmax(Q K^T * scale + causal mask) V on the current CUDA stream.

    q, k, v: contiguous CUDA [B, H, S, D] float16/bfloat16 (D in {64, 128}).
    Returns (o [B, H, S, D] in the input dtype, lse [B, H, S] float32, natural log).
    """
    B, H, S, D, scale, out, lse = _prepare(q, k, v, scale, out, lse)
    with _on_device(q.device):
        rc = lib().fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                          B, H, S, D, int(bool(causal)), float(scale), _DTYPE[q.dtype],
                          _stream_ptr(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd")
    return out, lse


def splitkv_workspace_bytes(B: int, H: int, S: int, D: int, causal: bool,
                            dtype=torch.bfloat16) -> int:
    """Workspace bytes fa_fwd_splitkv needs on the current device (0: no split)."""
    n = ctypes.c_size_t(0)
    rc = lib().fa_fwd_splitkv_workspace(B, H, S, D, int(bool(causal)), _DTYPE.get(dtype, 99),
                                        ctypes.byref(n))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_splitkv_workspace")
    return n.value


def fa_fwd_splitkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
                   scale: float | None = None, workspace: torch.Tensor | None = None,
                   out: torch.Tensor | None = None, lse: torch.Tensor | None = None, stream=None):
    """fa_fwd for problems too small to fill the GPU in one pass: key ranges are
    split into chunks whose partial results are merged by a second kernel.
    `workspace` (a CUDA byte tensor) defaults to a fresh torch allocation of
    the size splitkv_workspace_bytes reports."""
    B, H, S, D, scale, out, lse = _prepare(q, k, v, scale, out, lse)
    with _on_device(q.device):
        if workspace is None:
            need = splitkv_workspace_bytes(B, H, S, D, causal, q.dtype)
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
        if not isinstance(workspace, torch.Tensor) or workspace.device != q.device \
                or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor on q's device")
        ws_bytes = workspace.numel() * workspace.element_size()
        rc = lib().fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                  lse.data_ptr(), B, H, S, D, int(bool(causal)), float(scale),
                                  _DTYPE[q.dtype], workspace.data_ptr(), ws_bytes,
                                  _stream_ptr(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_splitkv")
    return out, lse


def fa_fwd_splitkv_static(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
                          scale: float | None = None, out: torch.Tensor | None = None,
                          lse: torch.Tensor | None = None, stream=None):
    """fa_fwd_splitkv without a workspace: for callers that cannot allocate
    device memory, the split scratch is a fixed 32 MiB array inside the library
    (shared by every call on a device; overlapping calls race on it).  Raises
    FaError with FA_ERR_SCRATCH when the problem needs more than that."""
    B, H, S, D, scale, out, lse = _prepare(q, k, v, scale, out, lse)
    with _on_device(q.device):
        rc = lib().fa_fwd_splitkv_static(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                         lse.data_ptr(), B, H, S, D, int(bool(causal)), float(scale),
                                         _DTYPE[q.dtype], _stream_ptr(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_splitkv_static")
    return out, lse


def fa_fwd_hostio(q_h, k_h, v_h, o_h, lse_h, q_d, k_d, v_d, o_d, lse_d, causal: bool = False,
                  scale: float | None = None, stream=None):
    """Host-buffer form: copies q/k/v in, runs the pass, copies o/lse out, all
    enqueued on the stream (the caller synchronises).  Host tensors should be
    pinned; device tensors are the caller's [B, H, S, D] / [B, H, S] buffers."""
    host = {"q_h": q_h, "k_h": k_h, "v_h": v_h, "o_h": o_h, "lse_h": lse_h}
    dev = {"q_d": q_d, "k_d": k_d, "v_d": v_d, "o_d": o_d, "lse_d": lse_d}
    for name, t in list(host.items()) + list(dev.items()):
        if not isinstance(t, torch.Tensor) or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous tensor")
    if q_h.dim() != 4:
        raise ValueError("q_h must be [B, H, S, D]")
    B, H, S, D = q_h.shape
    dt = q_h.dtype
    if dt not in _DTYPE:
        raise ValueError("dtype must be float16 or bfloat16")
    for name in ("k_h", "v_h", "o_h", "q_d", "k_d", "v_d", "o_d"):
        t = host.get(name, dev.get(name))
        if t.shape != q_h.shape or t.dtype != dt:
            raise ValueError(f"{name} must match q_h's shape and dtype")
    for name, t in (("lse_h", lse_h), ("lse_d", lse_d)):
        if t.shape != (B, H, S) or t.dtype != torch.float32:
            raise ValueError(f"{name} must be a float32 [B, H, S] tensor")
    for name, t in host.items():
        if t.is_cuda:
            raise ValueError(f"{name} must be a host tensor")
    for name, t in dev.items():
        if not t.is_cuda or t.device != q_d.device:
            raise ValueError(f"{name} must be a CUDA tensor on q_d's device")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with _on_device(q_d.device):
        rc = lib().fa_fwd_hostio(q_h.data_ptr(), k_h.data_ptr(), v_h.data_ptr(), o_h.data_ptr(),
                                 lse_h.data_ptr(), q_d.data_ptr(), k_d.data_ptr(), v_d.data_ptr(),
                                 o_d.data_ptr(), lse_d.data_ptr(), B, H, S, D, int(bool(causal)),
                                 float(scale), _DTYPE[dt], _stream_ptr(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_hostio")


def launch_info(B: int, H: int, S: int, D: int, causal: bool, dtype=torch.bfloat16) -> dict:
    """Launch geometry on the current device (host query, launches nothing)."""
    info = LaunchInfo()
    rc = lib().fa_fwd_launch_info(B, H, S, D, int(bool(causal)), _DTYPE.get(dtype, 99),
                                  ctypes.byref(info))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_launch_info")
    return info.as_dict()


def plan(B: int, H: int, S: int, D: int, causal: bool, num_sms: int, dtype=torch.bfloat16) -> dict:
    """Launch geometry for a device with `num_sms` SMs (pure host computation)."""
    info = LaunchInfo()
    rc = lib().fa_fwd_plan(B, H, S, D, int(bool(causal)), _DTYPE.get(dtype, 99), num_sms,
                           ctypes.byref(info))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_plan")
    return info.as_dict()


def schedule_table(B: int, H: int, S: int, D: int, causal: bool, num_sms: int, dtype=torch.bfloat16):
    """Per-CTA unit lists of the host list schedule (pure host computation):
    a list of `grid` lists of unit indices, or None when the launch uses a
    closed-form schedule."""
    cap = 1 << 16
    off = (ctypes.c_ushort * (cap + 1))()
    units = (ctypes.c_ushort * cap)()
    n_ctas, n_units = ctypes.c_int(0), ctypes.c_int(0)
    rc = lib().fa_fwd_schedule_table(B, H, S, D, int(bool(causal)), _DTYPE.get(dtype, 99), num_sms, off, cap + 1,
                                     units, cap, ctypes.byref(n_ctas), ctypes.byref(n_units))
    if rc == FA_ERR_UNSUPPORTED:
        return None
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_schedule_table")
    return [list(units[off[c]:off[c + 1]]) for c in range(n_ctas.value)]


def device_status(clear: bool = True, stream=None) -> tuple[int, int]:
    """(status, site) of the bounded in-kernel waits; synchronises the stream."""
    site = ctypes.c_uint(0)
    rc = lib().fa_device_status(_stream_ptr(stream), int(bool(clear)), ctypes.byref(site))
    if rc not in (FA_OK, FA_ERR_TIMEOUT, FA_ERR_RANGE):
        raise FaError(rc, "fa_device_status")
    return rc, site.value


_dbg_lib = None


def debug_stats(q, k, v, causal: bool = False, scale: float | None = None):
    """One pass through the debug-statistics build of the library (a separate
    .so, compiled on first use with -DFA_DEBUG_STATS), the debug mode of "CUDA
    手写masked multi-head attention", section 6.3: each row hands its running
    statistics to the host.  Returns (o, lse, stats, counts, rule): stats
    [B, H, S, 2] float32 holds each row's final base b and row sum
    l = sum 2^(x - b) (x the scaled score in base 2; ln2 * (b + log2 l) is the
    LSE); counts = (warp rescales of O, row re-bases after a row's first key
    tile); rule = (threshold T, overshoot) of the re-base rule for q's dtype."""
    global _dbg_lib
    B, H, S, D, scale, out, lse = _prepare(q, k, v, scale, None, None)
    if _dbg_lib is None:
        L = ctypes.CDLL(_build.build(debug_stats=True))
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
        L.fa_debug_stats_set.argtypes = [vp, vp]
        L.fa_debug_rebase_rule.argtypes = [i, ctypes.POINTER(f), ctypes.POINTER(f)]
        L.fa_device_status.argtypes = [vp, i, ctypes.POINTER(ctypes.c_uint)]
        for name in ("fa_fwd", "fa_debug_stats_set", "fa_debug_rebase_rule", "fa_device_status"):
            getattr(L, name).restype = i
        _dbg_lib = L
    L = _dbg_lib
    stats = torch.full((B, H, S, 2), float("nan"), device=q.device, dtype=torch.float32)
    counts = torch.zeros(2, device=q.device, dtype=torch.int64)
    with _on_device(q.device):
        stream = _stream_ptr(None)
        rc = L.fa_debug_stats_set(stats.data_ptr(), counts.data_ptr())
        if rc == FA_OK:
            rc = L.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, S, D,
                          int(bool(causal)), float(scale), _DTYPE[q.dtype], stream)
        site = ctypes.c_uint(0)
        st = L.fa_device_status(stream, 1, ctypes.byref(site))
        L.fa_debug_stats_set(None, None)
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd (debug statistics build)")
    if st != FA_OK:
        raise FaError(st, f"fa_fwd (debug statistics build), site {site.value:#x}")
    t, o_ = ctypes.c_float(0), ctypes.c_float(0)
    L.fa_debug_rebase_rule(_DTYPE[q.dtype], ctypes.byref(t), ctypes.byref(o_))
    c = counts.cpu().tolist()
    return out, lse, stats, (c[0], c[1]), (t.value, o_.value)


def selftest_wait_timeout(timeout_us: int, stream=None) -> None:
    rc = lib().fa_selftest_wait_timeout(int(timeout_us), _stream_ptr(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_selftest_wait_timeout")


def selftest_exp2_poly(x, stream=None):
    """2^x by the FMA-pipe exponential, element-wise, for a CUDA float32 tensor."""
    if not (isinstance(x, torch.Tensor) and x.is_cuda and x.dtype == torch.float32):
        raise TypeError("x must be a CUDA float32 tensor")
    x = x.contiguous()
    y = torch.empty_like(x)
    rc = lib().fa_selftest_exp2_poly(x.data_ptr(), y.data_ptr(), x.numel(), _stream_ptr(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_selftest_exp2_poly")
    return y
