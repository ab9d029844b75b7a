"""Thin Python binding over libmita.so (ctypes).

Names match the C ABI in include/mita.h.  This module only marshals torch
tensors to pointers and picks the bf16 or `_f32` entry point; every step of the
computation runs in the library's CUDA kernels.  There is no fallback: if
libmita.so is missing, every call raises.

Tensors must be contiguous; Q/K/V/out are [B, H, N, d].  Calls run on the
current torch CUDA stream unless `stream` is given.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libmita.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "mita.h")

_lock = threading.Lock()
_lib = None

MITA_OK = 0
MITA_ERR_DEVICE_CHECK = 5


class MitaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"[{status}] {message}")
        self.status = status


def load() -> ctypes.CDLL:
    """Load libmita.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m sparse_top_landmark_gb300.build` (there is no CPU fallback)")
            lib = ctypes.CDLL(LIB_PATH)
            P, I = ctypes.c_void_p, ctypes.c_int
            sigs = {
                "mita_pool": [P, I, I, I, I, I, I, I, P, P],
                "mita_landmark_topk_shared": [P, P, P, I, I, I, I, I, I, P, P, P],
                "mita_route": [P, P, P, I, I, I, I, I, I, P, P, P, P],
                "mita_expert_attn": [P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, P],
                "mita_forward": [P, P, P, I, I, I, I, I, I, I, I, I, P, P],
                "mita_forward_host": [P, P, P, I, I, I, I, I, I, I, I, I, P, P],
                "mita_forward_ex": [P, P, P, I, I, I, I, I, I, I, I, I, P, P, P],
                "mita_pool_grid": [P, I, I, I, I, I, I, I, I, P, P],
                "mita_dense_attn": [P, P, P, I, I, I, I, P, P],
                "mita_backward": [P, P, P, P, I, I, I, I, I, I, I, I, I, P, P, P, P, P],
            }
            for name, at in sigs.items():
                for suffix in ("", "_f32"):
                    f = getattr(lib, name + suffix)
                    f.argtypes = at
                    f.restype = I
            lib.mita_bucket.argtypes = [P, I, I, I, I, I, P, P, P]
            lib.mita_bucket.restype = I
            lib.mita_bucket_noalloc.argtypes = [P, I, I, I, I, I, P, P, P]
            lib.mita_bucket_noalloc.restype = I
            lib.mita_forward_workspace_bytes.argtypes = [I, I, I, I, I, I, I, I]
            lib.mita_forward_workspace_bytes.restype = ctypes.c_uint64
            lib.mita_status_string.argtypes = [I]
            lib.mita_status_string.restype = ctypes.c_char_p
            lib.mita_last_error_message.argtypes = []
            lib.mita_last_error_message.restype = ctypes.c_char_p
            lib.mita_get_last_device_error.argtypes = [P, ctypes.POINTER(I)]
            lib.mita_get_last_device_error.restype = I
            lib.mita_workspace_release.argtypes = []
            lib.mita_workspace_release.restype = I
            lib.mita_workspace_set_limit.argtypes = [ctypes.c_uint64]
            lib.mita_workspace_set_limit.restype = ctypes.c_uint64
            lib.mita_kernel_launches.argtypes = []
            lib.mita_kernel_launches.restype = ctypes.c_uint64
            lib.mita_check_bounded_wait.argtypes = [P, P]
            lib.mita_check_bounded_wait.restype = I
            _lib = lib
    return _lib


def declared_functions() -> list:
    """Names of every function include/mita.h declares."""
    import re
    with open(HEADER_PATH) as f:
        text = f.read()
    return sorted(set(re.findall(r"\b(mita_[a-z0-9_]+)\s*\(", text)))


# ---------------------------------------------------------------------------
def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(rc: int):
    if rc != MITA_OK:
        lib = load()
        raise MitaError(rc, f"{lib.mita_status_string(rc).decode()}: "
                            f"{lib.mita_last_error_message().decode()}")


def _fn(name: str, dtype: torch.dtype):
    lib = load()
    if dtype == torch.bfloat16:
        return getattr(lib, name)
    if dtype == torch.float32:
        return getattr(lib, name + "_f32")
    raise TypeError(f"unsupported dtype {dtype}: use bfloat16 or float32")


def _need(t: torch.Tensor, name: str, dtype=None, device=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    return t


class MitaOptions(ctypes.Structure):
    """mita_options of the C header."""
    _fields_ = [("shared_temperature", ctypes.c_int), ("landmark_grid_h", ctypes.c_int),
                ("landmark_grid_w", ctypes.c_int), ("branches", ctypes.c_int)]


SHARED_TEMPERATURES = {"sqrt_d": 0, "d": 1}
BRANCHES = {"both": 0, "routed": 1}


# ---------------------------------------------------------------------------
def mita_pool_grid(q, grid_h: int, grid_w: int, landmark_grid_h: int, landmark_grid_w: int,
                   q_tilde=None, stream=None):
    """Pooling onto an explicit landmark_grid_h x landmark_grid_w landmark grid."""
    _need(q, "q")
    B, H, N, d = q.shape
    m = landmark_grid_h * landmark_grid_w
    if q_tilde is None:
        q_tilde = torch.empty((B, H, m, d), dtype=q.dtype, device=q.device)
    _need(q_tilde, "q_tilde", q.dtype, q.device)
    _check(_fn("mita_pool_grid", q.dtype)(_ptr(q), B, H, N, d, grid_h, grid_w, landmark_grid_h,
                                          landmark_grid_w, _ptr(q_tilde),
                                          _stream(stream, q.device)))
    return q_tilde


def mita_forward_ex(q, k, v, grid_h: int, grid_w: int, m: int, topk: int, s: int = 1,
                    shared_temperature: str = "sqrt_d", landmark_grid=None,
                    branches: str = "both", out=None, stream=None):
    """mita_forward on device tensors with options: the shared logits' temperature
    ("sqrt_d": q.q~/sqrt(d), "d": q.q~/d), an explicit (rows, cols) landmark grid, and
    the branches ("both", or "routed": the routing-only ablation without shared pairs)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype, q.device)
    B, H, N, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", q.dtype, q.device)
    opt = _options(shared_temperature, landmark_grid, branches)
    _check(_fn("mita_forward_ex", q.dtype)(_ptr(q), _ptr(k), _ptr(v), B, H, N, d, grid_h, grid_w,
                                           m, topk, s, ctypes.byref(opt), _ptr(out),
                                           _stream(stream, q.device)))
    return out


def _options(shared_temperature, landmark_grid, branches):
    lh, lw = landmark_grid if landmark_grid is not None else (0, 0)
    return MitaOptions(SHARED_TEMPERATURES[shared_temperature], lh, lw, BRANCHES[branches])


def mita_backward(q, k, v, dout, grid_h: int, grid_w: int, m: int, topk: int, s: int = 1,
                  shared_temperature: str = "sqrt_d", landmark_grid=None, branches: str = "both",
                  stream=None):
    """(dq, dk, dv), fp32, of mita_forward_ex's output for the upstream gradient ``dout``,
    with the forward's selections held constant."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (dout, "dout")):
        _need(t, n, q.dtype, q.device)
    B, H, N, d = q.shape
    grads = [torch.empty(q.shape, dtype=torch.float32, device=q.device) for _ in range(3)]
    opt = _options(shared_temperature, landmark_grid, branches)
    _check(_fn("mita_backward", q.dtype)(
        _ptr(q), _ptr(k), _ptr(v), _ptr(dout), B, H, N, d, grid_h, grid_w, m, topk, s,
        ctypes.byref(opt), _ptr(grads[0]), _ptr(grads[1]), _ptr(grads[2]),
        _stream(stream, q.device)))
    return tuple(grads)


class MiTAFunction(torch.autograd.Function):
    """MiTA attention as an autograd function: forward through mita_forward_ex, backward
    through mita_backward (selections held constant; gradients cast to the input dtype)."""

    @staticmethod
    def forward(ctx, q, k, v, grid_h, grid_w, m, topk, s=1, shared_temperature="sqrt_d",
                landmark_grid=None, branches="both"):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        ctx.save_for_backward(q, k, v)
        ctx.cfg = (grid_h, grid_w, m, topk, s, shared_temperature, landmark_grid, branches)
        return mita_forward_ex(q, k, v, grid_h, grid_w, m, topk, s, shared_temperature,
                               landmark_grid, branches)

    @staticmethod
    def backward(ctx, dout):
        q, k, v = ctx.saved_tensors
        gh, gw, m, topk, s, temp, lg, br = ctx.cfg
        dq, dk, dv = mita_backward(q, k, v, dout.contiguous().to(q.dtype), gh, gw, m, topk, s,
                                   temp, lg, br)
        return (dq.to(q.dtype), dk.to(k.dtype), dv.to(v.dtype)) + (None,) * 8


def mita_dense_attn(q, k, v, out=None, stream=None):
    """Dense softmax attention over all N keys of each head (the comparison baseline)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype, q.device)
    B, H, N, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", q.dtype, q.device)
    _check(_fn("mita_dense_attn", q.dtype)(_ptr(q), _ptr(k), _ptr(v), B, H, N, d, _ptr(out),
                                           _stream(stream, q.device)))
    return out


def mita_pool(q, grid_h: int, grid_w: int, m: int, q_tilde=None, stream=None):
    _need(q, "q")
    B, H, N, d = q.shape
    if q_tilde is None:
        q_tilde = torch.empty((B, H, m, d), dtype=q.dtype, device=q.device)
    _need(q_tilde, "q_tilde", q.dtype, q.device)
    _check(_fn("mita_pool", q.dtype)(_ptr(q), B, H, N, d, grid_h, grid_w, m, _ptr(q_tilde),
                                     _stream(stream, q.device)))
    return q_tilde


def mita_landmark_topk_shared(q_tilde, k, v, topk: int, topk_idx=None, v_tilde=None,
                              stream=None):
    for t, n in ((q_tilde, "q_tilde"), (k, "k"), (v, "v")):
        _need(t, n, k.dtype, k.device)
    B, H, N, d = k.shape
    m = q_tilde.shape[2]
    if topk_idx is None:
        topk_idx = torch.empty((B, H, m, topk), dtype=torch.int32, device=k.device)
    if v_tilde is None:
        v_tilde = torch.empty((B, H, m, d), dtype=torch.float32, device=k.device)
    _need(topk_idx, "topk_idx", torch.int32, k.device)
    _need(v_tilde, "v_tilde", torch.float32, k.device)
    _check(_fn("mita_landmark_topk_shared", k.dtype)(
        _ptr(q_tilde), _ptr(k), _ptr(v), B, H, N, d, m, topk, _ptr(topk_idx), _ptr(v_tilde),
        _stream(stream, k.device)))
    return topk_idx, v_tilde


def mita_route(q, q_tilde, v_tilde=None, s: int = 1, route_idx=None, shared: bool = False,
               stream=None):
    _need(q, "q")
    _need(q_tilde, "q_tilde", q.dtype, q.device)
    B, H, N, d = q.shape
    m = q_tilde.shape[2]
    if route_idx is None:
        route_idx = torch.empty((B, H, N, s), dtype=torch.int32, device=q.device)
    _need(route_idx, "route_idx", torch.int32, q.device)
    lse = o = None
    if shared:
        _need(v_tilde, "v_tilde", torch.float32, q.device)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
        o = torch.empty((B, H, N, d), dtype=torch.float32, device=q.device)
    _check(_fn("mita_route", q.dtype)(
        _ptr(q), _ptr(q_tilde), _ptr(v_tilde), B, H, N, d, m, s, _ptr(route_idx), _ptr(lse),
        _ptr(o), _stream(stream, q.device)))
    return (route_idx, lse, o) if shared else route_idx


def mita_bucket(route_idx, m: int, bucket_off=None, bucket_qidx=None, stream=None):
    _need(route_idx, "route_idx", torch.int32)
    B, H, N, s = route_idx.shape
    if bucket_off is None:
        bucket_off = torch.empty((B, H, m + 1), dtype=torch.int32, device=route_idx.device)
    if bucket_qidx is None:
        bucket_qidx = torch.empty((B, H, N * s), dtype=torch.int32, device=route_idx.device)
    _need(bucket_off, "bucket_off", torch.int32, route_idx.device)
    _need(bucket_qidx, "bucket_qidx", torch.int32, route_idx.device)
    _check(load().mita_bucket(_ptr(route_idx), B, H, N, m, s, _ptr(bucket_off),
                              _ptr(bucket_qidx), _stream(stream, route_idx.device)))
    return bucket_off, bucket_qidx


def mita_bucket_noalloc(route_idx, m: int, bucket_off, bucket_qidx, stream=None):
    """mita_bucket for callers that cannot allocate device memory: the caller
    passes both outputs, and the library uses its fixed 4 MiB device scratch
    instead of its workspace cache (limit B*H*(ceil(N*s/4096)+1)*m <= 1048576).
    Calls that overlap on the GPU race on that scratch; order them."""
    _need(route_idx, "route_idx", torch.int32)
    B, H, N, s = route_idx.shape
    _need(bucket_off, "bucket_off", torch.int32, route_idx.device)
    _need(bucket_qidx, "bucket_qidx", torch.int32, route_idx.device)
    _check(load().mita_bucket_noalloc(_ptr(route_idx), B, H, N, m, s, _ptr(bucket_off),
                                      _ptr(bucket_qidx), _stream(stream, route_idx.device)))
    return bucket_off, bucket_qidx


def mita_expert_attn(q, k, v, q_tilde, v_tilde, topk_idx, bucket_off, bucket_qidx,
                     shared_lse=None, shared_o=None, s: int = 1, out=None, stream=None):
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype, q.device)
    B, H, N, d = q.shape
    m, topk = topk_idx.shape[-2], topk_idx.shape[-1]
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", q.dtype, q.device)
    for t, n in ((topk_idx, "topk_idx"), (bucket_off, "bucket_off"), (bucket_qidx, "bucket_qidx")):
        _need(t, n, torch.int32, q.device)
    if bucket_qidx.numel() != B * H * N * s:
        raise ValueError(f"bucket_qidx holds {bucket_qidx.numel()} entries, expected B*H*N*s = "
                         f"{B * H * N * s}")
    if q_tilde is not None:
        _need(q_tilde, "q_tilde", q.dtype, q.device)
    if v_tilde is not None:
        _need(v_tilde, "v_tilde", torch.float32, q.device)
    _check(_fn("mita_expert_attn", q.dtype)(
        _ptr(q), _ptr(k), _ptr(v), _ptr(q_tilde), _ptr(v_tilde), _ptr(topk_idx),
        _ptr(bucket_off), _ptr(bucket_qidx), _ptr(shared_lse), _ptr(shared_o), B, H, N, d, m,
        topk, s, _ptr(out), _stream(stream, q.device)))
    return out


def mita_forward(q, k, v, grid_h: int, grid_w: int, m: int, topk: int, s: int = 1, out=None,
                 stream=None, device=None):
    """The whole forward pass.

    Device tensors: runs on the GPU and returns the device output.  Host
    tensors (ideally pinned) go through the library's host entry point, which
    copies Q, K, V to `device` (default cuda:0), runs, copies the output back
    into `out` (or a new pinned tensor) and synchronises before returning.
    """
    if not q.is_cuda:
        # host buffers: the library copies in, runs and copies out (one C call)
        dev = torch.device(device if device is not None else "cuda:0")
        for t, n in ((q, "q"), (k, "k"), (v, "v")):
            if t.is_cuda or t.dtype != q.dtype or t.shape != q.shape or not t.is_contiguous():
                raise ValueError(f"{n}: expected a contiguous host tensor like q")
        if out is None:
            out = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
        if out.is_cuda or out.dtype != q.dtype or out.shape != q.shape or not out.is_contiguous():
            raise ValueError("out: expected a contiguous host tensor like q")
        B, H, N, d = q.shape
        with torch.cuda.device(dev):
            _check(_fn("mita_forward_host", q.dtype)(
                _ptr(q), _ptr(k), _ptr(v), B, H, N, d, grid_h, grid_w, m, topk, s, _ptr(out),
                _stream(stream, dev)))
        return out
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype, q.device)
    B, H, N, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", q.dtype, q.device)
    _check(_fn("mita_forward", q.dtype)(_ptr(q), _ptr(k), _ptr(v), B, H, N, d, grid_h, grid_w,
                                        m, topk, s, _ptr(out), _stream(stream, q.device)))
    return out


def forward_workspace_bytes(B, H, N, d, m, topk, dtype=torch.bfloat16, s: int = 1) -> int:
    return int(load().mita_forward_workspace_bytes(B, H, N, d, m, topk, s,
                                                    1 if dtype == torch.float32 else 0))


def get_last_device_error(stream=None, device=None) -> int:
    """Synchronise and return (and clear) the device status bits (0 = clean)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    bits = ctypes.c_int(0)
    rc = load().mita_get_last_device_error(_stream(stream, dev), ctypes.byref(bits))
    if rc not in (MITA_OK, MITA_ERR_DEVICE_CHECK):
        _check(rc)
    return bits.value


def workspace_release() -> None:
    _check(load().mita_workspace_release())


def workspace_set_limit(nbytes: int) -> int:
    """Cap the growth of each cached buffer (0: no cap); returns the previous cap.  Growth past
    it raises MitaError(MITA_ERR_OOM) before any allocation."""
    return int(load().mita_workspace_set_limit(int(nbytes)))


def kernel_launches() -> int:
    """Kernel launches this library has issued in this process so far."""
    return int(load().mita_kernel_launches())


def check_bounded_wait(stream=None, device=None) -> torch.Tensor:
    """Runs the library's wait-timeout probe (mita_check_bounded_wait): a kernel whose
    two bounded waits on a never-arrived mbarrier must give up after about a second.
    Returns the device int32[2] gave-up flags (1 = that wait gave up)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    gave_up = torch.full((2,), -1, dtype=torch.int32, device=dev)
    _check(load().mita_check_bounded_wait(_ptr(gave_up), _stream(stream, dev)))
    return gave_up
