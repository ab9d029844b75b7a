"""fp64 CPU oracle for the MiTA forward pass -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  The product library never does, and
this package imports nothing from the product (it shares no code with the CUDA
path).  The arithmetic lives in ``mita_oracle.cpp`` (plain loops, fp64,
OpenMP over rows); this file only marshals tensors.

Every function follows the pages' step list (MiTA tutorial, iwxt.cn, ch. 4,
restating paper Sec. 3.2 eq. 5-12; gist.science summary Sec. 2.3, Algorithm 1);
the exact citation is on each C function.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mita_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_DT = {torch.float32: 0, torch.bfloat16: 1, torch.float64: 2}


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (OpenMP) into oracle/liboracle.so."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["g++", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c++17",
                        "-o", tmp, _SRC], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P, I, L = ctypes.c_void_p, ctypes.c_int, ctypes.c_long
            lib.orc_pool.argtypes = [P, I, I, I, I, I, I, I, I, I, P]
            lib.orc_pool_grid.argtypes = [P, I, I, I, I, I, I, I, I, I, I, P]
            lib.orc_landmark_rows.argtypes = [P, P, P, I, I, I, I, I, I, I, L, P, P, P, P]
            lib.orc_route_rows.argtypes = [P, I, P, I, I, I, I, I, I, L, P, P, P]
            lib.orc_bucket.argtypes = [P, I, I, I, I, I, P, P]
            lib.orc_attend_rows.argtypes = [P, P, P, I, P, P, P, P, I, I, I, I, I, I, I, L, P, P]
            lib.orc_attend_rows_v.argtypes = [P, P, P, I, P, P, P, P, I, I, I, I, I, I, I, L, P,
                                              I, I, P]
            lib.orc_dense_rows.argtypes = [P, P, P, I, I, I, I, I, L, P, P]
            lib.orc_num_threads.restype = I
            lib.orc_set_num_threads.argtypes = [I]
            _lib = lib
    return _lib


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _cpu(t):
    return t.detach().to("cpu").contiguous()


def num_threads() -> int:
    return _load().orc_num_threads()


def set_num_threads(n: int) -> None:
    _load().orc_set_num_threads(int(n))


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments (rc={rc})")


def pool(q, grid_h: int, grid_w: int, m: int, landmark_grid=None):
    """Landmark queries q~ [B,H,m,d] (float64 holding values of q's dtype).

    ``landmark_grid`` = (mh, mw) with mh * mw = m pools onto that grid; by
    default 1D pools to 1 x m and 2D to sqrt(m) x sqrt(m)."""
    q = _cpu(q)
    B, H, N, d = q.shape
    out = torch.empty((B, H, m, d), dtype=torch.float64)
    if landmark_grid is None:
        _check(_load().orc_pool(_p(q), _DT[q.dtype], B, H, N, d, grid_h, grid_w, m,
                                _DT[q.dtype], _p(out)), "pool")
    else:
        mh, mw = landmark_grid
        if mh * mw != m:
            raise ValueError("landmark grid must hold m landmarks")
        _check(_load().orc_pool_grid(_p(q), _DT[q.dtype], B, H, N, d, grid_h, grid_w, mh, mw,
                                     _DT[q.dtype], _p(out)), "pool")
    return out


def landmark(q_tilde, k, v, topk: int, rows=None):
    """Routed experts and shared values.

    Returns (topk_idx int32, v_tilde float64, gap float64).  With ``rows``
    (flat ids bh*m+i) only those rows are computed and outputs are [R, ...];
    otherwise outputs are [B,H,m,topk], [B,H,m,d], [B,H,m].
    """
    k, v = _cpu(k), _cpu(v)
    assert k.dtype == v.dtype
    B, H, N, d = k.shape
    qt = _cpu(q_tilde).to(torch.float64)
    m = qt.shape[2]
    if rows is None:
        R, rsel = B * H * m, None
    else:
        rsel = torch.as_tensor(rows, dtype=torch.int64).contiguous()
        R = rsel.numel()
    idx = torch.empty((R, topk), dtype=torch.int32)
    vt = torch.empty((R, d), dtype=torch.float64)
    gap = torch.empty((R,), dtype=torch.float64)
    _check(_load().orc_landmark_rows(_p(qt), _p(k), _p(v), _DT[k.dtype], B, H, N, d, m,
                                     topk, R, _p(rsel), _p(idx), _p(vt), _p(gap)),
           "landmark")
    if rows is None:
        return idx.view(B, H, m, topk), vt.view(B, H, m, d), gap.view(B, H, m)
    return idx, vt, gap


def route(q, q_tilde, s: int = 1, queries=None):
    """Top-s landmarks per query: (route int32 [B,H,N,s] or [R,s], gap)."""
    q = _cpu(q)
    B, H, N, d = q.shape
    qt = _cpu(q_tilde).to(torch.float64)
    m = qt.shape[2]
    if queries is None:
        R, qsel = B * H * N, None
    else:
        qsel = torch.as_tensor(queries, dtype=torch.int64).contiguous()
        R = qsel.numel()
    r = torch.empty((R, s), dtype=torch.int32)
    gap = torch.empty((R,), dtype=torch.float64)
    _check(_load().orc_route_rows(_p(q), _DT[q.dtype], _p(qt), B, H, N, d, m, s, R,
                                  _p(qsel), _p(r), _p(gap)), "route")
    if queries is None:
        return r.view(B, H, N, s), gap.view(B, H, N)
    return r, gap


def bucket(route_idx, m: int):
    """Stable grouping by expert: (bucket_off [B,H,m+1], bucket_qidx [B,H,N*s])."""
    r = _cpu(route_idx).to(torch.int32)
    B, H, N, s = r.shape
    off = torch.empty((B, H, m + 1), dtype=torch.int32)
    qidx = torch.empty((B, H, N * s), dtype=torch.int32)
    _check(_load().orc_bucket(_p(r), B, H, N, m, s, _p(off), _p(qidx)), "bucket")
    return off, qidx


def attend(q, k, v, q_tilde, v_tilde, topk_idx, route_idx, queries=None,
           shared_temperature: str = "sqrt_d", branches: str = "both"):
    """Joint-softmax output (float64) for all queries [B,H,N,d] or a sample [R,d].

    ``route_idx`` is [B,H,N,s] for all queries, or [R,s] aligned with ``queries``.
    ``shared_temperature``: "sqrt_d" (every logit / sqrt(d)) or "d" (the shared
    logits q . q~ / d, raw logits still / sqrt(d)).
    ``branches``: "both" (the m shared pairs and the s*k raw pairs) or "routed"
    (the routing-only ablation: the s*k raw pairs alone).
    """
    temp = {"sqrt_d": 0, "d": 1}[shared_temperature]
    routed = {"both": 0, "routed": 1}[branches]
    q, k, v = _cpu(q), _cpu(k), _cpu(v)
    B, H, N, d = q.shape
    qt = _cpu(q_tilde).to(torch.float64)
    vt = _cpu(v_tilde).to(torch.float64)
    ti = _cpu(topk_idx).to(torch.int32)
    m, topk = ti.shape[-2], ti.shape[-1]
    r = _cpu(route_idx).to(torch.int32)
    s = r.shape[-1]
    if queries is None:
        R, qsel = B * H * N, None
    else:
        qsel = torch.as_tensor(queries, dtype=torch.int64).contiguous()
        R = qsel.numel()
    out = torch.empty((R, d), dtype=torch.float64)
    _check(_load().orc_attend_rows_v(_p(q), _p(k), _p(v), _DT[q.dtype], _p(qt), _p(vt),
                                     _p(ti), _p(r), B, H, N, d, m, topk, s, R, _p(qsel),
                                     temp, routed, _p(out)), "attend")
    return out.view(B, H, N, d) if queries is None else out


def dense(q, k, v, queries=None):
    """Dense softmax attention (float64): [B,H,N,d], or [R,d] for the flat query ids
    ``queries``."""
    q, k, v = _cpu(q), _cpu(k), _cpu(v)
    B, H, N, d = q.shape
    if queries is None:
        R, qsel = B * H * N, None
    else:
        qsel = torch.as_tensor(queries, dtype=torch.int64).contiguous()
        R = qsel.numel()
    out = torch.empty((R, d), dtype=torch.float64)
    _check(_load().orc_dense_rows(_p(q), _p(k), _p(v), _DT[q.dtype], B, H, N, d, R, _p(qsel),
                                  _p(out)), "dense")
    return out.view(B, H, N, d) if queries is None else out


def forward(q, k, v, grid_h: int, grid_w: int, m: int, topk: int, s: int = 1,
            shared_temperature: str = "sqrt_d", landmark_grid=None, branches: str = "both"):
    """All six steps for every query; returns a dict of every intermediate."""
    qt = pool(q, grid_h, grid_w, m, landmark_grid)
    ti, vt, tgap = landmark(qt, k, v, topk)
    r, rgap = route(q, qt, s)
    off, qidx = bucket(r, m)
    out = attend(q, k, v, qt, vt, ti, r, shared_temperature=shared_temperature,
                 branches=branches)
    return dict(q_tilde=qt, topk_idx=ti, v_tilde=vt, topk_gap=tgap, route=r,
                route_gap=rgap, bucket_off=off, bucket_qidx=qidx, out=out)
