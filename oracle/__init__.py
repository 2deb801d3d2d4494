"""fp64 CPU oracle of the MiTA forward pass -- TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline/reference
legs import this package. The CUDA library never uses it and shares no code
with it. The arithmetic lives in mita_oracle.cpp (plain C++17, OpenMP over
independent items); this file only builds it and marshals numpy arrays.

Pins: tests/test_oracle_pins.py checks every entry point against facts that
do not come from the oracle itself (see the header of mita_oracle.cpp).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mita_oracle.cpp")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile mita_oracle.cpp into _build/liboracle.so (g++, -O2, OpenMP)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-fopenmp", "-shared", "-fPIC", _SRC, "-o", tmp])
    os.replace(tmp, _LIB)
    return _LIB


def _bind(path: str):
    """Load a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    lib.oracle_window.argtypes = [i64, ci, ci, ci, ci, vp]
    lib.oracle_window.restype = i64
    lib.oracle_landmarks.argtypes = [vp, i64, i64, ci, ci, ci, ci, vp]
    lib.oracle_scores.argtypes = [vp, vp, i64, i64, ci, ci, i64, ci, vp]
    lib.oracle_scan.argtypes = [vp, vp, vp, i64, i64, ci, ci, ci, vp, i64, vp, vp, vp]
    lib.oracle_route.argtypes = [vp, vp, i64, i64, ci, ci, vp, i64, vp, vp]
    lib.oracle_attend.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, ci, ci, ci, vp, i64, ci, vp, vp]
    lib.oracle_forward.argtypes = [vp, vp, vp, i64, i64, i64, ci, ci, ci, ci, ci, ci] + [vp] * 8
    lib.oracle_route_multi.argtypes = [vp, vp, i64, i64, ci, ci, ci, vp, i64, vp, vp]
    lib.oracle_attend_multi.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, ci, ci, ci, ci, vp, i64, vp, vp]
    return lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a):
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, "bf16 inputs are passed as uint16 bit patterns"
    return a


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments (rc={rc})")


class Oracle:
    """The oracle's entry points over one loaded library (the default build, or
    a variant compiled by the tests to check that the pins catch mistakes)."""

    def __init__(self, path: str | None = None):
        self.lib = _bind(path or build())

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def window(self, N: int, grid_h: int, grid_w: int, m: int, i: int) -> np.ndarray:
        lib = self.lib
        n = lib.oracle_window(N, grid_h, grid_w, m, i, None)
        if n < 0:
            raise ValueError("invalid window arguments")
        out = np.empty(n, dtype=np.int64)
        lib.oracle_window(N, grid_h, grid_w, m, i, _p(out))
        return out

    def landmarks(self, q, grid_h: int, grid_w: int, m: int) -> np.ndarray:
        """q [..., N, d] bf16 -> Lq [..., m, d] float64."""
        q = _u16(q)
        *lead, N, d = q.shape
        BH = int(np.prod(lead)) if lead else 1
        out = np.empty((BH, m, d), dtype=np.float64)
        _check(self.lib.oracle_landmarks(_p(q), BH, N, d, grid_h, grid_w, m, _p(out)), "landmarks")
        return out.reshape(*lead, m, d)

    def scores(self, lq, k, bh: int, i: int) -> np.ndarray:
        """tau <Lq_i, K_j> for all keys j of flattened head bh."""
        k = _u16(k)
        *lead, N, d = k.shape
        BH = int(np.prod(lead)) if lead else 1
        lq = np.ascontiguousarray(lq, dtype=np.float64).reshape(BH, -1, d)
        out = np.empty(N, dtype=np.float64)
        _check(self.lib.oracle_scores(_p(lq), _p(k), BH, N, d, lq.shape[1], bh, i, _p(out)), "scores")
        return out

    def scan(self, lq, k, v, kk: int, which=None, want_lv=True, want_idx=True, want_gap=True):
        """Landmark scan. Returns (LV, E, gap), each None when not wanted.

        Without `which`: LV [BH,m,d], E [BH,m,kk], gap [BH,m] (flattened heads).
        With `which` (global ids bh*m+i): arrays indexed like `which`.
        """
        k, v = _u16(k), _u16(v)
        *lead, N, d = k.shape
        BH = int(np.prod(lead)) if lead else 1
        lq = np.ascontiguousarray(lq, dtype=np.float64).reshape(BH, -1, d)
        m = lq.shape[1]
        if which is not None:
            which = np.ascontiguousarray(which, dtype=np.int64)
            n = which.shape[0]
            shp = (n,)
        else:
            n = BH * m
            shp = (BH, m)
        lv = np.empty(shp + (d,), np.float64) if want_lv else None
        e = np.empty(shp + (kk,), np.int32) if want_idx else None
        g = np.empty(shp, np.float64) if want_gap else None
        _check(self.lib.oracle_scan(_p(lq), _p(k), _p(v), BH, N, d, m, kk, _p(which), n, _p(lv), _p(e), _p(g)), "scan")
        return lv, e, g

    def route(self, q, lq, which=None):
        """Routes and top-2 margins for the queries in `which` (global ids bh*N+n), or all."""
        q = _u16(q)
        *lead, N, d = q.shape
        BH = int(np.prod(lead)) if lead else 1
        lq = np.ascontiguousarray(lq, dtype=np.float64).reshape(BH, -1, d)
        m = lq.shape[1]
        if which is not None:
            which = np.ascontiguousarray(which, dtype=np.int64)
            n, shp = which.shape[0], (which.shape[0],)
        else:
            n, shp = BH * N, (BH, N)
        r = np.empty(shp, np.int32)
        g = np.empty(shp, np.float64)
        _check(self.lib.oracle_route(_p(q), _p(lq), BH, N, d, m, _p(which), n, _p(r), _p(g)), "route")
        return r, g

    def attend(self, q, lq, lv, k, v, eidx, route_, which=None, shared: bool = True):
        """Query-expert attention conditioned on the given routes and experts.

        Returns (out, wsum) for the queries in `which` (global ids) or all
        queries. shared=False: the routing-only ablation (no shared pairs).
        """
        q, k, v = _u16(q), _u16(k), _u16(v)
        *lead, N, d = q.shape
        BH = int(np.prod(lead)) if lead else 1
        lq = np.ascontiguousarray(lq, dtype=np.float64).reshape(BH, -1, d)
        lv = np.ascontiguousarray(lv, dtype=np.float64).reshape(BH, -1, d)
        m = lq.shape[1]
        eidx = np.ascontiguousarray(eidx, dtype=np.int32).reshape(BH, m, -1)
        kk = eidx.shape[2]
        route_ = np.ascontiguousarray(route_, dtype=np.int32).reshape(BH * N)
        if which is not None:
            which = np.ascontiguousarray(which, dtype=np.int64)
            n, shp = which.shape[0], (which.shape[0],)
        else:
            n, shp = BH * N, (BH, N)
        out = np.empty(shp + (d,), np.float64)
        ws = np.empty(shp, np.float64)
        _check(self.lib.oracle_attend(_p(q), _p(lq), _p(lv), _p(k), _p(v), _p(eidx), _p(route_), BH, N, d, m, kk,
                                     _p(which), n, int(shared), _p(out), _p(ws)), "attend")
        return out, ws

    def forward(self, q, k, v, grid_h: int, grid_w: int, m: int, kk: int, shared: bool = True):
        """Full forward with the oracle's own routes/experts (shared=False: the
        routing-only ablation, no shared pairs).

        q,k,v: [B,H,N,d] bf16 (uint16). Returns a dict of float64/int32 arrays:
        out [B,H,N,d], expert_idx [B,H,m,kk], route [B,H,N], lq, lv [B,H,m,d],
        gap [B,H,m], rgap [B,H,N], wsum [B,H,N].
        """
        q, k, v = _u16(q), _u16(k), _u16(v)
        B, H, N, d = q.shape
        r = dict(out=np.empty((B, H, N, d)), expert_idx=np.empty((B, H, m, kk), np.int32),
                 route=np.empty((B, H, N), np.int32), lq=np.empty((B, H, m, d)), lv=np.empty((B, H, m, d)),
                 gap=np.empty((B, H, m)), rgap=np.empty((B, H, N)), wsum=np.empty((B, H, N)))
        _check(self.lib.oracle_forward(_p(q), _p(k), _p(v), B, H, N, d, grid_h, grid_w, m, kk, int(shared), _p(r["out"]),
                                      _p(r["expert_idx"]), _p(r["route"]), _p(r["lq"]), _p(r["lv"]), _p(r["gap"]),
                                      _p(r["rgap"]), _p(r["wsum"])), "forward")
        return r


    def route_multi(self, q, lq, s: int, which=None):
        """Top-s routes (highest logit first, ties to the lower landmark) and
        the margin between the s-th and (s+1)-th logits, for the queries in
        `which` (global ids) or all: ([..., s] int32, [...] float64)."""
        q = _u16(q)
        *lead, N, d = q.shape
        BH = int(np.prod(lead)) if lead else 1
        lq = np.ascontiguousarray(lq, dtype=np.float64).reshape(BH, -1, d)
        m = lq.shape[1]
        if which is not None:
            which = np.ascontiguousarray(which, dtype=np.int64)
            n, shp = which.shape[0], (which.shape[0],)
        else:
            n, shp = BH * N, (BH, N)
        r = np.empty(shp + (s,), np.int32)
        g = np.empty(shp, np.float64)
        _check(self.lib.oracle_route_multi(_p(q), _p(lq), BH, N, d, m, s, _p(which), n, _p(r), _p(g)), "route_multi")
        return r, g

    def attend_multi(self, q, lq, lv, k, v, eidx, route_, which=None):
        """Attention over the shared pairs and the union of each query's s
        routed experts (route_ [B,H,N,s]); returns (out, wsum) like attend."""
        q, k, v = _u16(q), _u16(k), _u16(v)
        *lead, N, d = q.shape
        BH = int(np.prod(lead)) if lead else 1
        lq = np.ascontiguousarray(lq, dtype=np.float64).reshape(BH, -1, d)
        lv = np.ascontiguousarray(lv, dtype=np.float64).reshape(BH, -1, d)
        m = lq.shape[1]
        eidx = np.ascontiguousarray(eidx, dtype=np.int32).reshape(BH, m, -1)
        kk = eidx.shape[2]
        s = int(np.asarray(route_).shape[-1])
        route_ = np.ascontiguousarray(route_, dtype=np.int32).reshape(BH * N, s)
        if which is not None:
            which = np.ascontiguousarray(which, dtype=np.int64)
            n, shp = which.shape[0], (which.shape[0],)
        else:
            n, shp = BH * N, (BH, N)
        out = np.empty(shp + (d,), np.float64)
        ws = np.empty(shp, np.float64)
        _check(self.lib.oracle_attend_multi(_p(q), _p(lq), _p(lv), _p(k), _p(v), _p(eidx), _p(route_), BH, N, d, m,
                                           kk, s, _p(which), n, _p(out), _p(ws)), "attend_multi")
        return out, ws

    def forward_multi(self, q, k, v, grid_h: int, grid_w: int, m: int, kk: int, s: int):
        """The forward pass with s routed experts per query: landmarks, scan,
        top-s routes, attention over the shared pairs and the union of the s
        experts. Same keys as forward; route is [B,H,N,s]."""
        q, k, v = _u16(q), _u16(k), _u16(v)
        B, H, N, d = q.shape
        lq = self.landmarks(q, grid_h, grid_w, m)
        lv, e, gap = self.scan(lq, k, v, kk)
        r, rg = self.route_multi(q, lq, s)
        out, ws = self.attend_multi(q, lq, lv, k, v, e, r)
        return dict(out=out.reshape(B, H, N, d), expert_idx=e.reshape(B, H, m, kk), route=r.reshape(B, H, N, s),
                    lq=lq.reshape(B, H, m, d), lv=lv.reshape(B, H, m, d), gap=gap.reshape(B, H, m),
                    rgap=rg.reshape(B, H, N), wsum=ws.reshape(B, H, N))


def _default() -> Oracle:
    global _lib
    with _lock:
        if _lib is None:
            _lib = Oracle()
    return _lib


def num_threads():
    return _default().num_threads()


def window(*a, **kw):
    return _default().window(*a, **kw)


def landmarks(*a, **kw):
    return _default().landmarks(*a, **kw)


def scores(*a, **kw):
    return _default().scores(*a, **kw)


def scan(*a, **kw):
    return _default().scan(*a, **kw)


def route(*a, **kw):
    return _default().route(*a, **kw)


def attend(*a, **kw):
    return _default().attend(*a, **kw)


def forward(*a, **kw):
    return _default().forward(*a, **kw)


def route_multi(*a, **kw):
    return _default().route_multi(*a, **kw)


def attend_multi(*a, **kw):
    return _default().attend_multi(*a, **kw)


def forward_multi(*a, **kw):
    return _default().forward_multi(*a, **kw)
