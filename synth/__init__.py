"""Seeded synthetic inputs for the MiTA forward pass.

This module only draws random numbers and rounds them to bf16: it contains
none of the attention arithmetic, so both the CUDA path's tests/benchmark and
the oracle's checks can take their inputs from here.

Workload recipes (the pages give shapes and value structure only; the
datasets themselves are not used):

* ``tiny``      B=1,H=1,N=196 on a 14x14 grid, m=k=25; Q,K,V i.i.d. N(0,1).
* ``deit``      B=64,H=6,N=196 (14x14), m=k=25; K and Q from 16 Gaussian
                clusters per head (centres N(0,I), noise sigma 0.3, independent
                cluster draws for K and for Q); V i.i.d. N(0,1).
* ``seg1024``   B=16,H=6,N=1024 (32x32), m=k=49; same clustering as ``deit``.
* ``seg1600``   B=16,H=6,N=1600 (40x40), m=k=49; same clustering.
* ``lra``       B=32,H=8,N=4096, 1-D windows of 64, m=k=64; K and Q from 64
                clusters per head whose membership runs along the sequence in
                runs of length U{16..256}, cluster per run U{0..63}
                (independent run sequences for K and Q), noise sigma 0.3;
                V i.i.d. N(0,1).
* ``long64k``/``long256k``/``long1m``  B=1,H=8,N=2^16/2^18/2^20, 1-D windows
                of N/256, m=k=256; Q,K,V i.i.d. N(0,1); per head floor(N/100)
                key rows, uniform without replacement, scaled x4 before
                rounding (salient outliers).

Every config uses seed 0 by default. Stream tags: Q=0, K=1, V=2, cluster
centres=3, K cluster draws=4, Q cluster draws=5, outlier rows=6, K runs=7,
Q runs=8. The generator itself is defined in ``gen.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB = os.path.join(_HERE, "_build", "libsynth.so")
_lock = threading.Lock()
_lib = None

TAG_Q, TAG_K, TAG_V, TAG_CENTRE, TAG_KASSIGN, TAG_QASSIGN, TAG_OUTLIER, TAG_KRUN, TAG_QRUN = range(9)

CONFIGS = {
    "tiny": dict(B=1, H=1, N=196, d=64, grid_h=14, grid_w=14, m=25, k=25, recipe="iid"),
    "deit": dict(B=64, H=6, N=196, d=64, grid_h=14, grid_w=14, m=25, k=25, recipe="clusters", clusters=16),
    "seg1024": dict(B=16, H=6, N=1024, d=64, grid_h=32, grid_w=32, m=49, k=49, recipe="clusters", clusters=16),
    "seg1600": dict(B=16, H=6, N=1600, d=64, grid_h=40, grid_w=40, m=49, k=49, recipe="clusters", clusters=16),
    "lra": dict(B=32, H=8, N=4096, d=64, grid_h=0, grid_w=0, m=64, k=64, recipe="runs", clusters=64),
    "long64k": dict(B=1, H=8, N=65536, d=64, grid_h=0, grid_w=0, m=256, k=256, recipe="outliers"),
    "long256k": dict(B=1, H=8, N=262144, d=64, grid_h=0, grid_w=0, m=256, k=256, recipe="outliers"),
    "long1m": dict(B=1, H=8, N=1048576, d=64, grid_h=0, grid_w=0, m=256, k=256, recipe="outliers"),
}


def build(force: bool = False) -> str:
    """Compile gen.c into _build/libsynth.so (gcc, OpenMP)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            u64, i64, vp, f32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_float
            lib.synth_words.argtypes = [vp, i64, u64, u64, u64]
            lib.synth_normals.argtypes = [vp, i64, u64, u64, u64]
            lib.synth_rows_bf16.argtypes = [vp, i64, ctypes.c_int, u64, u64, vp, vp, f32, vp]
            lib.synth_stream_key.argtypes = [u64, u64]
            lib.synth_stream_key.restype = u64
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def words(n: int, seed: int, tag: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _load().synth_words(_ptr(out), n, seed, tag, offset)
    return out


def normals(n: int, seed: int, tag: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _load().synth_normals(_ptr(out), n, seed, tag, offset)
    return out


def uniform_int(w: np.ndarray, n) -> np.ndarray:
    """Map 64-bit words to integers in [0, n): ((w >> 32) * n) >> 32."""
    n = np.asarray(n, dtype=np.uint64)
    return (((w >> np.uint64(32)) * n) >> np.uint64(32)).astype(np.int64)


def rows_bf16(rows: int, d: int, seed: int, tag: int, centre=None, assign=None, sigma: float = 1.0,
              row_scale=None) -> np.ndarray:
    """rows x d bf16 bit patterns (uint16), see gen.c for the formula."""
    out = np.empty((rows, d), dtype=np.uint16)
    if centre is not None:
        centre = np.ascontiguousarray(centre, dtype=np.float32)
        assign = np.ascontiguousarray(assign, dtype=np.int32)
        assert assign.shape == (rows,)
    if row_scale is not None:
        row_scale = np.ascontiguousarray(row_scale, dtype=np.float32)
        assert row_scale.shape == (rows,)
    _load().synth_rows_bf16(_ptr(out), rows, d, seed, tag, _ptr(centre), _ptr(assign), sigma, _ptr(row_scale))
    return out


def normal_bf16(shape, seed: int, tag: int, scale: float = 1.0) -> np.ndarray:
    """i.i.d. N(0, scale^2) rounded to bf16, any shape whose last dim is d."""
    shape = tuple(shape)
    rows = int(np.prod(shape[:-1]))
    rs = None if scale == 1.0 else np.full(rows, scale, dtype=np.float32)
    return rows_bf16(rows, shape[-1], seed, tag, row_scale=rs).reshape(shape)


def bf16_to_f64(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def f64_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round float values to bf16 bit patterns (RNE via float32)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    return (u >> np.uint64(16)).astype(np.uint16)


def _cluster_assign_iid(BH, N, C, seed, tag):
    w = words(BH * N, seed, tag)
    c = uniform_int(w, C).reshape(BH, N)
    return (c + (np.arange(BH, dtype=np.int64) * C)[:, None]).reshape(-1)


def _cluster_assign_runs(BH, N, C, seed, tag):
    max_runs = N // 16 + 2
    out = np.empty((BH, N), dtype=np.int64)
    for bh in range(BH):
        w = words(2 * max_runs, seed, tag, offset=bh * 2 * max_runs)
        lengths = 16 + uniform_int(w[0::2], 241)
        clus = uniform_int(w[1::2], C)
        out[bh] = np.repeat(clus, lengths)[:N] + bh * C
    return out.reshape(-1)


def _outlier_scale(BH, N, seed):
    r = N // 100
    scale = np.ones((BH, N), dtype=np.float32)
    for bh in range(BH):
        w = words(r, seed, TAG_OUTLIER, offset=bh * r) if r else np.empty(0, np.uint64)
        perm = np.arange(N, dtype=np.int64)
        for t in range(r):
            j = t + int(uniform_int(w[t:t + 1], N - t)[0])
            perm[t], perm[j] = perm[j], perm[t]
        scale[bh, perm[:r]] = 4.0
    return scale.reshape(-1)


def make_inputs(cfg, seed: int = 0):
    """Q, K, V of a named config (or a config dict) as uint16 bf16 arrays [B,H,N,d]."""
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    B, H, N, d = cfg["B"], cfg["H"], cfg["N"], cfg["d"]
    BH, rows = B * H, B * H * N
    recipe = cfg.get("recipe", "iid")
    shape = (B, H, N, d)
    if recipe in ("iid", "outliers"):
        q = rows_bf16(rows, d, seed, TAG_Q)
        ks = _outlier_scale(BH, N, seed) if recipe == "outliers" else None
        k = rows_bf16(rows, d, seed, TAG_K, row_scale=ks)
    elif recipe in ("clusters", "runs"):
        C = cfg["clusters"]
        centre = normals(BH * C * d, seed, TAG_CENTRE).astype(np.float32).reshape(BH * C, d)
        if recipe == "clusters":
            ka = _cluster_assign_iid(BH, N, C, seed, TAG_KASSIGN)
            qa = _cluster_assign_iid(BH, N, C, seed, TAG_QASSIGN)
        else:
            ka = _cluster_assign_runs(BH, N, C, seed, TAG_KRUN)
            qa = _cluster_assign_runs(BH, N, C, seed, TAG_QRUN)
        sigma = float(cfg.get("sigma", 0.3))
        q = rows_bf16(rows, d, seed, TAG_Q, centre=centre, assign=qa, sigma=sigma)
        k = rows_bf16(rows, d, seed, TAG_K, centre=centre, assign=ka, sigma=sigma)
    else:
        raise ValueError(f"unknown recipe {recipe!r}")
    v = rows_bf16(rows, d, seed, TAG_V)
    return q.reshape(shape), k.reshape(shape), v.reshape(shape)
