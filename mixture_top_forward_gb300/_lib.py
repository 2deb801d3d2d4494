"""ctypes binding of libmita.so: the entry points of include/mita.h under the
same names. Only argument marshalling happens here; every step of the forward
pass runs in the library's CUDA kernels. There is no fallback: if the library
is missing or cannot load, importing the entry points raises."""
from __future__ import annotations

import ctypes
import os
import re
import threading

from . import build_lib

MITA_OK = 0
MITA_ERR_INVALID_ARG = -1
MITA_ERR_UNSUPPORTED = -2
MITA_ERR_ALLOC = -3
MITA_ERR_CUDA = -4
MITA_ERR_TIMEOUT = -5

_lock = threading.Lock()
_lib = None


class MitaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"mita error {code}: {msg}")
        self.code = code


def header_path() -> str:
    return os.path.join(build_lib.INCLUDE, "mita.h")


def declared_functions() -> list[str]:
    """Names of the functions include/mita.h declares."""
    text = open(header_path()).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(mita_\w+)\s*\(", text, flags=re.M)


def load(path: str | None = None, build_if_missing: bool = True) -> ctypes.CDLL:
    """Loads libmita.so (building it in-tree first when it is missing)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or build_lib.LIB
        if not os.path.exists(p):
            if not build_if_missing:
                raise ImportError(f"libmita.so not found at {p}; run __graft_entry__.build()")
            build_lib.build()
        lib = ctypes.CDLL(p)
        vp, ci, i32p, f32p, u16p = (ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_int32),
                                    ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_uint16))
        lib.mita_forward.argtypes = [vp, vp, vp] + [ci] * 8 + [vp, vp, vp, vp]
        lib.mita_forward.restype = ci
        lib.mita_forward_split.argtypes = [vp, vp, vp] + [ci] * 8 + [vp, vp, vp, vp]
        lib.mita_forward_split.restype = ci
        lib.mita_forward_routed.argtypes = [vp, vp, vp] + [ci] * 8 + [vp, vp, vp, vp]
        lib.mita_forward_routed.restype = ci
        lib.mita_forward_aux.argtypes = [vp, vp, vp] + [ci] * 8 + [vp, vp, vp, vp, vp, vp]
        lib.mita_forward_aux.restype = ci
        lib.mita_backward.argtypes = [vp, vp, vp, vp] + [ci] * 8 + [vp] * 6
        lib.mita_backward.restype = ci
        lib.mita_forward_multi.argtypes = [vp, vp, vp] + [ci] * 9 + [vp, vp, vp, vp]
        lib.mita_forward_multi.restype = ci
        lib.mita_forward_noalloc.argtypes = [vp, vp, vp] + [ci] * 8 + [vp, vp, vp, vp]
        lib.mita_forward_noalloc.restype = ci
        lib.mita_forward_host.argtypes = [vp, vp, vp] + [ci] * 8 + [vp, vp, vp, vp]
        lib.mita_forward_host.restype = ci
        lib.mita_workspace_bytes.argtypes = [ci] * 8
        lib.mita_workspace_bytes.restype = ctypes.c_size_t
        lib.mita_plan_info.argtypes = [ci] * 8 + [vp, ci]
        lib.mita_plan_info.restype = ci
        lib.mita_selftest_wait.argtypes = [ctypes.c_int64, vp]
        lib.mita_selftest_wait.restype = ci
        lib.mita_sync_status.argtypes = [vp]
        lib.mita_sync_status.restype = ci
        lib.mita_last_error.argtypes = []
        lib.mita_last_error.restype = ctypes.c_char_p
        lib.mita_profile_enable.argtypes = [ci]
        lib.mita_profile_enable.restype = ci
        lib.mita_profile_read.argtypes = [vp, vp, ci, vp]
        lib.mita_profile_read.restype = ci
        lib.mita_stage_name.argtypes = [ci]
        lib.mita_stage_name.restype = ctypes.c_char_p
        lib.mita_release_workspace.argtypes = []
        lib.mita_release_workspace.restype = None
        if path is None:
            _lib = lib
        return lib


def _raise(rc: int):
    if rc != MITA_OK:
        raise MitaError(rc, (load().mita_last_error() or b"").decode())


def _stream(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _dev_ptr(t, dtype_name, what):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if str(t.dtype) != dtype_name:
        raise ValueError(f"{what} must be {dtype_name}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    return t.data_ptr()


def _shape(Q, m, k, grid_h, grid_w):
    if Q.dim() != 4:
        raise ValueError("Q, K, V are [B, H, N, d]")
    B, H, N, d = Q.shape
    return B, H, N, d


def mita_forward(Q, K, V, grid_h: int, grid_w: int, m: int, k: int, out=None, expert_idx=None, route=None,
                 stream=None, _entry="mita_forward"):
    """MiTA forward on device tensors (torch, bf16 [B,H,N,d]).

    Returns (out bf16 [B,H,N,d], expert_idx int32 [B,H,m,k], route int32
    [B,H,N]); buffers are allocated with torch when not given.
    """
    import torch

    B, H, N, d = _shape(Q, m, k, grid_h, grid_w)
    for t, n in ((K, "K"), (V, "V")):
        if tuple(t.shape) != (B, H, N, d):
            raise ValueError(f"{n} must have the shape of Q")
    out = torch.empty_like(Q) if out is None else out
    expert_idx = torch.empty((B, H, m, k), dtype=torch.int32, device=Q.device) if expert_idx is None else expert_idx
    route = torch.empty((B, H, N), dtype=torch.int32, device=Q.device) if route is None else route
    rc = getattr(load(), _entry)(_dev_ptr(Q, "torch.bfloat16", "Q"), _dev_ptr(K, "torch.bfloat16", "K"),
                                 _dev_ptr(V, "torch.bfloat16", "V"), B, H, N, d, grid_h, grid_w, m, k,
                                 _dev_ptr(out, "torch.bfloat16", "out"),
                                 _dev_ptr(expert_idx, "torch.int32", "expert_idx"),
                                 _dev_ptr(route, "torch.int32", "route"), _stream(stream))
    _raise(rc)
    return out, expert_idx, route


def mita_forward_routed(Q, K, V, grid_h: int, grid_w: int, m: int, k: int, out=None, expert_idx=None, route=None,
                        stream=None):
    """The routing-only ablation (no shared pairs; each query attends to the
    k pairs of its routed expert alone), on device tensors; arguments and
    results as mita_forward."""
    return mita_forward(Q, K, V, grid_h, grid_w, m, k, out, expert_idx, route, stream, _entry="mita_forward_routed")


def mita_forward_split(Q, K, V, grid_h: int, grid_w: int, m: int, k: int, out=None, expert_idx=None, route=None,
                       stream=None):
    """mita_forward with the shared branch folded into the routing kernel
    (online-softmax combine of the two branches); same arguments and
    results as mita_forward."""
    return mita_forward(Q, K, V, grid_h, grid_w, m, k, out, expert_idx, route, stream, _entry="mita_forward_split")


def mita_forward_multi(Q, K, V, grid_h: int, grid_w: int, m: int, k: int, s: int, out=None, expert_idx=None,
                       route=None, stream=None):
    """MiTA with s routed experts per query, on device tensors. Returns (out,
    expert_idx, route int32 [B,H,N,s], each query's landmarks highest first);
    other arguments and results as mita_forward."""
    import torch

    B, H, N, d = _shape(Q, m, k, grid_h, grid_w)
    for t, n in ((K, "K"), (V, "V")):
        if tuple(t.shape) != (B, H, N, d):
            raise ValueError(f"{n} must have the shape of Q")
    out = torch.empty_like(Q) if out is None else out
    expert_idx = torch.empty((B, H, m, k), dtype=torch.int32, device=Q.device) if expert_idx is None else expert_idx
    route = torch.empty((B, H, N, s), dtype=torch.int32, device=Q.device) if route is None else route
    if route.numel() != B * H * N * max(s, 0):
        raise ValueError("route must hold B*H*N*s entries")
    rc = load().mita_forward_multi(_dev_ptr(Q, "torch.bfloat16", "Q"), _dev_ptr(K, "torch.bfloat16", "K"),
                                   _dev_ptr(V, "torch.bfloat16", "V"), B, H, N, d, grid_h, grid_w, m, k, s,
                                   _dev_ptr(out, "torch.bfloat16", "out"),
                                   _dev_ptr(expert_idx, "torch.int32", "expert_idx"),
                                   _dev_ptr(route, "torch.int32", "route"), _stream(stream))
    _raise(rc)
    return out, expert_idx, route


def mita_backward(Q, K, V, dO, grid_h: int, grid_w: int, m: int, k: int, expert_idx, route, dQ=None, dK=None,
                  dV=None, stream=None):
    """Gradients (float32 [B,H,N,d]) of sum(out * dO) for mita_forward's
    output, with its experts and routes held fixed. Q, K, V, dO: bf16 device
    tensors; expert_idx, route: as returned by mita_forward."""
    import torch

    B, H, N, d = _shape(Q, m, k, grid_h, grid_w)
    for t, n in ((K, "K"), (V, "V"), (dO, "dO")):
        if tuple(t.shape) != (B, H, N, d):
            raise ValueError(f"{n} must have the shape of Q")
    dQ = torch.empty((B, H, N, d), dtype=torch.float32, device=Q.device) if dQ is None else dQ
    dK = torch.empty_like(dQ) if dK is None else dK
    dV = torch.empty_like(dQ) if dV is None else dV
    rc = load().mita_backward(_dev_ptr(Q, "torch.bfloat16", "Q"), _dev_ptr(K, "torch.bfloat16", "K"),
                              _dev_ptr(V, "torch.bfloat16", "V"), _dev_ptr(dO, "torch.bfloat16", "dO"), B, H, N, d,
                              grid_h, grid_w, m, k, _dev_ptr(expert_idx, "torch.int32", "expert_idx"),
                              _dev_ptr(route, "torch.int32", "route"), _dev_ptr(dQ, "torch.float32", "dQ"),
                              _dev_ptr(dK, "torch.float32", "dK"), _dev_ptr(dV, "torch.float32", "dV"),
                              _stream(stream))
    _raise(rc)
    return dQ, dK, dV


def mita_forward_noalloc(Q, K, V, grid_h: int, grid_w: int, m: int, k: int, out, expert_idx, route, stream=None):
    """mita_forward through the no-allocation entry point: the library uses
    its static device scratch instead of its workspace, so the caller must
    pass every output buffer (nothing is allocated on this path)."""
    B, H, N, d = _shape(Q, m, k, grid_h, grid_w)
    rc = load().mita_forward_noalloc(_dev_ptr(Q, "torch.bfloat16", "Q"), _dev_ptr(K, "torch.bfloat16", "K"),
                                     _dev_ptr(V, "torch.bfloat16", "V"), B, H, N, d, grid_h, grid_w, m, k,
                                     _dev_ptr(out, "torch.bfloat16", "out"),
                                     _dev_ptr(expert_idx, "torch.int32", "expert_idx"),
                                     _dev_ptr(route, "torch.int32", "route"), _stream(stream))
    _raise(rc)
    return out, expert_idx, route


def mita_forward_aux(Q, K, V, grid_h: int, grid_w: int, m: int, k: int, stream=None):
    """mita_forward that also returns Lq and LV (float32 [B,H,m,d])."""
    import torch

    B, H, N, d = _shape(Q, m, k, grid_h, grid_w)
    out = torch.empty_like(Q)
    expert_idx = torch.empty((B, H, m, k), dtype=torch.int32, device=Q.device)
    route = torch.empty((B, H, N), dtype=torch.int32, device=Q.device)
    lq = torch.empty((B, H, m, d), dtype=torch.float32, device=Q.device)
    lv = torch.empty((B, H, m, d), dtype=torch.float32, device=Q.device)
    rc = load().mita_forward_aux(_dev_ptr(Q, "torch.bfloat16", "Q"), _dev_ptr(K, "torch.bfloat16", "K"),
                                 _dev_ptr(V, "torch.bfloat16", "V"), B, H, N, d, grid_h, grid_w, m, k,
                                 out.data_ptr(), expert_idx.data_ptr(), route.data_ptr(), lq.data_ptr(),
                                 lv.data_ptr(), _stream(stream))
    _raise(rc)
    return out, expert_idx, route, lq, lv


def mita_forward_host(Q, K, V, grid_h: int, grid_w: int, m: int, k: int, out=None, expert_idx=None, route=None,
                      stream=0):
    """MiTA forward on host numpy arrays (uint16 bf16 bit patterns [B,H,N,d]).

    Synchronous. Returns (out uint16, expert_idx int32, route int32) numpy
    arrays; pass preallocated (ideally pinned) ones to avoid allocation.
    """
    import numpy as np

    B, H, N, d = Q.shape
    for a, n in ((Q, "Q"), (K, "K"), (V, "V")):
        if a.dtype != np.uint16 or not a.flags["C_CONTIGUOUS"] or a.shape != (B, H, N, d):
            raise ValueError(f"{n} must be a C-contiguous uint16 array of shape {(B, H, N, d)}")
    out = np.empty_like(Q) if out is None else out
    expert_idx = np.empty((B, H, m, k), np.int32) if expert_idx is None else expert_idx
    route = np.empty((B, H, N), np.int32) if route is None else route
    rc = load().mita_forward_host(Q.ctypes.data, K.ctypes.data, V.ctypes.data, B, H, N, d, grid_h, grid_w, m, k,
                                  out.ctypes.data, expert_idx.ctypes.data, route.ctypes.data,
                                  stream if isinstance(stream, int) else stream.cuda_stream)
    _raise(rc)
    return out, expert_idx, route


def mita_workspace_bytes(B, H, N, d, grid_h, grid_w, m, k) -> int:
    return int(load().mita_workspace_bytes(B, H, N, d, grid_h, grid_w, m, k))


def mita_plan_info(B, H, N, d, grid_h, grid_w, m, k) -> dict | None:
    """The landmark scan's schedule (mita_plan_info in mita.h): the levels as
    (keys, stride, dense) tuples, whether the main scan ranks whole rows, and
    the speculative threshold key's rank (0: none). None for an invalid shape."""
    buf = (ctypes.c_int64 * 32)()
    n = int(load().mita_plan_info(B, H, N, d, grid_h, grid_w, m, k, ctypes.cast(buf, ctypes.c_void_p), 32))
    if n == 0:
        return None
    v = list(buf[:n])
    levels = [(int(v[3 + 3 * l]), int(v[4 + 3 * l]), bool(v[5 + 3 * l])) for l in range(int(v[0]))]
    return {"levels": levels, "dense_main": bool(v[1]), "spec_j": int(v[2])}


def mita_sync_status(stream=None) -> int:
    return int(load().mita_sync_status(_stream(stream)))


def mita_selftest_wait(limit_us: int, stream=None) -> None:
    """Enqueues the bounded-wait self-test kernel (a wait nothing completes,
    given up after limit_us microseconds); mita_sync_status then reports
    MITA_ERR_TIMEOUT once."""
    _raise(load().mita_selftest_wait(int(limit_us), _stream(stream)))


def mita_profile_enable(on: bool = True) -> None:
    _raise(load().mita_profile_enable(1 if on else 0))


def mita_profile_read(stream=None) -> dict:
    """{stage name: (milliseconds, kernel launches)} since the last read."""
    import numpy as np

    ms = np.zeros(16, np.float64)
    nl = np.zeros(16, np.int64)
    rc = load().mita_profile_read(ms.ctypes.data, nl.ctypes.data, 16, _stream(stream))
    if rc < 0:
        _raise(rc)
    lib = load()
    return {lib.mita_stage_name(i).decode(): (float(ms[i]), int(nl[i])) for i in range(rc)}


def mita_stage_name(i: int):
    s = load().mita_stage_name(i)
    return None if s is None else s.decode()


def mita_last_error() -> str:
    return (load().mita_last_error() or b"").decode()


def mita_release_workspace() -> None:
    load().mita_release_workspace()
