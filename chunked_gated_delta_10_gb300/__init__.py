"""GB300 (sm_103a) chunk-parallel Kimi Delta Attention: forward and backward.

Thin Python binding of the C ABI in ``include/kda.h`` (``lib/libkda_gb300.so``,
built by :func:`build`). This module only marshals arguments: it checks
shapes, allocates outputs and the workspace with PyTorch's caching allocator,
passes raw device pointers and the current CUDA stream, and turns status codes
into exceptions. Every step of the computation runs in the library's CUDA
kernels; there is no CPU or PyTorch fallback, and calling without the built
library raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from .build import LIB, build  # noqa: F401

__all__ = ["build", "load", "Dims", "prepare_chunks", "workspace_bytes", "saved_bytes", "chunk_fwd", "chunk_bwd",
           "chunk_fwd_save", "chunk_bwd_from_saved", "KdaError", "STATUS", "DTYPE_BF16", "DTYPE_F32", "PASS_FWD",
           "PASS_BWD"]

DTYPE_BF16, DTYPE_F32 = 0, 1
PASS_FWD, PASS_BWD = 0, 1
CHUNK = 64
STATUS = {0: "KDA_OK", 1: "KDA_ERR_INVALID_ARG", 2: "KDA_ERR_UNSUPPORTED", 3: "KDA_ERR_WORKSPACE", 4: "KDA_ERR_CUDA",
          5: "KDA_ERR_DEVICE_TIMEOUT"}


class KdaError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        msg = f"{where}: {STATUS.get(code, code)} ({load().kda_status_string(code).decode()})"
        if code == 4:
            msg += f" [{load().kda_last_cuda_error().decode()}]"
        super().__init__(msg)


class Dims(ctypes.Structure):
    """Mirror of ``kda_dims``."""
    _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int32), ("H", ctypes.c_int32), ("HV", ctypes.c_int32),
                ("K", ctypes.c_int32), ("V", ctypes.c_int32), ("chunk", ctypes.c_int32), ("num_seqs", ctypes.c_int32),
                ("num_chunks", ctypes.c_int64), ("dtype", ctypes.c_int32), ("scale", ctypes.c_float)]


_lib = None
_lock = threading.Lock()
_P = ctypes.c_void_p


def load():
    """Load the built library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB):
                raise RuntimeError(f"KDA CUDA library not built ({LIB}); call chunked_gated_delta_10_gb300.build()")
            lib = ctypes.CDLL(LIB)
            lib.kda_status_string.restype = ctypes.c_char_p
            lib.kda_status_string.argtypes = [ctypes.c_int]
            lib.kda_prepare_chunks.restype = ctypes.c_int
            lib.kda_prepare_chunks.argtypes = [_P, ctypes.c_int32, ctypes.c_int32, _P, _P, _P]
            lib.kda_workspace_bytes.restype = ctypes.c_size_t
            lib.kda_workspace_bytes.argtypes = [ctypes.POINTER(Dims), ctypes.c_int32]
            lib.kda_chunk_fwd.restype = ctypes.c_int
            lib.kda_chunk_fwd.argtypes = [ctypes.POINTER(Dims)] + [_P] * 13 + [ctypes.c_size_t, _P]
            lib.kda_chunk_bwd.restype = ctypes.c_int
            lib.kda_chunk_bwd.argtypes = [ctypes.POINTER(Dims)] + [_P] * 19 + [ctypes.c_size_t, _P]
            lib.kda_chunk_bwd_fused.restype = ctypes.c_int
            lib.kda_chunk_bwd_fused.argtypes = [ctypes.POINTER(Dims)] + [_P] * 19 + [ctypes.c_size_t, _P]
            lib.kda_saved_bytes.restype = ctypes.c_size_t
            lib.kda_saved_bytes.argtypes = [ctypes.POINTER(Dims)]
            lib.kda_chunk_fwd_save.restype = ctypes.c_int
            lib.kda_chunk_fwd_save.argtypes = [ctypes.POINTER(Dims)] + [_P] * 12 + [ctypes.c_size_t, _P]
            lib.kda_chunk_bwd_from_saved.restype = ctypes.c_int
            lib.kda_chunk_bwd_from_saved.argtypes = ([ctypes.POINTER(Dims)] + [_P] * 12 + [ctypes.c_size_t] +
                                                     [_P] * 6 + [_P])
            lib.kda_device_status.restype = ctypes.c_int
            lib.kda_device_status.argtypes = [_P, _P]
            lib.kda_set_profile_events.restype = ctypes.c_int
            lib.kda_set_profile_events.argtypes = [_P, ctypes.c_int32]
            lib.kda_last_launch_count.restype = ctypes.c_int32
            lib.kda_last_launch_count.argtypes = []
            lib.kda_last_cuda_error.restype = ctypes.c_char_p
            lib.kda_last_cuda_error.argtypes = []
            lib.kda_launch_name.restype = ctypes.c_char_p
            lib.kda_launch_name.argtypes = [ctypes.c_int32]
            _lib = lib
    return _lib


def _check(code, where):
    if code != 0:
        raise KdaError(code, where)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def prepare_chunks(cu_seqlens):
    """Host chunk table of packed sequences: (chunk_idx int32 [NT, 2], chunk_off int64 [N+1], NT), CPU tensors."""
    lib = load()
    cu = torch.as_tensor(cu_seqlens, dtype=torch.int64).cpu().contiguous()
    N = cu.numel() - 1
    nt = ctypes.c_int64(0)
    _check(lib.kda_prepare_chunks(_ptr(cu), N, CHUNK, None, None, ctypes.byref(nt)), "kda_prepare_chunks")
    idx = torch.empty(max(nt.value, 1), 2, dtype=torch.int32)
    off = torch.empty(N + 1, dtype=torch.int64)
    _check(lib.kda_prepare_chunks(_ptr(cu), N, CHUNK, _ptr(idx), _ptr(off), ctypes.byref(nt)), "kda_prepare_chunks")
    return idx[:nt.value], off, nt.value


def make_dims(q: torch.Tensor, v: torch.Tensor, scale: Optional[float], cu_seqlens=None) -> Dims:
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    if q.dtype == torch.bfloat16:
        dt = DTYPE_BF16
    elif q.dtype == torch.float32:
        dt = DTYPE_F32
    else:
        raise TypeError(f"unsupported dtype {q.dtype}")
    if cu_seqlens is None:
        N, NT = B, B * ((T + CHUNK - 1) // CHUNK)
    else:
        cu = torch.as_tensor(cu_seqlens).cpu().tolist()
        N = len(cu) - 1
        NT = sum((cu[i + 1] - cu[i] + CHUNK - 1) // CHUNK for i in range(N))
    return Dims(B, T, H, HV, K, V, CHUNK, N, NT, dt, float(K ** -0.5 if scale is None else scale))


def workspace_bytes(dims: Dims, which: int) -> int:
    return int(load().kda_workspace_bytes(ctypes.byref(dims), which))


class _Varlen:
    """Device copies of cu_seqlens and its chunk table."""

    def __init__(self, cu_seqlens, device):
        if cu_seqlens is None:
            self.cu = self.idx = self.off = None
            return
        idx, off, _ = prepare_chunks(cu_seqlens)
        self.cu = torch.as_tensor(cu_seqlens, dtype=torch.int64).to(device).contiguous()
        self.idx = idx.to(device).contiguous()
        self.off = off.to(device).contiguous()


def _req(t, name, dtype=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _opt(t, name, dtype=None):
    return None if t is None else _req(t, name, dtype)


def _workspace(dims, which, device, ws):
    need = workspace_bytes(dims, which)
    if need == 0:
        raise KdaError(1, "kda_workspace_bytes")
    if ws is None or ws.numel() < need:
        ws = torch.empty(need, dtype=torch.uint8, device=device)
    return ws


def chunk_fwd(q, k, v, g, beta, scale=None, h0=None, cu_seqlens=None, output_states=False, ws=None):
    """Chunked KDA forward. Returns (o, ht, states); states is [num_chunks, HV, K, V] fp32 when
    ``output_states`` (the state entering every chunk, for a backward that skips the recompute), else None."""
    lib = load()
    dt = q.dtype
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (beta, "beta")):
        _req(t, n, dt)
    _req(g, "g", torch.float32)
    _opt(h0, "h0", torch.float32)
    dims = make_dims(q, v, scale, cu_seqlens)
    dev = q.device
    vl = _Varlen(cu_seqlens, dev)
    o = torch.empty_like(v)
    ht = torch.empty(dims.num_seqs, dims.HV, dims.K, dims.V, dtype=torch.float32, device=dev)
    states = (torch.empty(dims.num_chunks, dims.HV, dims.K, dims.V, dtype=torch.float32, device=dev)
              if output_states else None)
    ws = _workspace(dims, PASS_FWD, dev, ws)
    _check(lib.kda_chunk_fwd(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                             _ptr(vl.cu), _ptr(vl.idx), _ptr(vl.off), _ptr(o), _ptr(ht), _ptr(states), _ptr(ws),
                             ws.numel(), _stream()), "kda_chunk_fwd")
    return o, ht, states


def chunk_bwd(q, k, v, g, beta, do, scale=None, h0=None, dht=None, cu_seqlens=None, states=None, ws=None,
              out=None):
    """Chunked KDA backward (recomputes the forward state pass unless ``states`` is given).

    Returns a dict with dq, dk ([B,T,H,K]), dv, dg (fp32), dbeta and dh0
    (fp32, or None without h0). ``out`` may pass preallocated outputs."""
    return _chunk_bwd("kda_chunk_bwd", q, k, v, g, beta, do, scale, h0, dht, cu_seqlens, states, ws, out)


def chunk_bwd_fused(q, k, v, g, beta, do, scale=None, h0=None, dht=None, cu_seqlens=None, states=None, ws=None,
                    out=None):
    """As :func:`chunk_bwd` through ``kda_chunk_bwd_fused`` (the reverse pass and the per-chunk gradients in
    one launch; bf16, K = V = 128, H == HV)."""
    return _chunk_bwd("kda_chunk_bwd_fused", q, k, v, g, beta, do, scale, h0, dht, cu_seqlens, states, ws, out)


def _chunk_bwd(entry, q, k, v, g, beta, do, scale, h0, dht, cu_seqlens, states, ws, out):
    lib = load()
    dt = q.dtype
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (beta, "beta"), (do, "do")):
        _req(t, n, dt)
    _req(g, "g", torch.float32)
    _opt(h0, "h0", torch.float32)
    _opt(dht, "dht", torch.float32)
    _opt(states, "states", torch.float32)
    dims = make_dims(q, v, scale, cu_seqlens)
    dev = q.device
    vl = _Varlen(cu_seqlens, dev)
    if out is None:
        out = dict(dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v),
                   dg=torch.empty_like(g), dbeta=torch.empty_like(beta),
                   dh0=torch.empty_like(h0) if h0 is not None else None)
    ws = _workspace(dims, PASS_BWD, dev, ws)
    _check(getattr(lib, entry)(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                                _ptr(vl.cu), _ptr(vl.idx), _ptr(vl.off), _ptr(do), _ptr(dht), _ptr(states),
                                _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dg"]),
                                _ptr(out["dbeta"]), _ptr(out.get("dh0")), _ptr(ws), ws.numel(), _stream()), entry)
    return out


def saved_bytes(dims: Dims) -> int:
    return int(load().kda_saved_bytes(ctypes.byref(dims)))


def chunk_fwd_save(q, k, v, g, beta, scale=None, h0=None, cu_seqlens=None):
    """Forward that also keeps the saved context for chunk_bwd_from_saved (bf16, K = V = 128).
    Returns (o, ht, saved); saved is a uint8 device tensor of saved_bytes(dims)."""
    lib = load()
    dt = q.dtype
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (beta, "beta")):
        _req(t, n, dt)
    _req(g, "g", torch.float32)
    _opt(h0, "h0", torch.float32)
    dims = make_dims(q, v, scale, cu_seqlens)
    dev = q.device
    vl = _Varlen(cu_seqlens, dev)
    need = saved_bytes(dims)
    if need == 0:
        raise KdaError(2, "kda_saved_bytes")
    saved = torch.empty(need, dtype=torch.uint8, device=dev)
    o = torch.empty_like(v)
    ht = torch.empty(dims.num_seqs, dims.HV, dims.K, dims.V, dtype=torch.float32, device=dev)
    _check(lib.kda_chunk_fwd_save(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                                  _ptr(vl.cu), _ptr(vl.idx), _ptr(vl.off), _ptr(o), _ptr(ht), _ptr(saved),
                                  saved.numel(), _stream()), "kda_chunk_fwd_save")
    return o, ht, saved


def chunk_bwd_from_saved(q, k, v, g, beta, do, saved, scale=None, h0=None, dht=None, cu_seqlens=None, out=None):
    """Backward from chunk_fwd_save's context: only the reverse pass and the per-chunk gradients run.
    Same returns as chunk_bwd, and the same values bit for bit."""
    lib = load()
    dt = q.dtype
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (beta, "beta"), (do, "do")):
        _req(t, n, dt)
    _req(g, "g", torch.float32)
    _opt(h0, "h0", torch.float32)
    _opt(dht, "dht", torch.float32)
    _req(saved, "saved", torch.uint8)
    dims = make_dims(q, v, scale, cu_seqlens)
    vl = _Varlen(cu_seqlens, q.device)
    if out is None:
        out = dict(dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v),
                   dg=torch.empty_like(g), dbeta=torch.empty_like(beta),
                   dh0=torch.empty_like(h0) if h0 is not None else None)
    _check(lib.kda_chunk_bwd_from_saved(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                                        _ptr(vl.cu), _ptr(vl.idx), _ptr(vl.off), _ptr(do), _ptr(dht), _ptr(saved),
                                        saved.numel(), _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]),
                                        _ptr(out["dg"]), _ptr(out["dbeta"]), _ptr(out.get("dh0")), _stream()),
           "kda_chunk_bwd_from_saved")
    return out


def device_status(ws: torch.Tensor) -> int:
    """Status word of the last call that used workspace ``ws`` (syncs the current stream)."""
    return int(load().kda_device_status(_ptr(ws), _stream()))
