"""KDA oracle: fp64 CPU reference for the chunked-backward CUDA library.

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product path
never does. It shares no code with the CUDA library.

Two independent forms of the same computation live here:

* ``kda_oracle.c`` (wrapped by :func:`run`): token-by-token recurrence in fp64
  with a hand-derived reverse-mode backward, threaded over (sequence, key-head
  group) units. This is the definition every parity test compares against.
* ``chunked.py`` (:func:`oracle.chunked.run_chunked`): the chunk-parallel form
  (WY representation within a chunk, state passing between chunks) in fp64
  numpy, following the chunked formulas of the FlashKDA backward page and the
  FLA ``chunk_bwd.py`` page. It exposes every per-chunk intermediate, and is
  pinned against the recurrence.

Parity pins of this package live in ``tests/test_oracle_*.py`` (finite
differences, torch fp64 autograd of an independent forward, closed forms,
invariances, chunk-form equality).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libkda_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the C oracle (gcc -O2, no fast-math) next to its source."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-D_GNU_SOURCE", "-o", tmp,
                               _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            lib.kda_oracle_run.restype = ctypes.c_int
            lib.kda_oracle_run.argtypes = [ctypes.c_int, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_double] + [P] * 18 + [ctypes.c_int]
            lib.kda_oracle_num_chunks.restype = ctypes.c_int64
            lib.kda_oracle_num_chunks.argtypes = [P, ctypes.c_int, ctypes.c_int]
            _lib = lib
    return _lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu")
        import torch

        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def run(q, k, v, g, beta, scale, h0=None, do=None, dht=None, cu_seqlens=None, *, chunk=64,
        backward=True, chunk_states=False, nthreads=0):
    """Run the fp64 recurrence (and its backward) on full tensors.

    Shapes follow the library: q, k ``[B, T, H, K]``; v, do ``[B, T, HV, V]``;
    g ``[B, T, HV, K]`` (natural-log per-token decay, not cumsummed); beta
    ``[B, T, HV]``; h0, dht ``[N, HV, K, V]``; ``cu_seqlens`` int64 ``[N+1]``
    (then B must be 1) or None. Inputs may be torch tensors or numpy arrays of
    any float dtype; they are widened exactly to float64.

    Returns a dict of float64 numpy arrays: o, ht and, with ``backward``, dq,
    dk (``[B, T, H, K]``, summed over each key head's value heads), dv, dg,
    dbeta, dh0; with ``chunk_states``, s_in / ds_out ``[num_chunks, HV, K, V]``
    (state entering each chunk, gradient of the state leaving it).
    """
    lib = _load()
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    h0, do, dht = _f64(h0), _f64(do), _f64(dht)
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    if cu_seqlens is None:
        cu = np.arange(B + 1, dtype=np.int64) * T
    else:
        if B != 1:
            raise ValueError("cu_seqlens requires B == 1")
        cu = np.ascontiguousarray(np.asarray(cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist")
                                             else cu_seqlens, dtype=np.int64))
    N = cu.size - 1
    nck = int(lib.kda_oracle_num_chunks(cu.ctypes.data_as(ctypes.c_void_p), N, chunk))
    out = {"o": np.zeros((B, T, HV, V)), "ht": np.zeros((N, HV, K, V))}
    if backward:
        out.update(dq=np.zeros((B, T, H, K)), dk=np.zeros((B, T, H, K)), dv=np.zeros((B, T, HV, V)),
                   dg=np.zeros((B, T, HV, K)), dbeta=np.zeros((B, T, HV)), dh0=np.zeros((N, HV, K, V)))
    if chunk_states:
        out.update(s_in=np.zeros((nck, HV, K, V)), ds_out=np.zeros((nck, HV, K, V)))
    rc = lib.kda_oracle_run(
        N, cu.ctypes.data_as(ctypes.c_void_p), H, HV, K, V, chunk, float(scale),
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(do), _ptr(dht),
        _ptr(out["o"]), _ptr(out["ht"]), _ptr(out.get("dq")), _ptr(out.get("dk")), _ptr(out.get("dv")),
        _ptr(out.get("dg")), _ptr(out.get("dbeta")), _ptr(out.get("dh0")),
        _ptr(out.get("s_in")), _ptr(out.get("ds_out")), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_run failed with code {rc}")
    return out


def run_inputs(inp, **kw):
    """:func:`run` on a :class:`kda_inputs.Inputs` bundle."""
    return run(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.scale, inp.h0, inp.do, inp.dht,
               inp.cu_seqlens, **kw)


def run_unit(inp, n, h, **kw):
    """Oracle outputs of one independent unit: sequence ``n``, key head ``h``
    and its value heads. Returns the same dict as :func:`run`, restricted to
    that unit (rows of sequence n; head axes of length 1 for keys, G for
    values; state axes of length 1 for the sequence)."""
    bos, eos = inp.seq_bounds[n]
    H, HV = inp.q.shape[2], inp.v.shape[2]
    G = HV // H

    def rows(x, heads):
        flat = x.reshape(-1, *x.shape[2:])
        return flat[bos:eos, heads].unsqueeze(0)

    hs = slice(h, h + 1)
    vs = slice(h * G, h * G + G)
    st = (lambda x: None if x is None else x[n:n + 1, vs])
    return run(rows(inp.q, hs), rows(inp.k, hs), rows(inp.v, vs), rows(inp.g, vs), rows(inp.beta, vs),
               inp.scale, st(inp.h0), rows(inp.do, vs), st(inp.dht), None, **kw)
