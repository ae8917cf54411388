"""Tests of kda_chunk_bwd_noalloc, the backward for callers that cannot
allocate device memory (for example a plugin running inside another engine's
execute phase, where allocation is forbidden or would synchronise the device).
It takes its scratch from a fixed array inside the library instead of a
caller workspace, so its results must match kda_chunk_bwd's, call after call,
even though every call reuses the same scratch.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import kda_inputs
from tests.util import to64

NOALLOC_BYTES = 64 * 1024 * 1024


def _lib():
    import chunked_gated_delta_10_gb300 as kda

    kda.build()
    lib = kda.load()
    P = ctypes.c_void_p
    lib.kda_chunk_bwd_noalloc.restype = ctypes.c_int
    lib.kda_chunk_bwd_noalloc.argtypes = [ctypes.POINTER(kda.Dims)] + [P] * 17 + [P]
    lib.kda_noalloc_prepare.restype = ctypes.c_int
    lib.kda_noalloc_prepare.argtypes = []
    lib.kda_noalloc_device_status.restype = ctypes.c_int
    lib.kda_noalloc_device_status.argtypes = [P]
    return kda, lib


def _noalloc_bwd(kda, lib, inp, x):
    """Call kda_chunk_bwd_noalloc through the C ABI on device tensors ``x``."""
    dims = kda.make_dims(x["q"], x["v"], inp.scale, inp.cu_seqlens)
    out = dict(dq=torch.empty_like(x["q"]), dk=torch.empty_like(x["k"]), dv=torch.empty_like(x["v"]),
               dg=torch.empty_like(x["g"]), dbeta=torch.empty_like(x["beta"]),
               dh0=torch.empty_like(x["h0"]) if x["h0"] is not None else None)
    vl = kda._Varlen(inp.cu_seqlens, x["q"].device)
    p = kda._ptr
    rc = lib.kda_chunk_bwd_noalloc(ctypes.byref(dims), p(x["q"]), p(x["k"]), p(x["v"]), p(x["g"]), p(x["beta"]),
                                   p(x["h0"]), p(vl.cu), p(vl.idx), p(vl.off), p(x["do"]), p(x["dht"]),
                                   p(out["dq"]), p(out["dk"]), p(out["dv"]), p(out["dg"]), p(out["dbeta"]),
                                   p(out["dh0"]), kda._stream())
    assert rc == 0, kda.STATUS.get(rc, rc)
    # the bounded device waits of this call left no time-out in the shared scratch's status word
    assert lib.kda_noalloc_device_status(kda._stream()) == 0
    return out


def _cuda(inp):
    c = lambda t: None if t is None else t.cuda().contiguous()
    return dict(q=c(inp.q), k=c(inp.k), v=c(inp.v), g=c(inp.g), beta=c(inp.beta), h0=c(inp.h0), do=c(inp.do),
                dht=c(inp.dht))


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    """Both entry points launch the same deterministic kernels, so their results must agree bit for bit.
    The larger case runs first, so the second call reads a scratch that still holds the first call's
    contents: a stale-scratch read would show as a mismatch."""
    kda, lib = _lib()
    torch.cuda.init()
    assert lib.kda_noalloc_prepare() == 0  # the set-up phase: module load and address look-up
    cases = [
        kda_inputs.small(seed=41, B=1, T=0, H=2, HV=4, K=128, V=128, dtype="bf16", seq_lens=[150, 3, 64]),
        kda_inputs.small(seed=42, B=2, T=97, H=1, HV=1, K=64, V=64, dtype="f32", dht=False),
    ]
    for inp in cases:  # two calls in a row share (and reuse) the same scratch
        x = _cuda(inp)
        got = _noalloc_bwd(kda, lib, inp, x)
        ref = kda.chunk_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"], scale=inp.scale, h0=x["h0"],
                            dht=x["dht"], cu_seqlens=inp.cu_seqlens)
        torch.cuda.synchronize()
        for key in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
            if ref[key] is None:
                continue
            assert torch.equal(got[key], ref[key]), key
            assert np.isfinite(to64(got[key])).all(), key


def test_noalloc_rejects_problems_larger_than_its_scratch():
    kda, lib = _lib()
    # a workload whose backward needs more scratch than the fixed array: rejected before any CUDA call
    dims = kda.Dims(8, 4096, 32, 32, 128, 128, 64, 8, 8 * 64, kda.DTYPE_BF16, 128 ** -0.5)
    assert kda.workspace_bytes(dims, kda.PASS_BWD) > NOALLOC_BYTES
    A = ctypes.c_void_p(1 << 20)
    args = [A] * 5 + [None] * 4 + [A, None] + [A] * 5 + [None]
    assert lib.kda_chunk_bwd_noalloc(ctypes.byref(dims), *args, None) == 3  # KDA_ERR_WORKSPACE
    bad = kda.Dims(1, 64, 1, 1, 96, 128, 64, 1, 1, kda.DTYPE_BF16, 0.1)
    assert lib.kda_chunk_bwd_noalloc(ctypes.byref(bad), *args, None) == 2   # unsupported K, as kda_chunk_bwd
