"""Host-side tests of the C ABI (no GPU): the library builds and loads, exports
every entry point that include/kda.h declares, builds chunk tables, sizes
workspaces, and rejects invalid arguments before any CUDA call."""
import ctypes
import os
import re

import pytest

import chunked_gated_delta_10_gb300 as kda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
A = 1 << 20  # a 16-byte aligned fake device address (never dereferenced: validation fails first)


@pytest.fixture(scope="module")
def lib():
    kda.build()
    return kda.load()


def test_exports_every_declared_symbol(lib):
    names = set()
    for hdr in os.listdir(os.path.join(ROOT, "include")):
        if hdr.endswith(".h"):
            src = open(os.path.join(ROOT, "include", hdr)).read()
            names |= set(re.findall(r"^\s*(?:const\s+)?[\w\*\s]+?\b(kda_\w+)\s*\(", src, re.M))
    assert {"kda_chunk_fwd", "kda_chunk_bwd", "kda_workspace_bytes", "kda_prepare_chunks"} <= names
    for n in sorted(names):
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code, name in kda.STATUS.items():
        assert lib.kda_status_string(code).decode().startswith(name)


def test_prepare_chunks_table():
    cu = [0, 1, 64, 65, 65, 200]
    idx, off, nt = kda.prepare_chunks(cu)
    lens = [1, 63, 1, 0, 135]
    per = [(L + 63) // 64 for L in lens]
    assert nt == sum(per) == 6
    assert off.tolist() == [0, 1, 2, 3, 3, 6]
    assert idx.tolist() == [[0, 0], [1, 0], [2, 0], [4, 0], [4, 1], [4, 2]]


@pytest.mark.parametrize("cu", [[1, 5], [0, 5, 3], [0]])
def test_prepare_chunks_rejects_bad_cu(lib, cu):
    arr = (ctypes.c_int64 * len(cu))(*cu)
    nt = ctypes.c_int64(0)
    assert lib.kda_prepare_chunks(arr, len(cu) - 1, 64, None, None, ctypes.byref(nt)) == 1


def _dims(**kw):
    d = dict(B=2, T=130, H=2, HV=4, K=64, V=128, chunk=64, num_seqs=2, num_chunks=6, dtype=0, scale=0.125)
    d.update(kw)
    return kda.Dims(**d)


def test_workspace_bytes(lib):
    d = _dims()
    fwd, bwd = kda.workspace_bytes(d, kda.PASS_FWD), kda.workspace_bytes(d, kda.PASS_BWD)
    assert 0 < fwd < bwd
    assert kda.workspace_bytes(_dims(T=300, num_chunks=10), kda.PASS_BWD) > bwd
    assert kda.workspace_bytes(_dims(K=96), kda.PASS_BWD) == 0
    assert kda.workspace_bytes(_dims(HV=3), kda.PASS_BWD) == 0
    assert kda.workspace_bytes(d, 7) == 0


def _bwd(lib, d, ws_bytes=None, entry="kda_chunk_bwd", **ptr):
    p = dict(q=A, k=A, v=A, g=A, beta=A, h0=None, cu=None, idx=None, off=None, do=A, dht=None, states=None,
             dq=A, dk=A, dv=A, dg=A, db=A, dh0=None, ws=A)
    p.update(ptr)
    if ws_bytes is None:
        ws_bytes = kda.workspace_bytes(d, kda.PASS_BWD)
    args = [p[n] for n in ("q", "k", "v", "g", "beta", "h0", "cu", "idx", "off", "do", "dht", "states", "dq", "dk",
                           "dv", "dg", "db", "dh0", "ws")]
    return getattr(lib, entry)(ctypes.byref(d), *[None if a is None else ctypes.c_void_p(a) for a in args],
                               ws_bytes, None)


def test_bwd_rejects_invalid_arguments_before_launch(lib):
    d = _dims()
    assert lib.kda_chunk_bwd(None, *([None] * 19), 0, None) == 1
    assert _bwd(lib, _dims(K=96)) == 2                     # unsupported head dim
    assert _bwd(lib, _dims(chunk=32)) == 2                 # unsupported chunk
    assert _bwd(lib, _dims(HV=3)) == 1                     # HV % H
    assert _bwd(lib, _dims(num_chunks=5)) == 1             # inconsistent chunk count
    assert _bwd(lib, d, q=A + 8) == 1                      # misaligned
    assert _bwd(lib, d, q=None) == 1                       # missing input
    assert _bwd(lib, d, ws_bytes=16) == 3                  # workspace too small
    assert _bwd(lib, d, ws=None) == 3                      # no workspace
    assert _bwd(lib, d, dh0=A) == 1                        # dh0 without h0
    assert _bwd(lib, d, cu=A) == 1                         # cu_seqlens without chunk table
    assert _bwd(lib, d, cu=A, idx=A, off=A) == 1           # packed sequences need B == 1


def test_fused_reverse_rejects_before_launch(lib):
    """kda_chunk_bwd_fused checks its arguments as kda_chunk_bwd does, and refuses, before any CUDA call,
    the cases it does not cover: the fp32 path (K = 64, or fp32 inputs) and grouped value heads."""
    fused = dict(entry="kda_chunk_bwd_fused")
    assert lib.kda_chunk_bwd_fused(None, *([None] * 19), 0, None) == 1
    assert _bwd(lib, _dims(HV=2), **fused) == 2                         # bf16 with K = 64: the fp32 path
    assert _bwd(lib, _dims(dtype=1, K=128, V=128, HV=2), **fused) == 2  # fp32 inputs
    assert _bwd(lib, _dims(K=128, V=128, HV=4), **fused) == 2           # grouped value heads (H = 2)
    d = _dims(K=128, V=128, HV=2)
    assert _bwd(lib, d, q=A + 8, **fused) == 1                          # misaligned
    assert _bwd(lib, d, ws_bytes=16, **fused) == 3                      # workspace too small
    assert _bwd(lib, d, dh0=A, **fused) == 1                            # dh0 without h0


def test_binding_requires_built_library(monkeypatch, tmp_path):
    import chunked_gated_delta_10_gb300 as m
    monkeypatch.setattr(m, "LIB", str(tmp_path / "missing.so"))
    monkeypatch.setattr(m, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        m.load()


def test_saved_context_size_and_argument_checks(lib):
    """kda_saved_bytes is the backward workspace size on the tensor-core path and 0 off it; the saved-context
    entry points reject a small buffer and unsupported dims before any CUDA call."""
    tc = kda.Dims(2, 130, 2, 4, 128, 128, 64, 2, 6, kda.DTYPE_BF16, 0.1)
    need = kda.saved_bytes(tc)
    assert need == kda.workspace_bytes(tc, kda.PASS_BWD) > 0
    for dims in (_dims(), _dims(dtype=1, K=128, V=128)):  # K = 64 bf16, fp32
        assert kda.saved_bytes(dims) == 0
    P = ctypes.c_void_p
    a = P(A)
    fwd_args = [a] * 5 + [None] * 4 + [a, None]
    assert lib.kda_chunk_fwd_save(ctypes.byref(tc), *fwd_args, a, need - 1, None) == 3  # KDA_ERR_WORKSPACE
    bwd_args = [a] * 5 + [None] * 4 + [a, None]
    outs = [a] * 5 + [None]
    assert lib.kda_chunk_bwd_from_saved(ctypes.byref(tc), *bwd_args, a, need - 1, *outs, None) == 3
    f32 = _dims(dtype=1, K=128, V=128)
    assert lib.kda_chunk_fwd_save(ctypes.byref(f32), *fwd_args, a, 1 << 40, None) == 2  # KDA_ERR_UNSUPPORTED
    assert lib.kda_chunk_bwd_from_saved(ctypes.byref(f32), *bwd_args, a, 1 << 40, *outs, None) == 2
