"""Stage-by-stage GPU parity of the tensor-core backward (bf16, K = V = 128):
the per-chunk intermediates each stage leaves in the workspace (bf16 tiles in
the library's swizzled operand layout) against the fp64 chunked-form oracle's
intermediates of the same chunk and value head."""
import ctypes

import numpy as np
import pytest
import torch

import kda_inputs
from oracle.chunked import run_chunked
from tests.util import rel_l2

pytestmark = pytest.mark.gpu


def tile_off(r, c, R):
    off = (c // 64) * R * 128 + r * 128 + (c % 64) * 2
    return off ^ (((off >> 7) & 7) << 4)


def untile(raw_u8: np.ndarray, R: int, C: int) -> np.ndarray:
    """bf16 tile bytes -> float64 [R, C]."""
    idx = np.array([[tile_off(r, c, R) // 2 for c in range(C)] for r in range(R)])
    as_u16 = raw_u8.view(np.uint16)
    vals = torch.from_numpy(as_u16[idx].astype(np.int16)).view(torch.bfloat16).double().numpy()
    return vals


@pytest.fixture(scope="module")
def setup():
    import chunked_gated_delta_10_gb300 as kda

    kda.build()
    lib = kda.load()
    P = ctypes.c_void_p
    lib.kda_debug_bwd_stages.restype = ctypes.c_int
    lib.kda_debug_bwd_stages.argtypes = [ctypes.POINTER(kda.Dims)] + [P] * 12 + [ctypes.c_int32, P, ctypes.c_size_t, P]
    lib.kda_debug_ws_region.restype = ctypes.c_int
    lib.kda_debug_ws_region.argtypes = [ctypes.POINTER(kda.Dims), ctypes.c_int32, ctypes.c_char_p,
                                        ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_size_t)]
    inp = kda_inputs.small(seed=51, B=1, T=0, H=2, HV=4, K=128, V=128, dtype="bf16", seq_lens=[150, 40, 64])
    c = lambda t: None if t is None else t.cuda().contiguous()
    x = dict(q=c(inp.q), k=c(inp.k), v=c(inp.v), g=c(inp.g), beta=c(inp.beta), h0=c(inp.h0), do=c(inp.do),
             dht=c(inp.dht))
    dims = kda.make_dims(x["q"], x["v"], inp.scale, inp.cu_seqlens)
    vl = kda._Varlen(inp.cu_seqlens, "cuda")
    wsb = kda.workspace_bytes(dims, kda.PASS_BWD)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    dh0 = torch.zeros_like(x["h0"])
    p = kda._ptr
    rc = lib.kda_debug_bwd_stages(ctypes.byref(dims), p(x["q"]), p(x["k"]), p(x["v"]), p(x["g"]), p(x["beta"]),
                                  p(x["h0"]), p(vl.cu), p(vl.idx), p(vl.off), p(x["do"]), p(x["dht"]), p(dh0), 3,
                                  p(ws), wsb, kda._stream())
    assert rc == 0, kda.STATUS.get(rc)
    torch.cuda.synchronize()
    status = int(ws[:4].view(torch.int32).item())
    assert status == 0, f"device status {status}"
    host = ws.cpu().numpy()

    def region(name):
        off, nb = ctypes.c_size_t(0), ctypes.c_size_t(0)
        assert lib.kda_debug_ws_region(ctypes.byref(dims), kda.PASS_BWD, name.encode(), ctypes.byref(off),
                                       ctypes.byref(nb)) == 0
        return host[off.value:off.value + nb.value]

    ref = run_chunked(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.scale, inp.h0, inp.do, inp.dht, inp.cu_seqlens,
                      keep=True)
    # rows of every global chunk, for the column scaling of INV diag(beta)
    idx, _, _ = kda.prepare_chunks(inp.cu_seqlens)
    cu = inp.cu_seqlens.tolist()
    rows = {gc: (cu[n] + 64 * i, min(cu[n + 1], cu[n] + 64 * (i + 1))) for gc, (n, i) in enumerate(idx.tolist())}
    beta = inp.beta[0].double().numpy()
    return dict(region=region, ref=ref, HV=4, dh0=dh0.cpu().double().numpy(), dims=dims, rows=rows, beta=beta)


# (workspace name, tile rows, tile cols, oracle key, transform of the oracle value)
TILES = [
    ("w", 64, 128, "w", None), ("invb", 64, 64, "INV", "beta_cols"), ("kh", 64, 128, "Kh", None),
    ("aqk", 64, 64, "Aqk", None), ("inv", 64, 64, "INV", None),
    ("sin", 128, 128, "S_in", None), ("vn", 64, 128, "delta", None),
    ("dso", 128, 128, "dS_out", None), ("dvn", 64, 128, "d_delta", None),
]


@pytest.mark.parametrize("name,R,C,key,tf", TILES, ids=[t[0] for t in TILES])
def test_stage_tiles(setup, name, R, C, key, tf):
    reg = setup["region"](name)
    size = R * C * 2
    HV = setup["HV"]
    got_all, ref_all = [], []
    for (gc, hv), ch in sorted(setup["ref"]["chunks"].items()):
        raw = reg[(gc * HV + hv) * size:(gc * HV + hv + 1) * size]
        got = untile(raw, R, C)
        want = ch[key]
        if tf == "beta_cols":  # INV diag(beta): column j scaled by beta of the chunk's row j
            r0, r1 = setup["rows"][gc]
            want = want * setup["beta"][r0:r1, hv][None, :]
        pad = np.zeros((R, C))
        if key == "INV" and tf is None:  # padded rows of a partial chunk: (I + Akk) is the identity there
            pad = np.eye(R)
        pad[:want.shape[0], :want.shape[1]] = want
        got_all.append(got)
        ref_all.append(pad)
    err = rel_l2(np.stack(got_all), np.stack(ref_all))
    print(f"{name}: rel L2 {err:.2e}")
    assert err < 1e-2, err


def test_stage_qs_and_egc(setup):
    ref, HV = setup["ref"], setup["HV"]
    reg_qs = setup["region"]("qs")
    reg_e = setup["region"]("egc").view(np.float32)
    got_q, want_q, got_e, want_e = [], [], [], []
    scale = 128 ** -0.5
    for (gc, hv), ch in sorted(ref["chunks"].items()):
        i = gc * HV + hv
        got_q.append(untile(reg_qs[i * 16384:(i + 1) * 16384], 64, 128)[:ch["Qt"].shape[0]])
        want_q.append(scale * ch["Qt"])
        got_e.append(reg_e[i * 128:(i + 1) * 128])
        want_e.append(np.exp(ch["Gamma"][-1]))
    assert rel_l2(np.concatenate(got_q), np.concatenate(want_q)) < 1e-2
    assert rel_l2(np.concatenate(got_e), np.concatenate(want_e)) < 1e-5


def test_stage_dh0(setup):
    assert rel_l2(setup["dh0"], setup["ref"]["dh0"]) < 1e-2


def test_sweep_order_longest_first(setup):
    """Packed sequences: the workspace's sweep order lists the sequences by decreasing chunk count, ties by
    index (empty and one-token sequences included), after a call that runs the state pass."""
    import chunked_gated_delta_10_gb300 as kda

    lib = kda.load()
    lens = [10, 200, 64, 65, 0, 200, 1, 130]
    inp = kda_inputs.small(seed=52, B=1, T=0, H=1, HV=1, K=128, V=128, dtype="bf16", seq_lens=lens)
    c = lambda t: None if t is None else t.cuda().contiguous()
    x = dict(q=c(inp.q), k=c(inp.k), v=c(inp.v), g=c(inp.g), beta=c(inp.beta), h0=c(inp.h0), do=c(inp.do),
             dht=c(inp.dht))
    dims = kda.make_dims(x["q"], x["v"], inp.scale, inp.cu_seqlens)
    vl = kda._Varlen(inp.cu_seqlens, "cuda")
    wsb = kda.workspace_bytes(dims, kda.PASS_BWD)
    ws = torch.full((wsb,), 255, dtype=torch.uint8, device="cuda")
    p = kda._ptr
    rc = lib.kda_debug_bwd_stages(ctypes.byref(dims), p(x["q"]), p(x["k"]), p(x["v"]), p(x["g"]), p(x["beta"]),
                                  p(x["h0"]), p(vl.cu), p(vl.idx), p(vl.off), p(x["do"]), p(x["dht"]), None, 2,
                                  p(ws), wsb, kda._stream())
    assert rc == 0, kda.STATUS.get(rc)
    torch.cuda.synchronize()
    off, nb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert lib.kda_debug_ws_region(ctypes.byref(dims), kda.PASS_BWD, b"order", ctypes.byref(off),
                                   ctypes.byref(nb)) == 0
    got = ws[off.value:off.value + 4 * len(lens)].cpu().view(torch.int32).tolist()
    chunks = [-(-n // 64) for n in lens]
    assert got == sorted(range(len(lens)), key=lambda i: (-chunks[i], i)), (got, chunks)
