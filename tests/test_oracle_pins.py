"""Pins of the fp64 oracle against things other than itself.

* central finite differences of the loss L = sum(o*do) + sum(ht*dht) for every
  input (q, k, v, g, beta, h0) and every output gradient;
* torch float64 autograd through an independent, literal implementation of the
  stated recurrence S_t = (I - beta k k^T) Diag(exp g_t) S_{t-1} + beta k v^T;
* equality of the chunk-parallel form (oracle/chunked.py) with the recurrence
  for several chunk sizes, partial last chunks, packed sequences and grouped
  value heads.
"""
import numpy as np
import pytest
import torch

import kda_inputs
import oracle
from oracle.chunked import run_chunked

GRAD_KEYS = ["dq", "dk", "dv", "dg", "dbeta", "dh0"]


def _f64_inputs(inp):
    f = lambda x: None if x is None else x.to(torch.float64).numpy().copy()
    return dict(q=f(inp.q), k=f(inp.k), v=f(inp.v), g=f(inp.g), beta=f(inp.beta), h0=f(inp.h0),
                do=f(inp.do), dht=f(inp.dht), cu=None if inp.cu_seqlens is None else inp.cu_seqlens.numpy(),
                scale=inp.scale)


def _loss(x, chunk):
    r = oracle.run(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"], None, None, x["cu"],
                   chunk=chunk, backward=False)
    L = np.sum(r["o"] * x["do"])
    if x["dht"] is not None:
        L += np.sum(r["ht"] * x["dht"])
    return L


@pytest.mark.parametrize("case", [
    dict(B=1, T=13, H=1, HV=2, K=3, V=2, seq_lens=None, chunk=4),
    dict(B=2, T=7, H=2, HV=2, K=2, V=3, seq_lens=None, chunk=3),
    dict(B=1, T=11, H=1, HV=1, K=3, V=3, seq_lens=[4, 7], chunk=4),
])
def test_finite_differences(case):
    case = dict(case)
    chunk = case.pop("chunk")
    inp = kda_inputs.small(seed=11, dtype="f32", g_mu=0.5, **case)
    x = _f64_inputs(inp)
    # make beta and g generic (not bf16-rounded, larger decay) so every term matters
    rng = np.random.default_rng(5)
    x["beta"] = rng.uniform(0.2, 0.9, size=x["beta"].shape)
    x["g"] = -rng.uniform(0.05, 0.6, size=x["g"].shape)
    r = oracle.run(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"], x["do"], x["dht"],
                   x["cu"], chunk=chunk)
    eps = 1e-6
    pairs = [("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("beta", "dbeta"), ("h0", "dh0")]
    for name, gname in pairs:
        arr = x[name]
        fd = np.zeros_like(arr)
        flat = arr.reshape(-1)
        for i in range(flat.size):
            old = flat[i]
            flat[i] = old + eps
            lp = _loss(x, chunk)
            flat[i] = old - eps
            lm = _loss(x, chunk)
            flat[i] = old
            fd.reshape(-1)[i] = (lp - lm) / (2 * eps)
        err = np.linalg.norm(fd - r[gname]) / np.linalg.norm(fd)
        assert err < 1e-7, (gname, err)


def _torch_literal(x, G):
    """Literal recurrence in torch fp64 (independent of the oracle's code)."""
    q, k, v, g, beta = (torch.tensor(x[n], requires_grad=True) for n in ("q", "k", "v", "g", "beta"))
    h0 = torch.tensor(x["h0"], requires_grad=True) if x["h0"] is not None else None
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    cu = x["cu"] if x["cu"] is not None else [b * T for b in range(B + 1)]
    qf, kf, vf, gf, bf = q.reshape(-1, H, K), k.reshape(-1, H, K), v.reshape(-1, HV, V), g.reshape(-1, HV, K), \
        beta.reshape(-1, HV)
    hmap = torch.arange(HV) // G
    eye = torch.eye(K, dtype=torch.float64)
    outs, finals = [None] * qf.shape[0], []
    for n in range(len(cu) - 1):
        S = h0[n] if h0 is not None else torch.zeros(HV, K, V, dtype=torch.float64)
        for t in range(int(cu[n]), int(cu[n + 1])):
            kt = kf[t, hmap]  # [HV, K]
            A = eye - bf[t][:, None, None] * kt[:, :, None] * kt[:, None, :]
            S = A @ (torch.exp(gf[t])[:, :, None] * S) + bf[t][:, None, None] * kt[:, :, None] * vf[t][:, None, :]
            outs[t] = x["scale"] * torch.einsum("hkv,hk->hv", S, qf[t, hmap])
        finals.append(S)
    o = torch.stack(outs).reshape(B, T, HV, V)
    ht = torch.stack(finals)
    L = (o * torch.tensor(x["do"])).sum()
    if x["dht"] is not None:
        L = L + (ht * torch.tensor(x["dht"])).sum()
    L.backward()
    res = dict(o=o.detach().numpy(), ht=ht.detach().numpy(), dq=q.grad.numpy(), dk=k.grad.numpy(),
               dv=v.grad.numpy(), dg=g.grad.numpy(), dbeta=beta.grad.numpy())
    if h0 is not None:
        res["dh0"] = h0.grad.numpy()
    return res


@pytest.mark.parametrize("case", [
    dict(B=1, T=40, H=2, HV=4, K=6, V=5, seq_lens=None),
    dict(B=1, T=0, H=1, HV=2, K=4, V=4, seq_lens=[9, 1, 17]),
    dict(B=2, T=19, H=1, HV=1, K=5, V=3, seq_lens=None),
])
def test_torch_autograd_literal_recurrence(case):
    inp = kda_inputs.small(seed=3, dtype="f32", **case)
    x = _f64_inputs(inp)
    G = x["v"].shape[2] // x["q"].shape[2]
    ref = _torch_literal(x, G)
    r = oracle.run(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"], x["do"], x["dht"], x["cu"],
                   chunk=8)
    for key, val in ref.items():
        err = np.linalg.norm(r[key] - val) / max(np.linalg.norm(val), 1e-300)
        assert err < 1e-12, (key, err)


@pytest.mark.parametrize("chunk", [16, 32, 64])
@pytest.mark.parametrize("case", [
    dict(B=2, T=150, H=2, HV=4, K=8, V=8, seq_lens=None, h0=True, dht=True),
    dict(B=1, T=0, H=2, HV=2, K=8, V=16, seq_lens=[1, 64, 65, 30], h0=True, dht=False),
    dict(B=1, T=200, H=1, HV=1, K=16, V=8, seq_lens=None, h0=False, dht=False),
])
def test_chunked_equals_recurrent(case, chunk):
    inp = kda_inputs.small(seed=7, dtype="f32", **case)
    a = oracle.run_inputs(inp, chunk=chunk, chunk_states=True)
    b = run_chunked(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.scale, inp.h0, inp.do, inp.dht, inp.cu_seqlens,
                    chunk=chunk)
    for key in ["o", "ht", "s_in", "ds_out"] + GRAD_KEYS:
        ref = a[key]
        err = np.abs(b[key] - ref).max() / max(np.abs(ref).max(), 1e-300)
        assert err < 1e-12, (key, err)


def test_chunk_size_invariance_of_chunked_form():
    inp = kda_inputs.small(seed=2, T=96, H=1, HV=2, K=8, V=8, dtype="f32")
    outs = [run_chunked(inp.q, inp.k, inp.v, inp.g, inp.beta, inp.scale, inp.h0, inp.do, inp.dht, chunk=c)
            for c in (16, 32, 64)]
    for key in ["o", "ht"] + GRAD_KEYS:
        for other in outs[1:]:
            assert np.allclose(outs[0][key], other[key], rtol=0, atol=1e-12 * max(1.0, np.abs(outs[0][key]).max()))


def test_oracle_thread_count_is_bitwise_irrelevant():
    inp = kda_inputs.small(seed=4, B=3, T=70, H=2, HV=4, K=8, V=8, dtype="f32")
    a = oracle.run_inputs(inp, nthreads=1)
    b = oracle.run_inputs(inp, nthreads=5)
    for key in a:
        assert np.array_equal(a[key], b[key]), key


def test_run_unit_matches_full_run():
    inp = kda_inputs.small(seed=9, T=0, H=2, HV=4, K=8, V=8, dtype="f32", seq_lens=[33, 70, 5])
    full = oracle.run_inputs(inp)
    bounds = inp.seq_bounds
    for n in range(3):
        for h in range(2):
            u = oracle.run_unit(inp, n, h)
            b, e = bounds[n]
            assert np.array_equal(u["dq"][0, :, 0], full["dq"][0, b:e, h])
            assert np.array_equal(u["dk"][0, :, 0], full["dk"][0, b:e, h])
            assert np.array_equal(u["dg"][0], full["dg"][0, b:e, 2 * h:2 * h + 2])
            assert np.array_equal(u["dh0"][0], full["dh0"][n, 2 * h:2 * h + 2])
