"""Closed forms, special cases and invariances that pin the fp64 oracle.

Exact reductions of the KDA recurrence used here (they follow from the
recurrence itself; the usual "beta = 0 gives gated linear attention" shorthand
is not literally true for this update, since beta = 0 writes nothing):

1. beta = 0: S_t = Diag(e^{G_t}) h0 with G_t the running sum of g, so
   o_t = scale (q_t e^{G_t})^T h0, dk = dv = 0, and dbeta, dq, dg, dh0 follow
   from Lambda_t = dL/dS_t = Diag(e^{G_T - G_t}) dht
                             + scale sum_{s>=t} Diag(e^{G_s - G_t}) q_s do_s^T.
2. Distinct one-hot keys (T <= K) and h0 = 0: the removal term S'^T k_t is
   zero, so KDA is gated linear attention with values beta_t v_t.
3. (2) with g = 0: plain causal linear attention.
4. do = 0 and dht = 0: every gradient is exactly zero.
5. o is linear in (v, h0) jointly and in scale.
6. Grouped value heads with identical per-value-head inputs: the key-head
   gradient is G times the single-head one.
7. Packed sequences give exactly the per-sequence results.
"""
import numpy as np
import pytest
import torch

import kda_inputs
import oracle


def _np(inp):
    f = lambda x: None if x is None else x.to(torch.float64).numpy().copy()
    return dict(q=f(inp.q), k=f(inp.k), v=f(inp.v), g=f(inp.g), beta=f(inp.beta), h0=f(inp.h0), do=f(inp.do),
                dht=f(inp.dht), scale=inp.scale)


def _run(x, **kw):
    return oracle.run(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], x["h0"], x["do"], x["dht"], **kw)


def _close(a, b, tol=1e-12):
    den = max(np.linalg.norm(b), 1e-300)
    return np.linalg.norm(a - b) / den < tol


def test_beta_zero_closed_form():
    x = _np(kda_inputs.small(seed=21, B=1, T=30, H=1, HV=1, K=5, V=4, dtype="f32", g_mu=0.0))
    x["beta"][:] = 0.0
    r = _run(x, chunk=8)
    q, k, v, g, do = (x[n][0, :, 0] for n in ("q", "k", "v", "g", "do"))
    h0, dht, sc = x["h0"][0, 0], x["dht"][0, 0], x["scale"]
    T = q.shape[0]
    Gc = np.cumsum(g, axis=0)  # G_t, [T, K]
    o = sc * np.einsum("tk,kv->tv", q * np.exp(Gc), h0)
    ht = np.exp(Gc[-1])[:, None] * h0
    assert _close(r["o"][0, :, 0], o) and _close(r["ht"][0, 0], ht)
    assert np.all(r["dk"] == 0) and np.all(r["dv"] == 0)
    # Lambda_t and the derived gradients
    dbeta, dq, dG = np.zeros(T), np.zeros_like(q), np.zeros_like(g)
    for t in range(T):
        lam = np.exp(Gc[-1] - Gc[t])[:, None] * dht
        for s in range(t, T):
            lam = lam + sc * np.exp(Gc[s] - Gc[t])[:, None] * np.outer(q[s], do[s])
        Sp = np.exp(Gc[t])[:, None] * h0
        u = v[t] - Sp.T @ k[t]
        dbeta[t] = k[t] @ lam @ u
        dq[t] = sc * (np.exp(Gc[t])[:, None] * h0) @ do[t]
        dG[t] = sc * np.sum((np.exp(Gc[t])[:, None] * h0) * np.outer(q[t], do[t]), axis=1)
    dG[-1] += np.sum(ht * dht, axis=1)
    dg = np.cumsum(dG[::-1], axis=0)[::-1]
    dh0 = np.exp(Gc[-1])[:, None] * dht + sum(sc * np.exp(Gc[s])[:, None] * np.outer(q[s], do[s]) for s in range(T))
    assert _close(r["dbeta"][0, :, 0], dbeta)
    assert _close(r["dq"][0, :, 0], dq)
    assert _close(r["dg"][0, :, 0], dg)
    assert _close(r["dh0"][0, 0], dh0)


def _gla_torch(q, k, v, g, beta, scale, do, perm):
    """Gated linear attention with values beta*v and one-hot keys e_perm[j],
    written as its closed form o_t = scale sum_{j<=t} q_t[p_j] e^{G_t[p_j]-G_j[p_j]} beta_j v_j;
    returns o and autograd gradients of sum(o*do)."""
    q, g, beta, v = (torch.tensor(a, requires_grad=True) for a in (q, g, beta, v))
    T = q.shape[0]
    Gc = torch.cumsum(g, 0)
    rows = []
    for t in range(T):
        acc = torch.zeros(v.shape[1], dtype=torch.float64)
        for j in range(t + 1):
            p = perm[j]
            acc = acc + q[t, p] * torch.exp(Gc[t, p] - Gc[j, p]) * beta[j] * v[j]
        rows.append(scale * acc)
    o = torch.stack(rows)
    (o * torch.tensor(do)).sum().backward()
    return o.detach().numpy(), q.grad.numpy(), g.grad.numpy(), beta.grad.numpy(), v.grad.numpy()


@pytest.mark.parametrize("zero_gate", [False, True])
def test_one_hot_keys_reduce_to_gla_and_linear_attention(zero_gate):
    T, K, V = 10, 12, 3
    x = _np(kda_inputs.small(seed=23, B=1, T=T, H=1, HV=1, K=K, V=V, dtype="f32", h0=False, dht=False))
    perm = np.random.default_rng(1).permutation(K)[:T]
    x["k"][:] = 0.0
    for t in range(T):
        x["k"][0, t, 0, perm[t]] = 1.0
    if zero_gate:
        x["g"][:] = 0.0
    r = _run(x, chunk=4)
    q, g, beta, v, do = x["q"][0, :, 0], x["g"][0, :, 0], x["beta"][0, :, 0], x["v"][0, :, 0], x["do"][0, :, 0]
    o, dq, dg, dbeta, dv = _gla_torch(q, None, v, g, beta, x["scale"], do, perm)
    assert _close(r["o"][0, :, 0], o)
    assert _close(r["dq"][0, :, 0], dq)
    assert _close(r["dv"][0, :, 0], dv)
    assert _close(r["dbeta"][0, :, 0], dbeta)
    assert _close(r["dg"][0, :, 0], dg, 1e-11)
    if zero_gate:
        # textbook causal linear attention with values beta v
        sc = x["scale"]
        A = np.tril(q @ x["k"][0, :, 0].T)
        assert _close(r["o"][0, :, 0], sc * A @ (beta[:, None] * v))
        assert _close(r["dv"][0, :, 0], sc * beta[:, None] * (A.T @ do))
        assert _close(r["dq"][0, :, 0], sc * np.tril(do @ (beta[:, None] * v).T) @ x["k"][0, :, 0])


def test_zero_cotangents_give_zero_gradients():
    x = _np(kda_inputs.small(seed=5, B=2, T=33, H=2, HV=4, K=6, V=6, dtype="f32"))
    x["do"][:] = 0.0
    x["dht"][:] = 0.0
    r = _run(x, chunk=8)
    for key in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        assert np.all(r[key] == 0.0), key


def test_linearity_in_values_state_and_scale():
    x = _np(kda_inputs.small(seed=6, B=1, T=40, H=1, HV=2, K=6, V=5, dtype="f32"))
    base = _run(x, chunk=8, backward=False)
    y = dict(x, v=2.5 * x["v"], h0=2.5 * x["h0"])
    r = _run(y, chunk=8, backward=False)
    assert _close(r["o"], 2.5 * base["o"]) and _close(r["ht"], 2.5 * base["ht"])
    z = dict(x, scale=3.0 * x["scale"])
    r = _run(z, chunk=8, backward=False)
    assert _close(r["o"], 3.0 * base["o"]) and np.array_equal(r["ht"], base["ht"])


def test_gva_identical_value_heads():
    G = 3
    single = _np(kda_inputs.small(seed=8, B=1, T=50, H=1, HV=1, K=6, V=4, dtype="f32"))
    grouped = dict(single)
    for n in ("v", "g", "beta", "do"):
        grouped[n] = np.repeat(single[n], G, axis=2)
    for n in ("h0", "dht"):
        grouped[n] = np.repeat(single[n], G, axis=1)
    a, b = _run(single, chunk=16), _run(grouped, chunk=16)
    assert _close(b["dq"], G * a["dq"]) and _close(b["dk"], G * a["dk"])
    for j in range(G):
        assert np.array_equal(b["dv"][:, :, j], a["dv"][:, :, 0])
        assert np.array_equal(b["dg"][:, :, j], a["dg"][:, :, 0])


def test_packed_sequences_equal_separate_runs():
    lens = [17, 64, 1, 90]
    inp = kda_inputs.small(seed=10, T=0, H=2, HV=2, K=6, V=6, dtype="f32", seq_lens=lens)
    full = oracle.run_inputs(inp, chunk=16)
    for n, (b, e) in enumerate(inp.seq_bounds):
        sl = lambda t: t[:, b:e]
        r = oracle.run(sl(inp.q), sl(inp.k), sl(inp.v), sl(inp.g), sl(inp.beta), inp.scale, inp.h0[n:n + 1],
                       sl(inp.do), inp.dht[n:n + 1], chunk=16)
        for key in ("o", "dq", "dk", "dv", "dg", "dbeta"):
            assert np.array_equal(r[key][0], full[key][0, b:e]), key
        for key in ("ht", "dh0"):
            assert np.array_equal(r[key][0], full[key][n]), key


def test_triangle_backward_product_identity():
    """The chunked oracle's dINV INV^T, with dINV = d_delta (beta V)^T + dw (beta K~)^T, equals
    d_delta delta^T in every chunk, partial chunks included (u = INV beta V, w = INV beta K~,
    dw = -d_delta S_in^T, delta = u - w S_in). The gradient kernel forms the product that way."""
    from oracle.chunked import run_chunked

    inp = kda_inputs.small(seed=41, B=1, T=0, H=1, HV=2, K=8, V=6, dtype="f32", seq_lens=[150, 37])
    t = lambda x: None if x is None else x.to(torch.float64)
    ref = run_chunked(t(inp.q), t(inp.k), t(inp.v), t(inp.g), t(inp.beta), inp.scale, t(inp.h0), t(inp.do),
                      t(inp.dht), inp.cu_seqlens, keep=True)
    assert len(ref["chunks"]) == 2 * (3 + 1)
    for key, ch in ref["chunks"].items():
        dINV = ch["d_delta"] @ ch["Xv"].T + ch["dw"] @ ch["Xk"].T
        lhs = dINV @ ch["INV"].T
        rhs = ch["d_delta"] @ ch["delta"].T
        assert _close(lhs, rhs, 1e-11), key
        # dropping the dw w^T term (a plausible slip) does not pass: S_in is nonzero (h0 given)
        assert not _close(ch["d_delta"] @ ch["u"].T, rhs, 1e-6), key
