"""Seeded synthetic inputs for the KDA chunked backward.

This module is the one piece shared by the CUDA library's tests/benchmark and
the CPU oracle: it draws inputs and nothing else (no step of the method's
arithmetic lives here). Every tensor is drawn on the CPU from a
``torch.Generator`` seeded per workload, in a fixed order:

    [lengths], q, k, v, g, beta, h0, do, dht

* q, k ~ N(0, 1), L2-normalised over the key dimension (per token and head)
  in fp32, then cast to the compute dtype;
* v, do ~ N(0, 1);
* g = logsigmoid(N(mu, 1)) per key channel, fp32 (natural-log per-token decay);
* beta = sigmoid(N(0, 1)), cast to the compute dtype;
* h0, dht ~ std * N(0, 1), fp32, when the workload has them.

bf16 casts round to nearest even (torch's ``.to``). The five named workloads
are the KDA forward-recompute + backward cases: fp32 B1 T256 H2 K64; bf16 B1
T2048 H16 K128; bf16 B8 T4096 H32 K128; bf16 varlen 16 sequences of U[1,4096]
tokens H32 K128; bf16 B1 T65536 H16/HV32 K128 with slow decay.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

CHUNK = 64


@dataclasses.dataclass
class Spec:
    name: str
    B: int
    T: int
    H: int
    HV: int
    K: int
    V: int
    dtype: str  # "bf16" or "f32"
    seed: int
    scale: Optional[float] = None  # None -> K ** -0.5
    g_mu: float = 3.0
    h0_std: Optional[float] = None  # None -> no initial state
    dht_std: Optional[float] = None  # None -> no final-state gradient
    varlen_n: int = 0  # > 0: B must be 1 and lengths ~ U[varlen_min, varlen_max]
    varlen_min: int = 1
    varlen_max: int = 4096
    seq_lens: Optional[tuple] = None  # explicit packed lengths (B must be 1)


WORKLOADS = {
    "fp32_b1_t256_h2_k64": Spec("fp32_b1_t256_h2_k64", B=1, T=256, H=2, HV=2, K=64, V=64,
                                 dtype="f32", seed=0, scale=1.0 / 8.0, h0_std=0.1, dht_std=1.0),
    "bf16_b1_t2048_h16_k128": Spec("bf16_b1_t2048_h16_k128", B=1, T=2048, H=16, HV=16, K=128, V=128,
                                    dtype="bf16", seed=1, scale=128 ** -0.5, h0_std=0.1, dht_std=1.0),
    "bf16_b8_t4096_h32_k128": Spec("bf16_b8_t4096_h32_k128", B=8, T=4096, H=32, HV=32, K=128, V=128,
                                    dtype="bf16", seed=2),
    "bf16_varlen16_h32_k128": Spec("bf16_varlen16_h32_k128", B=1, T=0, H=32, HV=32, K=128, V=128,
                                    dtype="bf16", seed=3, h0_std=0.1, varlen_n=16),
    "bf16_b1_t65536_h16_hv32_k128": Spec("bf16_b1_t65536_h16_hv32_k128", B=1, T=65536, H=16, HV=32,
                                          K=128, V=128, dtype="bf16", seed=4, g_mu=4.0,
                                          h0_std=0.1, dht_std=0.1),
}
WORKLOAD_ORDER = list(WORKLOADS)


@dataclasses.dataclass
class Inputs:
    spec: Spec
    q: torch.Tensor  # [B, T, H, K]
    k: torch.Tensor  # [B, T, H, K]
    v: torch.Tensor  # [B, T, HV, V]
    g: torch.Tensor  # [B, T, HV, K] fp32
    beta: torch.Tensor  # [B, T, HV]
    h0: Optional[torch.Tensor]  # [N, HV, K, V] fp32
    do: torch.Tensor  # [B, T, HV, V]
    dht: Optional[torch.Tensor]  # [N, HV, K, V] fp32
    cu_seqlens: Optional[torch.Tensor]  # int64 [N + 1] or None
    scale: float

    @property
    def B(self):
        return self.q.shape[0]

    @property
    def T(self):
        return self.q.shape[1]

    @property
    def num_seqs(self):
        return self.B if self.cu_seqlens is None else self.cu_seqlens.numel() - 1

    @property
    def seq_bounds(self):
        """List of (bos, eos) packed row ranges, one per sequence."""
        if self.cu_seqlens is None:
            return [(b * self.T, (b + 1) * self.T) for b in range(self.B)]
        cu = self.cu_seqlens.tolist()
        return [(cu[i], cu[i + 1]) for i in range(len(cu) - 1)]

    @property
    def tokens(self):
        return self.B * self.T

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.spec.dtype == "bf16" else torch.float32


def _l2norm(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-6)


def make(spec: Spec) -> Inputs:
    """Draw the inputs of ``spec`` (CPU tensors, final dtypes)."""
    gen = torch.Generator(device="cpu").manual_seed(spec.seed)
    B, T = spec.B, spec.T
    cu = None
    if spec.varlen_n > 0 or spec.seq_lens is not None:
        if B != 1:
            raise ValueError("packed sequences need B == 1")
        if spec.seq_lens is not None:
            lens = torch.tensor(spec.seq_lens, dtype=torch.int64)
        else:
            lens = torch.randint(spec.varlen_min, spec.varlen_max + 1, (spec.varlen_n,),
                                 generator=gen, dtype=torch.int64)
        cu = torch.zeros(lens.numel() + 1, dtype=torch.int64)
        cu[1:] = torch.cumsum(lens, 0)
        T = int(cu[-1])
    N = B if cu is None else cu.numel() - 1
    H, HV, K, V = spec.H, spec.HV, spec.K, spec.V
    dt = torch.bfloat16 if spec.dtype == "bf16" else torch.float32
    q = _l2norm(torch.randn(B, T, H, K, generator=gen)).to(dt)
    k = _l2norm(torch.randn(B, T, H, K, generator=gen)).to(dt)
    v = torch.randn(B, T, HV, V, generator=gen).to(dt)
    g = torch.nn.functional.logsigmoid(torch.randn(B, T, HV, K, generator=gen) + spec.g_mu)
    beta = torch.sigmoid(torch.randn(B, T, HV, generator=gen)).to(dt)
    h0 = None
    if spec.h0_std is not None:
        h0 = torch.randn(N, HV, K, V, generator=gen) * spec.h0_std
    do = torch.randn(B, T, HV, V, generator=gen).to(dt)
    dht = None
    if spec.dht_std is not None:
        dht = torch.randn(N, HV, K, V, generator=gen) * spec.dht_std
    scale = spec.scale if spec.scale is not None else K ** -0.5
    return Inputs(spec, q, k, v, g.contiguous(), beta, h0, do, dht, cu, float(scale))


def workload(name: str) -> Inputs:
    return make(WORKLOADS[name])


def small(seed=0, B=1, T=100, H=2, HV=2, K=16, V=16, dtype="f32", h0=True, dht=True,
          seq_lens=None, g_mu=3.0, scale=None) -> Inputs:
    """A small case for tests (any sizes the library accepts)."""
    sp = Spec("small", B=B, T=T, H=H, HV=HV, K=K, V=V, dtype=dtype, seed=seed, scale=scale,
              g_mu=g_mu, h0_std=0.1 if h0 else None, dht_std=1.0 if dht else None,
              seq_lens=tuple(seq_lens) if seq_lens is not None else None)
    return make(sp)


def num_chunks(inp: Inputs, chunk: int = CHUNK) -> int:
    return sum(math.ceil((e - b) / chunk) for b, e in inp.seq_bounds)
