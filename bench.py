"""Benchmark: KDA forward-recompute + backward tokens/s on GB300.

One step = one ``kda_chunk_bwd`` call with ``states = NULL`` (the call
recomputes the chunk forward it needs, then runs the whole backward) over the
bf16 workload B=8, T=4096, H=HV=32, K=V=128, chunk 64 (seeded synthetic
inputs; see kda_inputs.py). Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--pass bwd|fwd|bwd-states|bwd-saved|fwd-save|bwd-fused] [--workload NAME]

* ``value``: device-timed tokens/s (inputs resident in HBM; K steps between
  CUDA events, barrier + synchronize on both sides, max over ranks). The
  per-step working set (~10 GB) is far larger than the 129 MB L2, so no flush
  is needed between steps. The library also records one CUDA event after
  each of its kernel launches inside the timed region (its per-kernel timing
  hook); ``step_ms`` gives the median, minimum, maximum and standard
  deviation of the per-step spans those events bracket.
* ``e2e``: the same metric through the C ABI from pinned host buffers: every
  step copies its inputs host->device, runs the call, and copies every
  gradient back; with two device buffer sets the copies of neighbouring steps
  overlap the current step's compute on their own streams. It is bound by the
  host link: each step moves about 2.95 GB (bf16 inputs and gradients, fp32 g
  and dg).
* ``roofline``: the dominant kernel's algorithmic bytes (or FLOPs) per launch
  over its average launch time, measured with CUDA events that the library
  records between its own launches on the call's stream.
* ``cpu_baseline``: the fp64 oracle on the host cores on a bounded sample of
  the same workload (whole sequences x heads), scaled to tokens/s.
* ``--impl reference``: the fp64 oracle timed as the reference arm.
* ``--pass``: ``bwd`` (default, the headline step above); ``fwd`` times one
  ``kda_chunk_fwd`` call (o and ht) per step; ``bwd-states`` times the
  backward that consumes the fp32 chunk states a forward saved; ``bwd-saved``
  times ``kda_chunk_bwd_from_saved`` on the context ``kda_chunk_fwd_save``
  kept (the states or context are produced once before the timed region);
  ``bwd-fused`` times ``kda_chunk_bwd_fused`` (the step of ``bwd`` with the
  reverse pass and the per-chunk gradients fused into one launch).
* ``--workload``: one of the four bf16 workloads of kda_inputs.py (default
  the B=8 T=4096 H=HV=32 benchmark); the others (B=1 T=2048 H=16 with h0 and
  dht; 16 packed sequences of U[1,4096] tokens with h0; B=1 T=65536 with 16
  key heads over 32 value heads, h0 and dht) run with their initial states,
  final-state gradients and packed-sequence tables as drawn.

Multi-GPU (torchrun): every rank runs the full workload on its own GPU (weak
scaling, independent batches, no data-path collective); ``value`` is the sum
of tokens over ranks divided by the max over ranks of the timed span.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import kda_inputs  # noqa: E402

WORKLOAD = "bf16_b8_t4096_h32_k128"
METRIC = "KDA fwd-recompute+bwd tokens/s on 1 GB300 and % of roofline vs CPU oracle"
METRICS = {"bwd": METRIC, "fwd": "KDA chunk forward (o, ht) tokens/s on 1 GB300",
           "bwd-states": "KDA backward from saved chunk states tokens/s on 1 GB300",
           "bwd-saved": "KDA backward from the forward's saved context tokens/s on 1 GB300",
           "fwd-save": "KDA chunk forward (o, ht) keeping the backward's saved context tokens/s on 1 GB300",
           "bwd-fused": "KDA fwd-recompute+bwd with the fused reverse kernel tokens/s on 1 GB300"}
UNIT = "tokens/s"

# ----------------------------------------------------------------------------
# Algorithmic cost model (per launch) of each kernel, from the problem sizes.
# Bytes count what the step must read/write at its dtype, plus the fp32 chunk
# state written once and read once; FLOPs count each dense product once.
# ----------------------------------------------------------------------------


def step_cost(B, T, H, HV, K, V, in_bytes=2, C=64, nck=None, seq_states=0):
    """Algorithmic bytes / FLOPs of one backward step. ``nck``: chunk-heads when the sequences are packed
    (default B * ceil(T / C) * HV); ``seq_states``: fp32 [N, HV, K, V] tensors the step reads or writes
    besides the chunk states (h0, dht, dh0), given as their total element count."""
    th = B * T * HV  # token-heads
    tk = B * T * H
    if nck is None:
        nck = B * ((T + C - 1) // C) * HV
    io_in = tk * K * in_bytes * 2 + th * V * in_bytes * 2 + th * K * 4 + th * in_bytes
    io_out = tk * K * in_bytes * 2 + th * V * in_bytes + th * K * 4 + th * in_bytes
    io_in += seq_states * 4
    states = 2 * nck * K * V * 4
    flops = nck * (16 * C * K * V + 9 * C * C * K + 5 * C * C * V + C ** 3)
    return dict(bytes=io_in + io_out + states, flops=flops, io_in=io_in, io_out=io_out, states=states, nck=nck)


def pass_cost(mode, B, T, H, HV, K, V, in_bytes=2, C=64, nck=None, seq_states=0):
    """Algorithmic bytes / FLOPs of one step of ``mode`` (see step_cost for the backward)."""
    s = step_cost(B, T, H, HV, K, V, in_bytes, C, nck, seq_states)
    th, tk, nck = B * T * HV, B * T * H, s["nck"]
    if mode in ("fwd", "fwd-save"):  # q, k, v, g, beta in; o and ht out (fwd-save: plus the chunk state written once)
        b = tk * K * in_bytes * 2 + th * V * in_bytes + th * K * 4 + th * in_bytes + th * V * in_bytes
        b += B * HV * K * V * 4
        if mode == "fwd-save":
            b += s["states"] // 2
        f = nck * (6 * C * C * K + 2 * C * C * V + C ** 3 // 3 + 6 * C * K * V + 2 * C * C * V)
        return dict(s, bytes=b, flops=f)
    if mode in ("bwd-states", "bwd-saved"):  # the saved chunk states are read once instead of written and read
        return dict(s, bytes=s["io_in"] + s["io_out"] + s["states"] // 2)
    return s


def kernel_cost(name, B, T, H, HV, K, V, in_bytes=2, C=64, nck=None):
    """(bound, algorithmic bytes, algorithmic flops) of one launch of kernel ``name``. A ``_vhalf`` launch
    (each sweep split by state columns over two CTAs) has the algorithmic cost of the whole one."""
    name = name[: -len("_vhalf")] if name.endswith("_vhalf") else name
    s = step_cost(B, T, H, HV, K, V, in_bytes, C, nck)
    nck = s["nck"]
    th = B * T * HV
    tk = B * T * H
    st = nck * K * V * 4  # one pass over the fp32 chunk states
    if name == "simt_intra":
        b = tk * K * in_bytes * 2 + th * (V * in_bytes + K * 4 + in_bytes)
        f = nck * (4 * C * C * K + 2 * C * C * (K + V) + C ** 3 // 3)
        return "alu", b, f
    if name == "simt_state_fwd":
        return "alu", st + tk * K * in_bytes, nck * 4 * C * K * V
    if name == "simt_ds_rev":
        return "alu", th * V * in_bytes + tk * K * in_bytes * 2, nck * (6 * C * K * V + 2 * C * C * V)
    if name == "simt_grads_a":
        return "alu", 2 * st + th * V * in_bytes, nck * 6 * C * K * V
    if name == "simt_grads_b":
        b = s["io_out"] + tk * K * in_bytes * 2 + th * (2 * V * in_bytes + in_bytes)
        f = nck * (6 * C * C * V + 10 * C * C * K + 4 * C ** 3)
        return "alu", b, f
    if name == "gva_reduce":
        return "hbm", th * K * 4 * 2 + tk * K * in_bytes * 2, 0
    # Tensor-core path (bf16 K = V = 128): per chunk-head I/O of each kernel at
    # its dtypes (bf16 tiles CxK = 16 KB, CxC = 8 KB, KxV = 32 KB), read once
    # and written once; FLOPs of its dense products counted once.
    tcd, tcc, tdd = C * K * 2, C * C * 2, K * V * 2
    per_in = C * (2 * K * in_bytes + V * in_bytes + K * 4 + in_bytes)  # q, k, v, g, beta of one chunk-head
    if name == "tc_intra":  # q, k, g, beta in; w, K^, scale Q~, Aqk, INV, INV diag(beta), e^Gamma_C out
        b = nck * (per_in - C * V * in_bytes + 3 * tcd + 3 * tcc + K * 4)
        f = nck * (2 * 2 * C * C * K + 2 * 2 * C * C * (K + V) // 2 + C ** 3 // 3)
        return "hbm", b, f
    if name == "tc_state_fwd":  # w, INV diag(beta), V, K^, e^Gamma_C in; S_in, delta out
        return "hbm", nck * (3 * tcd + tcc + K * 4 + tdd + tcd), nck * 4 * C * K * V
    if name == "tc_state_both":  # tc_state_fwd and tc_ds_rev in one launch
        sf, sr = kernel_cost("tc_state_fwd", B, T, H, HV, K, V, in_bytes, C, nck), kernel_cost(
            "tc_ds_rev", B, T, H, HV, K, V, in_bytes, C, nck)
        return "hbm", sf[1] + sr[1], sf[2] + sr[2]
    if name == "tc_ds_rev":
        return "hbm", nck * (3 * tcd + tcc + C * V * in_bytes + K * 4 + tdd + tcd), nck * (6 * C * K * V + 2 * C * C * V)
    if name == "tc_grads":
        b = nck * (per_in + C * V * in_bytes + 2 * tcd + 2 * tdd + tcc + K * 4) + s["io_out"]
        return "hbm", b, s["flops"]
    if name == "tc_rev_fused":  # tc_ds_rev's and tc_grads' inputs (dO, e^Gamma_C once) and outputs, no
        # dS_out / d_delta round trip
        b = nck * (per_in + C * V * in_bytes + 4 * tcd + tdd + 2 * tcc + K * 4) + s["io_out"]
        return "hbm", b, s["flops"]
    if name == "tc_fwd_out":  # w, INV diag(beta), V, K^, scale Q~, Aqk, e^Gamma_C in; o out (state on chip)
        return "hbm", nck * (4 * tcd + 2 * tcc + K * 4 + C * V * in_bytes), nck * (6 * C * K * V + 2 * C * C * V)
    if name == "tc_state_load":  # fp32 state, w, INV diag(beta), V in; S_in, delta out
        return "hbm", nck * (K * V * 4 + 2 * tcd + tcc + tdd + tcd), nck * 2 * C * K * V
    return "hbm", s["bytes"], s["flops"]


# DRAM traffic per launch measured by ncu (dram__bytes_read.sum + dram__bytes_write.sum) on the
# B=2 case of the benchmark workload and scaled by chunk-heads; reported only while the kernel's
# source file is the revision named (sha1 prefix): the captured one, or a later one that leaves
# that kernel's code as it was (the entry says so).
MEASURED_TRAFFIC = {
    # tc_grads and tc_rev_fused captured at kda_tc_grads.cu 145f696ca185; the later revision changes only a comment
    "tc_grads": {"source": "chunked_gated_delta_10_gb300/csrc/kda_tc_grads.cu", "sha1": "519ea07f922c",
                 "bytes_per_chunk_head": (841.820928e6 + 302.801408e6) / 4096},
    "tc_rev_fused": {"source": "chunked_gated_delta_10_gb300/csrc/kda_tc_grads.cu", "sha1": "519ea07f922c",
                     "bytes_per_chunk_head": (875.679488e6 + 311.447296e6) / 4096},
    # captured at kda_tc.cu 5d4485ab5f02; the later revision changes only comments
    "tc_intra": {"source": "chunked_gated_delta_10_gb300/csrc/kda_tc.cu", "sha1": "126e2613ba82",
                 "bytes_per_chunk_head": (269.103104e6 + 249.853440e6) / 4096},
}


def measured_traffic(name, nck):
    import hashlib

    m = MEASURED_TRAFFIC.get(name)
    if not m:
        return None
    try:
        with open(os.path.join(ROOT, m["source"]), "rb") as f:
            if hashlib.sha1(f.read()).hexdigest()[:12] != m["sha1"]:
                return None
    except OSError:
        return None
    return m["bytes_per_chunk_head"] * nck


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "sm_max_mhz": 2070.0}, "fallback"


def alu_peak_tflops(sm_mhz):
    """FP32 FFMA peak: 152 SMs x 128 FP32 lanes x 2 FLOP x clock."""
    return 152 * 128 * 2 * sm_mhz * 1e6 / 1e12


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        mhz, mx, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                mhz.append(float(parts[1]))
                mx.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        load = [m for m, p in zip(mhz, power) if p > 0.3 * max(power)] or mhz
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(mhz), "power_w_max": max(power)}


# ----------------------------------------------------------------------------
# distributed helpers
# ----------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, device) -> float:
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device):
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        if device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def aggregate(tokens_per_rank: int, elapsed_s: float, world: int, device) -> tuple:
    """Whole-job tokens/s: every rank processed ``tokens_per_rank``; time is the max over ranks."""
    t = max_over_ranks(elapsed_s, device)
    return tokens_per_rank * world / t, t


# ----------------------------------------------------------------------------
# the CPU oracle leg
# ----------------------------------------------------------------------------

def oracle_sample(inp, n_seqs, n_heads):
    """Time the fp64 oracle on ``n_seqs`` whole sequences x ``n_heads`` key heads (all host cores)."""
    import oracle

    H = inp.q.shape[2]
    HV = inp.v.shape[2]
    G = HV // H
    T = inp.T
    sl = lambda x, hs: x[:n_seqs, :, hs].contiguous()
    hs, vs = slice(0, n_heads), slice(0, n_heads * G)
    args = (sl(inp.q, hs), sl(inp.k, hs), sl(inp.v, vs), sl(inp.g, vs), sl(inp.beta, vs), inp.scale,
            None if inp.h0 is None else inp.h0[:n_seqs, vs].contiguous(), sl(inp.do, vs),
            None if inp.dht is None else inp.dht[:n_seqs, vs].contiguous())
    oracle.build()
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    used = min(cores, n_seqs * n_heads)
    t0 = time.perf_counter()
    oracle.run(*args, nthreads=used)
    dt = time.perf_counter() - t0
    # tokens/s of the full-width problem: token-heads processed / heads / time
    token_heads = n_seqs * T * n_heads
    return token_heads / H / dt, used, dt, f"{n_seqs} sequence(s) x {n_heads} of {H} key heads x {T} tokens"


def workload_config(inp, world, extra=None):
    """The ``config`` object of a JSON line (the same keys on both arms)."""
    B, T, H, K = inp.q.shape
    HV = inp.v.shape[2]
    cfg = {"workload": inp.spec.name, "global_batch": B * world, "seq_len": T, "heads": H, "value_heads": HV,
           "head_dim": K, "chunk": 64, "parallelism": f"dp{world}" if world > 1 else "single",
           "l2": "inputs larger than L2 (several GB touched per step), no flush"}
    if inp.cu_seqlens is not None:
        cfg["packed_sequences"] = inp.num_seqs
    cfg.update(extra or {})
    return cfg


def oracle_sample_any(inp):
    """The bounded CPU sample of a workload: 16 key heads of the first sequence (its first 4096 tokens)."""
    if inp.cu_seqlens is None and inp.T <= 4096:
        return oracle_sample(inp, 1, min(16, inp.q.shape[2]))
    import oracle

    b, e = inp.seq_bounds[0]
    L = min(e - b, 4096)
    H, HV = inp.q.shape[2], inp.v.shape[2]
    G = HV // H
    nh = min(16, H)
    hs, vs = slice(0, nh), slice(0, nh * G)
    rows = lambda x, s: x.reshape(-1, *x.shape[2:])[b:b + L, s].unsqueeze(0).contiguous()
    st = lambda x: None if x is None else x[0:1, vs].contiguous()
    oracle.build()
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    used = min(cores, nh)
    t0 = time.perf_counter()
    oracle.run(rows(inp.q, hs), rows(inp.k, hs), rows(inp.v, vs), rows(inp.g, vs), rows(inp.beta, vs), inp.scale,
               st(inp.h0), rows(inp.do, vs), st(inp.dht), nthreads=used)
    dt = time.perf_counter() - t0
    return L * nh / H / dt, used, dt, f"first {L} tokens of sequence 0 x {nh} of {H} key heads"


def reference_arm(args):
    ws, rank, local = dist_env()
    if rank != 0:
        return
    inp = kda_inputs.workload(args.workload)
    vals = []
    for _ in range(args.warmup):
        oracle_sample_any(inp)
    used = 0
    sample = ""
    for _ in range(args.steps):
        v, used, dt, sample = oracle_sample_any(inp)
        vals.append(v)
    value = statistics.median(vals)
    tokens = int(inp.q.shape[0]) * int(inp.q.shape[1])
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": tokens / value * 1e3 if value > 0 else None,
            "timing": "each timed step runs the bounded sample (cpu_baseline.sample); value is the median rate over "
                      "the steps and ms_per_step the whole workload's step at that rate",
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(inp, ws),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# the GPU arm
# ----------------------------------------------------------------------------

def gpu_arm(args):
    import chunked_gated_delta_10_gb300 as kda

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    kda.build()
    lib = kda.load()

    spec = kda_inputs.WORKLOADS[args.workload]
    if args.batch or args.seq_len:
        import dataclasses

        spec = dataclasses.replace(spec, B=args.batch or spec.B, T=args.seq_len or spec.T)
    inp = kda_inputs.make(spec)
    B, T, H, K = inp.q.shape
    HV, V = inp.v.shape[2], inp.v.shape[3]
    N = inp.num_seqs
    tokens = B * T
    mode = args.mode
    fwd_like = mode in ("fwd", "fwd-save")
    host = dict(q=inp.q, k=inp.k, v=inp.v, g=inp.g, beta=inp.beta)
    if inp.h0 is not None:
        host["h0"] = inp.h0
    if not fwd_like:
        host["do"] = inp.do
        if inp.dht is not None:
            host["dht"] = inp.dht
    x = {n: t.to(device).contiguous() for n, t in host.items()}
    vl = kda._Varlen(inp.cu_seqlens, device)
    dims = kda.make_dims(x["q"], x["v"], inp.scale, inp.cu_seqlens)
    nck = int(dims.num_chunks) * HV
    wsb = (kda.workspace_bytes(dims, kda.PASS_FWD) if mode == "fwd" else
           kda.saved_bytes(dims) if mode == "fwd-save" else kda.workspace_bytes(dims, kda.PASS_BWD))
    ws = torch.empty(wsb, dtype=torch.uint8, device=device)
    if fwd_like:
        out = dict(o=torch.empty_like(x["v"]), ht=torch.empty(N, HV, K, V, dtype=torch.float32, device=device))
    else:
        out = dict(dq=torch.empty_like(x["q"]), dk=torch.empty_like(x["k"]), dv=torch.empty_like(x["v"]),
                   dg=torch.empty_like(x["g"]), dbeta=torch.empty_like(x["beta"]))
        if "h0" in x:
            out["dh0"] = torch.empty_like(x["h0"])
    stream = torch.cuda.current_stream(device)
    sptr = ctypes.c_void_p(stream.cuda_stream)
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    states = None
    if mode == "bwd-states":  # the forward's saved chunk states, produced once outside the timed region
        fwb = kda.workspace_bytes(dims, kda.PASS_FWD)
        fws = torch.empty(fwb, dtype=torch.uint8, device=device)
        states = torch.empty(dims.num_chunks, HV, K, V, dtype=torch.float32, device=device)
        o_tmp = torch.empty_like(x["v"])
        rc = lib.kda_chunk_fwd(ctypes.byref(dims), P(x["q"]), P(x["k"]), P(x["v"]), P(x["g"]), P(x["beta"]),
                               P(x.get("h0")), P(vl.cu), P(vl.idx), P(vl.off), P(o_tmp), None, P(states), P(fws),
                               fwb, sptr)
        if rc != 0:
            raise kda.KdaError(rc, "kda_chunk_fwd")
        del fws, o_tmp
    if mode == "bwd-saved":  # the forward's saved context, produced once outside the timed region; it is also
        wsb = kda.saved_bytes(dims)  # the backward's workspace
        ws = torch.empty(wsb, dtype=torch.uint8, device=device)
        o_tmp = torch.empty_like(x["v"])
        rc = lib.kda_chunk_fwd_save(ctypes.byref(dims), P(x["q"]), P(x["k"]), P(x["v"]), P(x["g"]), P(x["beta"]),
                                    P(x.get("h0")), P(vl.cu), P(vl.idx), P(vl.off), P(o_tmp), None, P(ws), wsb, sptr)
        if rc != 0:
            raise kda.KdaError(rc, "kda_chunk_fwd_save")
        del o_tmp

    def step(inputs, outs):
        if mode == "fwd":
            rc = lib.kda_chunk_fwd(ctypes.byref(dims), P(inputs["q"]), P(inputs["k"]), P(inputs["v"]),
                                   P(inputs["g"]), P(inputs["beta"]), P(inputs.get("h0")), P(vl.cu), P(vl.idx),
                                   P(vl.off), P(outs["o"]), P(outs["ht"]), None, P(ws), wsb, sptr)
        elif mode == "fwd-save":
            rc = lib.kda_chunk_fwd_save(ctypes.byref(dims), P(inputs["q"]), P(inputs["k"]), P(inputs["v"]),
                                        P(inputs["g"]), P(inputs["beta"]), P(inputs.get("h0")), P(vl.cu), P(vl.idx),
                                        P(vl.off), P(outs["o"]), P(outs["ht"]), P(ws), wsb, sptr)
        elif mode == "bwd-saved":
            rc = lib.kda_chunk_bwd_from_saved(ctypes.byref(dims), P(inputs["q"]), P(inputs["k"]), P(inputs["v"]),
                                              P(inputs["g"]), P(inputs["beta"]), P(inputs.get("h0")), P(vl.cu),
                                              P(vl.idx), P(vl.off), P(inputs["do"]), P(inputs.get("dht")), P(ws),
                                              wsb, P(outs["dq"]), P(outs["dk"]), P(outs["dv"]), P(outs["dg"]),
                                              P(outs["dbeta"]), P(outs.get("dh0")), sptr)
        else:
            entry = lib.kda_chunk_bwd_fused if mode == "bwd-fused" else lib.kda_chunk_bwd
            rc = entry(ctypes.byref(dims), P(inputs["q"]), P(inputs["k"]), P(inputs["v"]),
                                   P(inputs["g"]), P(inputs["beta"]), P(inputs.get("h0")), P(vl.cu), P(vl.idx),
                                   P(vl.off), P(inputs["do"]), P(inputs.get("dht")), P(states), P(outs["dq"]),
                                   P(outs["dk"]), P(outs["dv"]), P(outs["dg"]), P(outs["dbeta"]),
                                   P(outs.get("dh0")), P(ws), wsb, sptr)
        if rc != 0:
            raise kda.KdaError(rc, {"fwd": "kda_chunk_fwd", "fwd-save": "kda_chunk_fwd_save",
                                    "bwd-saved": "kda_chunk_bwd_from_saved",
                                    "bwd-fused": "kda_chunk_bwd_fused"}.get(mode, "kda_chunk_bwd"))

    for _ in range(args.warmup):
        step(x, out)
    torch.cuda.synchronize(device)
    launches = int(lib.kda_last_launch_count())
    names = [lib.kda_launch_name(i).decode() for i in range(launches)]

    # -- device-timed region, with per-launch events recorded by the library --
    nev = launches + 1
    ev_sets = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(args.steps)]
    clocks = ClockSampler(device.index)
    barrier(device)
    torch.cuda.synchronize(device)
    clocks.start()
    time.sleep(0.3)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for evs in ev_sets:
        for e in evs:
            e.record(stream)  # create the event objects before the timed region
    handle_sets = [(ctypes.c_void_p * nev)(*[e.cuda_event for e in evs]) for evs in ev_sets]
    torch.cuda.synchronize(device)
    start.record(stream)
    for i in range(args.steps):
        lib.kda_set_profile_events(handle_sets[i], nev)
        step(x, out)
    lib.kda_set_profile_events(None, 0)
    stop.record(stream)
    torch.cuda.synchronize(device)
    barrier(device)
    clk = clocks.stop()
    elapsed = start.elapsed_time(stop) / 1e3
    value, tmax = aggregate(tokens * args.steps, elapsed, world, device)

    per = {n: [] for n in names}
    for evs in ev_sets:
        for i, n in enumerate(names):
            per[n].append(evs[i].elapsed_time(evs[i + 1]) / 1e3)
    spans = [evs[0].elapsed_time(evs[-1]) for evs in ev_sets]  # ms, first to last launch of each step
    step_ms = {"mean": statistics.fmean(spans), "median": statistics.median(spans), "min": min(spans),
               "max": max(spans), "stdev": statistics.pstdev(spans), "n": len(spans)}
    tot = {n: sum(v) for n, v in per.items()}
    dom = max(tot, key=tot.get)
    avg = tot[dom] / len(per[dom])
    peaks, peak_src = load_peaks()
    ib = 2 if spec.dtype == "bf16" else 4
    bound, abytes, aflops = kernel_cost(dom, B, T, H, HV, K, V, in_bytes=ib, nck=nck)
    if bound == "hbm":
        ach, pk, unit = abytes / avg / 1e9, peaks["hbm_gbs"], "GB/s"
    elif bound == "tensor":
        ach, pk, unit = aflops / avg / 1e12, peaks["bf16_tflops_sustained"], "TFLOP/s"
    else:
        ach, pk, unit = aflops / avg / 1e12, alu_peak_tflops(clk.get("sm_mhz") or peaks["sm_max_mhz"]), "TFLOP/s"
    traffic = measured_traffic(dom, nck) if args.workload == WORKLOAD else None
    roofline = {"bound": bound, "kernel": dom, "achieved": ach, "peak": pk, "unit": unit, "frac": ach / pk,
                "traffic": traffic, "peak_source": peak_src if bound != "alu" else "152 SMs x 128 FFMA lanes x SM clock",
                "avg_launch_ms": avg * 1e3, "share": tot[dom] / sum(tot.values()),
                "kernels_ms": {n: 1e3 * tot[n] / len(per[n]) for n in names}}
    seq_states = N * HV * K * V * ((1 if "h0" in x else 0) + (0 if fwd_like else
                                                             (1 if "dht" in x else 0) + (1 if "h0" in x else 0)))
    sc = pass_cost(mode, B, T, H, HV, K, V, in_bytes=ib, nck=nck, seq_states=seq_states)
    step_s = elapsed / args.steps
    path = {"bytes_alg": sc["bytes"], "flops_alg": sc["flops"],
            "hbm_frac": sc["bytes"] / step_s / 1e9 / peaks["hbm_gbs"],
            "tensor_frac": sc["flops"] / step_s / 1e12 / peaks["bf16_tflops_sustained"]}

    # -- end to end through the C ABI from pinned host buffers: every step copies its inputs
    # host -> device and its results device -> host. With two device buffer sets, the copies of
    # neighbouring steps run on their own streams and overlap the compute of the current step.
    hin = {n: t.pin_memory() for n, t in host.items()}
    hout = {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for n, t in out.items()}
    h2d = sum(t.numel() * t.element_size() for t in hin.values())
    d2h = sum(t.numel() * t.element_size() for t in hout.values())
    # at least 20 steps (more when the timed run has more), so that the pipeline's fill and drain (the first
    # inputs in, the last results out, not overlapped) are amortised as in a long training run
    e2e_steps = max(20, args.steps)
    xs = [x, {n: torch.empty_like(t) for n, t in x.items()}]
    outs = [out, {n: torch.empty_like(t) for n, t in out.items()}]
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev = lambda: torch.cuda.Event()
    ev_in, ev_comp, ev_out = ([ev() for _ in range(e2e_steps)] for _ in range(3))
    barrier(device)
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(e2e_steps):
        b = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_comp[i - 2])  # buffer set b's inputs are free
            for n in hin:
                xs[b][n].copy_(hin[n], non_blocking=True)
            ev_in[i].record(s_in)
        stream.wait_event(ev_in[i])
        if i >= 2:
            stream.wait_event(ev_out[i - 2])  # buffer set b's results have been copied out
        step(xs[b], outs[b])
        ev_comp[i].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[i])
            for n in hout:
                hout[n].copy_(outs[b][n], non_blocking=True)
            ev_out[i].record(s_out)
    s_out.wait_event(ev_out[e2e_steps - 1])
    e1.record(s_out)
    torch.cuda.synchronize(device)
    e2e_val, _ = aggregate(tokens * e2e_steps, e0.elapsed_time(e1) / 1e3, world, device)

    extra = {}
    if args.batch or args.seq_len:
        extra["workload"] = f"{spec.name} with B={spec.B} T={spec.T}"
    if mode != "bwd":
        extra["pass"] = mode
    line = {"metric": METRICS[mode], "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": tmax / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if spec.dtype == "bf16" else "f32",
            "data": "synthetic", "config": workload_config(inp, world, extra),
            "timing": "value and ms_per_step: mean over the K back-to-back steps between two CUDA events; the "
                      "library records one CUDA event after each of its launches inside that region (per-kernel "
                      "times); step_ms: per-step spans from those events",
            "step_ms": step_ms, "roofline": roofline, "path": path, "clocks": clk,
            "gpu_launches": launches * args.steps,
            "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": e2e_steps}}
    if rank == 0 and world == 1 and not args.no_cpu_baseline and mode == "bwd":
        v, used, dt, sample = oracle_sample_any(inp)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": used, "kind": "oracle", "sample": sample,
                                "seconds": dt}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pass", dest="mode", default="bwd", choices=list(METRICS),
                    help="bwd: forward recompute + backward (the benchmark metric); fwd: forward only; "
                         "bwd-states: backward from the fp32 chunk states a forward saved; bwd-saved: backward "
                         "from the context kda_chunk_fwd_save kept (reverse pass and gradients only); fwd-save: "
                         "the forward that keeps that context; bwd-fused: bwd with the fused reverse kernel")
    ap.add_argument("--workload", default=WORKLOAD, choices=kda_inputs.WORKLOAD_ORDER,
                    help="the workload of the JSON line (default: the B=8 T=4096 H=HV=32 benchmark)")
    ap.add_argument("--seq-len", type=int, default=None,
                    help="override the tokens per sequence of a dense workload (smaller cases for profiling; not "
                         "the workload's own line)")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the batch size (smaller cases for profiling; not the benchmark workload)")
    args = ap.parse_args()
    if args.seq_len and kda_inputs.WORKLOADS[args.workload].varlen_n:
        ap.error("--seq-len applies to dense workloads only")
    if args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
