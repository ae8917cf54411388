"""GPU parity: the CUDA library (called through its C ABI) against the fp64
oracle on the same seeded inputs.

Tolerances (per-tensor relative L2, oracle rounded to the output dtype):
5e-3 for bf16 inputs (bf16 tensor-core operands, fp32 accumulation) and 1e-4
for fp32 inputs. Every case, the full-size workloads included, is compared
element by element over whole tensors (the oracle runs on all host cores), at
the sizes and in the launch configuration the benchmark times.
"""
import dataclasses
import functools

import numpy as np
import pytest
import torch

import kda_inputs
import oracle
from tests.util import TOL, rel_l2, round_like, to64

pytestmark = pytest.mark.gpu

GRADS = ("dq", "dk", "dv", "dg", "dbeta", "dh0")


@pytest.fixture(scope="session")
def kda():
    import chunked_gated_delta_10_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    m.build()
    m.load()
    return m


def _cuda(inp):
    c = lambda t: None if t is None else t.cuda().contiguous()
    return dict(q=c(inp.q), k=c(inp.k), v=c(inp.v), g=c(inp.g), beta=c(inp.beta), h0=c(inp.h0), do=c(inp.do),
                dht=c(inp.dht))


def gpu_bwd(kda, inp, states=None):
    x = _cuda(inp)
    out = kda.chunk_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"], scale=inp.scale, h0=x["h0"],
                        dht=x["dht"], cu_seqlens=inp.cu_seqlens, states=states)
    torch.cuda.synchronize()
    return out


def gpu_fwd(kda, inp):
    x = _cuda(inp)
    o, ht, st = kda.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], scale=inp.scale, h0=x["h0"],
                              cu_seqlens=inp.cu_seqlens, output_states=True)
    torch.cuda.synchronize()
    return o, ht, st


def _tol(inp):
    return TOL[inp.spec.dtype]


def _check(name, got, ref64, out_dtype, errs):
    errs[name] = rel_l2(to64(got), round_like(ref64, out_dtype))


def _report(name, errs):
    """One greppable line per workload: the whole-tensor errors behind the error table."""
    import json
    print("PARITY " + json.dumps({"workload": name, **{k: float(v) for k, v in errs.items()}}))


def compare_full(inp, out, ref):
    """Whole-tensor relative L2 of every gradient against the oracle (rounded to the output dtype);
    every tensor is measured before any is asserted, so a failure shows all of them."""
    dt, tol, errs = inp.torch_dtype, _tol(inp), {}
    for key in ("dq", "dk", "dv", "dbeta"):
        _check(key, out[key], ref[key], dt, errs)
    _check("dg", out["dg"], ref["dg"], torch.float32, errs)
    if inp.h0 is not None:
        _check("dh0", out["dh0"], ref["dh0"], torch.float32, errs)
    assert all(e <= tol for e in errs.values()), (errs, tol)
    return errs


# ---------------------------------------------------------------- small cases

SMALL = {
    "t1": dict(B=1, T=1, H=1, HV=1, K=64, V=64),
    "t63": dict(B=2, T=63, H=2, HV=2, K=64, V=64),
    "t64": dict(B=1, T=64, H=1, HV=2, K=128, V=128),
    "t65": dict(B=1, T=65, H=2, HV=2, K=64, V=128),
    "t200_gva": dict(B=2, T=200, H=2, HV=4, K=128, V=64),
    "varlen_empty": dict(B=1, T=0, H=2, HV=2, K=64, V=64, seq_lens=[5, 0, 70, 129, 1]),
    "no_state": dict(B=1, T=150, H=1, HV=1, K=128, V=128, h0=False, dht=False),
}


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("name", list(SMALL))
def test_small_cases_full(kda, name, dtype):
    inp = kda_inputs.small(seed=31, dtype=dtype, **SMALL[name])
    out = gpu_bwd(kda, inp)
    compare_full(inp, out, oracle.run_inputs(inp))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("name", ["t65", "t200_gva", "varlen_empty"])
def test_forward_outputs_and_states(kda, name, dtype):
    inp = kda_inputs.small(seed=32, dtype=dtype, **SMALL[name])
    o, ht, st = gpu_fwd(kda, inp)
    ref = oracle.run_inputs(inp, backward=False, chunk_states=True)
    tol = _tol(inp)
    assert rel_l2(to64(o), round_like(ref["o"], inp.torch_dtype)) <= tol
    assert rel_l2(to64(ht), ref["ht"]) <= tol
    assert rel_l2(to64(st), ref["s_in"]) <= tol


# Tensor-core forward (bf16, K = V = 128): o, ht and the fp32 chunk states.
FWD_TC = {
    "t64": SMALL["t64"],
    "no_state": SMALL["no_state"],
    "varlen_gva": dict(B=1, T=0, H=2, HV=4, K=128, V=128, seq_lens=[130, 1, 0, 64, 200]),
    "many_heads": dict(B=3, T=100, H=64, HV=64, K=128, V=128),
}


@pytest.mark.parametrize("name", list(FWD_TC))
def test_tensor_core_forward(kda, name):
    inp = kda_inputs.small(seed=35, dtype="bf16", **FWD_TC[name])
    o, ht, st = gpu_fwd(kda, inp)
    # the tensor-core path ran; with at most one (sequence, head) sweep per SM each sweep is split by columns
    sweeps, nsm = len(inp.seq_bounds) * FWD_TC[name]["HV"], torch.cuda.get_device_properties(0).multi_processor_count
    lib = kda.load()
    names = [lib.kda_launch_name(i) for i in range(lib.kda_last_launch_count())]
    assert (b"tc_fwd_out_vhalf" if sweeps <= nsm else b"tc_fwd_out") in names, names
    # packed sequences: the sweeps are launched longest first (a ranking launch before them)
    assert (b"tc_seq_order" in names) == (inp.cu_seqlens is not None and len(inp.seq_bounds) > 1), names
    ref = oracle.run_inputs(inp, backward=False, chunk_states=True)
    tol = _tol(inp)
    errs = dict(o=rel_l2(to64(o), round_like(ref["o"], inp.torch_dtype)), ht=rel_l2(to64(ht), ref["ht"]),
                states=rel_l2(to64(st), ref["s_in"]))
    print(name, errs)
    assert all(e <= tol for e in errs.values()), errs


def test_tensor_core_forward_workload(kda):
    inp = _workload("bf16_b1_t2048_h16_k128")
    o, ht, st = gpu_fwd(kda, inp)
    ref = oracle.run_inputs(inp, backward=False, chunk_states=True)
    errs = dict(o=rel_l2(to64(o), round_like(ref["o"], inp.torch_dtype)), ht=rel_l2(to64(ht), ref["ht"]),
                states=rel_l2(to64(st), ref["s_in"]))
    _report("bf16_b1_t2048_h16_k128 forward", errs)
    assert all(e <= _tol(inp) for e in errs.values()), errs


@pytest.mark.parametrize("name", ["varlen_gva", "no_state"])
def test_backward_from_saved_states_is_bitwise_recompute(kda, name):
    """The backward that loads the forward's chunk states (no sequential state
    pass) returns exactly what the recompute path returns."""
    inp = kda_inputs.small(seed=36, dtype="bf16", **FWD_TC[name])
    _, _, st = gpu_fwd(kda, inp)
    rec = gpu_bwd(kda, inp)
    lib = kda.load()
    names = [lib.kda_launch_name(i) for i in range(lib.kda_last_launch_count())]
    # (both state passes in one launch when the batch is small)
    assert b"tc_state_fwd" in names or any(x.startswith(b"tc_state_both") for x in names), names
    sv = gpu_bwd(kda, inp, states=st)
    names = [lib.kda_launch_name(i) for i in range(lib.kda_last_launch_count())]
    assert b"tc_state_load" in names and b"tc_state_fwd" not in names, names
    for key in GRADS:
        if rec[key] is not None:
            assert torch.equal(rec[key], sv[key]), key
    compare_full(inp, sv, oracle.run_inputs(inp))


def _launches(kda):
    lib = kda.load()
    return [lib.kda_launch_name(i) for i in range(lib.kda_last_launch_count())]


def _bwd_from_saved(kda, inp, x, saved):
    out = kda.chunk_bwd_from_saved(x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"], saved, scale=inp.scale,
                                   h0=x["h0"], dht=x["dht"], cu_seqlens=inp.cu_seqlens)
    torch.cuda.synchronize()
    return out


def _check_saved_context(kda, inp, oracle_parity=True):
    """chunk_fwd_save gives the forward's o and ht bit for bit; chunk_bwd_from_saved runs only the reverse
    pass and the gradient kernel and gives the recompute path's gradients bit for bit, twice in a row on
    the same saved buffer; and the oracle agrees."""
    x = _cuda(inp)
    o_ref, ht_ref, _ = gpu_fwd(kda, inp)
    o, ht, saved = kda.chunk_fwd_save(x["q"], x["k"], x["v"], x["g"], x["beta"], scale=inp.scale, h0=x["h0"],
                                      cu_seqlens=inp.cu_seqlens)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(ht, ht_ref)
    rec = gpu_bwd(kda, inp)
    for rep in range(2):
        sv = _bwd_from_saved(kda, inp, x, saved)
        names = _launches(kda)
        assert b"tc_grads" in names and not {b"tc_intra", b"tc_state_fwd", b"tc_state_both",
                                             b"tc_state_both_vhalf"} & set(names), names
        for key in GRADS:
            if rec[key] is not None:
                assert torch.equal(rec[key], sv[key]), (rep, key)
    assert kda.device_status(saved) == 0
    if oracle_parity:
        return compare_full(inp, sv, oracle.run_inputs(inp))


SAVED = {
    "varlen_gva": FWD_TC["varlen_gva"],
    "no_state": FWD_TC["no_state"],
    "t64": SMALL["t64"],
}


@pytest.mark.parametrize("name", list(SAVED))
def test_backward_from_saved_context_is_bitwise_recompute(kda, name):
    _check_saved_context(kda, kda_inputs.small(seed=44, dtype="bf16", **SAVED[name]))


def test_backward_from_saved_context_segmented(kda):
    """A long sequence with few sweeps: the forward runs segmented and keeps every chunk's S_in and delta;
    the backward's reverse pass runs segmented from the saved context."""
    inp = kda_inputs.small(seed=45, B=1, T=8192 + 37, H=1, HV=2, K=128, V=128, dtype="bf16")
    print("saved segmented", _check_saved_context(kda, inp))


def test_backward_from_saved_context_benchmark_workload(kda):
    _check_saved_context(kda, _workload("bf16_b8_t4096_h32_k128"), oracle_parity=False)


def test_saved_states_off_tensor_core_path_is_unsupported(kda):
    inp = kda_inputs.small(seed=37, dtype="f32", **SMALL["t65"])
    _, _, st = gpu_fwd(kda, inp)
    with pytest.raises(kda.KdaError) as err:
        gpu_bwd(kda, inp, states=st)
    assert err.value.code == 2  # KDA_ERR_UNSUPPORTED


def test_segmented_state_passes_long_sequence(kda):
    """A dense batch with few (sequence, head) sweeps over long sequences runs both state passes in
    segments (ends and transitions per segment, their chain, then the checkpoints): full parity."""
    inp = kda_inputs.small(seed=38, B=1, T=8192 + 37, H=1, HV=2, K=128, V=128, dtype="bf16")
    out = gpu_bwd(kda, inp)
    lib = kda.load()
    names = [lib.kda_launch_name(i) for i in range(lib.kda_last_launch_count())]
    assert b"tc_state_fwd_seg" in names and b"tc_ds_rev_seg" in names, names
    print("segmented", compare_full(inp, out, oracle.run_inputs(inp)))


def test_segmented_forward_long_sequence(kda):
    inp = kda_inputs.small(seed=39, B=1, T=8192 + 37, H=1, HV=2, K=128, V=128, dtype="bf16")
    o, ht, st = gpu_fwd(kda, inp)
    lib = kda.load()
    names = [lib.kda_launch_name(i) for i in range(lib.kda_last_launch_count())]
    assert b"tc_state_fwd_seg" in names, names
    ref = oracle.run_inputs(inp, backward=False, chunk_states=True)
    errs = dict(o=rel_l2(to64(o), round_like(ref["o"], inp.torch_dtype)), ht=rel_l2(to64(ht), ref["ht"]),
                states=rel_l2(to64(st), ref["s_in"]))
    print("segmented forward", errs)
    assert all(e <= _tol(inp) for e in errs.values()), errs


# Tensor-core gradient kernel with grouped value heads: a group's G value heads run back to back on one
# CTA, which carries their dq / dk sum; groups of 3 and 4, partial chunks, empty sequences, fewer groups
# than CTAs, and a group count that does not divide among the CTAs.
GROUPED = {
    "g4_one_head": dict(B=1, T=200, H=1, HV=4, K=128, V=128),
    "g3_varlen": dict(B=1, T=0, H=2, HV=6, K=128, V=128, seq_lens=[130, 1, 0, 64, 77]),
    "g2_many_groups": dict(B=2, T=64 * 90 + 5, H=1, HV=2, K=128, V=128),
}


@pytest.mark.parametrize("name", list(GROUPED))
def test_grouped_value_heads_tensor_core(kda, name):
    inp = kda_inputs.small(seed=46, dtype="bf16", **GROUPED[name])
    out = gpu_bwd(kda, inp)
    compare_full(inp, out, oracle.run_inputs(inp))


@pytest.mark.parametrize("dtype,K", [("f32", 64), ("bf16", 128)])
def test_packed_batch_of_empty_sequences(kda, dtype, K):
    """Packed sequences that are all empty own no chunk (chunk_idx is an empty array): the forward returns
    ht = h0 and the backward dh0 = dht exactly (the identity of a sequence with no token), on both paths and,
    for the tensor-core shape, through the fused reverse too."""
    inp = kda_inputs.small(seed=51, B=1, T=0, H=2, HV=2, K=K, V=K, dtype=dtype, seq_lens=[0, 0, 0])
    o, ht, st = gpu_fwd(kda, inp)
    assert o.numel() == 0 and st.numel() == 0
    assert torch.equal(ht.cpu(), inp.h0)
    outs = [gpu_bwd(kda, inp)]
    if dtype == "bf16":
        x = _cuda(inp)
        outs.append(kda.chunk_bwd_fused(x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"], scale=inp.scale,
                                        h0=x["h0"], dht=x["dht"], cu_seqlens=inp.cu_seqlens))
        torch.cuda.synchronize()
    for out in outs:
        assert torch.equal(out["dh0"].cpu(), inp.dht)
        assert all(out[key].numel() == 0 for key in ("dq", "dk", "dv", "dg", "dbeta"))


# ------------------------------------------------------- the five workloads

@functools.lru_cache(maxsize=1)
def _workload(name):
    return kda_inputs.workload(name)


def test_workload_fp32_b1_t256_full(kda):
    inp = _workload("fp32_b1_t256_h2_k64")
    out = gpu_bwd(kda, inp)
    errs = compare_full(inp, out, oracle.run_inputs(inp))
    _report("fp32_b1_t256_h2_k64", errs)


def test_workload_bf16_b1_t2048_full(kda):
    inp = _workload("bf16_b1_t2048_h16_k128")
    out = gpu_bwd(kda, inp)
    errs = compare_full(inp, out, oracle.run_inputs(inp))
    _report("bf16_b1_t2048_h16_k128", errs)


def _full_backward(kda, name):
    inp = _workload(name)
    out = gpu_bwd(kda, inp)
    got = {k: (None if v is None else v.cpu()) for k, v in out.items()}
    del out
    torch.cuda.empty_cache()
    errs = compare_full(inp, got, oracle.run_inputs(inp))
    _report(name, errs)
    return errs


def test_workload_bf16_b8_t4096_full(kda):
    """The benchmark workload (B=8 T=4096 H=HV=32), every element of every gradient."""
    _full_backward(kda, "bf16_b8_t4096_h32_k128")


def test_workload_bf16_varlen_full(kda):
    """16 packed sequences of U[1,4096] tokens, every element of every gradient and of dh0."""
    _full_backward(kda, "bf16_varlen16_h32_k128")


@pytest.mark.slow
def test_workload_bf16_t65536_gva_full(kda):
    """B=1 T=65536 with 16 key heads over 32 value heads (segmented state passes and the grouped
    dq/dk sum), every element of every gradient and of dh0."""
    _full_backward(kda, "bf16_b1_t65536_h16_hv32_k128")


@pytest.mark.parametrize("name", ["bf16_b8_t4096_h32_k128", "bf16_varlen16_h32_k128",
                                  "bf16_b1_t65536_h16_hv32_k128"])
def test_workload_forward_full(kda, name):
    """Forward o, ht and the fp32 chunk states on the large workloads, whole tensors."""
    inp = _workload(name)
    o, ht, st = gpu_fwd(kda, inp)
    o, ht, st = o.cpu(), ht.cpu(), st.cpu()
    torch.cuda.empty_cache()
    ref = oracle.run_inputs(inp, backward=False, chunk_states=True)
    errs = dict(o=rel_l2(to64(o), round_like(ref["o"], inp.torch_dtype)), ht=rel_l2(to64(ht), ref["ht"]),
                states=rel_l2(to64(st), ref["s_in"]))
    _report(name + " forward", errs)
    assert all(e <= _tol(inp) for e in errs.values()), errs


@pytest.mark.parametrize("seed", [11, 12, 13, 14, 15])
def test_workload_bf16_b1_t2048_seeds(kda, seed):
    """The B=1 T=2048 H=16 workload drawn from five more seeds: the bf16 error level is not a
    property of one draw."""
    inp = kda_inputs.make(dataclasses.replace(kda_inputs.WORKLOADS["bf16_b1_t2048_h16_k128"], seed=seed))
    out = gpu_bwd(kda, inp)
    errs = compare_full(inp, out, oracle.run_inputs(inp))
    o, ht, st = gpu_fwd(kda, inp)
    ref = oracle.run_inputs(inp, backward=False, chunk_states=True)
    errs.update(o=rel_l2(to64(o), round_like(ref["o"], inp.torch_dtype)), ht=rel_l2(to64(ht), ref["ht"]),
                states=rel_l2(to64(st), ref["s_in"]))
    _report(f"bf16_b1_t2048_h16_k128 seed {seed}", errs)
    assert all(e <= _tol(inp) for e in errs.values()), errs


# ------------------------------------------------------------ degenerate inputs

DEGENERATE = {
    "fp32_k64": dict(B=1, T=0, H=2, HV=2, K=64, V=64, seq_lens=[70, 1, 33], dtype="f32"),
    "bf16_k128": dict(B=1, T=0, H=2, HV=4, K=128, V=128, seq_lens=[130, 5, 64], dtype="bf16"),
}


@pytest.mark.parametrize("name", list(DEGENERATE))
def test_zero_cotangents_give_exactly_zero_gradients(kda, name):
    """do = 0 and dht = 0: every gradient is exactly zero (an exactly zero reference
    requires an exactly zero result)."""
    inp = kda_inputs.small(seed=41, **DEGENERATE[name])
    inp = dataclasses.replace(inp, do=torch.zeros_like(inp.do), dht=torch.zeros_like(inp.dht))
    out = gpu_bwd(kda, inp)
    for key in GRADS:
        assert torch.count_nonzero(out[key]) == 0, key


@pytest.mark.parametrize("name", list(DEGENERATE))
@pytest.mark.parametrize("case", ["beta_zero", "gate_zero"])
def test_degenerate_gates_match_the_oracle(kda, name, case):
    """beta = 0 (no delta-rule write: the state only decays) and g = 0 (no decay)."""
    inp = kda_inputs.small(seed=42, **DEGENERATE[name])
    if case == "beta_zero":
        inp = dataclasses.replace(inp, beta=torch.zeros_like(inp.beta))
    else:
        inp = dataclasses.replace(inp, g=torch.zeros_like(inp.g))
    out = gpu_bwd(kda, inp)
    errs = compare_full(inp, out, oracle.run_inputs(inp))
    print(name, case, errs)


# ------------------------------------------------------------ invariances

def test_rerun_is_bitwise_identical(kda):
    inp = kda_inputs.small(seed=33, B=1, T=0, H=2, HV=4, K=128, V=128, dtype="bf16", seq_lens=[300, 17, 64])
    a = gpu_bwd(kda, inp)
    b = gpu_bwd(kda, inp)
    for key in GRADS:
        assert torch.equal(a[key], b[key]), key


def test_rerun_is_bitwise_identical_benchmark_workload(kda):
    """The benchmark workload (16,384 chunk-heads, about 108 per persistent CTA, so every CTA runs its
    prefetch pipeline and its producer / SIMT hand-offs many times): two backward runs and two
    forward runs agree bit for bit."""
    inp = _workload("bf16_b8_t4096_h32_k128")
    a = gpu_bwd(kda, inp)
    b = gpu_bwd(kda, inp)
    for key in GRADS:
        if a[key] is not None:
            assert torch.equal(a[key], b[key]), key
    del a, b
    o1, ht1, _ = gpu_fwd(kda, inp)
    o2, ht2, _ = gpu_fwd(kda, inp)
    assert torch.equal(o1, o2) and torch.equal(ht1, ht2)


def test_packed_equals_separate_sequences_bitwise(kda):
    lens = [100, 1, 64, 257]
    inp = kda_inputs.small(seed=34, B=1, T=0, H=2, HV=2, K=128, V=128, dtype="bf16", seq_lens=lens)
    packed = gpu_bwd(kda, inp)
    for n, (b, e) in enumerate(inp.seq_bounds):
        sl = lambda t: t[:, b:e].contiguous()
        one = kda_inputs.Inputs(inp.spec, sl(inp.q), sl(inp.k), sl(inp.v), sl(inp.g), sl(inp.beta),
                                inp.h0[n:n + 1].contiguous(), sl(inp.do), inp.dht[n:n + 1].contiguous(), None,
                                inp.scale)
        single = gpu_bwd(kda, one)
        for key in ("dq", "dk", "dv", "dg", "dbeta"):
            assert torch.equal(single[key][0], packed[key][0, b:e]), (n, key)
        assert torch.equal(single["dh0"][0], packed["dh0"][n]), n
