"""GPU: the fused reverse (kda_chunk_bwd_fused: the reverse state-gradient sweep and the per-chunk
gradients in one launch, a cluster of three CTAs per (sequence, head), the sweep CTA passing dS_out and
d_delta to two gradient CTAs through shared memory) against the split backward (kda_chunk_bwd) bit for
bit, and against the fp64 oracle over whole tensors.

The two paths run the same arithmetic on the same operand values (the sweep CTA forms each chunk's
dS_out and d_delta tiles exactly as the split reverse pass does), so every gradient must be equal, not
merely close. Cases: a single token (one gradient CTA without chunks), one exact chunk, ragged tails,
packed sequences with empty and length-1 members, no initial state and no dht, a long sequence whose
forward state pass runs in segments, and the benchmark-sized workloads.
"""
import functools

import pytest
import torch

import kda_inputs
import oracle
from tests.test_gpu_parity import GRADS, _cuda, compare_full, gpu_bwd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="session")
def kda():
    import chunked_gated_delta_10_gb300 as m
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    m.build()
    m.load()
    return m


def _launches(kda):
    lib = kda.load()
    return [lib.kda_launch_name(i) for i in range(lib.kda_last_launch_count())]


def fused_bwd(kda, inp, ws=None, states=None):
    x = _cuda(inp)
    out = kda.chunk_bwd_fused(x["q"], x["k"], x["v"], x["g"], x["beta"], x["do"], scale=inp.scale, h0=x["h0"],
                              dht=x["dht"], cu_seqlens=inp.cu_seqlens, states=states, ws=ws)
    torch.cuda.synchronize()
    return out


def _workspace(kda, inp):
    dims = kda.make_dims(_cuda(inp)["q"], _cuda(inp)["v"], inp.scale, inp.cu_seqlens)
    return torch.empty(kda.workspace_bytes(dims, kda.PASS_BWD), dtype=torch.uint8, device="cuda")


def _check_bitwise(kda, inp, reps=2):
    """The fused path, twice on one workspace, equals the split path bit for bit; clean status word.
    (With at most one (sequence, head) sweep per SM the split path runs its two state passes as one launch,
    tc_state_both, and with at most one per two SMs splits each sweep by columns over two CTAs,
    tc_state_both_vhalf; the fused path runs tc_state_fwd on its own.)"""
    split = gpu_bwd(kda, inp)
    split_names = _launches(kda)
    ws = _workspace(kda, inp)
    for rep in range(reps):
        got = fused_bwd(kda, inp, ws=ws)
        names = _launches(kda)
        assert b"tc_rev_fused" in names and b"tc_ds_rev" not in names and b"tc_grads" not in names, names
        assert kda.device_status(ws) == 0
        for key in GRADS:
            if split[key] is None:
                assert got[key] is None, key
            else:
                assert torch.equal(split[key], got[key]), (rep, key)
    return got, split_names


FUSED = {
    "t1": dict(B=1, T=1, H=1, HV=1, K=128, V=128),
    "t64": dict(B=1, T=64, H=2, HV=2, K=128, V=128),
    "ragged": dict(B=2, T=64 * 5 + 17, H=2, HV=2, K=128, V=128),
    "varlen": dict(B=1, T=0, H=2, HV=2, K=128, V=128, seq_lens=[130, 1, 0, 64, 77, 0]),
    "no_state": dict(B=1, T=150, H=1, HV=1, K=128, V=128, h0=False, dht=False),
    "many_sweeps": dict(B=3, T=64 * 3 + 40, H=64, HV=64, K=128, V=128),
    "sweeps_100": dict(B=2, T=64 * 2 + 9, H=50, HV=50, K=128, V=128),
}


@pytest.mark.parametrize("name", list(FUSED))
def test_fused_reverse_bitwise_and_oracle(kda, name):
    inp = kda_inputs.small(seed=47, dtype="bf16", **FUSED[name])
    got, split_names = _check_bitwise(kda, inp)
    # the split path's state passes: side by side with each sweep split by columns up to one sweep per two SMs,
    # side by side up to one per SM, else one after the other
    sweeps, nsm = len(inp.seq_bounds) * FUSED[name]["HV"], torch.cuda.get_device_properties(0).multi_processor_count
    want = (b"tc_state_both_vhalf" if 2 * sweeps <= nsm else b"tc_state_both" if sweeps <= nsm
            else b"tc_state_fwd")
    assert want in split_names, (sweeps, split_names)
    print(name, compare_full(inp, got, oracle.run_inputs(inp)))


def test_fused_reverse_long_sequence(kda):
    """129 chunks in one sweep, after a segmented forward state pass."""
    inp = kda_inputs.small(seed=48, B=1, T=8192 + 37, H=1, HV=1, K=128, V=128, dtype="bf16")
    got, _ = _check_bitwise(kda, inp, reps=1)
    print("long", compare_full(inp, got, oracle.run_inputs(inp)))


def test_fused_reverse_with_saved_states(kda):
    """With the forward's fp32 chunk states (the chunk-parallel state load) the fused path equals the
    split path given the same states."""
    inp = kda_inputs.small(seed=49, dtype="bf16", **FUSED["varlen"])
    x = _cuda(inp)
    _, _, st = kda.chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], scale=inp.scale, h0=x["h0"],
                             cu_seqlens=inp.cu_seqlens, output_states=True)
    split = gpu_bwd(kda, inp, states=st)
    got = fused_bwd(kda, inp, states=st)
    names = _launches(kda)
    assert b"tc_state_load" in names and b"tc_rev_fused" in names, names
    for key in GRADS:
        assert torch.equal(split[key], got[key]), key


@functools.lru_cache(maxsize=1)
def _workload(name):
    return kda_inputs.workload(name)


@pytest.mark.parametrize("name", ["bf16_b1_t2048_h16_k128", "bf16_b8_t4096_h32_k128", "bf16_varlen16_h32_k128"])
def test_fused_reverse_workloads_bitwise(kda, name):
    """The workloads with equal key and value heads, in the launch configuration the benchmark times:
    bit for bit the split path's gradients (whose whole-tensor oracle parity the parity tests check)."""
    inp = _workload(name)
    got, split_names = _check_bitwise(kda, inp, reps=1)
    side_by_side = name == "bf16_b1_t2048_h16_k128"  # 16 sweeps (each split by columns); the others 256, 512
    assert (b"tc_state_both_vhalf" in split_names) == side_by_side, split_names
    assert (b"tc_ds_rev" in split_names) != side_by_side, split_names
    if name == "bf16_b1_t2048_h16_k128":
        print(name, compare_full(inp, {k: (None if v is None else v.cpu()) for k, v in got.items()},
                                 oracle.run_inputs(inp)))


def test_fused_reverse_unsupported_cases(kda):
    """Grouped value heads (the dq/dk group sum runs across sweeps) and the fp32 path are refused
    before any launch."""
    for dtype, dims in (("bf16", dict(B=1, T=100, H=1, HV=2, K=128, V=128)),
                        ("f32", dict(B=1, T=100, H=2, HV=2, K=64, V=64))):
        inp = kda_inputs.small(seed=50, dtype=dtype, **dims)
        with pytest.raises(kda.KdaError) as err:
            fused_bwd(kda, inp)
        assert err.value.code == 2, (dtype, dims)  # KDA_ERR_UNSUPPORTED
