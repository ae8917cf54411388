"""The benchmark's algorithmic cost model (the numerators of its roofline fractions), checked on the CPU
against the per-unit figures worked out by hand from the tensor sizes: 4,868 bytes per token-head for a
backward step at K = V = 128 in bf16, and each tensor-core kernel's bytes per chunk-head."""
import bench

B, T, H, K, C = 8, 4096, 32, 128, 64
NCK = B * (T // C) * H  # 16,384 chunk-heads


def test_step_bytes_per_token_head():
    s = bench.step_cost(B, T, H, H, K, K)
    # in: q, k, v, do 256 B each, g 512, beta 2; out: dq, dk, dv 256 each, dg 512, dbeta 2; fp32 state 2 x 1024
    assert s["bytes"] == B * T * H * (4 * 256 + 512 + 2 + 3 * 256 + 512 + 2 + 2 * 1024)
    assert s["nck"] == NCK
    assert abs(s["bytes"] / 1e9 - 5.104) < 1e-3
    assert s["flops"] == NCK * (16 * C * K * K + 9 * C * C * K + 5 * C * C * K + C ** 3)


def _kb_per_chunk_head(name):
    bound, b, _ = bench.kernel_cost(name, B, T, H, H, K, K)
    assert bound == "hbm"
    return b / NCK / 1024


def test_tensor_core_kernel_bytes():
    # tc_intra: q, k 16 KB each, g 32 KB, beta 128 B in; w, K^, scale Q~ 16 KB each, Aqk, INV, INV diag(beta)
    # 8 KB each, e^Gamma_C 512 B out
    assert _kb_per_chunk_head("tc_intra") == (2 * 16 + 32 + 0.125) + (3 * 16 + 3 * 8 + 0.5)
    # tc_state_fwd: w, V, K^ 16 KB each, INV diag(beta) 8 KB, e^Gamma_C 512 B in; S_in 32 KB, delta 16 KB out
    assert _kb_per_chunk_head("tc_state_fwd") == 3 * 16 + 8 + 0.5 + 32 + 16
    # tc_ds_rev: K^, scale Q~, w, dO 16 KB each, Aqk 8 KB, e^Gamma_C in; dS_out 32 KB, d_delta 16 KB out
    assert _kb_per_chunk_head("tc_ds_rev") == 4 * 16 + 8 + 0.5 + 32 + 16
    # tc_grads: q, k, v, g, beta, dO, delta, d_delta, S_in, dS_out, INV, e^Gamma_C in; dq, dk, dv, dg, dbeta out
    grads_in = (3 * 16 + 32 + 0.125) + 16 + 2 * 16 + 2 * 32 + 8 + 0.5
    grads_out = 3 * 16 + 32 + 0.125
    assert _kb_per_chunk_head("tc_grads") == grads_in + grads_out == 280.75
    # the fused reverse: both kernels' inputs without dS_out and d_delta (dO and e^Gamma_C once), tc_grads' outputs
    fused_in = (3 * 16 + 32 + 0.125) + 16 + 16 + 32 + 8 + 0.5 + (3 * 16 + 8)
    assert _kb_per_chunk_head("tc_rev_fused") == fused_in + grads_out == 288.75


def test_forward_and_state_load_bytes():
    # tc_fwd_out: w, V, K^, scale Q~ 16 KB each, INV diag(beta), Aqk 8 KB each, e^Gamma_C in; o 16 KB out
    assert _kb_per_chunk_head("tc_fwd_out") == 4 * 16 + 2 * 8 + 0.5 + 16
    # tc_state_load: the fp32 state 64 KB, w, V 16 KB each, INV diag(beta) 8 KB in; S_in 32 KB, delta 16 KB out
    assert _kb_per_chunk_head("tc_state_load") == 64 + 2 * 16 + 8 + 32 + 16


def test_merged_state_passes_bytes():
    both = _kb_per_chunk_head("tc_state_fwd") + _kb_per_chunk_head("tc_ds_rev")
    assert _kb_per_chunk_head("tc_state_both") == _kb_per_chunk_head("tc_state_both_vhalf") == both

    for name in ("tc_state_fwd", "tc_ds_rev"):
        assert _kb_per_chunk_head(name + "_vhalf") == _kb_per_chunk_head(name)
