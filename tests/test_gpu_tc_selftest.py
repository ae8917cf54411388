"""GPU checks of the tensor-core building blocks (tcgen05.mma over 128-byte
swizzled shared-memory tiles, K-major and MN-major operands, TMA loads, TMEM
read-back) against a host matmul of the same bf16 values."""
import ctypes
import itertools

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import chunked_gated_delta_10_gb300 as kda

    kda.build()
    lib = kda.load()
    lib.kda_selftest_umma.restype = ctypes.c_int
    lib.kda_selftest_umma.argtypes = [ctypes.c_int32] * 4 + [ctypes.c_void_p] * 5
    return lib


def _run(lib, M, N, Kd, mode, seed=0):
    g = torch.Generator().manual_seed(seed)
    A = torch.randn(M, Kd, generator=g).to(torch.bfloat16)  # logical A[m, k]
    B = torch.randn(N, Kd, generator=g).to(torch.bfloat16)  # logical B[n, k]
    a_dev = (A.t() if mode & 1 else A).contiguous().cuda()
    b_dev = (B.t() if mode & 2 else B).contiguous().cuda()
    raw = torch.zeros(128, N, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.kda_selftest_umma(M, N, Kd, mode, a_dev.data_ptr(), b_dev.data_ptr(), raw.data_ptr(),
                               status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "bounded wait gave up"
    ref = (A.double() @ B.double().t()).numpy()
    return raw.cpu().double().numpy(), ref


@pytest.mark.parametrize("N,Kd,mode", list(itertools.product([64, 128, 256], [64, 128], [0, 1, 2, 3, 4, 6])))
def test_m128_layouts(lib, N, Kd, mode):
    raw, ref = _run(lib, 128, N, Kd, mode)
    err = np.abs(raw - ref).max() / np.abs(ref).max()
    assert err < 1e-5, err


# Accumulator rows of an M = 64 MMA live in lanes 16 of each 32-lane quarter:
# row r -> lane 32 * (r // 16) + r % 16.
M64_LANES = np.array([32 * (r // 16) + r % 16 for r in range(64)])


@pytest.mark.parametrize("N,Kd,mode", [(64, 128, 0), (128, 64, 3), (256, 128, 1), (64, 64, 2), (128, 128, 4)])
def test_m64_lane_layout(lib, N, Kd, mode):
    raw, ref = _run(lib, 64, N, Kd, mode, seed=1)
    err = np.abs(raw[M64_LANES] - ref).max() / np.abs(ref).max()
    alt = np.abs(raw[:64] - ref).max() / np.abs(ref).max()
    print(f"M=64 N={N} Kd={Kd} mode={mode}: quarter-lane layout err {err:.2e}, lanes 0..63 err {alt:.2e}")
    assert err < 1e-5


def test_bounded_wait_reports_timeout_and_context_stays_usable(lib):
    """A device wait on a barrier that nothing completes gives up, records a
    status code the host reads, and leaves the CUDA context usable."""
    A = torch.zeros(128, 64, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    raw = torch.zeros(128, 64, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.kda_selftest_umma(128, 64, 64, 8, A.data_ptr(), B.data_ptr(), raw.data_ptr(), status.data_ptr(),
                               torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 7
    got, ref = _run(lib, 128, 64, 64, 0)  # the next launch on the same context works
    assert np.abs(got - ref).max() / np.abs(ref).max() < 1e-5
