"""GPU checks of w4a16_gemm_host_io: the GEMM with activations and output in host memory.

The call enqueues the host-to-device copy of A, the GEMM and the device-to-host
copy of Y on one stream. Its Y must equal, bit for bit, the device-buffer
w4a16_gemm on the same inputs (same kernels, same split), with launch overlap
off and on, on both kernel paths; a small case is also compared with the float64
oracle under the MatMulNBits pull request's "Validation" bound.
"""
import numpy as np
import pytest
import torch

import oracle
from w4a16_inputs import make_case

pytestmark = pytest.mark.gpu


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.fixture
def w4(gpu_lib):
    yield gpu_lib
    gpu_lib.w4a16_set_launch_overlap(False)


@pytest.mark.parametrize("overlap", [False, True])
@pytest.mark.parametrize("M,N,K,group", [(8, 13824, 5120, 128), (1, 4096, 4096, 128), (300, 2048, 1024, 64)])
def test_host_io_matches_device_call(w4, overlap, M, N, K, group):
    c = make_case(M, N, K, group, seed=120 + M)
    q, s, z = w4.w4a16_repack(dev(c.bq)), dev(c.scales), dev(c.zp)
    A_h = torch.from_numpy(c.A).pin_memory()
    Y_h = torch.empty((M, N), dtype=torch.float16).pin_memory()
    A_d = torch.empty((M, K), dtype=torch.float16, device="cuda")
    Y_d = torch.empty((M, N), dtype=torch.float16, device="cuda")
    w4.w4a16_set_launch_overlap(overlap)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for _ in range(3):  # back-to-back calls reuse the same buffers
            w4.w4a16_gemm_host_io(A_h, A_d, q, s, z, group, Y_d, Y_h, stream=stream)
    stream.synchronize()
    ref = w4.w4a16_gemm(dev(c.A), q, s, z, group)
    torch.cuda.synchronize()
    assert torch.equal(A_d.cpu(), A_h)
    assert torch.equal(Y_h, ref.cpu())
    assert w4.w4a16_device_error() == w4.W4A16_OK


def test_host_io_against_oracle(w4):
    c = make_case(8, 256, 512, 64, seed=130)
    q, s, z = w4.w4a16_repack(dev(c.bq)), dev(c.scales), dev(c.zp)
    A_h = torch.from_numpy(c.A).pin_memory()
    Y_h = torch.zeros((8, 256), dtype=torch.float16).pin_memory()
    A_d = torch.empty((8, 512), dtype=torch.float16, device="cuda")
    Y_d = torch.empty((8, 256), dtype=torch.float16, device="cuda")
    w4.w4a16_gemm_host_io(A_h, A_d, q, s, z, 64, Y_d, Y_h)
    torch.cuda.synchronize()
    ref = oracle.gemm(c.A, c.bq, c.scales, c.zp, 64)
    y = Y_h.float().double().numpy()
    err = np.abs(y - ref).max()
    assert err <= 2e-2 * np.abs(ref).max(), err
