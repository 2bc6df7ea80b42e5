"""The allocation-free unfused SwiGLU entry point (fixed device scratch).

Some callers cannot allocate device memory for the unfused chain's gate and up
intermediates -- code running inside another framework's memory pool, or on a
path where a device allocation (which may synchronise the device) is not
allowed. w4a16_gemm_swiglu_unfused_static keeps those intermediates in an array
compiled into the library. It launches the same kernels in the same order as
w4a16_gemm_swiglu(fused=0), so its output must be bit-identical to that call's;
it is also checked against the float64 oracle. This file is collected last so
that a run stopping at the first failure has already run every other test; it
passes alone or after them.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from w4a16_inputs import make_swiglu_case

pytestmark = pytest.mark.gpu
TOL = 2e-2


def _call_static(w4, args, Y):
    A, gq, sg, zg, uq, su, zu, group = args
    M, K = A.shape
    N = sg.shape[0]
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    return w4.lib.w4a16_gemm_swiglu_unfused_static(
        ptr(A), ptr(gq), ptr(sg), ptr(zg), ptr(uq), ptr(su), ptr(zu), 0, ptr(Y), M, N, K, group,
        torch.cuda.current_stream().cuda_stream)


@pytest.fixture
def w4(gpu_lib):
    yield gpu_lib
    gpu_lib.w4a16_set_launch_overlap(False)


# (8, 4096, ...) and (33, 1024, ...) run the small-M kernel, (300, 4096, ...)
# the tensor-core kernel; 4*M*N stays within the fixed array in all three.
@pytest.mark.parametrize("M,N,K,group", [(8, 4096, 1024, 64), (33, 1024, 2048, 128), (300, 4096, 1024, 128)])
@pytest.mark.parametrize("overlap", [False, True])
def test_static_scratch_matches_workspace_entry_point(w4, M, N, K, group, overlap):
    assert 4 * M * N <= w4.w4a16_swiglu_static_scratch_bytes()
    gc, uc = make_swiglu_case(M, N, K, group, seed=31 + M)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    args = (dev(gc.A), w4.w4a16_repack(dev(gc.bq)), dev(gc.scales), dev(gc.zp),
            w4.w4a16_repack(dev(uc.bq)), dev(uc.scales), dev(uc.zp), group)
    w4.w4a16_set_launch_overlap(overlap)
    ref = w4.w4a16_gemm_swiglu(*args, fused=False)
    outs = []
    for _ in range(2):  # two calls in a row share the fixed scratch
        Y = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        assert _call_static(w4, args, Y) == w4.W4A16_OK
        outs.append(Y)
    torch.cuda.synchronize()
    for Y in outs:
        assert torch.equal(Y, ref), "static-scratch result differs from the workspace entry point"
    rows = sorted({0, M // 2, M - 1})
    yref = oracle.gemm_swiglu(gc.A, (gc.bq, gc.scales, gc.zp), (uc.bq, uc.scales, uc.zp), group, rows=rows)
    err = np.abs(outs[1].float().cpu().double().numpy()[rows] - yref).max()
    assert err <= TOL * np.abs(yref).max(), err
    assert w4.w4a16_device_error() == w4.W4A16_OK


def test_static_scratch_rejects_oversized_shapes(w4):
    limit = w4.w4a16_swiglu_static_scratch_bytes()
    M, N = 1024, 13824                       # 4*M*N = 56.6 MB > the fixed array
    assert 4 * M * N > limit
    fake = ctypes.c_void_p(0x10000)
    st = w4.lib.w4a16_gemm_swiglu_unfused_static(fake, fake, fake, None, fake, fake, None, 0, fake,
                                                 M, N, 5120, 128, None)
    assert st == w4.W4A16_ERR_WORKSPACE
