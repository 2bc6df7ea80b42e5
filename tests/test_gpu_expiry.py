"""The expiry path of the bounded device-side waits, run for real.

Every mbarrier wait in the kernels gives up after a limit (2 s by default),
records W4A16_ERR_TIMEOUT in the device error word, stops issuing work, waits
for the copies and tensor-core operations it already issued and returns. With
the limit set to 0 the first poll that finds a copy still in flight gives up,
so a call runs that path while its bulk copies are genuinely outstanding; every
barrier it waits on is fed (nothing is left to wait forever) and the drain
waits keep their own fixed limit. The tests check that the error comes back
through w4a16_device_error, that reading it clears it, and that the next call
with the default limit matches the oracle (the context stays usable).
"""
import numpy as np
import pytest
import torch

import oracle
from w4a16_inputs import make_case, make_swiglu_case

pytestmark = pytest.mark.gpu


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.fixture
def w4(gpu_lib):
    torch.cuda.synchronize()
    assert gpu_lib.w4a16_device_error() == gpu_lib.W4A16_OK
    yield gpu_lib
    gpu_lib.w4a16_set_wait_limit_ns(gpu_lib.WAIT_LIMIT_DEFAULT_NS)
    gpu_lib.w4a16_set_tuning(0)
    torch.cuda.synchronize()
    gpu_lib.w4a16_device_error()


def expire_then_recover(w4, call, ref):
    w4.w4a16_set_wait_limit_ns(0)
    call()
    torch.cuda.synchronize()
    assert w4.w4a16_device_error() == w4.W4A16_ERR_TIMEOUT
    assert w4.w4a16_device_error() == w4.W4A16_OK  # reading cleared it
    w4.w4a16_set_wait_limit_ns(w4.WAIT_LIMIT_DEFAULT_NS)
    y = call().float().cpu().double().numpy()
    torch.cuda.synchronize()
    assert w4.w4a16_device_error() == w4.W4A16_OK
    err = np.abs(y - ref).max()
    assert err <= 2e-2 * np.abs(ref).max(), err


# Shapes whose CTAs stream more ring stages than their ring holds: the producer
# reuses the first slot before the consumers can have released it (its data is
# still in flight), so that wait is certainly incomplete when first tested.
@pytest.mark.parametrize("M,N,K,split", [(8, 13824, 5120, 0), (8, 4096, 14336, 1), (1, 2048, 28672, 2),
                                         (33, 4096, 14336, 2)])
def test_small_m_wait_expiry(w4, M, N, K, split):
    c = make_case(M, N, K, 128, seed=70 + M)
    A, q, s, z = dev(c.A), w4.w4a16_repack(dev(c.bq)), dev(c.scales), dev(c.zp)
    info = w4.w4a16_gemm_launch_info(M, N, K, 128, split)
    assert info["path"] == w4.W4A16_PATH_SMALL_M
    stages_per_cta = -(-(K // 64 // info["split"]) // 4)
    assert info["stages"] < stages_per_cta, info
    ref = oracle.gemm(c.A, c.bq, c.scales, c.zp, 128)
    expire_then_recover(w4, lambda: w4.w4a16_gemm(A, q, s, z, 128, split_k=split), ref)


@pytest.mark.parametrize("M,N", [(256, 2048), (1024, 13824)])
def test_tcgen05_wait_expiry(w4, M, N):
    K = 5120
    c = make_case(M, N, K, 128, seed=80 + M)
    A, q, s, z = dev(c.A), w4.w4a16_repack(dev(c.bq)), dev(c.scales), dev(c.zp)
    w4.w4a16_set_tuning(-1)
    assert w4.w4a16_gemm_plan(M, N, K, 128)[0] == w4.W4A16_PATH_TCGEN05
    rows = [0, M // 2, M - 1]
    ref = oracle.gemm(c.A, c.bq, c.scales, c.zp, 128, rows=rows)
    full = lambda: w4.w4a16_gemm(A, q, s, z, 128)  # noqa: E731
    w4.w4a16_set_wait_limit_ns(0)
    full()
    torch.cuda.synchronize()
    assert w4.w4a16_device_error() == w4.W4A16_ERR_TIMEOUT
    w4.w4a16_set_wait_limit_ns(w4.WAIT_LIMIT_DEFAULT_NS)
    y = full().float().cpu().double().numpy()
    assert w4.w4a16_device_error() == w4.W4A16_OK
    assert np.abs(y[rows] - ref).max() <= 2e-2 * np.abs(ref).max()


@pytest.mark.parametrize("M,N,K", [(8, 13824, 5120), (300, 1024, 2048)])
def test_swiglu_fused_wait_expiry(w4, M, N, K):
    gc, uc = make_swiglu_case(M, N, K, 64, seed=90 + M)
    args = (dev(gc.A), w4.w4a16_repack(dev(gc.bq)), dev(gc.scales), dev(gc.zp),
            w4.w4a16_repack(dev(uc.bq)), dev(uc.scales), dev(uc.zp), 64)
    ref = oracle.gemm_swiglu(gc.A, (gc.bq, gc.scales, gc.zp), (uc.bq, uc.scales, uc.zp), 64)
    expire_then_recover(w4, lambda: w4.w4a16_gemm_swiglu(*args, fused=True), ref)
