"""GPU parity of the RMS-norm prologue entry points against the float64 oracle.

The prologue (the pull request github.com/justinchuby/onnx-genai pull 960,
"Update -- fused RMS-norm epilogue + e2e PASS" and "Update -- P1 COMPLETE")
normalises each activation row, stages it, then runs the GEMM or the gate/up
SwiGLU on it. Checked against oracle.gemm_rmsnorm / gemm_swiglu_rmsnorm with
the same bound as the GEMM (2e-2 * max|Y_ref|), on both kernels, for every
group size, fused and unfused SwiGLU, run-to-run bit identity and launch
overlap on/off bit identity.
"""
import numpy as np
import pytest
import torch

import oracle
from w4a16_inputs import draw_norm_weight, make_case, make_swiglu_case

pytestmark = pytest.mark.gpu
TOL = 2e-2


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def check(y, ref, label):
    err = np.abs(y - ref).max()
    bound = TOL * np.abs(ref).max()
    print(f"{label} worst_abs={err:.5f} tol={bound:.5f}")
    assert np.all(np.isfinite(y)) and err <= bound, f"{label}: {err} > {bound}"


@pytest.fixture
def w4(gpu_lib):
    yield gpu_lib
    gpu_lib.w4a16_set_launch_overlap(False)


@pytest.mark.parametrize("M,N,K,group,eps", [(1, 4096, 4096, 128, 1e-5), (8, 13824, 5120, 128, 1e-6),
                                             (33, 512, 2048, 32, 1e-5), (5, 400, 768, 16, 0.1),
                                             (256, 2048, 1024, 64, 1e-5), (1024, 13824, 5120, 128, 1e-5)])
def test_gemm_rmsnorm(w4, M, N, K, group, eps):
    c = make_case(M, N, K, group, seed=200 + M)
    gamma = draw_norm_weight(np.random.default_rng(M), K)
    q = w4.w4a16_repack(dev(c.bq))
    args = (dev(c.A), dev(gamma), eps, q, dev(c.scales), dev(c.zp), group)
    Y1 = w4.w4a16_gemm_rmsnorm(*args)
    Y2 = w4.w4a16_gemm_rmsnorm(*args)
    w4.w4a16_set_launch_overlap(True)
    Y3 = w4.w4a16_gemm_rmsnorm(*args)
    torch.cuda.synchronize()
    assert torch.equal(Y1, Y2) and torch.equal(Y1, Y3)
    rows = None if M <= 64 else sorted({0, 1, M // 2, M - 1})
    ref = oracle.gemm_rmsnorm(c.A, gamma, eps, c.bq, c.scales, c.zp, group, rows=rows)
    y = Y1.float().cpu().double().numpy()
    check(y if rows is None else y[rows], ref, f"rmsnorm gemm M={M} N={N} K={K} g={group}")
    assert w4.w4a16_device_error() == w4.W4A16_OK


@pytest.mark.parametrize("M", [8, 300])
@pytest.mark.parametrize("fused", [True, False])
def test_swiglu_rmsnorm(w4, M, fused):
    N, K, group = 1024, 2048, 64
    gc, uc = make_swiglu_case(M, N, K, group, seed=300 + M)
    gamma = draw_norm_weight(np.random.default_rng(M + 1), K)
    args = (dev(gc.A), dev(gamma), 1e-5, w4.w4a16_repack(dev(gc.bq)), dev(gc.scales), dev(gc.zp),
            w4.w4a16_repack(dev(uc.bq)), dev(uc.scales), dev(uc.zp), group)
    Y1 = w4.w4a16_gemm_swiglu_rmsnorm(*args, fused=fused)
    Y2 = w4.w4a16_gemm_swiglu_rmsnorm(*args, fused=fused)
    torch.cuda.synchronize()
    assert torch.equal(Y1, Y2)
    ref = oracle.gemm_swiglu_rmsnorm(gc.A, gamma, 1e-5, (gc.bq, gc.scales, gc.zp), (uc.bq, uc.scales, uc.zp),
                                     group)
    check(Y1.float().cpu().double().numpy(), ref, f"rmsnorm swiglu M={M} fused={fused}")


def test_rmsnorm_of_scaled_rows_matches(w4):
    # Scaling a row by a power of two leaves the normalised activation, and so Y,
    # unchanged (the definition is scale-free for eps = 0).
    M, N, K, group = 8, 1024, 2048, 128
    c = make_case(M, N, K, group, seed=7)
    gamma = draw_norm_weight(np.random.default_rng(3), K)
    q = w4.w4a16_repack(dev(c.bq))
    A2 = (c.A.astype(np.float32) * 4.0).astype(np.float16)
    Ya = w4.w4a16_gemm_rmsnorm(dev(c.A), dev(gamma), 0.0, q, dev(c.scales), dev(c.zp), group)
    Yb = w4.w4a16_gemm_rmsnorm(dev(A2), dev(gamma), 0.0, q, dev(c.scales), dev(c.zp), group)
    torch.cuda.synchronize()
    assert torch.equal(Ya, Yb)
