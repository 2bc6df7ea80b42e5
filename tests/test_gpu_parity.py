"""GPU parity: the CUDA path against the float64 oracle on the same seeded inputs.

Accept rule for the GEMM (the MatMulNBits pull request's "Validation": abs error
<= 2e-2 * max|out| against an f64 dequant -> GEMM oracle):
    max |Y - Y_ref| <= 2e-2 * max |Y_ref|
The repack is integer work and must match the oracle's layout byte for byte.
Every GPU result is also checked for run-to-run determinism (bit-identical).
"""
import numpy as np
import pytest
import torch

import oracle
from w4a16_inputs import make_case, make_swiglu_case

pytestmark = pytest.mark.gpu
TOL = 2e-2


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def check(Y, ref, label=""):
    y = Y.float().cpu().double().numpy()
    assert np.all(np.isfinite(y)), label
    err = np.abs(y - ref).max()
    bound = TOL * np.abs(ref).max()
    print(f"{label} worst_abs={err:.5f} tol={bound:.5f} rel={err / max(np.abs(ref).max(), 1e-30):.2e} "
          f"mean_abs={np.abs(y - ref).mean():.2e}")
    assert err <= bound, f"{label}: max|Y-Yref|={err} > {bound}"


def upload(c):
    return dict(q_rep=None, q=dev(c.bq), s=dev(c.scales), z=None if c.zp is None else dev(c.zp),
                A=dev(c.A))


# ---------------------------------------------------------------------------
# Repack
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("N,K", [(16, 64), (256, 256), (400, 192), (4096, 4096), (13824, 5120)])
def test_repack_matches_oracle_layout(gpu_lib, N, K):
    w4 = gpu_lib
    bq = np.random.default_rng(N + K).integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    rep = w4.w4a16_repack(dev(bq))
    torch.cuda.synchronize()
    got = rep.cpu().numpy()
    np.testing.assert_array_equal(got, oracle.repack(bq))
    np.testing.assert_array_equal(w4.w4a16_unpack_host(got, N, K), bq)


# ---------------------------------------------------------------------------
# GEMM, small-M path
# ---------------------------------------------------------------------------
def run_gemm(w4, c, split_k=0):
    t = upload(c)
    q_rep = w4.w4a16_repack(t["q"])
    Y = w4.w4a16_gemm(t["A"], q_rep, t["s"], t["z"], c.group, split_k=split_k)
    Y2 = w4.w4a16_gemm(t["A"], q_rep, t["s"], t["z"], c.group, split_k=split_k)
    torch.cuda.synchronize()
    assert torch.equal(Y, Y2), "non-deterministic result"
    return Y


def test_tiny_config(gpu_lib):
    c = make_case(2, 256, 256, 32, seed=0, asym=False)
    check(run_gemm(gpu_lib, c), oracle.gemm(c.A, c.bq, c.scales, None, 32), "tiny")


@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_decode_config(gpu_lib, M):
    c = make_case(M, 4096, 4096, 128, seed=1)
    check(run_gemm(gpu_lib, c), oracle.gemm(c.A, c.bq, c.scales, c.zp, 128), f"decode M={M}")


@pytest.mark.parametrize("M", [1, 2, 4, 8, 16, 32, 64])
def test_mlp_config(gpu_lib, M):
    c = make_case(M, 13824, 5120, 128, seed=2)
    check(run_gemm(gpu_lib, c), oracle.gemm(c.A, c.bq, c.scales, c.zp, 128), f"mlp M={M}")


@pytest.mark.parametrize("M", [1, 2, 7, 16, 33, 64])
@pytest.mark.parametrize("group", [16, 32, 64, 128])
@pytest.mark.parametrize("sdt", [np.float16, np.float32])
@pytest.mark.parametrize("asym", [False, True])
def test_format_sweep(gpu_lib, M, group, sdt, asym):
    c = make_case(M, 5120, 5120, group, seed=3, scale_dtype=sdt, asym=asym)
    check(run_gemm(gpu_lib, c), oracle.gemm(c.A, c.bq, c.scales, c.zp, group),
          f"format M={M} g={group} {np.dtype(sdt).name} asym={asym}")


@pytest.mark.parametrize("split", [1, 2, 3, 4, 5, 6, 7, 8])
def test_forced_split_factors(gpu_lib, split):
    c = make_case(8, 512, 1024, 64, seed=21)
    ref = oracle.gemm(c.A, c.bq, c.scales, c.zp, 64)
    check(run_gemm(gpu_lib, c, split_k=split), ref, f"split={split}")


@pytest.mark.parametrize("M,N,K,group", [(3, 400, 384, 128), (9, 144, 192, 64), (33, 16, 64, 16),
                                         (64, 272, 320, 32), (5, 13824, 64, 64)])
def test_ragged_shapes(gpu_lib, M, N, K, group):
    c = make_case(M, N, K, group, seed=M + N + K)
    check(run_gemm(gpu_lib, c), oracle.gemm(c.A, c.bq, c.scales, c.zp, group), f"ragged {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K,group", [(8, 8192, 28672, 128), (8, 28672, 8192, 64), (1, 8192, 28672, 16),
                                         (300, 8192, 28672, 128), (48, 28672, 8192, 128)])
def test_large_shapes_sampled_rows(gpu_lib, M, N, K, group):
    # 70B-class projections (long K for the down projection): every column of a
    # few token rows against the oracle.
    c = make_case(M, N, K, group, seed=M + K)
    rows = sorted({0, M // 2, M - 1})
    Y = run_gemm(gpu_lib, c)[rows]
    check(Y, oracle.gemm(c.A, c.bq, c.scales, c.zp, group, rows=rows), f"large {M}x{N}x{K} g={group}")


def test_split_results_differ_only_by_rounding(gpu_lib):
    c = make_case(4, 1024, 2048, 128, seed=22)
    Ys = [run_gemm(gpu_lib, c, split_k=s).float() for s in (1, 2, 8)]
    for Y in Ys[1:]:
        assert (Y - Ys[0]).abs().max().item() < 1e-2


# ---------------------------------------------------------------------------
# SwiGLU, fused and unfused
# ---------------------------------------------------------------------------
def run_swiglu(w4, gc, uc, fused):
    A = dev(gc.A)
    gq = w4.w4a16_repack(dev(gc.bq))
    uq = w4.w4a16_repack(dev(uc.bq))
    zg = None if gc.zp is None else dev(gc.zp)
    zu = None if uc.zp is None else dev(uc.zp)
    args = (A, gq, dev(gc.scales), zg, uq, dev(uc.scales), zu, gc.group)
    Y = w4.w4a16_gemm_swiglu(*args, fused=fused)
    Y2 = w4.w4a16_gemm_swiglu(*args, fused=fused)
    torch.cuda.synchronize()
    assert torch.equal(Y, Y2)
    return Y


@pytest.mark.parametrize("M", [1, 8, 33])
@pytest.mark.parametrize("fused", [True, False])
def test_swiglu(gpu_lib, M, fused):
    gc, uc = make_swiglu_case(M, 13824, 5120, 128, seed=4)
    ref = oracle.gemm_swiglu(gc.A, (gc.bq, gc.scales, gc.zp), (uc.bq, uc.scales, uc.zp), 128)
    check(run_swiglu(gpu_lib, gc, uc, fused), ref, f"swiglu M={M} fused={fused}")


@pytest.mark.parametrize("group", [16, 32, 64])
def test_swiglu_groups(gpu_lib, group):
    gc, uc = make_swiglu_case(5, 512, 1024, group, seed=23, scale_dtype=np.float32)
    ref = oracle.gemm_swiglu(gc.A, (gc.bq, gc.scales, gc.zp), (uc.bq, uc.scales, uc.zp), group)
    Yf = run_swiglu(gpu_lib, gc, uc, True)
    Yu = run_swiglu(gpu_lib, gc, uc, False)
    check(Yf, ref, f"swiglu fused g={group}")
    check(Yu, ref, f"swiglu unfused g={group}")
