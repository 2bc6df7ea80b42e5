"""GPU parity of the tensor-core (tcgen05) path against the float64 oracle.

Large M runs on the tcgen05 kernel. At the full MLP sizes the oracle computes a
sample of rows (all columns) one by one; smaller shapes are compared in full.
`w4a16_set_tuning(-1)` routes every M to the tensor-core path so small shapes,
ragged tiles and every group/scale format are covered there too.
Accept rule: max |Y - Y_ref| <= 2e-2 * max |Y_ref| (the MatMulNBits pull
request's "Validation" bound); results must be run-to-run bit-identical.
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


def check(y, ref, label):
    assert np.all(np.isfinite(y)), label
    err = np.abs(y - ref).max()
    bound = TOL * np.abs(ref).max()
    print(f"{label} worst_abs={err:.5f} tol={bound:.5f} mean_abs={np.abs(y - ref).mean():.2e}")
    assert err <= bound, f"{label}: {err} > {bound}"


@pytest.fixture
def tc_only(gpu_lib):
    gpu_lib.w4a16_set_tuning(-1)
    yield gpu_lib
    gpu_lib.w4a16_set_tuning(0)


def run(w4, c, rows=None):
    q = w4.w4a16_repack(dev(c.bq))
    A, s, z = dev(c.A), dev(c.scales), None if c.zp is None else dev(c.zp)
    Y1 = w4.w4a16_gemm(A, q, s, z, c.group)
    Y2 = w4.w4a16_gemm(A, q, s, z, c.group)
    torch.cuda.synchronize()
    assert torch.equal(Y1, Y2), "non-deterministic"
    y = Y1.float().cpu().double().numpy()
    return y if rows is None else y[rows]


@pytest.mark.parametrize("M", [65, 128, 200, 256, 1024, 4096])
def test_mlp_large_m_sampled_rows(gpu_lib, M):
    assert gpu_lib.w4a16_gemm_plan(M, 13824, 5120, 128)[0] == gpu_lib.W4A16_PATH_TCGEN05
    c = make_case(M, 13824, 5120, 128, seed=2)
    rows = sorted(set(np.random.default_rng(M).choice(M, size=min(M, 12), replace=False).tolist()) | {0, M - 1})
    ref = oracle.gemm(c.A, c.bq, c.scales, c.zp, 128, rows=rows)
    check(run(gpu_lib, c, rows), ref, f"tc mlp M={M}")


def test_path_choice(gpu_lib):
    small, tc = gpu_lib.W4A16_PATH_SMALL_M, gpu_lib.W4A16_PATH_TCGEN05
    assert gpu_lib.w4a16_gemm_plan(8, 13824, 5120, 128)[0] == small
    assert gpu_lib.w4a16_gemm_plan(32, 13824, 5120, 128)[0] == small
    assert gpu_lib.w4a16_gemm_plan(33, 13824, 5120, 128)[0] == tc
    # From 33 tokens on, a grid of 108 tiles makes the tensor-core kernel faster ...
    assert gpu_lib.w4a16_gemm_plan(48, 13824, 5120, 128)[0] == tc
    # ... but not one of 32 tiles, and a forced K split keeps the small-M path.
    assert gpu_lib.w4a16_gemm_plan(48, 4096, 4096, 128)[0] == small
    assert gpu_lib.w4a16_gemm_plan(48, 13824, 5120, 128, split_k=2) == (small, 2)


@pytest.mark.parametrize("M", [1, 8, 33, 100, 300])
@pytest.mark.parametrize("group", [16, 32, 64, 128])
@pytest.mark.parametrize("sdt", [np.float16, np.float32])
@pytest.mark.parametrize("asym", [False, True])
def test_formats_forced_tc(tc_only, M, group, sdt, asym):
    c = make_case(M, 256, 1024, group, seed=M + group, scale_dtype=sdt, asym=asym)
    check(run(tc_only, c), oracle.gemm(c.A, c.bq, c.scales, c.zp, group), f"tc M={M} g={group}")


@pytest.mark.parametrize("M,N,K,group", [(70, 400, 384, 128), (257, 144, 192, 64), (96, 16, 64, 16),
                                         (130, 13824, 64, 64)])
def test_ragged_forced_tc(tc_only, M, N, K, group):
    c = make_case(M, N, K, group, seed=M + N + K)
    check(run(tc_only, c), oracle.gemm(c.A, c.bq, c.scales, c.zp, group), f"tc ragged {M}x{N}x{K}")


def test_small_and_tc_paths_agree(gpu_lib):
    c = make_case(40, 512, 2048, 64, seed=77)
    y_small = run(gpu_lib, c)
    gpu_lib.w4a16_set_tuning(-1)
    try:
        y_tc = run(gpu_lib, c)
    finally:
        gpu_lib.w4a16_set_tuning(0)
    ref = oracle.gemm(c.A, c.bq, c.scales, c.zp, 64)
    check(y_small, ref, "small-M path")
    check(y_tc, ref, "tc path")


@pytest.mark.parametrize("M", [256, 1024, 4096, 8192])
@pytest.mark.parametrize("fused", [True, False])
def test_swiglu_large_m(gpu_lib, M, fused):
    gc, uc = make_swiglu_case(M, 13824, 5120, 128, seed=4)
    rows = [0, 1, 17, M // 2, M - 1]
    ref = oracle.gemm_swiglu(gc.A, (gc.bq, gc.scales, gc.zp), (uc.bq, uc.scales, uc.zp), 128, rows=rows)
    A = dev(gc.A)
    args = (A, gpu_lib.w4a16_repack(dev(gc.bq)), dev(gc.scales), dev(gc.zp),
            gpu_lib.w4a16_repack(dev(uc.bq)), dev(uc.scales), dev(uc.zp), 128)
    Y1 = gpu_lib.w4a16_gemm_swiglu(*args, fused=fused)
    Y2 = gpu_lib.w4a16_gemm_swiglu(*args, fused=fused)
    torch.cuda.synchronize()
    assert torch.equal(Y1, Y2)
    check(Y1.float().cpu().double().numpy()[rows], ref, f"tc swiglu M={M} fused={fused}")


@pytest.mark.parametrize("M,N,group", [(20, 384, 32), (150, 384, 16), (300, 384, 128),
                                       (100, 400, 64), (70, 208, 128), (33, 16, 16), (257, 80, 64)])
def test_swiglu_forced_tc(tc_only, M, N, group):
    # N = 400, 208, 80, 16: output halves of 64 columns that end inside a ragged
    # 128-row tile of the repacked layout (or are the whole of one).
    gc, uc = make_swiglu_case(M, N, 512, group, seed=M)
    ref = oracle.gemm_swiglu(gc.A, (gc.bq, gc.scales, gc.zp), (uc.bq, uc.scales, uc.zp), group)
    A = dev(gc.A)
    args = (A, tc_only.w4a16_repack(dev(gc.bq)), dev(gc.scales), dev(gc.zp),
            tc_only.w4a16_repack(dev(uc.bq)), dev(uc.scales), dev(uc.zp), group)
    Y = tc_only.w4a16_gemm_swiglu(*args, fused=True)
    torch.cuda.synchronize()
    check(Y.float().cpu().double().numpy(), ref, f"tc swiglu forced M={M}")


def test_no_device_error_recorded(gpu_lib):
    torch.cuda.synchronize()
    assert gpu_lib.w4a16_device_error() == gpu_lib.W4A16_OK


@pytest.mark.parametrize("M,N,K", [(1, 4096, 4096), (8, 13824, 5120), (32, 13824, 5120), (33, 13824, 5120),
                                   (300, 1024, 2048), (1024, 13824, 5120)])
def test_launch_info_matches_plan(gpu_lib, M, N, K):
    # The launch-shape query reports the plan w4a16_gemm_plan reports, and a grid
    # that covers the output: tiles of 128 columns (64 for fused SwiGLU on the
    # tensor-core path) times the K split (x2 for SwiGLU on the small-M path).
    path, split = gpu_lib.w4a16_gemm_plan(M, N, K, 128)
    info = gpu_lib.w4a16_gemm_launch_info(M, N, K, 128)
    assert (info["path"], info["split"]) == (path, split)
    assert info["threads"] % 32 == 0 and 0 < info["smem_bytes"] <= 227 * 1024 + 1024
    assert info["stages"] >= 2
    if path == gpu_lib.W4A16_PATH_SMALL_M:
        assert info["ctas"] == -(-N // 128) * split
    else:
        T = min(256, -(-M // 16) * 16)
        assert info["ctas"] == -(-M // T) * -(-N // 128)
    fused = gpu_lib.w4a16_gemm_launch_info(M, N, K, 128, 0, True)
    if fused["path"] == gpu_lib.W4A16_PATH_SMALL_M:
        assert fused["ctas"] == -(-N // 128) * fused["split"] * 2
    else:
        assert fused["ctas"] % -(-N // 64) == 0
