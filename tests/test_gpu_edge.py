"""GPU parity on the method's edge cases, on both kernels.

Random N(0,1) activations with uniform nibbles hide the numerically delicate
step of the small-M kernel: it accumulates (1024 + f*q)*a on the tensor cores
and subtracts (s/f)*(1024 + f*zp) times the group's activation sum afterwards,
so a large activation mean cancels two large fp32 terms. These cases exercise
that and the structural special cases of the definition
    Y = A . W^T,   W[n,k] = (q[n,k] - zp[n,k/g]) * s[n,k/g]
(the MatMulNBits pull request, github.com/justinchuby/onnx-genai pull 960,
"What's landed" and "Validation"):
  * zp == q in every group: Y == 0 exactly in the oracle; the GPU result is
    bounded by 2e-2 * max|Y_ref| of a random case with the same activations;
  * one-hot activation rows: Y[m, :] is one dequantised weight column;
  * constant weights: Y = s * (q - zp) * rowsum(A);
  * activations with a large mean (N(4, 1)) and large magnitude (N(500, 50)).
Each runs on the small-M path (every forced split 1..8 for the first two), on
the tensor-core path (w4a16_set_tuning(-1)), and through SwiGLU fused and
unfused. Inputs are built here from seeded numpy draws; expected values come
from the oracle only.
"""
import numpy as np
import pytest
import torch

import oracle
from w4a16_inputs import draw_activations, make_case, make_swiglu_case

pytestmark = pytest.mark.gpu
TOL = 2e-2


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def pack(q):
    """Nibbles [N][K] -> input-format bytes [N][K/2] (low nibble = even k)."""
    q = q.astype(np.uint8)
    return (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)


def zp_equal_q(N, K, group, seed):
    """Weights whose nibbles equal their group's zero point."""
    rng = np.random.default_rng(seed)
    G = K // group
    v = rng.integers(0, 16, size=(N, G))
    bq = pack(np.repeat(v, group, axis=1))
    vz = np.zeros((N, 2 * ((G + 1) // 2)), dtype=np.int64)
    vz[:, :G] = v
    zp = pack(vz)
    s = rng.uniform(0.005, 0.02, size=(N, G)).astype(np.float16)
    return bq, s, zp


def constant_weights(N, K, group, seed, q=11, z=3):
    rng = np.random.default_rng(seed)
    G = K // group
    bq = np.full((N, K // 2), q | (q << 4), dtype=np.uint8)
    zp = np.full((N, (G + 1) // 2), z | (z << 4), dtype=np.uint8)
    srow = rng.uniform(0.005, 0.02, size=N).astype(np.float16)
    s = np.repeat(srow[:, None], G, axis=1)
    return bq, s, zp


def one_hot_rows(M, K, seed):
    rng = np.random.default_rng(seed)
    A = np.zeros((M, K), dtype=np.float16)
    cols = rng.choice(K, size=M, replace=False)
    A[np.arange(M), cols] = 1.0
    return A


def large_mean(M, K, seed, mean, std):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((M, K)) * std + mean).astype(np.float16)


def gemm(w4, A, bq, s, zp, group, split_k=0):
    q = w4.w4a16_repack(dev(bq))
    args = (dev(A), q, dev(s), None if zp is None else dev(zp), group)
    Y1 = w4.w4a16_gemm(*args, split_k=split_k)
    Y2 = w4.w4a16_gemm(*args, split_k=split_k)
    torch.cuda.synchronize()
    assert torch.equal(Y1, Y2), "non-deterministic"
    y = Y1.float().cpu().double().numpy()
    assert np.all(np.isfinite(y))
    return y


def check(y, ref, label, bound=None):
    err = np.abs(y - ref).max()
    if bound is None:
        bound = TOL * np.abs(ref).max()
    print(f"{label} worst_abs={err:.6f} bound={bound:.6f}")
    assert err <= bound, f"{label}: {err} > {bound}"


@pytest.fixture(params=["small_m", "tcgen05"])
def path(request, gpu_lib):
    if request.param == "tcgen05":
        gpu_lib.w4a16_set_tuning(-1)
    yield request.param
    gpu_lib.w4a16_set_tuning(0)


SHAPES = [(8, 1024, 2048, 128), (3, 512, 1024, 64), (16, 256, 1024, 32), (1, 400, 768, 16)]


@pytest.mark.parametrize("M,N,K,group", SHAPES)
def test_zp_equal_q_gives_zero(gpu_lib, path, M, N, K, group):
    w4 = gpu_lib
    bq, s, zp = zp_equal_q(N, K, group, seed=M + N)
    A = large_mean(M, K, seed=K, mean=4.0, std=1.0)
    ref = oracle.gemm(A, bq, s, zp, group)
    assert np.all(ref == 0.0)
    comp = make_case(M, N, K, group, seed=M + K)
    bound = TOL * np.abs(oracle.gemm(A, comp.bq, comp.scales, comp.zp, group)).max()
    check(gemm(w4, A, bq, s, zp, group), ref, f"{path} zp==q {M}x{N}x{K} g={group}", bound)


@pytest.mark.parametrize("M,N,K,group", SHAPES)
def test_one_hot_rows_select_weight_columns(gpu_lib, path, M, N, K, group):
    w4 = gpu_lib
    c = make_case(M, N, K, group, seed=N + group)
    A = one_hot_rows(M, K, seed=M)
    ref = oracle.gemm(A, c.bq, c.scales, c.zp, group)
    W = oracle.dequant(c.bq, c.scales, c.zp, K, group)
    np.testing.assert_array_equal(ref, W[:, np.argmax(A, axis=1)].T)
    check(gemm(w4, A, c.bq, c.scales, c.zp, group), ref, f"{path} one-hot {M}x{N}x{K} g={group}")


@pytest.mark.parametrize("M,N,K,group", SHAPES)
def test_constant_weights(gpu_lib, path, M, N, K, group):
    w4 = gpu_lib
    bq, s, zp = constant_weights(N, K, group, seed=K)
    A = draw_activations(np.random.default_rng(M), M, K)
    ref = oracle.gemm(A, bq, s, zp, group)
    check(gemm(w4, A, bq, s, zp, group), ref, f"{path} constant {M}x{N}x{K} g={group}")


@pytest.mark.parametrize("mean,std", [(4.0, 1.0), (500.0, 50.0), (0.0, 500.0)])
@pytest.mark.parametrize("M,N,K,group", [(8, 1024, 5120, 128), (5, 256, 2048, 16), (33, 512, 1024, 64)])
def test_large_mean_and_magnitude_activations(gpu_lib, path, mean, std, M, N, K, group):
    w4 = gpu_lib
    c = make_case(M, N, K, group, seed=3 * M + K)
    A = large_mean(M, K, seed=M, mean=mean, std=std)
    ref = oracle.gemm(A, c.bq, c.scales, c.zp, group)
    while np.abs(ref).max() >= 3e4:  # keep Y inside fp16: halve A (exact) until it is
        A = (A.astype(np.float32) * 0.5).astype(np.float16)
        ref = oracle.gemm(A, c.bq, c.scales, c.zp, group)
    check(gemm(w4, A, c.bq, c.scales, c.zp, group), ref,
          f"{path} A~N({mean},{std}) {M}x{N}x{K} g={group}")


@pytest.mark.parametrize("split", [1, 2, 3, 4, 5, 6, 7, 8])
def test_edge_cases_every_split(gpu_lib, split):
    w4 = gpu_lib
    M, N, K, group = 8, 512, 2048, 64
    A = large_mean(M, K, seed=split, mean=4.0, std=1.0)
    bq, s, zp = zp_equal_q(N, K, group, seed=split)
    comp = make_case(M, N, K, group, seed=40 + split)
    bound = TOL * np.abs(oracle.gemm(A, comp.bq, comp.scales, comp.zp, group)).max()
    check(gemm(w4, A, bq, s, zp, group, split_k=split), np.zeros((M, N)), f"split {split} zp==q", bound)
    Ah = one_hot_rows(M, K, seed=split)
    check(gemm(w4, Ah, comp.bq, comp.scales, comp.zp, group, split_k=split),
          oracle.gemm(Ah, comp.bq, comp.scales, comp.zp, group), f"split {split} one-hot")
    Al = large_mean(M, K, seed=split, mean=500.0, std=50.0)
    check(gemm(w4, Al, comp.bq, comp.scales, comp.zp, group, split_k=split),
          oracle.gemm(Al, comp.bq, comp.scales, comp.zp, group), f"split {split} A~N(500,50)")


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("M", [8, 300])
def test_swiglu_edge_cases(gpu_lib, fused, M):
    w4 = gpu_lib
    N, K, group = 512, 1024, 64
    gc, uc = make_swiglu_case(M, N, K, group, seed=M)
    # Gate weights with zp == q (gate output 0, so silu(0) * up == 0) and
    # large-mean activations; then constant up weights with one-hot rows.
    bq0, s0, z0 = zp_equal_q(N, K, group, seed=M + 1)
    A = large_mean(M, K, seed=M + 2, mean=4.0, std=1.0)
    cases = [
        ("gate zp==q", A, (bq0, s0, z0), (uc.bq, uc.scales, uc.zp)),
        ("A~N(4,1)", A, (gc.bq, gc.scales, gc.zp), (uc.bq, uc.scales, uc.zp)),
        ("one-hot, constant up", one_hot_rows(M, K, seed=M) if M <= K else A,
         (gc.bq, gc.scales, gc.zp), constant_weights(N, K, group, seed=M)),
    ]
    for label, Ax, g, u in cases:
        ref = oracle.gemm_swiglu(Ax, g, u, group)
        args = (dev(Ax), w4.w4a16_repack(dev(g[0])), dev(g[1]), dev(g[2]),
                w4.w4a16_repack(dev(u[0])), dev(u[1]), dev(u[2]), group)
        Y1 = w4.w4a16_gemm_swiglu(*args, fused=fused)
        Y2 = w4.w4a16_gemm_swiglu(*args, fused=fused)
        torch.cuda.synchronize()
        assert torch.equal(Y1, Y2)
        y = Y1.float().cpu().double().numpy()
        bound = None
        if not np.abs(ref).max():
            comp = oracle.gemm_swiglu(Ax, (gc.bq, gc.scales, gc.zp), (uc.bq, uc.scales, uc.zp), group)
            bound = TOL * np.abs(comp).max()
        check(y, ref, f"swiglu fused={fused} M={M} {label}", bound)
