"""Pins for the oracle's RMS-norm prologue (CPU only).

The prologue normalises each activation row before the W4A16 GEMM (the pull
request github.com/justinchuby/onnx-genai pull 960, "Update -- fused RMS-norm
epilogue + e2e PASS"). Pinned by hand-worked examples (tests/golden), by the
properties of the definition (a constant row normalises to the weight vector,
scaling a row by a power of two leaves the result unchanged, a zero row stays
zero), and by PyTorch's float64 rms_norm on random inputs.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from w4a16_inputs import draw_activations, make_case, make_swiglu_case

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "rmsnorm_worked_examples.txt")


def load_golden():
    cases, cur = [], {}
    for line in open(GOLDEN):
        line = line.strip()
        if line.startswith("#"):
            continue
        if not line:
            if cur:
                cases.append(cur)
                cur = {}
            continue
        k, v = line.split(":", 1)
        cur[k.strip()] = v.strip()
    if cur:
        cases.append(cur)
    return cases


@pytest.mark.parametrize("case", load_golden(), ids=lambda c: c["name"])
def test_golden_worked_examples(case):
    f = lambda key: np.array([[float(x) for x in r.split()] for r in case[key].split("|")])  # noqa: E731
    A, xn, Y = f("A"), f("xn"), f("Y")
    gamma = f("gamma")[0]
    eps = float(case["eps"])
    bq = np.array([[int(x, 16) for x in case["bq"].split()]], dtype=np.uint8)
    scales = f("scales")
    group = int(case["group"])
    np.testing.assert_array_equal(oracle.rmsnorm(A, gamma, eps), xn)
    np.testing.assert_array_equal(oracle.gemm_rmsnorm(A, gamma, eps, bq, scales, None, group), Y.T)


def test_constant_row_normalises_to_gamma():
    K = 256
    gamma = draw_activations(np.random.default_rng(1), 1, K)[0]
    for c in (0.5, 3.0, -2.0):
        A = np.full((1, K), c)
        np.testing.assert_allclose(oracle.rmsnorm(A, gamma, 0.0)[0], np.sign(c) * gamma.astype(np.float64),
                                   rtol=1e-15, atol=0)


def test_power_of_two_scaling_leaves_rows_unchanged():
    A = draw_activations(np.random.default_rng(2), 4, 512).astype(np.float64)
    gamma = draw_activations(np.random.default_rng(3), 1, 512)[0]
    base = oracle.rmsnorm(A, gamma, 0.0)
    for alpha in (0.25, 4.0, 1024.0):
        np.testing.assert_array_equal(oracle.rmsnorm(alpha * A, gamma, 0.0), base)


def test_zero_row_stays_zero():
    A = np.zeros((2, 128))
    assert np.all(oracle.rmsnorm(A, np.ones(128), 1e-5) == 0.0)


@pytest.mark.parametrize("eps", [1e-6, 1e-5, 0.1])
def test_matches_torch_rms_norm(eps):
    A = draw_activations(np.random.default_rng(4), 6, 1024)
    gamma = draw_activations(np.random.default_rng(5), 1, 1024)[0]
    ref = torch.nn.functional.rms_norm(torch.from_numpy(A.astype(np.float64)), (1024,),
                                       weight=torch.from_numpy(gamma.astype(np.float64)), eps=eps).numpy()
    np.testing.assert_allclose(oracle.rmsnorm(A, gamma, eps), ref, rtol=1e-12, atol=1e-12)


def test_gemm_rmsnorm_matches_numpy_and_row_subsets():
    c = make_case(5, 48, 256, 64, seed=14)
    gamma = draw_activations(np.random.default_rng(6), 1, 256)[0]
    W = oracle.dequant(c.bq, c.scales, c.zp, c.K, c.group)
    xn = torch.nn.functional.rms_norm(torch.from_numpy(c.A.astype(np.float64)), (256,),
                                      weight=torch.from_numpy(gamma.astype(np.float64)), eps=1e-5).numpy()
    Y = oracle.gemm_rmsnorm(c.A, gamma, 1e-5, c.bq, c.scales, c.zp, c.group)
    np.testing.assert_allclose(Y, xn @ W.T, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(oracle.gemm_rmsnorm(c.A, gamma, 1e-5, c.bq, c.scales, c.zp, c.group,
                                                      rows=[4, 1]), Y[[4, 1]])


def test_swiglu_rmsnorm_matches_composition():
    gc, uc = make_swiglu_case(3, 32, 256, 32, seed=15)
    gamma = draw_activations(np.random.default_rng(7), 1, 256)[0]
    xn = oracle.rmsnorm(gc.A, gamma, 1e-5)
    Y = oracle.gemm_swiglu_rmsnorm(gc.A, gamma, 1e-5, (gc.bq, gc.scales, gc.zp), (uc.bq, uc.scales, uc.zp), 32)
    np.testing.assert_array_equal(Y, oracle.gemm_swiglu(xn, (gc.bq, gc.scales, gc.zp),
                                                        (uc.bq, uc.scales, uc.zp), 32))
