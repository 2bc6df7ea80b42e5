"""Pins for the float64 oracle: checks against things other than the oracle itself.

Hand-worked examples (tests/golden), closed forms on structured inputs,
invariants (zp == q gives zero, power-of-two linearity in the scale, a one-hot
activation row selects a weight row), and library routines (numpy matmul,
scipy's logistic function) on tiny random inputs.
"""
import os

import numpy as np
import pytest
from scipy.special import expit

import oracle
from w4a16_inputs import make_case, make_swiglu_case

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "dequant_worked_examples.txt")


def _parse_rows(text, conv):
    return [[conv(v) for v in row.split()] for row in text.split("|")]


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
        key, val = line.split(":", 1)
        cur[key.strip()] = val.strip()
    if cur:
        cases.append(cur)
    out = []
    for c in cases:
        N, K, group = int(c["N"]), int(c["K"]), int(c["group"])
        bq = np.array(_parse_rows(c["bq"], lambda v: int(v, 16)), dtype=np.uint8)
        zp = None if c["zp"] == "-" else np.array(_parse_rows(c["zp"], lambda v: int(v, 16)),
                                                  dtype=np.uint8)
        scales = np.array(_parse_rows(c["scales"], float), dtype=np.float64)
        A = np.array(_parse_rows(c["A"], float), dtype=np.float64)
        W = np.array(_parse_rows(c["W"], float), dtype=np.float64)
        Y = np.array(_parse_rows(c["Y"], float), dtype=np.float64)
        assert bq.shape == (N, K // 2)
        out.append((c["name"], N, K, group, bq, zp, scales, A, W, Y))
    return out


@pytest.mark.parametrize("case", load_golden(), ids=lambda c: c[0])
def test_golden_worked_examples(case):
    name, N, K, group, bq, zp, scales, A, W, Y = case
    np.testing.assert_array_equal(oracle.dequant(bq, scales, zp, K, group), W)
    np.testing.assert_array_equal(oracle.gemm(A, bq, scales, zp, group), Y)


def test_group_index_closed_form():
    # q = 9 everywhere, symmetric (zp 8) and scale 2**j for group j: W[n,k] = 2**(k//g).
    N, K = 3, 256
    for g in (16, 32, 64, 128):
        G = K // g
        bq = np.full((N, K // 2), 0x99, dtype=np.uint8)
        scales = np.tile(2.0 ** np.arange(G), (N, 1))
        W = oracle.dequant(bq, scales, None, K, g)
        np.testing.assert_array_equal(W, np.tile(2.0 ** (np.arange(K) // g), (N, 1)))


def test_nibble_order_closed_form():
    # Only even-k nibbles (low) set to 5, odd-k (high) to 0, zp 0: W = 5*s on even k.
    N, K, g = 2, 64, 16
    bq = np.full((N, K // 2), 0x05, dtype=np.uint8)
    zp = np.zeros((N, (K // g + 1) // 2), dtype=np.uint8)
    s = np.full((N, K // g), 0.5)
    W = oracle.dequant(bq, s, zp, K, g)
    assert np.all(W[:, 0::2] == 2.5) and np.all(W[:, 1::2] == 0.0)


def test_zero_point_order_closed_form():
    # zp byte 0x53: group 0 -> 3, group 1 -> 5; q = 8: W = 5 on group 0, 3 on group 1.
    N, K, g = 1, 64, 32
    bq = np.full((N, K // 2), 0x88, dtype=np.uint8)
    zp = np.array([[0x53]], dtype=np.uint8)
    W = oracle.dequant(bq, np.ones((N, 2)), zp, K, g)
    np.testing.assert_array_equal(W[0, :32], 5.0)
    np.testing.assert_array_equal(W[0, 32:], 3.0)


def test_zp_equal_q_gives_zero():
    rng = np.random.default_rng(11)
    M, N, K, g = 3, 32, 128, 32
    G = K // g
    v = rng.integers(0, 16, size=(N, G)).astype(np.uint8)       # one value per group
    qk = np.repeat(v, g, axis=1)                                 # q[n,k] = v[n, k//g]
    bq = (qk[:, 0::2] | (qk[:, 1::2] << 4)).astype(np.uint8)
    zp = (v[:, 0::2] | (v[:, 1::2] << 4)).astype(np.uint8)
    A = rng.standard_normal((M, K)).astype(np.float16)
    s = rng.uniform(0.005, 0.02, size=(N, G)).astype(np.float16)
    Y = oracle.gemm(A, bq, s, zp, g)
    assert np.all(Y == 0.0)


def test_scale_linearity_power_of_two():
    c = make_case(4, 48, 256, 64, seed=5)
    Y1 = oracle.gemm(c.A, c.bq, c.scales, c.zp, c.group)
    Y2 = oracle.gemm(c.A, c.bq, c.scales.astype(np.float64) * 4.0, c.zp, c.group)
    np.testing.assert_array_equal(Y2, 4.0 * Y1)


def test_one_hot_row_selects_weight_column():
    c = make_case(1, 64, 256, 32, seed=6)
    W = oracle.dequant(c.bq, c.scales, c.zp, c.K, c.group)
    for i in (0, 1, 31, 32, 255):
        A = np.zeros((1, c.K), dtype=np.float16)
        A[0, i] = 1
        np.testing.assert_array_equal(oracle.gemm(A, c.bq, c.scales, c.zp, c.group)[0], W[:, i])


def test_constant_weights_closed_form():
    # q = 11, zp = 3 (asym), scale s_n per row: Y[m,n] = s_n * 8 * sum_k A[m,k].
    rng = np.random.default_rng(7)
    M, N, K, g = 5, 16, 192, 64
    G = K // g
    bq = np.full((N, K // 2), 0xBB, dtype=np.uint8)
    zp = np.full((N, (G + 1) // 2), 0x33, dtype=np.uint8)
    srow = rng.uniform(0.005, 0.02, size=N).astype(np.float16).astype(np.float64)
    s = np.repeat(srow[:, None], G, axis=1)
    A = rng.standard_normal((M, K)).astype(np.float16)
    Y = oracle.gemm(A, bq, s, zp, g)
    expect = np.outer(A.astype(np.float64).sum(axis=1), 8.0 * srow)
    np.testing.assert_allclose(Y, expect, rtol=1e-12, atol=1e-12)


def test_symmetric_equals_explicit_eight():
    c = make_case(3, 32, 128, 16, seed=8, asym=False)
    zp8 = np.full((c.N, (c.G + 1) // 2), 0x88, dtype=np.uint8)
    np.testing.assert_array_equal(oracle.gemm(c.A, c.bq, c.scales, None, c.group),
                                  oracle.gemm(c.A, c.bq, c.scales, zp8, c.group))


@pytest.mark.parametrize("g", [16, 32, 64, 128])
@pytest.mark.parametrize("sdt", [np.float16, np.float32])
@pytest.mark.parametrize("asym", [False, True])
def test_gemm_matches_numpy_matmul(g, sdt, asym):
    c = make_case(7, 48, 256, g, seed=9, scale_dtype=sdt, asym=asym)
    W = oracle.dequant(c.bq, c.scales, c.zp, c.K, c.group)
    Y = oracle.gemm(c.A, c.bq, c.scales, c.zp, c.group)
    np.testing.assert_allclose(Y, c.A.astype(np.float64) @ W.T, rtol=1e-12, atol=1e-12)


def test_row_and_column_subsets():
    c = make_case(9, 64, 256, 32, seed=10)
    full = oracle.gemm(c.A, c.bq, c.scales, c.zp, c.group)
    rows, cols = [8, 0, 3], [63, 1, 17, 17]
    sub = oracle.gemm(c.A, c.bq, c.scales, c.zp, c.group, rows=rows, cols=cols)
    np.testing.assert_array_equal(sub, full[np.ix_(rows, cols)])
    np.testing.assert_array_equal(oracle.gemm(c.A, c.bq, c.scales, c.zp, c.group, nthreads=1),
                                  full)


def test_swiglu_unit_up_reduces_to_rowsum():
    # Up weights dequantise to exactly 1 (q = 9, symmetric zp 8, scale 1).
    g_case, _ = make_swiglu_case(4, 32, 256, 64, seed=12)
    N, K, G = g_case.N, g_case.K, g_case.G
    up = (np.full((N, K // 2), 0x99, dtype=np.uint8), np.ones((N, G)), None)
    gate = (g_case.bq, g_case.scales, g_case.zp)
    Y = oracle.gemm_swiglu(g_case.A, gate, up, g_case.group)
    x = oracle.gemm(g_case.A, *gate, g_case.group)
    rowsum = g_case.A.astype(np.float64).sum(axis=1, keepdims=True)
    np.testing.assert_allclose(Y, x * expit(x) * rowsum, rtol=1e-12, atol=1e-12)


def test_swiglu_matches_library_composition():
    gc, uc = make_swiglu_case(3, 64, 256, 32, seed=13)
    Y = oracle.gemm_swiglu(gc.A, (gc.bq, gc.scales, gc.zp), (uc.bq, uc.scales, uc.zp), 32)
    Wg = oracle.dequant(gc.bq, gc.scales, gc.zp, gc.K, 32)
    Wu = oracle.dequant(uc.bq, uc.scales, uc.zp, uc.K, 32)
    A = gc.A.astype(np.float64)
    xg, xu = A @ Wg.T, A @ Wu.T
    np.testing.assert_allclose(Y, xg * expit(xg) * xu, rtol=1e-12, atol=1e-12)
    # silu special values: silu(0) = 0.
    zero_gate = (np.full_like(gc.bq, 0x88), gc.scales, None)
    assert np.all(oracle.gemm_swiglu(gc.A, zero_gate, (uc.bq, uc.scales, uc.zp), 32) == 0.0)


def test_oracle_rejects_bad_shapes():
    c = make_case(1, 16, 64, 16, seed=1)
    with pytest.raises(ValueError):
        oracle.gemm(c.A, c.bq[:, :-1], c.scales, c.zp, 16)
    with pytest.raises(ValueError):
        oracle.gemm(c.A, c.bq, c.scales[:, :-1], c.zp, 16)


def test_oracle_does_not_import_the_product():
    import subprocess
    import sys
    code = ("import sys, oracle, numpy as np; from w4a16_inputs import make_case;"
            "c = make_case(1, 16, 64, 16, seed=0); oracle.gemm(c.A, c.bq, c.scales, c.zp, 16);"
            "bad = [m for m in sys.modules if m.startswith('weight_only_int4_repack_gb300')];"
            "assert not bad, bad")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    subprocess.check_call([sys.executable, "-c", code], cwd=root)
