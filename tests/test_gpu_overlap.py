"""Small-M calls launched as programmatic dependents (w4a16_set_launch_overlap).

Such a launch streams weights before the previous kernel on the stream has
finished and waits for it only before it reads A or writes Y. These tests issue
chains where A is the previous call's Y, where calls overwrite one Y, and where
a torch kernel rewrites A just before each call, with no synchronisation in
between (directly and inside a CUDA graph), and require results bit-identical
to the same chain with the switch off; the first layer is also checked against
the oracle.
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


def layers(w4, dims, M, group=128):
    """Weights of a chain of GEMMs whose N is the next one's K."""
    out = []
    for i, (N, K) in enumerate(zip(dims[1:], dims[:-1])):
        c = make_case(M, N, K, group, seed=100 + i)
        out.append((w4.w4a16_repack(dev(c.bq)), dev(c.scales), dev(c.zp), N, K, c))
    return out


def chain(w4, A0, ws, Ys, group=128):
    a = A0
    for (q, s, z, N, K, _), Y in zip(ws, Ys):
        w4.w4a16_gemm(a, q, s, z, group, out=Y)
        a = Y
    return a


def run_both(w4, fn):
    w4.w4a16_set_launch_overlap(False)
    ref = fn()
    torch.cuda.synchronize()
    ref = [r.clone() for r in ref]
    w4.w4a16_set_launch_overlap(True)
    got = fn()
    torch.cuda.synchronize()
    w4.w4a16_set_launch_overlap(False)
    assert w4.w4a16_device_error() == w4.W4A16_OK
    return ref, got


@pytest.mark.parametrize("M", [1, 8, 33])
def test_layer_chain_matches_and_first_layer_is_exact(w4, M):
    dims = [4096, 1024, 2048, 1024, 4096, 13824]
    ws = layers(w4, dims, M)
    A0 = dev(ws[0][5].A)
    Ys = [torch.empty((M, N), dtype=torch.float16, device="cuda") for (_, _, _, N, _, _) in ws]
    def fn():
        chain(w4, A0, ws, Ys)
        return Ys
    ref, got = run_both(w4, fn)
    for i, (r, g) in enumerate(zip(ref, got)):
        assert torch.equal(r, g), f"layer {i} differs with overlap on"
    c = ws[0][5]
    yref = oracle.gemm(c.A, c.bq, c.scales, c.zp, 128)
    y = got[0].float().cpu().double().numpy()
    assert np.abs(y - yref).max() <= 2e-2 * np.abs(yref).max()


def test_overwrites_of_one_output(w4):
    M, K, N = 8, 5120, 13824
    cs = [make_case(M, N, K, 128, seed=s) for s in (7, 8, 9)]
    A = dev(cs[0].A)
    wts = [(w4.w4a16_repack(dev(c.bq)), dev(c.scales), dev(c.zp)) for c in cs]
    Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    snaps = torch.empty((3, M, N), dtype=torch.float16, device="cuda")

    def fn():
        for i, (q, s, z) in enumerate(wts):
            w4.w4a16_gemm(A, q, s, z, 128, out=Y)
            snaps[i].copy_(Y)
        return [snaps]
    ref, got = run_both(w4, fn)
    assert torch.equal(ref[0], got[0])


def test_activation_rewritten_by_torch_before_each_call(w4):
    M, K, N = 8, 5120, 13824
    c = make_case(M, N, K, 128, seed=21)
    q, s, z = w4.w4a16_repack(dev(c.bq)), dev(c.scales), dev(c.zp)
    srcs = [torch.randn((M, K), device="cuda").half() for _ in range(4)]
    A = torch.empty((M, K), dtype=torch.float16, device="cuda")
    Ys = torch.empty((4, M, N), dtype=torch.float16, device="cuda")

    def fn():
        for i in range(4):
            A.copy_(srcs[i])
            w4.w4a16_gemm(A, q, s, z, 128, out=Ys[i])
        return [Ys]
    ref, got = run_both(w4, fn)
    assert torch.equal(ref[0], got[0])
    assert not torch.equal(Ys[0], Ys[1])


def test_chain_inside_cuda_graph(w4):
    M = 8
    dims = [5120, 13824, 5120]
    ws = layers(w4, dims, M)
    A0 = dev(ws[0][5].A)
    Ys = [torch.empty((M, N), dtype=torch.float16, device="cuda") for (_, _, _, N, _, _) in ws]
    w4.w4a16_set_launch_overlap(False)
    chain(w4, A0, ws, Ys)
    torch.cuda.synchronize()
    ref = [y.clone() for y in Ys]
    for y in Ys:
        y.zero_()
    w4.w4a16_set_launch_overlap(True)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        chain(w4, A0, ws, Ys)  # warm-up outside capture
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(3):
                chain(w4, A0, ws, Ys)
    torch.cuda.current_stream().wait_stream(stream)
    for y in Ys:
        y.zero_()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        g.replay()
        g.replay()
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()
    w4.w4a16_set_launch_overlap(False)
    for r, y in zip(ref, Ys):
        assert torch.equal(r, y)
    assert w4.w4a16_device_error() == w4.W4A16_OK
