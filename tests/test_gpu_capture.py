"""CUDA-graph capture of every compute call, warm.

The MatMulNBits pull request (github.com/justinchuby/onnx-genai pull 960,
"What's landed" and "Validation") requires its GEMM to be capture-safe once
warm: a static launch grid, no allocation and no host read-back inside the call,
and replays byte-identical to eager execution. Here each call is made once
eagerly (the first call on a device looks up per-device state), then captured
in torch's global capture mode, which fails the capture if anything in the
process makes a call that is unsafe during capture. The tests check
  * the device's free memory is the same before and after eager calls and graph
    replays (the library itself never allocates device memory);
  * capture in global mode succeeds (no synchronising or otherwise unsafe call);
  * two replays give output byte-identical to the eager call.
Covered: w4a16_gemm on the small-M and tensor-core paths (plain launches and
launch overlap), w4a16_gemm_swiglu fused and unfused on both paths.
"""
import numpy as np
import pytest
import torch

from w4a16_inputs import make_case, make_swiglu_case

pytestmark = pytest.mark.gpu


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def free_bytes():
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0]


def capture_and_replay(fn, out):
    """Eager call, capture, two replays; returns (eager, replayed) outputs."""
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        fn()
        fn()
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()
    eager = out.clone()

    before = free_bytes()
    with torch.cuda.stream(stream):
        for _ in range(3):
            fn()
    torch.cuda.current_stream().wait_stream(stream)
    assert free_bytes() == before, "eager calls changed the device's free memory"

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="global"):
        fn()

    out.zero_()
    torch.cuda.synchronize()
    before = free_bytes()
    with torch.cuda.stream(stream):
        g.replay()
        g.replay()
    torch.cuda.current_stream().wait_stream(stream)
    assert free_bytes() == before, "graph replays changed the device's free memory"
    return eager, out.clone()


@pytest.fixture
def w4(gpu_lib):
    yield gpu_lib
    gpu_lib.w4a16_set_launch_overlap(False)
    gpu_lib.w4a16_set_tuning(0)


@pytest.mark.parametrize("M,overlap", [(8, False), (8, True), (33, False), (256, False), (1024, False)])
def test_gemm_capture(w4, M, overlap):
    N, K, group = 13824 if M >= 256 else 4096, 5120, 128
    c = make_case(M, N, K, group, seed=50 + M)
    A, q, s, z = dev(c.A), w4.w4a16_repack(dev(c.bq)), dev(c.scales), dev(c.zp)
    Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    w4.w4a16_set_launch_overlap(overlap)
    path = w4.w4a16_gemm_plan(M, N, K, group)[0]
    eager, replay = capture_and_replay(lambda: w4.w4a16_gemm(A, q, s, z, group, out=Y), Y)
    assert torch.equal(eager, replay), f"path {path}: replay differs from eager"
    assert w4.w4a16_device_error() == w4.W4A16_OK


@pytest.mark.parametrize("M", [8, 256])
@pytest.mark.parametrize("fused", [True, False])
def test_swiglu_capture(w4, M, fused):
    N, K, group = 13824 if M >= 256 else 2048, 5120, 128
    gc, uc = make_swiglu_case(M, N, K, group, seed=60 + M)
    args = (dev(gc.A), w4.w4a16_repack(dev(gc.bq)), dev(gc.scales), dev(gc.zp),
            w4.w4a16_repack(dev(uc.bq)), dev(uc.scales), dev(uc.zp), group)
    Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
    ws = torch.empty(max(1, w4.w4a16_swiglu_workspace_bytes(M, N, K, group, fused)), dtype=torch.uint8,
                     device="cuda")
    eager, replay = capture_and_replay(
        lambda: w4.w4a16_gemm_swiglu(*args, fused=fused, out=Y, workspace=ws), Y)
    assert torch.equal(eager, replay)
    assert w4.w4a16_device_error() == w4.W4A16_OK
