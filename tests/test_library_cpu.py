"""CPU-only checks of the C ABI: the library loads, exports every declared symbol,
validates arguments on the host, and its host unpack inverts the oracle's
statement of the repacked layout bit for bit. No compute call reaches a GPU."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a16.h")


@pytest.fixture(scope="module")
def w4():
    import weight_only_int4_repack_gb300 as w4
    return w4


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(w4a16_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("w4a16_repack", "w4a16_gemm", "w4a16_gemm_swiglu", "w4a16_unpack_host"):
        assert required in names


def test_library_exports_every_declared_symbol(w4):
    for name in declared_functions():
        assert hasattr(w4.lib, name), name
        assert name in w4.EXPORTS, name


def test_status_strings(w4):
    for code in range(6):
        assert w4.w4a16_status_string(code)
    assert w4.w4a16_status_string(0) == "ok"


def test_sizes(w4):
    assert w4.w4a16_repacked_bytes(13824, 5120) == 13824 * 5120 // 2
    assert w4.w4a16_repacked_bytes(0, 64) == 0
    assert w4.w4a16_gemm_workspace_bytes(8, 13824, 5120, 128, 0) == 0
    assert w4.w4a16_swiglu_workspace_bytes(8, 256, 512, 64, 1) == 0
    assert w4.w4a16_swiglu_workspace_bytes(8, 256, 512, 64, 0) >= 4 * 8 * 256


@pytest.mark.parametrize("N,K", [(16, 64), (128, 64), (144, 128), (400, 192), (256, 512)])
def test_unpack_host_inverts_oracle_layout(w4, N, K):
    bq = np.random.default_rng(N * 7 + K).integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    rep = oracle.repack(bq)
    np.testing.assert_array_equal(w4.w4a16_unpack_host(rep, N, K), bq)


def test_unpack_host_rejects_bad_dims(w4):
    buf = np.zeros(64, dtype=np.uint8)
    out = np.zeros(64, dtype=np.uint8)
    lib = w4.lib
    assert lib.w4a16_unpack_host(buf.ctypes.data, out.ctypes.data, 8, 16) == w4.W4A16_ERR_UNSUPPORTED
    assert lib.w4a16_unpack_host(None, out.ctypes.data, 16, 64) == w4.W4A16_ERR_INVALID_ARG
    assert lib.w4a16_unpack_host(buf.ctypes.data, out.ctypes.data, 0, 64) == w4.W4A16_ERR_INVALID_ARG


# Fake, never-dereferenced device addresses: validation fails before any launch.
A16 = 0x10000
BAD = 0x10002


def _gemm(w4, A=A16, q=A16, s=A16, sdt=0, zp=None, Y=A16, M=8, N=256, K=512, group=64, split=0):
    return w4.lib.w4a16_gemm(A, q, s, sdt, zp, Y, M, N, K, group, split, None, 0, None)


@pytest.mark.parametrize("kw,status", [
    (dict(M=0), 1), (dict(N=-16), 1), (dict(K=0), 1),
    (dict(group=48), 2), (dict(group=8), 2), (dict(K=96, group=64), 1),
    (dict(N=200), 2), (dict(K=96, group=32), 2),
    (dict(A=None), 1), (dict(Y=None), 1), (dict(q=None), 1), (dict(s=None), 1),
    (dict(A=BAD), 1), (dict(q=BAD), 1), (dict(Y=BAD), 1), (dict(sdt=7), 1),
    (dict(s=BAD, sdt=1), 1), (dict(split=9), 1), (dict(split=-1), 1),
])
def test_gemm_validation(w4, kw, status):
    assert _gemm(w4, **kw) == status


def _host_io(w4, Ah=0x30000, A=A16, q=A16, s=A16, sdt=0, zp=None, Y=A16, Yh=0x40000, M=8, N=256, K=512,
             group=64, split=0):
    return w4.lib.w4a16_gemm_host_io(Ah, A, q, s, sdt, zp, Y, Yh, M, N, K, group, split, None)


@pytest.mark.parametrize("kw,status", [
    (dict(Ah=None), 1), (dict(Yh=None), 1), (dict(A=None), 1), (dict(Y=None), 1),
    (dict(A=BAD), 1), (dict(Y=BAD), 1), (dict(q=None), 1), (dict(sdt=7), 1),
    (dict(M=0), 1), (dict(N=200), 2), (dict(group=48), 2), (dict(split=9), 1),
])
def test_host_io_validation(w4, kw, status):
    # Every check runs before the first copy is enqueued (no device is touched).
    assert _host_io(w4, **kw) == status


def test_swiglu_workspace_validation(w4):
    lib = w4.lib
    args = [A16, A16, A16, None, A16, A16, None, 0, A16, 8, 256, 512, 64]
    # unfused without workspace -> WORKSPACE
    assert lib.w4a16_gemm_swiglu(*args, 0, None, 0, None) == w4.W4A16_ERR_WORKSPACE
    need = w4.w4a16_swiglu_workspace_bytes(8, 256, 512, 64, 0)
    assert lib.w4a16_gemm_swiglu(*args, 0, A16, need - 1, None) == w4.W4A16_ERR_WORKSPACE
    bad = list(args)
    bad[1] = None
    assert lib.w4a16_gemm_swiglu(*bad, 1, None, 0, None) == w4.W4A16_ERR_INVALID_ARG


def test_rmsnorm_validation(w4):
    lib = w4.lib
    need = w4.w4a16_rmsnorm_workspace_bytes(8, 256, 512, 64, 0)
    assert need >= 8 * 512 * 2
    assert w4.w4a16_rmsnorm_workspace_bytes(8, 256, 512, 64, 2) >= need + 4 * 8 * 256
    assert w4.w4a16_rmsnorm_workspace_bytes(8, 256, 512, 64, 3) == 0
    base = dict(A=A16, gamma=A16, eps=1e-5, q=A16, s=A16, sdt=0, zp=None, Y=A16, M=8, N=256, K=512, group=64,
                split=0, ws=A16 * 16, ws_bytes=need)

    def call(**kw):
        a = dict(base, **kw)
        return lib.w4a16_gemm_rmsnorm(a["A"], a["gamma"], a["eps"], a["q"], a["s"], a["sdt"], a["zp"], a["Y"],
                                      a["M"], a["N"], a["K"], a["group"], a["split"], a["ws"], a["ws_bytes"],
                                      None)
    assert call(gamma=None) == w4.W4A16_ERR_INVALID_ARG
    assert call(gamma=BAD) == w4.W4A16_ERR_INVALID_ARG
    assert call(eps=-1.0) == w4.W4A16_ERR_INVALID_ARG
    assert call(ws_bytes=need - 1) == w4.W4A16_ERR_WORKSPACE
    assert call(ws=None) == w4.W4A16_ERR_WORKSPACE
    assert call(group=48) == w4.W4A16_ERR_UNSUPPORTED
    assert call(q=None) == w4.W4A16_ERR_INVALID_ARG


def test_repack_validation(w4):
    lib = w4.lib
    assert lib.w4a16_repack(A16, 0x20000, 8, 64, None) == w4.W4A16_ERR_UNSUPPORTED
    assert lib.w4a16_repack(A16, 0x20000, 16, 96, None) == w4.W4A16_ERR_UNSUPPORTED
    assert lib.w4a16_repack(None, 0x20000, 16, 64, None) == w4.W4A16_ERR_INVALID_ARG
    assert lib.w4a16_repack(A16, A16 + 16, 16, 64, None) == w4.W4A16_ERR_INVALID_ARG  # overlap
    assert lib.w4a16_repack(A16, 0x20008, 16, 64, None) == w4.W4A16_ERR_INVALID_ARG   # misaligned


def test_tuning_validation(w4):
    assert w4.lib.w4a16_set_tuning(65) == w4.W4A16_ERR_INVALID_ARG
    assert w4.lib.w4a16_set_tuning(-2) == w4.W4A16_ERR_INVALID_ARG
    assert w4.lib.w4a16_set_tuning(0) == 0


def test_launch_overlap_validation(w4):
    assert w4.lib.w4a16_set_launch_overlap(2) == w4.W4A16_ERR_INVALID_ARG
    assert w4.lib.w4a16_set_launch_overlap(-1) == w4.W4A16_ERR_INVALID_ARG
    assert w4.lib.w4a16_set_launch_overlap(1) == 0
    assert w4.lib.w4a16_set_launch_overlap(0) == 0


def test_product_path_has_no_oracle_dependency():
    """The binding and the CUDA sources never reference the oracle."""
    pkg = os.path.join(ROOT, "weight_only_int4_repack_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".h", ".cuh")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "w4a16_oracle" not in text and "liboracle" not in text, f
