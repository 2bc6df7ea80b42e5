"""Python binding of libw4a16.so (fp16 x int4 group-quantized GEMM for GB300).

Argument marshalling only: every step of the computation runs in the CUDA
library. PyTorch supplies device memory and the current stream. The functions
carry the C ABI's names (include/w4a16.h); `lib` is the raw ctypes handle.

Importing fails loudly when the compiled library is missing: there is no CPU or
PyTorch fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libw4a16.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; "
                      f"g.build()'` (needs nvcc); there is no fallback implementation")

# torch first: the library links the shared CUDA runtime by soname, so it must
# resolve to the runtime torch already loaded (one runtime per process).
import torch  # noqa: E402,F401

lib = ctypes.CDLL(LIB_PATH)

# Status codes and enums (mirror include/w4a16.h).
W4A16_OK = 0
W4A16_ERR_INVALID_ARG = 1
W4A16_ERR_UNSUPPORTED = 2
W4A16_ERR_WORKSPACE = 3
W4A16_ERR_CUDA = 4
W4A16_ERR_TIMEOUT = 5
W4A16_SCALE_F16 = 0
W4A16_SCALE_F32 = 1
W4A16_PATH_SMALL_M = 0
W4A16_PATH_TCGEN05 = 1

EXPORTS = (
    "w4a16_status_string", "w4a16_repacked_bytes", "w4a16_repack", "w4a16_unpack_host",
    "w4a16_gemm_workspace_bytes", "w4a16_gemm_plan", "w4a16_gemm",
    "w4a16_swiglu_workspace_bytes", "w4a16_gemm_swiglu", "w4a16_set_tuning", "w4a16_set_launch_overlap",
    "w4a16_device_error", "w4a16_swiglu_static_scratch_bytes", "w4a16_gemm_swiglu_unfused_static",
    "w4a16_set_wait_limit_ns", "w4a16_rmsnorm_workspace_bytes", "w4a16_gemm_rmsnorm",
    "w4a16_gemm_swiglu_rmsnorm", "w4a16_gemm_launch_info", "w4a16_gemm_host_io",
)

_vp, _ci, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t


class LaunchInfo(ctypes.Structure):
    """w4a16_launch_info: launch shape of the kernel a call would run."""
    _fields_ = [("path", _ci), ("split", _ci), ("ctas", _ci), ("threads", _ci), ("smem_bytes", _ci),
                ("stages", _ci)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


_sig = {
    "w4a16_status_string": (ctypes.c_char_p, [_ci]),
    "w4a16_repacked_bytes": (_sz, [_ci, _ci]),
    "w4a16_repack": (_ci, [_vp, _vp, _ci, _ci, _vp]),
    "w4a16_unpack_host": (_ci, [_vp, _vp, _ci, _ci]),
    "w4a16_gemm_workspace_bytes": (_sz, [_ci, _ci, _ci, _ci, _ci]),
    "w4a16_gemm_plan": (_ci, [_ci, _ci, _ci, _ci, _ci, ctypes.POINTER(_ci), ctypes.POINTER(_ci)]),
    "w4a16_gemm_launch_info": (_ci, [_ci, _ci, _ci, _ci, _ci, _ci, ctypes.POINTER(LaunchInfo)]),
    "w4a16_gemm": (_ci, [_vp, _vp, _vp, _ci, _vp, _vp, _ci, _ci, _ci, _ci, _ci, _vp, _sz, _vp]),
    "w4a16_gemm_host_io": (_ci, [_vp, _vp, _vp, _vp, _ci, _vp, _vp, _vp, _ci, _ci, _ci, _ci, _ci, _vp]),
    "w4a16_swiglu_workspace_bytes": (_sz, [_ci, _ci, _ci, _ci, _ci]),
    "w4a16_gemm_swiglu": (_ci, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _ci, _vp,
                                _ci, _ci, _ci, _ci, _ci, _vp, _sz, _vp]),
    "w4a16_set_tuning": (_ci, [_ci]),
    "w4a16_set_launch_overlap": (_ci, [_ci]),
    "w4a16_device_error": (_ci, [_vp]),
    "w4a16_set_wait_limit_ns": (_ci, [ctypes.c_ulonglong]),
    "w4a16_rmsnorm_workspace_bytes": (_sz, [_ci, _ci, _ci, _ci, _ci]),
    "w4a16_gemm_rmsnorm": (_ci, [_vp, _vp, ctypes.c_float, _vp, _vp, _ci, _vp, _vp, _ci, _ci, _ci, _ci, _ci,
                                 _vp, _sz, _vp]),
    "w4a16_gemm_swiglu_rmsnorm": (_ci, [_vp, _vp, ctypes.c_float, _vp, _vp, _vp, _vp, _vp, _vp, _ci, _vp,
                                        _ci, _ci, _ci, _ci, _ci, _vp, _sz, _vp]),
    "w4a16_swiglu_static_scratch_bytes": (_sz, []),
    "w4a16_gemm_swiglu_unfused_static": (_ci, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _ci, _vp,
                                               _ci, _ci, _ci, _ci, _vp]),
}
for _name, (_res, _args) in _sig.items():
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args


class W4A16Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {w4a16_status_string(status)} (status {status})")


def w4a16_status_string(status: int) -> str:
    return lib.w4a16_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != W4A16_OK:
        raise W4A16Error(status, where)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def w4a16_repacked_bytes(N: int, K: int) -> int:
    return int(lib.w4a16_repacked_bytes(N, K))


def w4a16_repack(q, out=None, stream=None):
    """q: uint8 CUDA tensor [N, K/2] -> repacked uint8 CUDA tensor [N*K/2]."""
    import torch
    N, K = q.shape[0], 2 * q.shape[1]
    if out is None:
        out = torch.empty(w4a16_repacked_bytes(N, K), dtype=torch.uint8, device=q.device)
    _check(lib.w4a16_repack(_ptr(q), _ptr(out), N, K, _stream(stream)), "w4a16_repack")
    return out


def w4a16_unpack_host(q_rep, N: int, K: int):
    """Host inverse of the repack (numpy in, numpy out)."""
    import numpy as np
    src = np.ascontiguousarray(np.asarray(q_rep, dtype=np.uint8).reshape(-1))
    if src.size != N * K // 2:
        raise ValueError("q_rep has the wrong size")
    dst = np.empty((N, K // 2), dtype=np.uint8)
    _check(lib.w4a16_unpack_host(src.ctypes.data, dst.ctypes.data, N, K), "w4a16_unpack_host")
    return dst


def w4a16_gemm_workspace_bytes(M, N, K, group, split_k=0) -> int:
    return int(lib.w4a16_gemm_workspace_bytes(M, N, K, group, split_k))


def w4a16_gemm_plan(M, N, K, group, split_k=0) -> Tuple[int, int]:
    path, split = _ci(), _ci()
    _check(lib.w4a16_gemm_plan(M, N, K, group, split_k, ctypes.byref(path), ctypes.byref(split)),
           "w4a16_gemm_plan")
    return path.value, split.value


def w4a16_gemm_launch_info(M, N, K, group, split_k=0, swiglu_fused=False) -> dict:
    """Launch shape of w4a16_gemm (or fused w4a16_gemm_swiglu): path, split, ctas,
    threads, smem_bytes, stages."""
    info = LaunchInfo()
    _check(lib.w4a16_gemm_launch_info(M, N, K, group, split_k, int(bool(swiglu_fused)), ctypes.byref(info)),
           "w4a16_gemm_launch_info")
    return info.as_dict()


def _scale_dtype(scales) -> int:
    import torch
    if scales.dtype == torch.float16:
        return W4A16_SCALE_F16
    if scales.dtype == torch.float32:
        return W4A16_SCALE_F32
    raise TypeError("scales must be float16 or float32")


def w4a16_gemm(A, q_rep, scales, zp, group: int, out=None, split_k: int = 0, workspace=None,
               stream=None):
    """Y[M, N] = A[M, K] . dequant(q_rep)^T (all CUDA tensors; zp may be None)."""
    import torch
    M, K = A.shape
    N = scales.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=A.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.w4a16_gemm(_ptr(A), _ptr(q_rep), _ptr(scales), _scale_dtype(scales), _ptr(zp),
                          _ptr(out), M, N, K, group, split_k, _ptr(workspace), ws_bytes,
                          _stream(stream)), "w4a16_gemm")
    return out


def w4a16_gemm_host_io(A_host, A_dev, q_rep, scales, zp, group: int, Y_dev, Y_host, split_k: int = 0,
                       stream=None):
    """Copy A_host (pinned CPU fp16 [M, K]) into A_dev, run the GEMM into Y_dev and
    copy it into Y_host (pinned CPU fp16 [M, N]), all enqueued on the stream; no
    synchronisation (Y_host is valid once the stream has passed the call)."""
    M, K = A_host.shape
    N = scales.shape[0]
    _check(lib.w4a16_gemm_host_io(_ptr(A_host), _ptr(A_dev), _ptr(q_rep), _ptr(scales), _scale_dtype(scales),
                                  _ptr(zp), _ptr(Y_dev), _ptr(Y_host), M, N, K, group, split_k,
                                  _stream(stream)), "w4a16_gemm_host_io")
    return Y_host


def w4a16_swiglu_workspace_bytes(M, N, K, group, fused) -> int:
    return int(lib.w4a16_swiglu_workspace_bytes(M, N, K, group, int(bool(fused))))


def w4a16_gemm_swiglu(A, qg_rep, sg, zg, qu_rep, su, zu, group: int, fused: bool = True,
                      out=None, workspace=None, stream=None):
    """Y = silu(A . Wg^T) * (A . Wu^T); fused or the unfused three-kernel chain."""
    import torch
    M, K = A.shape
    N = sg.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=A.device)
    need = w4a16_swiglu_workspace_bytes(M, N, K, group, fused)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=A.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.w4a16_gemm_swiglu(_ptr(A), _ptr(qg_rep), _ptr(sg), _ptr(zg), _ptr(qu_rep),
                                 _ptr(su), _ptr(zu), _scale_dtype(sg), _ptr(out), M, N, K, group,
                                 int(bool(fused)), _ptr(workspace), ws_bytes, _stream(stream)),
           "w4a16_gemm_swiglu")
    return out


def w4a16_rmsnorm_workspace_bytes(M, N, K, group, mode) -> int:
    return int(lib.w4a16_rmsnorm_workspace_bytes(M, N, K, group, mode))


def w4a16_gemm_rmsnorm(A, gamma, eps: float, q_rep, scales, zp, group: int, out=None, split_k: int = 0,
                       workspace=None, stream=None):
    """Y = rmsnorm(A; gamma, eps) . dequant(q_rep)^T (normalised A staged in the workspace)."""
    import torch
    M, K = A.shape
    N = scales.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=A.device)
    if workspace is None:
        workspace = torch.empty(w4a16_rmsnorm_workspace_bytes(M, N, K, group, 0), dtype=torch.uint8,
                                device=A.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib.w4a16_gemm_rmsnorm(_ptr(A), _ptr(gamma), float(eps), _ptr(q_rep), _ptr(scales),
                                  _scale_dtype(scales), _ptr(zp), _ptr(out), M, N, K, group, split_k,
                                  _ptr(workspace), ws_bytes, _stream(stream)), "w4a16_gemm_rmsnorm")
    return out


def w4a16_gemm_swiglu_rmsnorm(A, gamma, eps: float, qg_rep, sg, zg, qu_rep, su, zu, group: int,
                              fused: bool = True, out=None, workspace=None, stream=None):
    """Y = silu(An . Wg^T) * (An . Wu^T), An = rmsnorm(A; gamma, eps)."""
    import torch
    M, K = A.shape
    N = sg.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=A.device)
    if workspace is None:
        workspace = torch.empty(w4a16_rmsnorm_workspace_bytes(M, N, K, group, 1 if fused else 2),
                                dtype=torch.uint8, device=A.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib.w4a16_gemm_swiglu_rmsnorm(_ptr(A), _ptr(gamma), float(eps), _ptr(qg_rep), _ptr(sg), _ptr(zg),
                                         _ptr(qu_rep), _ptr(su), _ptr(zu), _scale_dtype(sg), _ptr(out),
                                         M, N, K, group, int(bool(fused)), _ptr(workspace), ws_bytes,
                                         _stream(stream)), "w4a16_gemm_swiglu_rmsnorm")
    return out


def w4a16_swiglu_static_scratch_bytes() -> int:
    return int(lib.w4a16_swiglu_static_scratch_bytes())


def w4a16_gemm_swiglu_unfused_static(A, qg_rep, sg, zg, qu_rep, su, zu, group: int, out=None,
                                     stream=None):
    """Unfused SwiGLU whose intermediates live in the library's fixed device
    array: for callers that cannot allocate device memory (see include/w4a16.h)."""
    import torch
    M, K = A.shape
    N = sg.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=A.device)
    _check(lib.w4a16_gemm_swiglu_unfused_static(_ptr(A), _ptr(qg_rep), _ptr(sg), _ptr(zg),
                                                _ptr(qu_rep), _ptr(su), _ptr(zu),
                                                _scale_dtype(sg), _ptr(out), M, N, K, group,
                                                _stream(stream)),
           "w4a16_gemm_swiglu_unfused_static")
    return out


def w4a16_set_tuning(smallm_max: int) -> None:
    _check(lib.w4a16_set_tuning(smallm_max), "w4a16_set_tuning")


def w4a16_set_launch_overlap(enable: bool) -> None:
    """Let small-M GEMM calls start while the work before them finishes
    (weights must not be written by that work); see include/w4a16.h."""
    _check(lib.w4a16_set_launch_overlap(int(enable)), "w4a16_set_launch_overlap")


WAIT_LIMIT_DEFAULT_NS = 2_000_000_000


def w4a16_set_wait_limit_ns(limit_ns: int) -> None:
    """Limit of every bounded device-side wait (tests of the failure path)."""
    _check(lib.w4a16_set_wait_limit_ns(int(limit_ns)), "w4a16_set_wait_limit_ns")


def w4a16_device_error(stream=None) -> int:
    return int(lib.w4a16_device_error(_stream(stream)))
