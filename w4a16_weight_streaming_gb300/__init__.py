"""Python binding of libw4a16 (the W4A16 weight-streaming GEMM for GB300, sm_103a).

Argument marshalling only: every step of the GEMM runs in the CUDA kernels of
``libw4a16.so`` (built in-tree by ``_build.build()``), reached through the C ABI declared in
``include/w4a16.h``. PyTorch provides device memory and streams. There is no fallback: if the
library is missing or fails to load, importing this package raises.

Function names mirror the C entry points (``w4a16_repack``, ``w4a16_gemm`` ...), plus two
conveniences (``repack``, ``gemm``) that allocate the outputs with torch.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

LIB_PATH = _build.LIB_PATH
DEBUG_LIB_PATH = _build.DEBUG_LIB_PATH

OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED_SHAPE = 2
ERR_MISALIGNED = 3
ERR_CUDA = 4
ERR_DEVICE_TIMEOUT = 5
ERR_BOUNDS = 6

PATH_AUTO = 0
PATH_GEMV = 1
PATH_TC = 2

# every symbol include/w4a16.h declares
EXPORTED = [
    "w4a16_version", "w4a16_status_string", "w4a16_repacked_qweight_bytes", "w4a16_repacked_scales_bytes",
    "w4a16_repack", "w4a16_unrepack", "w4a16_gemm", "w4a16_gemm_ex", "w4a16_plan_for", "w4a16_last_dispatch",
    "w4a16_device_status", "w4a16_set_wait_timeout_ns", "w4a16_selftest_wait_timeout", "w4a16_gemm_host",
    "w4a16_silu_mul", "w4a16_debug_bounds", "w4a16_repacked_nvfp4_scales_bytes", "w4a16_repack_nvfp4",
    "w4a16_unrepack_nvfp4", "w4a16_gemm_nvfp4", "w4a16_gemm_nvfp4_ex", "w4a16_plan_for_nvfp4",
    "w4a16_quantize_x_int8", "w4a16_gemm_w4a8", "w4a16_gemm_w4a8_ex", "w4a16_plan_for_w4a8",
    "w4a16_quantize_gemm_w4a8",
]


class Plan(ctypes.Structure):
    """Mirror of ``w4a16_plan``; zero fields mean automatic."""

    _fields_ = [("path", ctypes.c_int), ("split_k", ctypes.c_int), ("m_tile", ctypes.c_int),
                ("k_chunk", ctypes.c_int), ("stages", ctypes.c_int), ("tmem_stages", ctypes.c_int),
                ("mma_issuers", ctypes.c_int), ("clusters", ctypes.c_int),
                ("dequant_warps", ctypes.c_int), ("tail_split", ctypes.c_int)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class W4A16Error(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)}")


def _load(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"{os.path.basename(path)} is not built ({path}); run __graft_entry__.build() first")
    lib = ctypes.CDLL(path)
    P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.w4a16_version.restype = I
    lib.w4a16_debug_bounds.restype = I
    lib.w4a16_status_string.restype = ctypes.c_char_p
    lib.w4a16_status_string.argtypes = [I]
    for n in ("w4a16_repacked_qweight_bytes", "w4a16_repacked_scales_bytes"):
        getattr(lib, n).restype = S
        getattr(lib, n).argtypes = [I, I, I]
    for n in ("w4a16_repack", "w4a16_unrepack"):
        getattr(lib, n).restype = I
        getattr(lib, n).argtypes = [P, P, P, P, I, I, I, P]
    lib.w4a16_gemm.restype = I
    lib.w4a16_gemm.argtypes = [P, P, P, P, I, I, I, I, P]
    lib.w4a16_gemm_ex.restype = I
    lib.w4a16_gemm_ex.argtypes = [P, P, P, P, I, I, I, I, ctypes.POINTER(Plan), P]
    lib.w4a16_gemm_host.restype = I
    lib.w4a16_gemm_host.argtypes = [P, P, P, P, P, P, I, I, I, I, P]
    lib.w4a16_silu_mul.restype = I
    lib.w4a16_silu_mul.argtypes = [P, P, I, I, P]
    lib.w4a16_plan_for.restype = I
    lib.w4a16_plan_for.argtypes = [I, I, I, I, ctypes.POINTER(Plan)]
    lib.w4a16_last_dispatch.restype = I
    lib.w4a16_last_dispatch.argtypes = [ctypes.c_char_p, S]
    lib.w4a16_device_status.restype = I
    lib.w4a16_device_status.argtypes = [P]
    lib.w4a16_set_wait_timeout_ns.restype = I
    lib.w4a16_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
    lib.w4a16_selftest_wait_timeout.restype = I
    lib.w4a16_selftest_wait_timeout.argtypes = [I, P]
    F = ctypes.c_float
    lib.w4a16_repacked_nvfp4_scales_bytes.restype = S
    lib.w4a16_repacked_nvfp4_scales_bytes.argtypes = [I, I]
    for n in ("w4a16_repack_nvfp4", "w4a16_unrepack_nvfp4"):
        getattr(lib, n).restype = I
        getattr(lib, n).argtypes = [P, P, P, P, I, I, P]
    lib.w4a16_gemm_nvfp4.restype = I
    lib.w4a16_gemm_nvfp4.argtypes = [P, P, P, F, P, I, I, I, P]
    lib.w4a16_gemm_nvfp4_ex.restype = I
    lib.w4a16_gemm_nvfp4_ex.argtypes = [P, P, P, F, P, I, I, I, ctypes.POINTER(Plan), P]
    lib.w4a16_plan_for_nvfp4.restype = I
    lib.w4a16_plan_for_nvfp4.argtypes = [I, I, I, ctypes.POINTER(Plan)]
    lib.w4a16_quantize_x_int8.restype = I
    lib.w4a16_quantize_x_int8.argtypes = [P, P, P, P, I, I, P]
    lib.w4a16_gemm_w4a8.restype = I
    lib.w4a16_gemm_w4a8.argtypes = [P, P, P, P, P, P, I, I, I, I, P]
    lib.w4a16_gemm_w4a8_ex.restype = I
    lib.w4a16_gemm_w4a8_ex.argtypes = [P, P, P, P, P, P, I, I, I, I, ctypes.POINTER(Plan), P]
    lib.w4a16_quantize_gemm_w4a8.restype = I
    lib.w4a16_quantize_gemm_w4a8.argtypes = [P, P, P, P, P, P, P, I, I, I, I, ctypes.POINTER(Plan), P]
    lib.w4a16_plan_for_w4a8.restype = I
    lib.w4a16_plan_for_w4a8.argtypes = [I, I, I, I, ctypes.POINTER(Plan)]
    return lib


lib = _load()


def load_debug_bounds() -> ctypes.CDLL:
    """The debug-bounds build (libw4a16_debug.so) as a second, independent handle with the same C
    entry points: every kernel checks its indices and reports W4A16_ERR_BOUNDS instead of accessing
    out of range."""
    return _load(DEBUG_LIB_PATH)


# ------------------------------------------------------------------------------ raw C ABI
def status_string(code: int) -> str:
    return lib.w4a16_status_string(int(code)).decode()


def w4a16_version() -> int:
    return lib.w4a16_version()


def w4a16_repacked_qweight_bytes(N: int, K: int, group: int) -> int:
    return lib.w4a16_repacked_qweight_bytes(N, K, group)


def w4a16_repacked_scales_bytes(N: int, K: int, group: int) -> int:
    return lib.w4a16_repacked_scales_bytes(N, K, group)


def w4a16_repack(qweight: int, scales: int, qweight_r: int, scales_r: int, N: int, K: int, group: int,
                 stream: int | None) -> int:
    return lib.w4a16_repack(qweight, scales, qweight_r, scales_r, N, K, group, stream)


def w4a16_unrepack(qweight_r: int, scales_r: int, qweight: int, scales: int, N: int, K: int, group: int,
                   stream: int | None) -> int:
    return lib.w4a16_unrepack(qweight_r, scales_r, qweight, scales, N, K, group, stream)


def w4a16_gemm(x: int, qweight_r: int, scales_r: int, y: int, M: int, N: int, K: int, group: int,
               stream: int | None) -> int:
    return lib.w4a16_gemm(x, qweight_r, scales_r, y, M, N, K, group, stream)


def w4a16_gemm_ex(x: int, qweight_r: int, scales_r: int, y: int, M: int, N: int, K: int, group: int,
                  plan: Plan | None, stream: int | None) -> int:
    return lib.w4a16_gemm_ex(x, qweight_r, scales_r, y, M, N, K, group,
                             ctypes.byref(plan) if plan is not None else None, stream)


def w4a16_gemm_host(x_host: int, x_dev: int, qweight_r: int, scales_r: int, y_dev: int, y_host: int, M: int, N: int,
                    K: int, group: int, stream: int | None) -> int:
    return lib.w4a16_gemm_host(x_host, x_dev, qweight_r, scales_r, y_dev, y_host, M, N, K, group, stream)


def w4a16_silu_mul(gu: int, act: int, M: int, I: int, stream: int | None) -> int:
    return lib.w4a16_silu_mul(gu, act, M, I, stream)


def w4a16_repacked_nvfp4_scales_bytes(N: int, K: int) -> int:
    return lib.w4a16_repacked_nvfp4_scales_bytes(N, K)


def w4a16_repack_nvfp4(qweight: int, scales8: int, qweight_r: int, scales_r: int, N: int, K: int,
                       stream: int | None) -> int:
    return lib.w4a16_repack_nvfp4(qweight, scales8, qweight_r, scales_r, N, K, stream)


def w4a16_unrepack_nvfp4(qweight_r: int, scales_r: int, qweight: int, scales8: int, N: int, K: int,
                         stream: int | None) -> int:
    return lib.w4a16_unrepack_nvfp4(qweight_r, scales_r, qweight, scales8, N, K, stream)


def w4a16_gemm_nvfp4(x: int, qweight_r: int, scales_r: int, tensor_scale: float, y: int, M: int, N: int, K: int,
                     stream: int | None) -> int:
    return lib.w4a16_gemm_nvfp4(x, qweight_r, scales_r, tensor_scale, y, M, N, K, stream)


def w4a16_gemm_nvfp4_ex(x: int, qweight_r: int, scales_r: int, tensor_scale: float, y: int, M: int, N: int, K: int,
                        plan: Plan | None, stream: int | None) -> int:
    return lib.w4a16_gemm_nvfp4_ex(x, qweight_r, scales_r, tensor_scale, y, M, N, K,
                                   ctypes.byref(plan) if plan is not None else None, stream)


def w4a16_plan_for_nvfp4(M: int, N: int, K: int) -> Plan:
    p = Plan()
    rc = lib.w4a16_plan_for_nvfp4(M, N, K, ctypes.byref(p))
    if rc != OK:
        raise W4A16Error(rc, "w4a16_plan_for_nvfp4")
    return p


def w4a16_plan_for(M: int, N: int, K: int, group: int) -> Plan:
    p = Plan()
    rc = lib.w4a16_plan_for(M, N, K, group, ctypes.byref(p))
    if rc != OK:
        raise W4A16Error(rc, "w4a16_plan_for")
    return p


def w4a16_last_dispatch() -> str:
    buf = ctypes.create_string_buffer(512)
    lib.w4a16_last_dispatch(buf, len(buf))
    return buf.value.decode()


def w4a16_device_status(stream: int | None = None) -> int:
    return lib.w4a16_device_status(stream)


def w4a16_set_wait_timeout_ns(ns: int) -> int:
    return lib.w4a16_set_wait_timeout_ns(int(ns))


def w4a16_selftest_wait_timeout(mode: int, stream: int | None = None) -> int:
    """Raw C ABI: `stream` is a cudaStream_t handle (None = the legacy default stream)."""
    return lib.w4a16_selftest_wait_timeout(int(mode), stream)


# ------------------------------------------------------------------------------ torch conveniences
def _stream_handle(stream: torch.cuda.Stream | None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(rc: int, where: str):
    if rc != OK:
        raise W4A16Error(rc, where)


def repack(qweight: torch.Tensor, scales: torch.Tensor, group: int = 128, stream=None):
    """Device layout from canonical device tensors (int32 [K/8, N], float16/int16 [K/G, N])."""
    K, N = qweight.shape[0] * 8, qweight.shape[1]
    qw_r = torch.empty(w4a16_repacked_qweight_bytes(N, K, group) // 4, dtype=torch.int32, device=qweight.device)
    sc_r = torch.empty(max(w4a16_repacked_scales_bytes(N, K, group) // 2, 1), dtype=torch.int16,
                       device=qweight.device)
    _check(w4a16_repack(qweight.data_ptr(), scales.data_ptr(), qw_r.data_ptr(), sc_r.data_ptr(), N, K, group,
                        _stream_handle(stream)), "w4a16_repack")
    return qw_r, sc_r


def w4a16_quantize_x_int8(x: int, xq: int, xq_f16: int | None, sx: int, M: int, K: int, stream: int | None) -> int:
    return lib.w4a16_quantize_x_int8(x, xq, xq_f16, sx, M, K, stream)


def w4a16_gemm_w4a8(xq: int, xq_f16: int | None, sx: int, qweight_r: int, scales_r: int, y: int, M: int, N: int,
                    K: int, group: int, stream: int | None) -> int:
    return lib.w4a16_gemm_w4a8(xq, xq_f16, sx, qweight_r, scales_r, y, M, N, K, group, stream)


def w4a16_gemm_w4a8_ex(xq: int, xq_f16: int | None, sx: int, qweight_r: int, scales_r: int, y: int, M: int, N: int,
                       K: int, group: int, plan: Plan | None, stream: int | None) -> int:
    return lib.w4a16_gemm_w4a8_ex(xq, xq_f16, sx, qweight_r, scales_r, y, M, N, K, group,
                                  ctypes.byref(plan) if plan is not None else None, stream)


def w4a16_quantize_gemm_w4a8(x: int, xq: int, xq_f16: int | None, sx: int, qweight_r: int, scales_r: int, y: int,
                             M: int, N: int, K: int, group: int, plan: Plan | None, stream: int | None) -> int:
    return lib.w4a16_quantize_gemm_w4a8(x, xq, xq_f16, sx, qweight_r, scales_r, y, M, N, K, group,
                                        ctypes.byref(plan) if plan is not None else None, stream)


def w4a16_plan_for_w4a8(M: int, N: int, K: int, group: int = 128) -> Plan:
    p = Plan()
    rc = lib.w4a16_plan_for_w4a8(M, N, K, group, ctypes.byref(p))
    if rc != OK:
        raise W4A16Error(rc, "w4a16_plan_for_w4a8")
    return p


def gemm_host(x_host: torch.Tensor, x_dev: torch.Tensor, qweight_r: torch.Tensor, scales_r: torch.Tensor,
              y_dev: torch.Tensor, y_host: torch.Tensor, N: int, K: int, group: int = 128, stream=None) -> None:
    """w4a16_gemm_host on tensors: x_host / y_host fp16 on the CPU (pinned), x_dev / y_dev on cuda.
    Queues the three operations on `stream`; y_host is valid after that stream is synchronised."""
    M = x_host.shape[0]
    _check(w4a16_gemm_host(x_host.data_ptr(), x_dev.data_ptr(), qweight_r.data_ptr(), scales_r.data_ptr(),
                           y_dev.data_ptr(), y_host.data_ptr(), M, N, K, group, _stream_handle(stream)),
           "w4a16_gemm_host")


def unrepack(qweight_r: torch.Tensor, scales_r: torch.Tensor, N: int, K: int, group: int = 128, stream=None):
    qw = torch.empty((K // 8, N), dtype=torch.int32, device=qweight_r.device)
    sc = torch.empty((K // group, N), dtype=torch.int16, device=qweight_r.device)
    _check(w4a16_unrepack(qweight_r.data_ptr(), scales_r.data_ptr(), qw.data_ptr(), sc.data_ptr(), N, K, group,
                          _stream_handle(stream)), "w4a16_unrepack")
    return qw, sc


def silu_mul(gu: torch.Tensor, act: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """act[M, I] = silu(gu[:, :I]) * gu[:, I:] (float16, CUDA) through w4a16_silu_mul."""
    M, I = gu.shape[0], gu.shape[1] // 2
    if act is None:
        act = torch.empty((M, I), dtype=torch.float16, device=gu.device)
    _check(w4a16_silu_mul(gu.data_ptr(), act.data_ptr(), M, I, _stream_handle(stream)), "w4a16_silu_mul")
    return act


def gemm(x: torch.Tensor, qweight_r: torch.Tensor, scales_r: torch.Tensor, N: int, K: int, group: int = 128,
         y: torch.Tensor | None = None, plan: Plan | dict | None = None, stream=None) -> torch.Tensor:
    """y[M, N] (float16) = x[M, K] (float16, CUDA) . dequant(W) through w4a16_gemm / w4a16_gemm_ex."""
    M = x.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=x.device)
    if isinstance(plan, dict):
        plan = Plan(**plan)
    _check(w4a16_gemm_ex(x.data_ptr(), qweight_r.data_ptr(), scales_r.data_ptr(), y.data_ptr(), M, N, K, group, plan,
                         _stream_handle(stream)), "w4a16_gemm")
    return y


# ------------------------------------------------------------------------------ NVFP4 weights
def repack_nvfp4(qweight: torch.Tensor, scales8: torch.Tensor, stream=None):
    """Device layout from canonical NVFP4 device tensors (int32 [K/8, N] of E2M1 codes, uint8
    [K/16, N] of E4M3 patterns): (qweight_r int32, scales_r int16 of fp16 bits)."""
    K, N = qweight.shape[0] * 8, qweight.shape[1]
    qw_r = torch.empty(N * K // 8, dtype=torch.int32, device=qweight.device)
    sc_r = torch.empty(max(w4a16_repacked_nvfp4_scales_bytes(N, K) // 2, 1), dtype=torch.int16, device=qweight.device)
    _check(w4a16_repack_nvfp4(qweight.data_ptr(), scales8.data_ptr(), qw_r.data_ptr(), sc_r.data_ptr(), N, K,
                              _stream_handle(stream)), "w4a16_repack_nvfp4")
    return qw_r, sc_r


def unrepack_nvfp4(qweight_r: torch.Tensor, scales_r: torch.Tensor, N: int, K: int, stream=None):
    qw = torch.empty((K // 8, N), dtype=torch.int32, device=qweight_r.device)
    s8 = torch.empty((K // 16, N), dtype=torch.uint8, device=qweight_r.device)
    _check(w4a16_unrepack_nvfp4(qweight_r.data_ptr(), scales_r.data_ptr(), qw.data_ptr(), s8.data_ptr(), N, K,
                                _stream_handle(stream)), "w4a16_unrepack_nvfp4")
    return qw, s8


def gemm_nvfp4(x: torch.Tensor, qweight_r: torch.Tensor, scales_r: torch.Tensor, tensor_scale: float, N: int, K: int,
               y: torch.Tensor | None = None, plan: Plan | dict | None = None, stream=None) -> torch.Tensor:
    """y[M, N] (float16) = x[M, K] (float16, CUDA) . dequant(W) for repacked NVFP4 weights."""
    M = x.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=x.device)
    if isinstance(plan, dict):
        plan = Plan(**plan)
    _check(w4a16_gemm_nvfp4_ex(x.data_ptr(), qweight_r.data_ptr(), scales_r.data_ptr(), float(tensor_scale),
                               y.data_ptr(), M, N, K, plan, _stream_handle(stream)), "w4a16_gemm_nvfp4")
    return y


# ------------------------------------------------------------------------------ W4A8 (int8 activations)
def quantize_x_int8(x: torch.Tensor, with_f16: bool = True, out=None, stream=None):
    """Per-token symmetric int8 quantisation of x (float16 [M, K], CUDA) through w4a16_quantize_x_int8:
    (xq int8 [M, K], xq_f16 float16 [M, K] holding the same integers or None, sx float32 [M])."""
    M, K = x.shape
    if out is None:
        xq = torch.empty((M, K), dtype=torch.int8, device=x.device)
        xh = torch.empty((M, K), dtype=torch.float16, device=x.device) if with_f16 else None
        sx = torch.empty(M, dtype=torch.float32, device=x.device)
    else:
        xq, xh, sx = out
    _check(w4a16_quantize_x_int8(x.data_ptr(), xq.data_ptr(), xh.data_ptr() if xh is not None else None,
                                 sx.data_ptr(), M, K, _stream_handle(stream)), "w4a16_quantize_x_int8")
    return xq, xh, sx


def gemm_w4a8(xq: torch.Tensor, xq_f16: torch.Tensor | None, sx: torch.Tensor, qweight_r: torch.Tensor,
              scales_r: torch.Tensor, N: int, K: int, group: int = 128, y: torch.Tensor | None = None,
              plan: Plan | dict | None = None, stream=None) -> torch.Tensor:
    """y[M, N] (float16) for int8 activations (from quantize_x_int8) and repacked int4 weights."""
    M = xq.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=xq.device)
    if isinstance(plan, dict):
        plan = Plan(**plan)
    _check(w4a16_gemm_w4a8_ex(xq.data_ptr(), xq_f16.data_ptr() if xq_f16 is not None else None, sx.data_ptr(),
                              qweight_r.data_ptr(), scales_r.data_ptr(), y.data_ptr(), M, N, K, group, plan,
                              _stream_handle(stream)), "w4a16_gemm_w4a8")
    return y


def quantize_gemm_w4a8(x: torch.Tensor, qweight_r: torch.Tensor, scales_r: torch.Tensor, N: int, K: int,
                       group: int = 128, out=None, y: torch.Tensor | None = None, plan: Plan | dict | None = None,
                       with_f16: bool = True, stream=None):
    """(y, (xq, xq_f16, sx)): quantise x (float16 [M, K], CUDA) and multiply in one call
    (w4a16_quantize_gemm_w4a8); the quantised activations are returned for other GEMMs of the same x."""
    M = x.shape[0]
    if out is None:
        out = (torch.empty((M, K), dtype=torch.int8, device=x.device),
               torch.empty((M, K), dtype=torch.float16, device=x.device) if with_f16 else None,
               torch.empty(M, dtype=torch.float32, device=x.device))
    xq, xh, sx = out
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=x.device)
    if isinstance(plan, dict):
        plan = Plan(**plan)
    _check(w4a16_quantize_gemm_w4a8(x.data_ptr(), xq.data_ptr(), xh.data_ptr() if xh is not None else None,
                                    sx.data_ptr(), qweight_r.data_ptr(), scales_r.data_ptr(), y.data_ptr(), M, N, K,
                                    group, plan, _stream_handle(stream)), "w4a16_quantize_gemm_w4a8")
    return y, out
