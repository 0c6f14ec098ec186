"""W4A16 GEMM oracle: plain fp64 CPU statement of what the GPU path computes.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
``cpu_baseline`` leg (and its ``--impl reference`` arm) may import this package. The product
path never does, and this package shares no code with the CUDA library: the arithmetic lives
in ``w4a16_oracle.c`` (plain C, no CUDA), loaded here through ctypes.

Functions and the passage each follows:

* ``gemm`` / ``gemm_sampled`` / ``gemm_xf64`` -- y[m,n] = sum_k x[m,k] * w[k,n] in fp64,
  ascending k. W4A16 = 4-bit weights, 16-bit activations: "RTX 3090 Tested: Qwen's 381 tok/s
  Myth Busted" (kongchang.com), section "What Exactly Is This Stack". One weight read shared by
  every activation row: "Qwen3.8-27B at 764, 1,035 and 1,623 tok/s" (ai.satyajit.si), section
  "One weight read, shared by every stream".
* ``dequant`` / ``unpack`` -- the canonical workload format (8 nibbles per int32 along K, low
  nibble first; fp16 scales per group of G rows; w = fp16_rne((q - 8) * s)). The pages do not
  print the format; this is the plainest reading of the workload definition.
* ``silu_mul`` -- the activation of the dense layer's MLP between the fused gate+up projection
  and the down projection, act = silu(gate) * up ("Qwen3.8-27B at 764, 1,035 and 1,623 tok/s",
  section "Where the line bends": the 17,408-wide MLPs; SwiGLU is the reading taken).
* ``repack`` / ``unrepack`` -- the library's own device layout, restated from its definition.
* ``e2m1_to_double`` / ``e4m3_to_double`` / ``dequant_nvfp4`` / ``gemm_nvfp4`` /
  ``gemm_nvfp4_sampled`` / ``repack_nvfp4`` / ``unrepack_nvfp4`` -- NVFP4 weights (the RTX 5090
  runs of "Qwen3.8-27B at 764, 1,035 and 1,623 tok/s", section "One weight read, shared by every
  stream"): E2M1 codes, one E4M3 scale per 16 weights along K, one fp32 tensor scale g, fp16
  activations; y = g * sum_k x * e2m1 * e4m3. The pages print no format: the reading is the
  published NVFP4 definition.
* ``quantize_x_int8`` / ``gemm_w4a8`` / ``gemm_w4a8_sampled`` -- int8 activations (W4A8: the MLP
  GEMMs past the bend in "Qwen3.8-27B at 764, 1,035 and 1,623 tok/s", section "Where the line
  bends"): per-token symmetric int8 (sx = fl32(amax / 127), xq = rne(fl32(x / sx))), and
  y = sx * sum_g s * sum_{k in g} (q - 8) * xq with exact integer group sums. The pages print no
  quantisation: the reading is the plainest per-token one.
* ``half_to_double`` / ``double_to_half`` -- the binary16 codec, written out bit by bit.

Parity status of each function is recorded in the test suite that pins it
(``tests/test_oracle_pins.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4a16_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None  # the default Oracle instance


def _compile(src: str, out: str) -> str:
    """gcc the C source into a shared library (OpenMP when the compiler has it)."""
    tmp = out + ".tmp"
    # IEEE semantics: no -ffast-math anywhere near the oracle.
    common = ["-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", src, "-o", tmp, "-lm"]
    err = ""
    for extra in (["-fopenmp"], []):
        r = subprocess.run(["gcc"] + extra + common, capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(tmp, out)
            return out
        err = r.stderr
    raise RuntimeError(f"oracle build failed: {err}")


def build(force: bool = False) -> str:
    """Compile ``w4a16_oracle.c`` into ``liboracle.so`` next to it."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    return _compile(_SRC, _LIB_PATH)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


class Oracle:
    """numpy front end over one compiled copy of ``w4a16_oracle.c``."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        P, I, L = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        lib.w4o_half_to_double_array.argtypes = [P, P, L]
        lib.w4o_double_to_half_array.argtypes = [P, P, L]
        lib.w4o_unpack.argtypes = [P, I, I, P]
        lib.w4o_dequant.argtypes = [P, P, I, I, I, P]
        for name in ("w4o_gemm", "w4o_gemm_xf64"):
            getattr(lib, name).restype = I
            getattr(lib, name).argtypes = [P, P, P, I, I, I, I, P, P, I]
        lib.w4o_gemm_sampled.restype = I
        lib.w4o_gemm_sampled.argtypes = [P, P, P, I, I, I, I, P, P, L, P, P, I]
        for name in ("w4o_repack", "w4o_unrepack"):
            getattr(lib, name).restype = I
            getattr(lib, name).argtypes = [P, P, I, I, I, P, P]
        lib.w4o_silu_mul.argtypes = [P, I, I, P, P]
        D = ctypes.c_double
        lib.w4o_e2m1_to_double.restype = D
        lib.w4o_e2m1_to_double.argtypes = [I]
        lib.w4o_e4m3_to_double_array.argtypes = [P, P, L]
        lib.w4o_dequant_nvfp4.argtypes = [P, P, I, I, P]
        lib.w4o_gemm_nvfp4.restype = I
        lib.w4o_gemm_nvfp4.argtypes = [P, P, P, D, I, I, I, P, P, I]
        lib.w4o_gemm_nvfp4_sampled.restype = I
        lib.w4o_gemm_nvfp4_sampled.argtypes = [P, P, P, D, I, I, I, P, P, L, P, P]
        for name in ("w4o_repack_nvfp4", "w4o_unrepack_nvfp4"):
            getattr(lib, name).restype = I
            getattr(lib, name).argtypes = [P, P, I, I, P, P]
        lib.w4o_quantize_x_int8.restype = I
        lib.w4o_quantize_x_int8.argtypes = [P, I, I, P, P]
        lib.w4o_gemm_w4a8.restype = I
        lib.w4o_gemm_w4a8.argtypes = [P, P, P, P, I, I, I, I, P, P, I]
        lib.w4o_gemm_w4a8_sampled.restype = I
        lib.w4o_gemm_w4a8_sampled.argtypes = [P, P, P, P, I, I, I, I, P, P, L, P, P]
        lib.w4o_max_threads.restype = I
        lib.w4o_has_openmp.restype = I
        self.lib = lib
        self.path = lib_path

    def has_openmp(self) -> bool:
        return bool(self.lib.w4o_has_openmp())

    # ---------------------------------------------------------------------------- codec
    def half_to_double(self, bits) -> np.ndarray:
        b = _c(bits, np.uint16)
        out = np.empty(b.shape, np.float64)
        self.lib.w4o_half_to_double_array(_ptr(b), _ptr(out), b.size)
        return out

    def double_to_half(self, values) -> np.ndarray:
        v = _c(values, np.float64)
        out = np.empty(v.shape, np.uint16)
        self.lib.w4o_double_to_half_array(_ptr(v), _ptr(out), v.size)
        return out

    # ---------------------------------------------------------------------------- format
    def unpack(self, qweight) -> np.ndarray:
        """uint8 q[K, N] from canonical int32 qweight[K/8, N]."""
        qw = _c(qweight, np.int32)
        K, N = qw.shape[0] * 8, qw.shape[1]
        out = np.empty((K, N), np.uint8)
        self.lib.w4o_unpack(_ptr(qw), K, N, _ptr(out))
        return out

    def dequant(self, qweight, scales, group: int) -> np.ndarray:
        """float64 w[K, N] = fp16_rne((q - 8) * s); every value is exactly an fp16 number."""
        qw = _c(qweight, np.int32)
        sc = _c(scales, np.uint16)
        K, N = qw.shape[0] * 8, qw.shape[1]
        out = np.empty((K, N), np.float64)
        self.lib.w4o_dequant(_ptr(qw), _ptr(sc), K, N, group, _ptr(out))
        return out

    # ---------------------------------------------------------------------------- GEMM
    def gemm(self, x_bits, qweight, scales, group: int, nthreads: int | None = None):
        """(y, absy) float64 [M, N]: y = sum_k x*w, absy = sum_k |x*w| (the tolerance scale)."""
        x = _c(x_bits, np.uint16)
        qw = _c(qweight, np.int32)
        sc = _c(scales, np.uint16)
        M, K = x.shape
        N = qw.shape[1]
        if qw.shape[0] * 8 != K:
            raise ValueError("qweight must have K/8 rows")
        y = np.empty((M, N), np.float64)
        a = np.empty((M, N), np.float64)
        rc = self.lib.w4o_gemm(_ptr(x), _ptr(qw), _ptr(sc), M, N, K, group, _ptr(y), _ptr(a),
                               nthreads or default_threads())
        if rc != 0:
            raise ValueError(f"oracle gemm rejected the shape (rc={rc})")
        return y, a

    def gemm_xf64(self, x, qweight, scales, group: int, nthreads: int | None = None):
        """As ``gemm`` with the activations given directly as float64 (linearity pin)."""
        xd = _c(x, np.float64)
        qw = _c(qweight, np.int32)
        sc = _c(scales, np.uint16)
        M, K = xd.shape
        N = qw.shape[1]
        y = np.empty((M, N), np.float64)
        a = np.empty((M, N), np.float64)
        rc = self.lib.w4o_gemm_xf64(_ptr(xd), _ptr(qw), _ptr(sc), M, N, K, group, _ptr(y), _ptr(a),
                                    nthreads or default_threads())
        if rc != 0:
            raise ValueError(f"oracle gemm rejected the shape (rc={rc})")
        return y, a

    def gemm_sampled(self, x_bits, qweight, scales, group: int, ms, ns, nthreads: int | None = None):
        """(y, absy) float64 [count] for the listed (m, n) pairs only."""
        x = _c(x_bits, np.uint16)
        qw = _c(qweight, np.int32)
        sc = _c(scales, np.uint16)
        msa = _c(ms, np.int64)
        nsa = _c(ns, np.int64)
        M, K = x.shape
        N = qw.shape[1]
        y = np.empty(msa.shape, np.float64)
        a = np.empty(msa.shape, np.float64)
        rc = self.lib.w4o_gemm_sampled(_ptr(x), _ptr(qw), _ptr(sc), M, N, K, group, _ptr(msa), _ptr(nsa),
                                       msa.size, _ptr(y), _ptr(a), nthreads or default_threads())
        if rc != 0:
            raise ValueError(f"oracle gemm_sampled rejected the input (rc={rc})")
        return y, a

    # ---------------------------------------------------------------------------- NVFP4
    def e2m1_to_double(self, codes) -> np.ndarray:
        """float64 values of 4-bit E2M1 codes."""
        c = np.asarray(codes)
        return np.array([self.lib.w4o_e2m1_to_double(int(v)) for v in c.reshape(-1)], np.float64).reshape(c.shape)

    def e4m3_to_double(self, bits) -> np.ndarray:
        """float64 values of E4M3 bit patterns (NaN for the NaN patterns)."""
        b = _c(bits, np.uint8)
        out = np.empty(b.shape, np.float64)
        self.lib.w4o_e4m3_to_double_array(_ptr(b), _ptr(out), b.size)
        return out

    def dequant_nvfp4(self, qweight, scales8) -> np.ndarray:
        """float64 w[K, N] = e2m1(q) * e4m3(s[k/16]) (without the tensor scale)."""
        qw = _c(qweight, np.int32)
        sc = _c(scales8, np.uint8)
        K, N = qw.shape[0] * 8, qw.shape[1]
        out = np.empty((K, N), np.float64)
        self.lib.w4o_dequant_nvfp4(_ptr(qw), _ptr(sc), K, N, _ptr(out))
        return out

    def gemm_nvfp4(self, x_bits, qweight, scales8, g: float, nthreads: int | None = None):
        """(y, absy) float64 [M, N]: y = g * sum_k x*w, absy = |g| * sum_k |x*w|."""
        x = _c(x_bits, np.uint16)
        qw = _c(qweight, np.int32)
        sc = _c(scales8, np.uint8)
        M, K = x.shape
        N = qw.shape[1]
        if qw.shape[0] * 8 != K or sc.shape != (K // 16, N):
            raise ValueError("qweight must be [K/8, N] and scales8 [K/16, N]")
        y = np.empty((M, N), np.float64)
        a = np.empty((M, N), np.float64)
        rc = self.lib.w4o_gemm_nvfp4(_ptr(x), _ptr(qw), _ptr(sc), float(g), M, N, K, _ptr(y), _ptr(a),
                                     nthreads or default_threads())
        if rc != 0:
            raise ValueError(f"oracle gemm_nvfp4 rejected the shape (rc={rc})")
        return y, a

    def gemm_nvfp4_sampled(self, x_bits, qweight, scales8, g: float, ms, ns):
        """(y, absy) float64 [count] for the listed (m, n) pairs only."""
        x = _c(x_bits, np.uint16)
        qw = _c(qweight, np.int32)
        sc = _c(scales8, np.uint8)
        msa = _c(ms, np.int64)
        nsa = _c(ns, np.int64)
        M, K = x.shape
        N = qw.shape[1]
        y = np.empty(msa.shape, np.float64)
        a = np.empty(msa.shape, np.float64)
        rc = self.lib.w4o_gemm_nvfp4_sampled(_ptr(x), _ptr(qw), _ptr(sc), float(g), M, N, K, _ptr(msa), _ptr(nsa),
                                             msa.size, _ptr(y), _ptr(a))
        if rc != 0:
            raise ValueError(f"oracle gemm_nvfp4_sampled rejected the input (rc={rc})")
        return y, a

    # ---------------------------------------------------------------------------- W4A8
    def quantize_x_int8(self, x_bits):
        """(xq int8 [M, K], sx float32 [M]): per-token symmetric int8 quantisation of fp16 x."""
        x = _c(x_bits, np.uint16)
        M, K = x.shape
        xq = np.empty((M, K), np.int8)
        sx = np.empty(M, np.float32)
        rc = self.lib.w4o_quantize_x_int8(_ptr(x), M, K, _ptr(xq), _ptr(sx))
        if rc != 0:
            raise ValueError(f"oracle quantize_x_int8 rejected the shape (rc={rc})")
        return xq, sx

    def gemm_w4a8(self, xq, sx, qweight, scales, G: int, nthreads: int | None = None):
        """(y, absy) float64 [M, N]: y = sx * sum_g s * sum (q - 8) xq; absy = sum_k |sx xq (q - 8) s|."""
        xa = _c(xq, np.int8)
        sa = _c(sx, np.float32)
        qw = _c(qweight, np.int32)
        sc = _c(scales, np.uint16)
        M, K = xa.shape
        N = qw.shape[1]
        if qw.shape[0] * 8 != K or sc.shape != (K // G, N) or sa.shape != (M,):
            raise ValueError("xq [M, K], sx [M], qweight [K/8, N], scales [K/G, N] expected")
        y = np.empty((M, N), np.float64)
        a = np.empty((M, N), np.float64)
        rc = self.lib.w4o_gemm_w4a8(_ptr(xa), _ptr(sa), _ptr(qw), _ptr(sc), M, N, K, G, _ptr(y), _ptr(a),
                                    nthreads or default_threads())
        if rc != 0:
            raise ValueError(f"oracle gemm_w4a8 rejected the shape (rc={rc})")
        return y, a

    def gemm_w4a8_sampled(self, xq, sx, qweight, scales, G: int, ms, ns):
        """(y, absy) float64 [count] for the listed (m, n) pairs only."""
        xa = _c(xq, np.int8)
        sa = _c(sx, np.float32)
        qw = _c(qweight, np.int32)
        sc = _c(scales, np.uint16)
        msa = _c(ms, np.int64)
        nsa = _c(ns, np.int64)
        M, K = xa.shape
        N = qw.shape[1]
        y = np.empty(msa.shape, np.float64)
        a = np.empty(msa.shape, np.float64)
        rc = self.lib.w4o_gemm_w4a8_sampled(_ptr(xa), _ptr(sa), _ptr(qw), _ptr(sc), M, N, K, G, _ptr(msa),
                                            _ptr(nsa), msa.size, _ptr(y), _ptr(a))
        if rc != 0:
            raise ValueError(f"oracle gemm_w4a8_sampled rejected the input (rc={rc})")
        return y, a

    def repack_nvfp4(self, qweight, scales8):
        """(wr uint32 [N*K/8], sr uint16 [N*K/16]): the NVFP4 device layout (flat)."""
        qw = _c(qweight, np.int32)
        sc = _c(scales8, np.uint8)
        K, N = qw.shape[0] * 8, qw.shape[1]
        wr = np.empty(N * K // 8, np.uint32)
        sr = np.empty(N * (K // 16), np.uint16)
        rc = self.lib.w4o_repack_nvfp4(_ptr(qw), _ptr(sc), K, N, _ptr(wr), _ptr(sr))
        if rc != 0:
            raise ValueError(f"oracle repack_nvfp4 rejected the shape (rc={rc})")
        return wr, sr

    def unrepack_nvfp4(self, wr, sr, K: int, N: int):
        """Inverse of ``repack_nvfp4``: (qweight int32 [K/8, N], scales8 uint8 [K/16, N])."""
        w = _c(wr, np.uint32)
        s = _c(sr, np.uint16)
        qw = np.empty((K // 8, N), np.int32)
        sc = np.empty((K // 16, N), np.uint8)
        rc = self.lib.w4o_unrepack_nvfp4(_ptr(w), _ptr(s), K, N, _ptr(qw), _ptr(sc))
        if rc != 0:
            raise ValueError(f"oracle unrepack_nvfp4 rejected the input (rc={rc})")
        return qw, sc

    # ---------------------------------------------------------------------------- activation
    def silu_mul(self, gu_bits):
        """(act float64 [M, I], act_half uint16 [M, I]) for fp16 bits gu [M, 2I] (gate, then up):
        act = silu(gate) * up in double and its fp16 rounding."""
        gu = _c(gu_bits, np.uint16)
        M, I2 = gu.shape
        if I2 % 2:
            raise ValueError("gu must have an even number of columns")
        I = I2 // 2
        act = np.empty((M, I), np.float64)
        half = np.empty((M, I), np.uint16)
        self.lib.w4o_silu_mul(_ptr(gu), M, I, _ptr(act), _ptr(half))
        return act, half

    # ---------------------------------------------------------------------------- layout
    def repack(self, qweight, scales, group: int):
        """(wr uint32 [N*K/8], sr uint16 [N*K/G]): the device layout (flat; see w4a16_oracle.c)."""
        qw = _c(qweight, np.int32)
        sc = _c(scales, np.uint16)
        K, N = qw.shape[0] * 8, qw.shape[1]
        wr = np.empty(N * K // 8, np.uint32)
        sr = np.empty(N * (K // group), np.uint16)
        rc = self.lib.w4o_repack(_ptr(qw), _ptr(sc), K, N, group, _ptr(wr), _ptr(sr))
        if rc != 0:
            raise ValueError(f"oracle repack rejected the shape (rc={rc})")
        return wr, sr

    def unrepack(self, wr, sr, K: int, N: int, group: int):
        """Inverse of ``repack``: (qweight int32 [K/8, N], scales uint16 [K/G, N])."""
        w = _c(wr, np.uint32)
        s = _c(sr, np.uint16)
        qw = np.empty((K // 8, N), np.int32)
        sc = np.empty((K // group, N), np.uint16)
        rc = self.lib.w4o_unrepack(_ptr(w), _ptr(s), K, N, group, _ptr(qw), _ptr(sc))
        if rc != 0:
            raise ValueError(f"oracle unrepack rejected the shape (rc={rc})")
        return qw, sc


def load() -> Oracle:
    """The oracle built from this directory's source (built on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = Oracle(build())
        return _lib


def load_from_source(c_source: str, workdir: str) -> Oracle:
    """Compile an alternative C source text (tests use this to plant mistakes) and load it."""
    src = os.path.join(workdir, "variant.c")
    with open(src, "w") as f:
        f.write(c_source)
    out = os.path.join(workdir, f"libvariant_{abs(hash(c_source))}.so")
    return Oracle(_compile(src, out))


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def has_openmp() -> bool:
    return load().has_openmp()


def half_to_double(bits):
    return load().half_to_double(bits)


def double_to_half(values):
    return load().double_to_half(values)


def unpack(qweight):
    return load().unpack(qweight)


def dequant(qweight, scales, group: int):
    return load().dequant(qweight, scales, group)


def gemm(x_bits, qweight, scales, group: int, nthreads: int | None = None):
    return load().gemm(x_bits, qweight, scales, group, nthreads)


def gemm_xf64(x, qweight, scales, group: int, nthreads: int | None = None):
    return load().gemm_xf64(x, qweight, scales, group, nthreads)


def gemm_sampled(x_bits, qweight, scales, group: int, ms, ns, nthreads: int | None = None):
    return load().gemm_sampled(x_bits, qweight, scales, group, ms, ns, nthreads)


def silu_mul(gu_bits):
    return load().silu_mul(gu_bits)


def repack(qweight, scales, group: int):
    return load().repack(qweight, scales, group)


def unrepack(wr, sr, K: int, N: int, group: int):
    return load().unrepack(wr, sr, K, N, group)


def e2m1_to_double(codes):
    return load().e2m1_to_double(codes)


def e4m3_to_double(bits):
    return load().e4m3_to_double(bits)


def dequant_nvfp4(qweight, scales8):
    return load().dequant_nvfp4(qweight, scales8)


def gemm_nvfp4(x_bits, qweight, scales8, g: float, nthreads: int | None = None):
    return load().gemm_nvfp4(x_bits, qweight, scales8, g, nthreads)


def gemm_nvfp4_sampled(x_bits, qweight, scales8, g: float, ms, ns):
    return load().gemm_nvfp4_sampled(x_bits, qweight, scales8, g, ms, ns)


def repack_nvfp4(qweight, scales8):
    return load().repack_nvfp4(qweight, scales8)


def unrepack_nvfp4(wr, sr, K: int, N: int):
    return load().unrepack_nvfp4(wr, sr, K, N)


def quantize_x_int8(x_bits):
    return load().quantize_x_int8(x_bits)


def gemm_w4a8(xq, sx, qweight, scales, G: int, nthreads: int | None = None):
    return load().gemm_w4a8(xq, sx, qweight, scales, G, nthreads)


def gemm_w4a8_sampled(xq, sx, qweight, scales, G: int, ms, ns):
    return load().gemm_w4a8_sampled(xq, sx, qweight, scales, G, ms, ns)


# ------------------------------------------------------------------------------------ check
TOL_REL = 2.0 ** -10
TOL_ABS_SCALE = 2.0 ** -10


def within_tolerance(y_gpu_f64: np.ndarray, y_ref: np.ndarray, abs_ref: np.ndarray):
    """Acceptance per element: |y - y_ref| <= 2^-10 |y_ref| + 2^-10 sum_k |x w|, all finite.

    Returns (ok: bool, worst_ratio: float, n_bad: int); worst_ratio is max |err| / bound.
    """
    bound = TOL_REL * np.abs(y_ref) + TOL_ABS_SCALE * abs_ref
    err = np.abs(y_gpu_f64 - y_ref)
    finite = np.isfinite(y_gpu_f64)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / np.where(bound > 0, bound, 1.0), np.where(err == 0, 0.0, np.inf))
    ratio = np.where(finite, ratio, np.inf)
    bad = ~(err <= bound) | ~finite
    worst = float(ratio.max()) if ratio.size else 0.0
    return (not bool(bad.any())), worst, int(bad.sum())
