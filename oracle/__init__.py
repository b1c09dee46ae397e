"""CPU oracle for out[M,N] = x[M,K] @ W[N,K]^T (+ bias[N]), bf16 in, bf16 out.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference legs of ``bench.py`` may import this package.  The
CUDA library (``moe_router_gemm_gb300``) never imports it and shares no code
with it; the only thing both sides use is the seeded input generator in
``workloads.py``, which holds none of the method's arithmetic.

The arithmetic lives in ``oracle.c`` (plain C, f64): widen every bf16 input to
f64, sum the products in ascending k, add the bias, round once to bf16 (round
to nearest, ties to even, written from the IEEE format definition).  The
definition follows the header comment of the TGV BF16 GEMM kernel on the sglang
PR #30117 page ("关键源码片段"): out[M, N] = x[M, K] @ weight[N, K].T
(+ bias[N]), bf16 in and out, fp32 accumulation inside.

Pins (tests/test_oracle_pins.py): rounding against an exact-rational
re-derivation and against torch's float32->bfloat16 cast; one-hot rows; all-ones
closed form; power-of-two scaling; linearity of the unrounded sum; bias
exactness; exact-rational brute force on tiny shapes; numpy's f64 matmul.

Arrays cross the boundary as numpy uint16 bit patterns (bf16) in C order.

Per-tensor FP8 (oracle.c, second part; the sglang PR #28333 page): e4m3
decoding from the format definition, the static quantisation of the page's
kernel (binary32 reciprocal and product, clamp to +-448, round to nearest
even), and the FP8 linear (exact f64 sum of e4m3 products, times both scales,
plus bias, one rounding to bf16).  e4m3 codes cross the boundary as uint8.

MXFP8 (oracle.c, third part; the sglang PR #34042 page, read as the OCP
microscaling format): 32-element blocks along K sharing one E8M0 scale byte,
the block quantisation (scale exponent floor(log2 max|v|) - 8, elements
rounded to nearest even e4m3 with saturation), and the block-scaled linear
(exact f64 terms summed in ascending k, plus bias, one rounding to bf16).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")


_u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_u32p = np.ctypeslib.ndpointer(dtype=np.uint32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_i64 = ctypes.c_int64


def compile_source(src: str, out_path: str) -> str:
    """Compile one C source of the oracle into a shared object with gcc."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    tmp = out_path + f".tmp{os.getpid()}"
    # -ffp-contract=off keeps a*b+c as two roundings on every host (the products
    # are exact in f64 anyway, so this only removes a needless source of variation).
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC",
                           "-shared", "-o", tmp, src])
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so for the host it runs on."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


class Oracle:
    """ctypes view of one build of oracle.c (the default build, or a test mutant)."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        lib.oracle_rne_bf16.argtypes = [ctypes.c_double]
        lib.oracle_rne_bf16.restype = ctypes.c_uint16
        lib.oracle_rne_f32.argtypes = [ctypes.c_double]
        lib.oracle_rne_f32.restype = ctypes.c_uint32
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        opt = ctypes.c_void_p  # bias may be NULL: passed as a raw pointer
        lib.oracle_linear_f64.argtypes = [_u16p, _u16p, opt, _i64, _i64, _i64, _f64p]
        lib.oracle_linear_bf16.argtypes = [_u16p, _u16p, opt, _i64, _i64, _i64, _u16p]
        lib.oracle_linear_f32.argtypes = [_u16p, _u16p, opt, _i64, _i64, _i64, _u32p]
        lib.oracle_linear_rows_bf16.argtypes = [_u16p, _u16p, opt, _i64, _i64, _i64,
                                                _i64p, _i64, _u16p]
        lib.oracle_linear_rows_f64.argtypes = [_u16p, _u16p, opt, _i64, _i64, _i64,
                                               _i64p, _i64, _f64p]
        lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_f64.restype = ctypes.c_double
        lib.oracle_rne_e4m3.argtypes = [ctypes.c_double]
        lib.oracle_rne_e4m3.restype = ctypes.c_uint8
        lib.oracle_quant_fp8.argtypes = [_u16p, _i64, ctypes.c_float, _u8p]
        lib.oracle_linear_fp8.argtypes = [_u8p, _u8p, ctypes.c_float, ctypes.c_float, opt, _i64, _i64, _i64, _u16p]
        lib.oracle_linear_fp8_f64.argtypes = [_u8p, _u8p, ctypes.c_float, ctypes.c_float, opt, _i64, _i64, _i64,
                                              _f64p]
        lib.oracle_e8m0_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_e8m0_to_f64.restype = ctypes.c_double
        lib.oracle_quant_mxfp8.argtypes = [_u16p, _i64, _i64, _u8p, _u8p]
        lib.oracle_linear_mxfp8.argtypes = [_u8p, _u8p, _u8p, _u8p, opt, _i64, _i64, _i64, _u16p]
        lib.oracle_linear_mxfp8_f64.argtypes = [_u8p, _u8p, _u8p, _u8p, opt, _i64, _i64, _i64, _f64p]
        lib.oracle_linear_rows_mxfp8.argtypes = [_u8p, _u8p, _u8p, _u8p, opt, _i64, _i64, _i64, _i64p, _i64,
                                                 _u16p]
        for fn in ("oracle_linear_f64", "oracle_linear_bf16", "oracle_linear_f32",
                   "oracle_linear_rows_bf16", "oracle_linear_rows_f64", "oracle_quant_fp8",
                   "oracle_linear_fp8", "oracle_linear_fp8_f64", "oracle_quant_mxfp8",
                   "oracle_linear_mxfp8", "oracle_linear_mxfp8_f64", "oracle_linear_rows_mxfp8"):
            getattr(lib, fn).restype = None
        self.lib = lib
        self.path = lib_path

    # ---- the oracle's entry points (numpy uint16 bf16 bit patterns in) ----

    def linear_bf16(self, x, W, bias=None) -> np.ndarray:
        """bf16 bits out[M,N] of the defined result (one rounding of the f64 sum)."""
        x, W, bias, M, N, K = _prep(x, W, bias)
        out = np.empty((M, N), dtype=np.uint16)
        self.lib.oracle_linear_bf16(x, W, _bias_ptr(bias), M, N, K, out)
        return out

    def linear_f64(self, x, W, bias=None) -> np.ndarray:
        """The unrounded f64 sums acc[M,N] (for invariant checks)."""
        x, W, bias, M, N, K = _prep(x, W, bias)
        out = np.empty((M, N), dtype=np.float64)
        self.lib.oracle_linear_f64(x, W, _bias_ptr(bias), M, N, K, out)
        return out

    def linear_f32(self, x, W, bias=None) -> np.ndarray:
        """binary32 bits out[M,N]: the f64 sum rounded once to fp32 (router-logits variant)."""
        x, W, bias, M, N, K = _prep(x, W, bias)
        out = np.empty((M, N), dtype=np.uint32)
        self.lib.oracle_linear_f32(x, W, _bias_ptr(bias), M, N, K, out)
        return out

    def linear_rows_bf16(self, x, W, bias, rows) -> np.ndarray:
        """bf16 bits of the selected output rows only: out[len(rows), N]."""
        x, W, bias, M, N, K = _prep(x, W, bias)
        rows = _rows(rows, M)
        out = np.empty((rows.size, N), dtype=np.uint16)
        self.lib.oracle_linear_rows_bf16(x, W, _bias_ptr(bias), M, N, K, rows, rows.size, out)
        return out

    def linear_rows_f64(self, x, W, bias, rows) -> np.ndarray:
        """Unrounded f64 sums of the selected output rows: acc[len(rows), N]."""
        x, W, bias, M, N, K = _prep(x, W, bias)
        rows = _rows(rows, M)
        out = np.empty((rows.size, N), dtype=np.float64)
        self.lib.oracle_linear_rows_f64(x, W, _bias_ptr(bias), M, N, K, rows, rows.size, out)
        return out

    def rne_bf16(self, values) -> np.ndarray:
        """Round each f64 value to bf16 (bits), ties to even."""
        v = np.asarray(values, dtype=np.float64).ravel()
        f = self.lib.oracle_rne_bf16
        return np.array([f(float(a)) for a in v], dtype=np.uint16)

    def rne_f32(self, values) -> np.ndarray:
        """Round each f64 value to binary32 (bits), ties to even."""
        v = np.asarray(values, dtype=np.float64).ravel()
        f = self.lib.oracle_rne_f32
        return np.array([f(float(a)) for a in v], dtype=np.uint32)

    def bf16_to_f64(self, bits) -> np.ndarray:
        """Exact widening of bf16 bit patterns to f64."""
        b = np.asarray(bits, dtype=np.uint16).ravel()
        f = self.lib.oracle_bf16_to_f64
        return np.array([f(int(h)) for h in b], dtype=np.float64)

    # ---- per-tensor FP8 (e4m3 codes as numpy uint8) ----

    def e4m3_to_f64(self, codes) -> np.ndarray:
        """Exact value of each e4m3 code (NaN for 0x7F / 0xFF)."""
        c = np.asarray(codes, dtype=np.uint8).ravel()
        f = self.lib.oracle_e4m3_to_f64
        return np.array([f(int(v)) for v in c], dtype=np.float64)

    def rne_e4m3(self, values) -> np.ndarray:
        """Round each value (|v| <= 448) to the nearest e4m3 code, ties to even."""
        v = np.asarray(values, dtype=np.float64).ravel()
        f = self.lib.oracle_rne_e4m3
        return np.array([f(float(a)) for a in v], dtype=np.uint8)

    def quant_fp8(self, x, scale: float) -> np.ndarray:
        """Static per-tensor quantisation of bf16 bits x to e4m3 codes (same shape)."""
        x = np.ascontiguousarray(x, dtype=np.uint16)
        q = np.empty(x.shape, dtype=np.uint8)
        self.lib.oracle_quant_fp8(x.ravel(), x.size, float(scale), q.reshape(-1))
        return q

    def _fp8_prep(self, xq, wq, bias):
        xq = np.ascontiguousarray(xq, dtype=np.uint8)
        wq = np.ascontiguousarray(wq, dtype=np.uint8)
        if xq.ndim != 2 or wq.ndim != 2 or xq.shape[1] != wq.shape[1]:
            raise ValueError(f"shapes xq{xq.shape} wq{wq.shape}: need xq[M,K], wq[N,K]")
        M, K = xq.shape
        N = wq.shape[0]
        if bias is not None:
            bias = np.ascontiguousarray(bias, dtype=np.uint16)
            if bias.shape != (N,):
                raise ValueError(f"bias shape {bias.shape}: need ({N},)")
        return xq, wq, bias, M, N, K

    def linear_fp8(self, xq, wq, sx: float, sw: float, bias=None) -> np.ndarray:
        """bf16 bits of the FP8 linear: RNE_bf16(sx * sw * sum_k e4m3(xq) e4m3(wq) + bias)."""
        xq, wq, bias, M, N, K = self._fp8_prep(xq, wq, bias)
        out = np.empty((M, N), dtype=np.uint16)
        self.lib.oracle_linear_fp8(xq, wq, float(sx), float(sw), _bias_ptr(bias), M, N, K, out)
        return out

    def linear_fp8_f64(self, xq, wq, sx: float, sw: float, bias=None) -> np.ndarray:
        """The unrounded FP8 result (f64)."""
        xq, wq, bias, M, N, K = self._fp8_prep(xq, wq, bias)
        out = np.empty((M, N), dtype=np.float64)
        self.lib.oracle_linear_fp8_f64(xq, wq, float(sx), float(sw), _bias_ptr(bias), M, N, K, out)
        return out

    # ---- MXFP8: e4m3 codes (uint8) with one E8M0 scale byte per 32 elements along K ----

    def e8m0_to_f64(self, scales) -> np.ndarray:
        """Exact value 2^(e - 127) of each E8M0 scale byte (NaN for 255)."""
        c = np.asarray(scales, dtype=np.uint8).ravel()
        f = self.lib.oracle_e8m0_to_f64
        return np.array([f(int(v)) for v in c], dtype=np.float64)

    def quant_mxfp8(self, x):
        """MXFP8 quantisation of bf16 bits x[rows, K] (K % 32 == 0): (codes[rows, K], scales[rows, K/32])."""
        x = np.ascontiguousarray(x, dtype=np.uint16)
        if x.ndim != 2 or x.shape[1] % 32:
            raise ValueError(f"x shape {x.shape}: need [rows, K] with K % 32 == 0")
        rows, K = x.shape
        q = np.empty((rows, K), dtype=np.uint8)
        s = np.empty((rows, K // 32), dtype=np.uint8)
        self.lib.oracle_quant_mxfp8(x.reshape(-1), rows, K, q.reshape(-1), s.reshape(-1))
        return q, s

    def _mx_prep(self, xq, sx, wq, sw, bias):
        xq, wq, bias, M, N, K = self._fp8_prep(xq, wq, bias)
        if K % 32:
            raise ValueError(f"K = {K}: need K % 32 == 0")
        sx = np.ascontiguousarray(sx, dtype=np.uint8)
        sw = np.ascontiguousarray(sw, dtype=np.uint8)
        if sx.shape != (M, K // 32) or sw.shape != (N, K // 32):
            raise ValueError(f"scale shapes {sx.shape}, {sw.shape}: need ({M}, {K // 32}), ({N}, {K // 32})")
        return xq, sx, wq, sw, bias, M, N, K

    def linear_mxfp8(self, xq, sx, wq, sw, bias=None) -> np.ndarray:
        """bf16 bits of the MXFP8 linear (block-scaled e4m3 operands, bias, one rounding)."""
        xq, sx, wq, sw, bias, M, N, K = self._mx_prep(xq, sx, wq, sw, bias)
        out = np.empty((M, N), dtype=np.uint16)
        self.lib.oracle_linear_mxfp8(xq, sx, wq, sw, _bias_ptr(bias), M, N, K, out)
        return out

    def linear_mxfp8_f64(self, xq, sx, wq, sw, bias=None) -> np.ndarray:
        """The unrounded MXFP8 result (f64)."""
        xq, sx, wq, sw, bias, M, N, K = self._mx_prep(xq, sx, wq, sw, bias)
        out = np.empty((M, N), dtype=np.float64)
        self.lib.oracle_linear_mxfp8_f64(xq, sx, wq, sw, _bias_ptr(bias), M, N, K, out)
        return out

    def linear_rows_mxfp8(self, xq, sx, wq, sw, bias, rows) -> np.ndarray:
        """bf16 bits of the selected output rows of the MXFP8 linear."""
        xq, sx, wq, sw, bias, M, N, K = self._mx_prep(xq, sx, wq, sw, bias)
        rows = _rows(rows, M)
        out = np.empty((rows.size, N), dtype=np.uint16)
        self.lib.oracle_linear_rows_mxfp8(xq, sx, wq, sw, _bias_ptr(bias), M, N, K, rows, rows.size, out)
        return out


def _prep(x, W, bias):
    x = np.ascontiguousarray(x, dtype=np.uint16)
    W = np.ascontiguousarray(W, dtype=np.uint16)
    if x.ndim != 2 or W.ndim != 2 or x.shape[1] != W.shape[1]:
        raise ValueError(f"shapes x{x.shape} W{W.shape}: need x[M,K], W[N,K]")
    M, K = x.shape
    N = W.shape[0]
    if bias is not None:
        bias = np.ascontiguousarray(bias, dtype=np.uint16)
        if bias.shape != (N,):
            raise ValueError(f"bias shape {bias.shape}: need ({N},)")
    return x, W, bias, M, N, K


def _rows(rows, M):
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    if rows.size and (rows.min() < 0 or rows.max() >= M):
        raise ValueError("row index out of range")
    return rows


def _bias_ptr(bias):
    return None if bias is None else bias.ctypes.data


_default = None
_lock = threading.Lock()


def default() -> Oracle:
    """The oracle built from oracle.c (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default


def linear_bf16(x, W, bias=None):
    return default().linear_bf16(x, W, bias)


def linear_f64(x, W, bias=None):
    return default().linear_f64(x, W, bias)


def linear_f32(x, W, bias=None):
    return default().linear_f32(x, W, bias)


def linear_rows_bf16(x, W, bias, rows):
    return default().linear_rows_bf16(x, W, bias, rows)


def linear_rows_f64(x, W, bias, rows):
    return default().linear_rows_f64(x, W, bias, rows)


def rne_bf16(values):
    return default().rne_bf16(values)


def rne_f32(values):
    return default().rne_f32(values)


def bf16_to_f64(bits):
    return default().bf16_to_f64(bits)


def e4m3_to_f64(codes):
    return default().e4m3_to_f64(codes)


def rne_e4m3(values):
    return default().rne_e4m3(values)


def quant_fp8(x, scale):
    return default().quant_fp8(x, scale)


def linear_fp8(xq, wq, sx, sw, bias=None):
    return default().linear_fp8(xq, wq, sx, sw, bias)


def linear_fp8_f64(xq, wq, sx, sw, bias=None):
    return default().linear_fp8_f64(xq, wq, sx, sw, bias)


def e8m0_to_f64(scales):
    return default().e8m0_to_f64(scales)


def quant_mxfp8(x):
    return default().quant_mxfp8(x)


def linear_mxfp8(xq, sx, wq, sw, bias=None):
    return default().linear_mxfp8(xq, sx, wq, sw, bias)


def linear_mxfp8_f64(xq, sx, wq, sw, bias=None):
    return default().linear_mxfp8_f64(xq, sx, wq, sw, bias)


def linear_rows_mxfp8(xq, sx, wq, sw, bias, rows):
    return default().linear_rows_mxfp8(xq, sx, wq, sw, bias, rows)
