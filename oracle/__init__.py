"""Oracle for the LLM.int8() mixed-precision decomposition linear.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the CPU-baseline / reference leg of ``bench.py`` may import this package.
The CUDA path never imports it and shares no code with it.

Two independent statements of the method:

* ``oracle.c`` (through :class:`Oracle`): plain C loops with OpenMP, int64
  accumulation checked to fit int32, epilogue in double with one final
  rounding to fp16 (or bf16).  Usable at full size for S1-S3 and on sampled
  rows for S4-S6.  Forms: fp16 or bf16 data (``fmt``), an optional bias, and
  the outlier weights from W16 or, with ``W16=None``, from the int8 codes
  dequantized; and the blockwise 8-bit codec of optimizer states.
* :mod:`oracle.brute`: pure Python with exact integers and
  :class:`fractions.Fraction`, for tiny inputs.

Every function follows the statement of LLM.int8() on the pages:
outlier feature dimensions computed in 16-bit, the rest vector-wise int8,
converted back to 16-bit at the end ("Hugging Face Quantization with
bitsandbytes: 4-bit & 8-bit Models Explained", section 2; threshold default
6.0 in section 3; "bitsandbytes: GPU-Accelerated Inference and Training at
Lower Bit Depths", section "How LLM.int8() quantizes weights and
activations").  The readings taken where the pages are silent are listed in
``oracle.c``'s header.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build_oracle

_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_P)


_FMT = {"fp16": 0, "bf16": 1}


def _bits16(a, fmt: str) -> np.ndarray:
    """16-bit element bit patterns, C-contiguous: float16 arrays for fp16,
    uint16 arrays of bfloat16 bit patterns for bf16."""
    if fmt == "fp16":
        return np.ascontiguousarray(a, dtype=np.float16).view(np.uint16)
    if fmt == "bf16":
        a = np.asarray(a)
        if a.dtype != np.uint16:
            raise TypeError("bf16 data is passed as uint16 bit patterns")
        return np.ascontiguousarray(a)
    raise ValueError(fmt)


class Oracle:
    """ctypes front of ``liboracle.so`` (compiled on first use)."""

    def __init__(self, lib_path: str | None = None):
        path = lib_path or build_oracle.build()
        lib = ctypes.CDLL(path)
        lib.orc_half_to_double.restype = ctypes.c_double
        lib.orc_half_to_double.argtypes = [ctypes.c_uint16]
        lib.orc_double_to_half.restype = ctypes.c_uint16
        lib.orc_double_to_half.argtypes = [ctypes.c_double]
        lib.orc_bf16_to_double.restype = ctypes.c_double
        lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.orc_double_to_bf16.restype = ctypes.c_uint16
        lib.orc_double_to_bf16.argtypes = [ctypes.c_double]
        for name in ("orc_quantize_weight", "orc_outlier_columns",
                     "orc_quantize_activations", "orc_int8_matmul_rows",
                     "orc_linear_rows", "orc_quantize_blockwise", "orc_dequantize_blockwise"):
            getattr(lib, name).restype = ctypes.c_int
        self.lib = lib

    def num_threads(self) -> int:
        return int(self.lib.orc_num_threads())

    # ---- elementwise helpers -------------------------------------------------
    def half_to_double(self, bits: int) -> float:
        return self.lib.orc_half_to_double(bits)

    def double_to_half(self, v: float) -> int:
        return self.lib.orc_double_to_half(v)

    def bf16_to_double(self, bits: int) -> float:
        return self.lib.orc_bf16_to_double(bits)

    def double_to_bf16(self, v: float) -> int:
        return self.lib.orc_double_to_bf16(v)

    # ---- the blockwise 8-bit codec of optimizer states ---------------------------
    def quantize_blockwise(self, x: np.ndarray, block: int):
        """fp32 values -> (int8 codes, fp32 absmax per block of ``block``)."""
        x = np.ascontiguousarray(x, dtype=np.float32).ravel()
        n = x.size
        q = np.empty(n, np.int8)
        absmax = np.empty((n + block - 1) // block, np.float32)
        rc = self.lib.orc_quantize_blockwise(_ptr(x), _I64(n), _I64(block), _ptr(q),
                                             _ptr(absmax))
        assert rc == 0, rc
        return q, absmax

    def dequantize_blockwise(self, q: np.ndarray, absmax: np.ndarray, block: int):
        q = np.ascontiguousarray(q, dtype=np.int8).ravel()
        absmax = np.ascontiguousarray(absmax, dtype=np.float32)
        y = np.empty(q.size, np.float32)
        rc = self.lib.orc_dequantize_blockwise(_ptr(q), _ptr(absmax), _I64(q.size),
                                               _I64(block), _ptr(y))
        assert rc == 0, rc
        return y

    # ---- S1 -------------------------------------------------------------------
    def quantize_weight(self, W16: np.ndarray, fmt: str = "fp16"):
        """fmt "fp16": W16 float16; fmt "bf16": W16 holds bfloat16 bit
        patterns (uint16)."""
        W16 = _bits16(W16, fmt)
        N, K = W16.shape
        Wq = np.empty((N, K), np.int8)
        sw = np.empty(N, np.float32)
        rc = self.lib.orc_quantize_weight(_ptr(W16), _I64(N), _I64(K),
                                          _ptr(Wq), _ptr(sw), _FMT[fmt])
        assert rc == 0, rc
        return Wq, sw

    # ---- S2 -------------------------------------------------------------------
    def outlier_columns(self, X16: np.ndarray, tau: float, fmt: str = "fp16"):
        X16 = _bits16(X16, fmt)
        T, K = X16.shape
        O = np.empty(max(K, 1), np.int32)
        n = ctypes.c_int32(0)
        rc = self.lib.orc_outlier_columns(_ptr(X16), _I64(T), _I64(K),
                                          ctypes.c_float(tau), _ptr(O), ctypes.byref(n),
                                          _FMT[fmt])
        assert rc == 0, rc
        return O[: n.value].copy()

    # ---- S3 -------------------------------------------------------------------
    def quantize_activations(self, X16: np.ndarray, O: np.ndarray, fmt: str = "fp16"):
        X16 = _bits16(X16, fmt)
        T, K = X16.shape
        O = np.ascontiguousarray(O, dtype=np.int32)
        Xq = np.empty((T, K), np.int8)
        sx = np.empty(T, np.float32)
        XO = np.empty((T, len(O)), np.uint16)
        rc = self.lib.orc_quantize_activations(
            _ptr(X16), _I64(T), _I64(K), _ptr(O), ctypes.c_int32(len(O)),
            _ptr(Xq), _ptr(sx), _ptr(XO) if len(O) else None, _FMT[fmt])
        if fmt == "fp16":
            XO = XO.view(np.float16)
        assert rc == 0, rc
        return Xq, sx, XO

    # ---- S4 -------------------------------------------------------------------
    def int8_matmul(self, Xq: np.ndarray, Wq: np.ndarray, rows=None):
        Xq = np.ascontiguousarray(Xq, dtype=np.int8)
        Wq = np.ascontiguousarray(Wq, dtype=np.int8)
        T, K = Xq.shape
        N = Wq.shape[0]
        rows = np.arange(T, dtype=np.int64) if rows is None else np.asarray(rows, np.int64)
        acc = np.empty((len(rows), N), np.int32)
        rc = self.lib.orc_int8_matmul_rows(_ptr(Xq), _ptr(Wq), _I64(T), _I64(N), _I64(K),
                                           _ptr(rows), _I64(len(rows)), _ptr(acc))
        assert rc == 0, "int32 accumulator overflow"
        return acc

    # ---- S2..S6 ---------------------------------------------------------------
    def linear(self, X16: np.ndarray, Wq: np.ndarray, sw: np.ndarray, W16: np.ndarray,
               tau: float, rows=None, bias=None, fmt: str = "fp16"):
        """Whole layer.  Returns a dict with O, Xq, sx (all rows) and, for
        ``rows`` (default: all), acc (int32), out (float64) and Y (float16).
        ``W16=None``: only the int8 weight is kept and the outlier weights are
        its codes dequantized, Wq * sw / 127.  fmt "bf16": X16, W16, bias
        and the returned Y are bfloat16 bit patterns (uint16)."""
        X16 = _bits16(X16, fmt)
        if W16 is not None:
            W16 = _bits16(W16, fmt)
        Wq = np.ascontiguousarray(Wq, dtype=np.int8)
        sw = np.ascontiguousarray(sw, dtype=np.float32)
        T, K = X16.shape
        N = Wq.shape[0]
        rows = np.arange(T, dtype=np.int64) if rows is None else np.asarray(rows, np.int64)
        R = len(rows)
        Xq = np.empty((T, K), np.int8)
        sx = np.empty(T, np.float32)
        O = np.empty(max(K, 1), np.int32)
        nO = ctypes.c_int32(0)
        acc = np.empty((R, N), np.int32)
        out = np.empty((R, N), np.float64)
        Y = np.empty((R, N), np.uint16)
        bias = None if bias is None else _bits16(bias, fmt)
        rc = self.lib.orc_linear_rows(
            _ptr(X16), _I64(T), _I64(K), _ptr(Wq), _ptr(sw),
            None if W16 is None else _ptr(W16), _I64(N), ctypes.c_float(tau),
            None if bias is None else _ptr(bias), _ptr(rows), _I64(R),
            _ptr(Xq), _ptr(sx), _ptr(O), ctypes.byref(nO), _ptr(acc), _ptr(out),
            _ptr(Y), _FMT[fmt])
        assert rc == 0, "int32 accumulator overflow"
        if fmt == "fp16":
            Y = Y.view(np.float16)
        return {"O": O[: nO.value].copy(), "Xq": Xq, "sx": sx, "acc": acc, "out": out,
                "Y": Y, "rows": rows}


_default = None


def get() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def lib_path() -> str:
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "liboracle.so")
