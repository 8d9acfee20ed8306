"""Thin ctypes binding of ``libbnbint8.so`` (argument marshalling only).

Every function here has the name and arguments of a C entry point in
``include/bnb_int8.h``; tensors are passed as device pointers, the stream as
torch's current stream handle.  All arithmetic happens in the CUDA library.
The library must have been built (``build.py`` / ``__graft_entry__.build``):
there is no fallback, a missing library raises.
"""

from __future__ import annotations

import ctypes
import enum
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libbnbint8.so")

_P = ctypes.c_void_p
_I64 = ctypes.c_int64


class Status(enum.IntEnum):
    OK = 0
    INVALID_ARG = 1
    UNSUPPORTED = 2
    CUDA = 3
    TIMEOUT = 4


class BnbError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = Status(status) if status in Status._value2member_map_ else status
        super().__init__(f"{where}: {self.status!r}")


class Lib:
    """The loaded C library with typed entry points."""

    SYMBOLS = ("bnb_int8_linear_workspace_bytes", "bnb_int8_quantize_weight",
               "bnb_int8_linear", "bnb_int8_linear_debug", "bnb_last_device_status",
               "bnb_status_string", "bnb_launch_count", "bnb_int8_linear_path",
               "bnb_int8_decode_cluster",
               "bnb_int8_linear_opts", "bnb_int8_linear_noalloc",
               "bnb_int8_linear_from_host", "bnb_int8_quantize_blockwise",
               "bnb_int8_dequantize_blockwise", "bnb_int8_linear_bias",
               "bnb_int8_linear_wq_only", "bnb_int8_quantize_weight_ex", "bnb_int8_linear_ex",
               "bnb_int8_linear_from_host_ex", "bnb_int8_linear_debug_ex")

    def __init__(self, path: str = LIB_PATH):
        if not os.path.exists(path):
            raise FileNotFoundError(
                f"{path} is not built; run `python -m int8_mixed_precision_04_b300.build`")
        self.path = path
        L = ctypes.CDLL(path)
        L.bnb_int8_linear_workspace_bytes.restype = ctypes.c_size_t
        L.bnb_int8_linear_workspace_bytes.argtypes = [_I64, _I64, _I64]
        L.bnb_int8_quantize_weight.restype = ctypes.c_int
        L.bnb_int8_quantize_weight.argtypes = [_P, _I64, _I64, _P, _P, _P]
        L.bnb_int8_linear.restype = ctypes.c_int
        L.bnb_int8_linear.argtypes = [_P, _I64, _I64, _P, _P, _P, _I64, ctypes.c_float, _P, _P,
                                      ctypes.c_size_t, _P]
        L.bnb_int8_linear_bias.restype = ctypes.c_int
        L.bnb_int8_linear_bias.argtypes = [_P, _I64, _I64, _P, _P, _P, _P, _I64, ctypes.c_float,
                                           _P, _P, ctypes.c_size_t, _P]
        L.bnb_int8_linear_wq_only.restype = ctypes.c_int
        L.bnb_int8_linear_wq_only.argtypes = [_P, _I64, _I64, _P, _P, _P, _I64, ctypes.c_float,
                                              _P, _P, ctypes.c_size_t, _P]
        L.bnb_int8_quantize_weight_ex.restype = ctypes.c_int
        L.bnb_int8_quantize_weight_ex.argtypes = [_P, _I64, _I64, ctypes.c_int, _P, _P, _P]
        L.bnb_int8_linear_ex.restype = ctypes.c_int
        L.bnb_int8_linear_ex.argtypes = [_P, _I64, _I64, _P, _P, _P, _P, _I64, ctypes.c_float,
                                         ctypes.c_int, _P, _P, ctypes.c_size_t, _P]
        L.bnb_int8_linear_from_host_ex.restype = ctypes.c_int
        L.bnb_int8_linear_from_host_ex.argtypes = [_P, _I64, _I64, _P, _P, _P, _P, _I64,
                                                   ctypes.c_float, ctypes.c_int, _P, _P, _P, _P,
                                                   ctypes.c_size_t, _P]
        L.bnb_int8_linear_debug_ex.restype = ctypes.c_int
        L.bnb_int8_linear_debug_ex.argtypes = L.bnb_int8_linear_ex.argtypes + [_P, _P, _P, _P, _P]
        L.bnb_int8_linear_debug.restype = ctypes.c_int
        L.bnb_int8_linear_debug.argtypes = L.bnb_int8_linear.argtypes + [_P, _P, _P, _P, _P]
        L.bnb_int8_linear_noalloc.restype = ctypes.c_int
        L.bnb_int8_linear_noalloc.argtypes = [_P, _I64, _I64, _P, _P, _P, _I64, ctypes.c_float,
                                              _P, _P]
        L.bnb_int8_linear_from_host.restype = ctypes.c_int
        L.bnb_int8_linear_from_host.argtypes = [_P, _I64, _I64, _P, _P, _P, _P, _I64, ctypes.c_float,
                                                _P, _P, _P, _P, ctypes.c_size_t, _P]
        L.bnb_int8_quantize_blockwise.restype = ctypes.c_int
        L.bnb_int8_quantize_blockwise.argtypes = [_P, _I64, _I64, _P, _P, _P]
        L.bnb_int8_dequantize_blockwise.restype = ctypes.c_int
        L.bnb_int8_dequantize_blockwise.argtypes = [_P, _P, _I64, _I64, _P, _P]
        L.bnb_last_device_status.restype = ctypes.c_int
        L.bnb_last_device_status.argtypes = [_P, _P, ctypes.POINTER(ctypes.c_int32)]
        L.bnb_status_string.restype = ctypes.c_char_p
        L.bnb_status_string.argtypes = [ctypes.c_int]
        L.bnb_launch_count.restype = ctypes.c_uint64
        L.bnb_launch_count.argtypes = []
        L.bnb_int8_linear_path.restype = ctypes.c_int
        L.bnb_int8_linear_path.argtypes = [_I64, _I64, _I64]
        L.bnb_int8_decode_cluster.restype = ctypes.c_int
        L.bnb_int8_decode_cluster.argtypes = [_I64, _I64, _I64]
        L.bnb_int8_linear_opts.restype = ctypes.c_int
        L.bnb_int8_linear_opts.argtypes = L.bnb_int8_linear_debug_ex.argtypes + [ctypes.c_uint32]
        self.c = L

    def __getattr__(self, name):
        return getattr(self.c, name)


_lib = None


def load() -> Lib:
    global _lib
    if _lib is None:
        _lib = Lib()
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc, where):
    if rc != 0:
        raise BnbError(rc, where)


def _dtype_code(t) -> int:
    """bnb_dtype_t of a tensor: 0 fp16, 1 bf16 (anything else raises)."""
    import torch
    if t.dtype == torch.float16:
        return 0
    if t.dtype == torch.bfloat16:
        return 1
    raise TypeError(f"fp16 or bf16 tensors only, got {t.dtype}")


def workspace_bytes(T: int, N: int, K: int) -> int:
    return load().bnb_int8_linear_workspace_bytes(T, N, K)


def quantize_weight(W16, Wq=None, Wscale=None, stream=None):
    """bnb_int8_quantize_weight(_ex): W16 [N,K] fp16 or bf16 (cuda) -> (Wq int8
    [N,K], sw fp32 [N])."""
    import torch
    N, K = W16.shape
    if Wq is None:
        Wq = torch.empty((N, K), dtype=torch.int8, device=W16.device)
    if Wscale is None:
        Wscale = torch.empty((N,), dtype=torch.float32, device=W16.device)
    dt = _dtype_code(W16)
    if dt == 0:
        rc = load().bnb_int8_quantize_weight(_ptr(W16), N, K, _ptr(Wq), _ptr(Wscale),
                                             _stream(stream))
    else:
        rc = load().bnb_int8_quantize_weight_ex(_ptr(W16), N, K, dt, _ptr(Wq), _ptr(Wscale),
                                                _stream(stream))
    _check(rc, "bnb_int8_quantize_weight")
    return Wq, Wscale


def _alloc_ws(T, N, K, device):
    import torch
    return torch.empty((workspace_bytes(T, N, K),), dtype=torch.uint8, device=device)


def linear_ex(X, Wq, Wscale, W16, bias, tau: float, Y=None, workspace=None, stream=None):
    """bnb_int8_linear_ex: X [T,K] fp16 or bf16 -> Y [T,N] in X's dtype; W16
    (X's dtype) and bias (X's dtype, [N]) may be None."""
    import torch
    T, K = X.shape
    N = Wq.shape[0]
    for name, t in (("W16", W16), ("bias", bias), ("Y", Y)):
        if t is not None and t.dtype != X.dtype:  # one element format per call
            raise TypeError(f"{name} is {t.dtype}, X is {X.dtype}")
    if Y is None:
        Y = torch.empty((T, N), dtype=X.dtype, device=X.device)
    if workspace is None:
        workspace = _alloc_ws(T, N, K, X.device)
    rc = load().bnb_int8_linear_ex(_ptr(X), T, K, _ptr(Wq), _ptr(Wscale), _ptr(W16), _ptr(bias),
                                   N, float(tau), _dtype_code(X), _ptr(Y), _ptr(workspace),
                                   workspace.numel(), _stream(stream))
    _check(rc, "bnb_int8_linear_ex")
    return Y


def linear(X, Wq, Wscale, W16, tau: float, Y=None, workspace=None, stream=None):
    """bnb_int8_linear: X [T,K] fp16 -> Y [T,N] fp16 (all cuda tensors); bf16
    X goes through bnb_int8_linear_ex."""
    import torch
    if _dtype_code(X) != 0:
        return linear_ex(X, Wq, Wscale, W16, None, tau, Y, workspace, stream)
    T, K = X.shape
    N = Wq.shape[0]
    if Y is None:
        Y = torch.empty((T, N), dtype=torch.float16, device=X.device)
    if workspace is None:
        workspace = _alloc_ws(T, N, K, X.device)
    rc = load().bnb_int8_linear(_ptr(X), T, K, _ptr(Wq), _ptr(Wscale), _ptr(W16), N,
                                float(tau), _ptr(Y), _ptr(workspace), workspace.numel(),
                                _stream(stream))
    _check(rc, "bnb_int8_linear")
    return Y


def linear_bias(X, Wq, Wscale, W16, bias, tau: float, Y=None, workspace=None, stream=None):
    """bnb_int8_linear_bias: as :func:`linear`, plus an fp16 bias [N] (cuda)
    added before the rounding of Y; ``bias=None`` passes NULL."""
    import torch
    if _dtype_code(X) != 0:
        return linear_ex(X, Wq, Wscale, W16, bias, tau, Y, workspace, stream)
    T, K = X.shape
    N = Wq.shape[0]
    if Y is None:
        Y = torch.empty((T, N), dtype=torch.float16, device=X.device)
    if workspace is None:
        workspace = _alloc_ws(T, N, K, X.device)
    rc = load().bnb_int8_linear_bias(_ptr(X), T, K, _ptr(Wq), _ptr(Wscale), _ptr(W16),
                                     _ptr(bias), N, float(tau), _ptr(Y), _ptr(workspace),
                                     workspace.numel(), _stream(stream))
    _check(rc, "bnb_int8_linear_bias")
    return Y


def linear_wq_only(X, Wq, Wscale, bias, tau: float, Y=None, workspace=None, stream=None):
    """bnb_int8_linear_wq_only: the layer with only the int8 weight resident
    (outlier weights dequantized from the codes); ``bias`` an fp16 [N] cuda
    tensor or None."""
    import torch
    if _dtype_code(X) != 0:
        return linear_ex(X, Wq, Wscale, None, bias, tau, Y, workspace, stream)
    T, K = X.shape
    N = Wq.shape[0]
    if Y is None:
        Y = torch.empty((T, N), dtype=torch.float16, device=X.device)
    if workspace is None:
        workspace = _alloc_ws(T, N, K, X.device)
    rc = load().bnb_int8_linear_wq_only(_ptr(X), T, K, _ptr(Wq), _ptr(Wscale), _ptr(bias), N,
                                        float(tau), _ptr(Y), _ptr(workspace), workspace.numel(),
                                        _stream(stream))
    _check(rc, "bnb_int8_linear_wq_only")
    return Y


def linear_from_host(X_host, Wq, Wscale, W16, tau: float, Y_host, X_dev, Y_dev, workspace,
                     stream=None, bias=None):
    """bnb_int8_linear_from_host: X_host [T,K] fp16 (pinned cpu tensor) -> Y_host
    [T,N] fp16 (pinned cpu tensor), through the caller's device buffers X_dev,
    Y_dev and workspace, all enqueued on `stream`; ``bias`` an optional fp16
    [N] cuda tensor; ``W16=None`` runs the int8-weight-only layer."""
    T, K = X_host.shape
    N = Wq.shape[0]
    rc = load().bnb_int8_linear_from_host_ex(_ptr(X_host), T, K, _ptr(Wq), _ptr(Wscale),
                                             _ptr(W16), _ptr(bias), N, float(tau),
                                             _dtype_code(X_host), _ptr(Y_host), _ptr(X_dev),
                                             _ptr(Y_dev), _ptr(workspace), workspace.numel(),
                                             _stream(stream))
    _check(rc, "bnb_int8_linear_from_host")
    return Y_host


BLOCKWISE_DEFAULT = 256  # the pages give no block size


def quantize_blockwise(x, block: int = BLOCKWISE_DEFAULT, codes=None, absmax=None, stream=None):
    """bnb_int8_quantize_blockwise: fp32 cuda tensor -> (int8 codes, fp32
    absmax per block of ``block`` values)."""
    import torch
    n = x.numel()
    if codes is None:
        codes = torch.empty(n, dtype=torch.int8, device=x.device)
    if absmax is None:
        absmax = torch.empty((n + block - 1) // block, dtype=torch.float32, device=x.device)
    rc = load().bnb_int8_quantize_blockwise(_ptr(x), n, block, _ptr(codes), _ptr(absmax),
                                            _stream(stream))
    _check(rc, "bnb_int8_quantize_blockwise")
    return codes, absmax


def dequantize_blockwise(codes, absmax, block: int = BLOCKWISE_DEFAULT, y=None, stream=None):
    """bnb_int8_dequantize_blockwise: (int8 codes, fp32 absmax) -> fp32."""
    import torch
    n = codes.numel()
    if y is None:
        y = torch.empty(n, dtype=torch.float32, device=codes.device)
    rc = load().bnb_int8_dequantize_blockwise(_ptr(codes), _ptr(absmax), n, block, _ptr(y),
                                              _stream(stream))
    _check(rc, "bnb_int8_dequantize_blockwise")
    return y


def linear_noalloc(X, Wq, Wscale, W16, tau: float, Y=None, stream=None):
    """bnb_int8_linear_noalloc: as :func:`linear`, with the library's static
    scratch array instead of a workspace (for callers that cannot allocate).
    The C entry point is fp16 only: X, W16 and a given Y must be fp16."""
    import torch
    for name, t in (("X", X), ("W16", W16), ("Y", Y)):
        if t is not None and t.dtype != torch.float16:
            raise TypeError(f"bnb_int8_linear_noalloc takes fp16 tensors, {name} is {t.dtype}")
    if Wq.dtype != torch.int8 or Wscale.dtype != torch.float32:
        raise TypeError("Wq must be int8 and Wscale float32")
    T, K = X.shape
    N = Wq.shape[0]
    if Y is None:
        Y = torch.empty((T, N), dtype=torch.float16, device=X.device)
    rc = load().bnb_int8_linear_noalloc(_ptr(X), T, K, _ptr(Wq), _ptr(Wscale), _ptr(W16), N,
                                        float(tau), _ptr(Y), _stream(stream))
    _check(rc, "bnb_int8_linear_noalloc")
    return Y


def linear_debug(X, Wq, Wscale, W16, tau: float, stream=None, want_acc: bool = True,
                 bias=None):
    """bnb_int8_linear_debug_ex (X fp16 or bf16, W16 and bias may be None);
    returns dict(Y, Xq, sx, O, acc) as cuda tensors."""
    import torch
    T, K = X.shape
    N = Wq.shape[0]
    dev = X.device
    Y = torch.empty((T, N), dtype=X.dtype, device=dev)
    Xq = torch.empty((T, K), dtype=torch.int8, device=dev)
    sx = torch.empty((T,), dtype=torch.float32, device=dev)
    O = torch.empty((K,), dtype=torch.int32, device=dev)
    nO = torch.empty((1,), dtype=torch.int32, device=dev)
    acc = torch.empty((T, N), dtype=torch.int32, device=dev) if want_acc else None
    ws = _alloc_ws(T, N, K, dev)
    rc = load().bnb_int8_linear_debug_ex(_ptr(X), T, K, _ptr(Wq), _ptr(Wscale), _ptr(W16),
                                         _ptr(bias), N, float(tau), _dtype_code(X), _ptr(Y),
                                         _ptr(ws), ws.numel(), _stream(stream), _ptr(Xq),
                                         _ptr(sx), _ptr(O), _ptr(nO), _ptr(acc))
    _check(rc, "bnb_int8_linear_debug_ex")
    return {"Y": Y, "Xq": Xq, "sx": sx, "O": O, "nO": nO, "acc": acc, "workspace": ws}


def last_device_status(workspace, stream=None) -> int:
    out = ctypes.c_int32(0)
    rc = load().bnb_last_device_status(_ptr(workspace), _stream(stream), ctypes.byref(out))
    _check(rc, "bnb_last_device_status")
    return out.value


def launch_count() -> int:
    return load().bnb_launch_count()


def linear_path(T: int, N: int, K: int) -> int:
    return load().bnb_int8_linear_path(T, N, K)


def decode_cluster(T: int, N: int, K: int) -> int:
    """The decode kernel's form for this shape (16, 8, 4: clusters; 1: none;
    0: not the decode path)."""
    return load().bnb_int8_decode_cluster(T, N, K)


# Flags of bnb_int8_linear_opts (include/bnb_int8.h): per-call options for
# benchmarks and tests.
OPT_MAIN_ONLY = 0x1
OPT_ACT_ONLY = 0x2
OPT_NO_PDL = 0x4
OPT_LEGACY_MMA = 0x8
OPT_FORCE_TIMEOUT = 0x10
OPT_SINGLE_CTA = 0x20
OPT_GEMM = 0x40


def OPT_CLUSTER(c: int) -> int:
    return int(c) << 8


def linear_opts(X, Wq, Wscale, W16, tau: float, opts: int, bias=None, Y=None, workspace=None,
                stream=None, debug: bool = False, want_acc: bool = True):
    """bnb_int8_linear_opts: the layer with per-call options (``OPT_*``).
    With ``debug`` the intermediates are exported as in :func:`linear_debug`
    and a dict is returned; otherwise Y."""
    import torch
    T, K = X.shape
    N = Wq.shape[0]
    dev = X.device
    if Y is None:
        Y = torch.empty((T, N), dtype=X.dtype, device=dev)
    if workspace is None:
        workspace = _alloc_ws(T, N, K, dev)
    d = {}
    if debug:
        d = {"Xq": torch.empty((T, K), dtype=torch.int8, device=dev),
             "sx": torch.empty((T,), dtype=torch.float32, device=dev),
             "O": torch.empty((K,), dtype=torch.int32, device=dev),
             "nO": torch.empty((1,), dtype=torch.int32, device=dev),
             "acc": torch.empty((T, N), dtype=torch.int32, device=dev) if want_acc else None}
    rc = load().bnb_int8_linear_opts(_ptr(X), T, K, _ptr(Wq), _ptr(Wscale), _ptr(W16), _ptr(bias),
                                     N, float(tau), _dtype_code(X), _ptr(Y), _ptr(workspace),
                                     workspace.numel(), _stream(stream), _ptr(d.get("Xq")),
                                     _ptr(d.get("sx")), _ptr(d.get("O")), _ptr(d.get("nO")),
                                     _ptr(d.get("acc")), ctypes.c_uint32(int(opts)))
    _check(rc, "bnb_int8_linear_opts")
    if debug:
        d["Y"] = Y
        d["workspace"] = workspace
        return d
    return Y
