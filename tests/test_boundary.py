"""The C-ABI library: it loads, exports every declared symbol, and rejects bad
arguments on the host before touching a device (CPU only)."""

import ctypes
import math
import os
import re

import pytest

from int8_mixed_precision_04_b300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.Lib()


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b(bnb_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("bnb_int8_quantize_weight", "bnb_int8_linear", "bnb_int8_linear_debug",
                 "bnb_int8_linear_workspace_bytes", "bnb_last_device_status", "bnb_status_string"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib.c, name), name
    for name in binding.Lib.SYMBOLS:
        assert name in declared_functions(), name


def test_status_strings(lib):
    for s in binding.Status:
        assert lib.bnb_status_string(int(s)).decode() == "BNB_ERR_" + s.name if s else True
    assert lib.bnb_status_string(0) == b"BNB_OK"
    assert lib.bnb_status_string(99) == b"BNB_ERR_UNKNOWN"


def test_workspace_bytes(lib):
    assert lib.bnb_int8_linear_workspace_bytes(0, 1, 16) == 0
    assert lib.bnb_int8_linear_workspace_bytes(1, 0, 16) == 0
    assert lib.bnb_int8_linear_workspace_bytes(-1, 1, 16) == 0
    small = lib.bnb_int8_linear_workspace_bytes(16, 256, 256)
    big = lib.bnb_int8_linear_workspace_bytes(4096, 28672, 8192)
    # at least the codes (2 B/elem worst case) and the padded outlier block
    assert big >= 4096 * 8192 * 4
    assert small < big
    assert lib.bnb_int8_linear_workspace_bytes(1 << 23, 16, 16) == 0  # beyond BNB_MAX_T


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every case fails on the host


def _linear(lib, X=FAKE, T=16, K=256, Wq=FAKE, sw=FAKE, W16=FAKE, N=256, tau=6.0, Y=FAKE * 64,
            ws=FAKE * 256, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = lib.bnb_int8_linear_workspace_bytes(T, N, K) if T > 0 and N > 0 and K > 0 else 0
    return lib.bnb_int8_linear(X, T, K, Wq, sw, W16, N, ctypes.c_float(tau), Y, ws, ws_bytes, None)


@pytest.mark.parametrize("case,want", [
    (dict(X=None), binding.Status.INVALID_ARG),
    (dict(Wq=None), binding.Status.INVALID_ARG),
    (dict(sw=None), binding.Status.INVALID_ARG),
    (dict(W16=None), binding.Status.INVALID_ARG),
    (dict(Y=None), binding.Status.INVALID_ARG),
    (dict(ws=None), binding.Status.INVALID_ARG),
    (dict(T=0), binding.Status.INVALID_ARG),
    (dict(N=-3), binding.Status.INVALID_ARG),
    (dict(K=0), binding.Status.INVALID_ARG),
    (dict(tau=math.nan), binding.Status.INVALID_ARG),
    (dict(tau=-1.0), binding.Status.INVALID_ARG),
    (dict(ws_bytes=100), binding.Status.INVALID_ARG),
    (dict(K=24, ws_bytes=1 << 30), binding.Status.UNSUPPORTED),
    (dict(X=FAKE + 8), binding.Status.UNSUPPORTED),
    (dict(Y=FAKE * 64 + 4), binding.Status.UNSUPPORTED),
    (dict(T=1 << 23, ws_bytes=1 << 40), binding.Status.UNSUPPORTED),
    (dict(Y=FAKE), binding.Status.INVALID_ARG),  # Y aliases X
])
def test_linear_rejects_on_host(lib, case, want):
    assert _linear(lib, **case) == want


@pytest.mark.parametrize("args,want", [
    ((None, 4, 16, FAKE, FAKE), binding.Status.INVALID_ARG),
    ((FAKE, 0, 16, FAKE, FAKE), binding.Status.INVALID_ARG),
    ((FAKE, 4, 20, FAKE, FAKE), binding.Status.UNSUPPORTED),
    ((FAKE, 4, 16, FAKE + 1, FAKE), binding.Status.UNSUPPORTED),
    ((FAKE, 4, 16, FAKE, None), binding.Status.INVALID_ARG),
])
def test_quantize_weight_rejects_on_host(lib, args, want):
    assert lib.bnb_int8_quantize_weight(*args, None) == want


def test_last_device_status_rejects_null(lib):
    out = ctypes.c_int32(0)
    assert lib.bnb_last_device_status(None, None, ctypes.byref(out)) == binding.Status.INVALID_ARG


def test_paths(lib):
    assert lib.bnb_int8_linear_path(16, 4096, 4096) == 1
    assert lib.bnb_int8_linear_path(1, 4096, 4096) == 1
    assert lib.bnb_int8_linear_path(17, 4096, 4096) in (2, 3)
    assert lib.bnb_int8_linear_path(2048, 11008, 4096) in (2, 3)
    assert lib.bnb_int8_linear_path(0, 1, 16) == 0
    # the decode kernel's form: a cluster size, 1 for no clusters, 0 off the decode path
    assert lib.bnb_int8_decode_cluster(16, 4096, 4096) in (4, 8, 16)
    assert lib.bnb_int8_decode_cluster(1, 4096, 4096) in (1, 4, 8, 16)
    assert lib.bnb_int8_decode_cluster(17, 4096, 4096) == 0
    assert lib.bnb_int8_decode_cluster(0, 1, 16) == 0


def test_missing_library_raises(tmp_path):
    with pytest.raises(FileNotFoundError):
        binding.Lib(str(tmp_path / "nope.so"))


@pytest.mark.parametrize("case,want", [
    (dict(xh=None), binding.Status.INVALID_ARG),
    (dict(yh=None), binding.Status.INVALID_ARG),
    (dict(xd=None), binding.Status.INVALID_ARG),
    (dict(yd=None), binding.Status.INVALID_ARG),
    (dict(yd=FAKE * 64 + 16), binding.Status.INVALID_ARG),   # Y_dev overlaps X_dev
    (dict(T=0), binding.Status.INVALID_ARG),
    (dict(tau=-1.0), binding.Status.INVALID_ARG),
    (dict(K=250), binding.Status.UNSUPPORTED),
    (dict(bias=FAKE * 3 + 4), binding.Status.UNSUPPORTED),     # misaligned bias
    (dict(bias=FAKE * 96 + 64), binding.Status.INVALID_ARG),   # bias inside Y_dev
])
def test_from_host_rejects_on_host(lib, case, want):
    """bnb_int8_linear_from_host checks its buffers and the layer's arguments
    before enqueuing a copy."""
    a = dict(xh=FAKE, T=16, K=256, N=256, tau=6.0, yh=FAKE * 2, xd=FAKE * 64,
             yd=FAKE * 96, ws=FAKE * 256, bias=None)
    a.update(case)
    T, K, N = a["T"], a["K"], a["N"]
    ws_bytes = lib.bnb_int8_linear_workspace_bytes(T, N, K) if min(T, K, N) > 0 else 0
    rc = lib.bnb_int8_linear_from_host(a["xh"], T, K, FAKE, FAKE, FAKE, a["bias"], N,
                                       ctypes.c_float(a["tau"]), a["yh"], a["xd"], a["yd"],
                                       a["ws"], ws_bytes, None)
    assert rc == want


@pytest.mark.parametrize("case,want", [
    (dict(x=None), binding.Status.INVALID_ARG),
    (dict(q=None), binding.Status.INVALID_ARG),
    (dict(a=None), binding.Status.INVALID_ARG),
    (dict(n=0), binding.Status.INVALID_ARG),
    (dict(block=100), binding.Status.UNSUPPORTED),
    (dict(block=32), binding.Status.UNSUPPORTED),
    (dict(block=4096), binding.Status.UNSUPPORTED),
    (dict(x=FAKE + 4), binding.Status.UNSUPPORTED),
    (dict(q=FAKE + 64), binding.Status.INVALID_ARG),  # codes inside x
])
def test_blockwise_rejects_on_host(lib, case, want):
    """The blockwise codec checks its arguments before touching a device."""
    a = dict(x=FAKE, n=1 << 16, block=256, q=FAKE * 64, a=FAKE * 128)
    a.update(case)
    assert lib.bnb_int8_quantize_blockwise(a["x"], a["n"], a["block"], a["q"], a["a"], None) == want
    if "x" not in case:  # the decoder's own checks, same buffers reversed
        rc = lib.bnb_int8_dequantize_blockwise(a["q"], a["a"], a["n"], a["block"], FAKE * 256, None)
        if case.get("q", 1) is None or case.get("a", 1) is None or "n" in case or "block" in case:
            assert rc == want


@pytest.mark.parametrize("case,want", [
    (dict(X=None), binding.Status.INVALID_ARG),
    (dict(tau=math.nan), binding.Status.INVALID_ARG),
    (dict(bias=FAKE * 64 + 8), binding.Status.UNSUPPORTED),    # misaligned bias
    (dict(bias=FAKE * 64 + 256), binding.Status.INVALID_ARG),  # bias inside Y
])
def test_linear_bias_rejects_on_host(lib, case, want):
    """bnb_int8_linear_bias runs the layer's checks, then its own on the bias."""
    a = dict(X=FAKE, T=16, K=256, N=256, tau=6.0, bias=FAKE * 32, Y=FAKE * 64, ws=FAKE * 256)
    a.update(case)
    ws_bytes = lib.bnb_int8_linear_workspace_bytes(a["T"], a["N"], a["K"])
    rc = lib.bnb_int8_linear_bias(a["X"], a["T"], a["K"], FAKE, FAKE, FAKE, a["bias"], a["N"],
                                  ctypes.c_float(a["tau"]), a["Y"], a["ws"], ws_bytes, None)
    assert rc == want


@pytest.mark.parametrize("case,want", [
    (dict(X=None), binding.Status.INVALID_ARG),
    (dict(Wq=None), binding.Status.INVALID_ARG),
    (dict(K=24), binding.Status.UNSUPPORTED),
    (dict(bias=FAKE * 64 + 8), binding.Status.UNSUPPORTED),
    (dict(Y=FAKE), binding.Status.INVALID_ARG),                # Y aliases X
])
def test_linear_wq_only_rejects_on_host(lib, case, want):
    """bnb_int8_linear_wq_only checks its arguments (no W16 to check)."""
    a = dict(X=FAKE, T=16, K=256, N=256, tau=6.0, Wq=FAKE * 16, bias=None, Y=FAKE * 64,
             ws=FAKE * 256)
    a.update(case)
    ws_bytes = lib.bnb_int8_linear_workspace_bytes(a["T"], a["N"], max(a["K"], 16))
    rc = lib.bnb_int8_linear_wq_only(a["X"], a["T"], a["K"], a["Wq"], FAKE * 8, a["bias"], a["N"],
                                     ctypes.c_float(a["tau"]), a["Y"], a["ws"], ws_bytes, None)
    assert rc == want


def test_fp16_weight_entry_points_need_w16(lib):
    """Only the int8-weight-only entry points accept a NULL W16."""
    ws_bytes = lib.bnb_int8_linear_workspace_bytes(16, 256, 256)
    assert lib.bnb_int8_linear_bias(FAKE, 16, 256, FAKE, FAKE, None, None, 256,
                                    ctypes.c_float(6.0), FAKE * 64, FAKE * 256, ws_bytes,
                                    None) == binding.Status.INVALID_ARG


def test_ex_entry_points_check_dtype_on_host(lib):
    """The general entry points reject an unknown element format, and run the
    same argument checks as the fp16 ones, before touching a device."""
    ws_bytes = lib.bnb_int8_linear_workspace_bytes(16, 256, 256)
    tau = ctypes.c_float(6.0)
    for dt in (2, -1):
        assert lib.bnb_int8_quantize_weight_ex(FAKE, 256, 256, dt, FAKE * 8, FAKE * 16,
                                               None) == binding.Status.INVALID_ARG
        assert lib.bnb_int8_linear_ex(FAKE, 16, 256, FAKE * 8, FAKE * 16, FAKE * 24, None, 256,
                                      tau, dt, FAKE * 64, FAKE * 256, ws_bytes,
                                      None) == binding.Status.INVALID_ARG
        assert lib.bnb_int8_linear_from_host_ex(FAKE, 16, 256, FAKE * 8, FAKE * 16, FAKE * 24,
                                                None, 256, tau, dt, FAKE * 2, FAKE * 64,
                                                FAKE * 96, FAKE * 256, ws_bytes,
                                                None) == binding.Status.INVALID_ARG
        assert lib.bnb_int8_linear_debug_ex(FAKE, 16, 256, FAKE * 8, FAKE * 16, FAKE * 24, None,
                                            256, tau, dt, FAKE * 64, FAKE * 256, ws_bytes, None,
                                            None, None, None, None,
                                            None) == binding.Status.INVALID_ARG
    # bf16 with the layer's own argument errors
    assert lib.bnb_int8_quantize_weight_ex(FAKE, 256, 24, 1, FAKE * 8, FAKE * 16,
                                           None) == binding.Status.UNSUPPORTED
    assert lib.bnb_int8_linear_ex(FAKE, 16, 256, FAKE * 8, FAKE * 16, None, None, 256,
                                  ctypes.c_float(math.nan), 1, FAKE * 64, FAKE * 256, ws_bytes,
                                  None) == binding.Status.INVALID_ARG
    assert lib.bnb_int8_linear_ex(FAKE, 16, 256, FAKE * 8, FAKE * 16, None, FAKE * 64 + 8, 256,
                                  tau, 1, FAKE * 64, FAKE * 256, ws_bytes,
                                  None) == binding.Status.UNSUPPORTED


def test_binding_dtype_codes():
    """The binding maps torch dtypes to bnb_dtype_t and refuses the rest."""
    import torch
    assert binding._dtype_code(torch.empty(1, dtype=torch.float16)) == 0
    assert binding._dtype_code(torch.empty(1, dtype=torch.bfloat16)) == 1
    with pytest.raises(TypeError):
        binding._dtype_code(torch.empty(1, dtype=torch.float32))


def test_binding_rejects_mixed_formats():
    """One element format per call: the binding refuses a W16, bias or Y whose
    dtype differs from X's before calling the library."""
    import torch
    X = torch.empty((16, 256), dtype=torch.bfloat16)
    Wq = torch.empty((8, 256), dtype=torch.int8)
    sw = torch.empty(8)
    with pytest.raises(TypeError):
        binding.linear_ex(X, Wq, sw, torch.empty((8, 256), dtype=torch.float16), None, 6.0)
    with pytest.raises(TypeError):
        binding.linear_ex(X, Wq, sw, None, torch.empty(8, dtype=torch.float16), 6.0)


def test_linear8bitlt_checks_its_weight():
    """The module wants a 2-D fp16 or bf16 CUDA weight and a matching bias;
    host tensors are refused before anything is quantized."""
    import torch

    from int8_mixed_precision_04_b300 import Linear8bitLt
    with pytest.raises(ValueError):
        Linear8bitLt(torch.zeros((8, 16), dtype=torch.float16))          # not on a GPU
    with pytest.raises(ValueError):
        Linear8bitLt(torch.zeros((8, 16), dtype=torch.float32))          # not 16-bit
    with pytest.raises(ValueError):
        Linear8bitLt(torch.zeros(16, dtype=torch.float16))               # not 2-D


def test_cuda_failure_surfaces_as_status(lib):
    """A failing CUDA layer (here: no device at all) reaches the caller as
    BNB_ERR_CUDA from every entry point once its argument checks pass, with
    nothing enqueued and nothing crashing.  The pointers are fake, so where a
    GPU is visible the test runs again in a child process that sees none
    (CUDA_VISIBLE_DEVICES empty)."""
    import torch
    if torch.cuda.is_available():
        import subprocess
        import sys
        env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
        r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", __file__,
                            "-k", "test_cuda_failure_surfaces_as_status",
                            "-p", "no:cacheprovider"],
                           env=env, capture_output=True, text=True, timeout=600)
        assert r.returncode == 0 and " passed" in r.stdout, r.stdout[-3000:] + r.stderr[-2000:]
        return
    ws_bytes = lib.bnb_int8_linear_workspace_bytes(16, 256, 256)
    tau = ctypes.c_float(6.0)
    cuda = binding.Status.CUDA
    assert lib.bnb_int8_quantize_weight(FAKE, 256, 256, FAKE * 8, FAKE * 16, None) == cuda
    assert lib.bnb_int8_linear(FAKE, 16, 256, FAKE * 8, FAKE * 16, FAKE * 24, 256, tau,
                               FAKE * 64, FAKE * 256, ws_bytes, None) == cuda
    assert lib.bnb_int8_linear_ex(FAKE, 16, 256, FAKE * 8, FAKE * 16, None, None, 256, tau, 1,
                                  FAKE * 64, FAKE * 256, ws_bytes, None) == cuda
    assert lib.bnb_int8_quantize_blockwise(FAKE, 1 << 16, 256, FAKE * 64, FAKE * 128,
                                           None) == cuda
    out = ctypes.c_int32(0)
    assert lib.bnb_last_device_status(FAKE * 256, None, ctypes.byref(out)) == cuda
