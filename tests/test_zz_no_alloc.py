"""bnb_int8_linear_noalloc: the entry point for callers that cannot allocate
device memory (a runtime that plans all memory ahead of time, a serving loop
where cudaMalloc may not be called, a host framework that hands out no
workspace).  It runs the same kernels as bnb_int8_linear on a static scratch
array inside the library.

The GPU test compares it with bnb_int8_linear through the C ABI, on two calls
in a row whose inputs differ, so that stale scratch contents from the first
call would show in the second.  This file sorts last so that a run stopping at
the first failure has already run every other test; it also passes alone in a
fresh process.
"""

import ctypes
import math

import pytest

import inputs
from int8_mixed_precision_04_b300 import binding, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def _noalloc(lib, T, K, N, X=0x10000, tau=6.0):
    return lib.bnb_int8_linear_noalloc(X, T, K, 0x20000, 0x30000, 0x40000, N,
                                       ctypes.c_float(tau), 0x80000000, None)


def test_noalloc_rejects_on_host(lib):
    """Argument and size errors come back before anything touches a device."""
    assert _noalloc(lib, 16, 256, 256, X=None) == binding.Status.INVALID_ARG
    assert _noalloc(lib, 0, 256, 256) == binding.Status.INVALID_ARG
    # a workspace larger than the static scratch array
    assert lib.bnb_int8_linear_workspace_bytes(4096, 28672, 8192) > (8 << 20)
    assert _noalloc(lib, 4096, 8192, 28672) == binding.Status.UNSUPPORTED


@pytest.mark.gpu
@pytest.mark.parametrize("T,K,N", [(16, 4096, 4096), (130, 512, 200)])
def test_noalloc_matches_linear_two_calls(lib, T, K, N):
    import torch
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    w1 = inputs.random_small(T, K, N, 4, seed=T + K)
    w2 = inputs.random_small(T, K, N, 9, seed=T + K + 1)
    W = torch.from_numpy(w1.W).cuda()
    Wq, sw = binding.quantize_weight(W)
    for w, tau in ((w1, 6.0), (w2, 3.0)):
        X = torch.from_numpy(w.X).cuda()
        Y_ref = binding.linear(X, Wq, sw, W, tau)
        Y = binding.linear_noalloc(X, Wq, sw, W, tau)
        torch.cuda.synchronize()
        # the same kernels on the same inputs: bit for bit, so that stale
        # scratch contents that perturb only low bits would show
        assert torch.equal(Y, Y_ref), f"noalloc T{T} K{K} N{N} tau{tau}"
    assert math.isfinite(float(Y.float().abs().max()))


@pytest.mark.gpu
def test_noalloc_rejects_other_dtypes(lib):
    """The binding refuses what the fp16-only C entry point would misread."""
    import torch
    X = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((32, 64), dtype=torch.float16, device="cuda")
    Wq, sw = binding.quantize_weight(W)
    with pytest.raises(TypeError):
        binding.linear_noalloc(X, Wq, sw, W, 6.0)
    with pytest.raises(TypeError):
        binding.linear_noalloc(X.half(), Wq, sw, W.bfloat16(), 6.0)
