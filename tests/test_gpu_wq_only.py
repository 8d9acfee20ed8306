"""The layer with only the int8 weight resident (bnb_int8_linear_wq_only):
the outlier columns use the codes dequantized, Wq sw / 127.  Against the
oracle's int8-weight-only leg on every path: decode (T <= 16, with more
outlier columns than the exchange carries), the tcgen05 GEMM with a sparse and
a dense outlier set (the legacy mma GEMM in test_gpu_options.py) (GPU)."""

import math
import numpy as np
import pytest

import inputs
from parity import check_y

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from int8_mixed_precision_04_b300 import binding, build
    build.build()
    binding.load()


@pytest.mark.parametrize("T,K,N,ncols", [
    (1, 256, 64, 2), (16, 4096, 4096, 4), (11, 1040, 520, 9), (16, 1040, 96, 70),
    (16, 4096, 3900, 20), (17, 272, 129, 3), (300, 1024, 200, 4), (257, 2064, 1000, 7),
    (130, 512, 257, 40), (2, 512, 100, 2), (3, 2048, 300, 5), (6, 4096, 500, 3),
])
@pytest.mark.parametrize("tau", [6.0, 0.0, math.inf])
@pytest.mark.parametrize("with_bias", [False, True])
def test_wq_only_parity(orc, T, K, N, ncols, tau, with_bias):
    import torch

    from int8_mixed_precision_04_b300 import binding
    w = inputs.random_small(T, K, N, ncols, seed=T + 5 * N + K, tau=tau)
    b = inputs.bias(N, K, seed=N) if with_bias else None
    Wq, sw = binding.quantize_weight(torch.from_numpy(w.W).cuda())
    Y = binding.linear_wq_only(torch.from_numpy(w.X).cuda(), Wq, sw,
                               None if b is None else torch.from_numpy(b).cuda(), tau)
    Wq_o, sw_o = orc.quantize_weight(w.W)
    ref = orc.linear(w.X, Wq_o, sw_o, None, tau, bias=b)
    check_y(Y.cpu().numpy(), ref["Y"], f"wq only T{T} K{K} N{N} tau{tau} bias {with_bias}")


def test_wq_only_full_decode(orc):
    """The decode workload at full size, sampled rows and all channels."""
    import torch

    from int8_mixed_precision_04_b300 import binding
    w = inputs.decode(T=16)
    Wq, sw = binding.quantize_weight(torch.from_numpy(w.W).cuda())
    Y = binding.linear_wq_only(torch.from_numpy(w.X).cuda(), Wq, sw, None, w.tau).cpu().numpy()
    Wq_o, sw_o = orc.quantize_weight(w.W)
    ref = orc.linear(w.X, Wq_o, sw_o, None, w.tau)
    assert len(ref["O"]) == 4
    check_y(Y, ref["Y"], "wq only decode")


def test_wq_only_from_host_and_module(orc):
    """bnb_int8_linear_from_host with W16 NULL, and Linear8bitLt without its
    fp16 weight, give the same Y as bnb_int8_linear_wq_only."""
    import torch

    from int8_mixed_precision_04_b300 import Linear8bitLt, binding
    T, K, N = 40, 1024, 300
    w = inputs.random_small(T, K, N, 5, seed=21)
    b = inputs.bias(N, K, seed=3)
    W = torch.from_numpy(w.W).cuda()
    Wq, sw = binding.quantize_weight(W)
    bd = torch.from_numpy(b).cuda()
    Y_ref = binding.linear_wq_only(torch.from_numpy(w.X).cuda(), Wq, sw, bd, 6.0)
    Xh = torch.from_numpy(w.X).pin_memory()
    Yh = torch.empty((T, N), dtype=torch.float16).pin_memory()
    Xd = torch.empty((T, K), dtype=torch.float16, device="cuda")
    Yd = torch.empty((T, N), dtype=torch.float16, device="cuda")
    ws = torch.empty(binding.workspace_bytes(T, N, K), dtype=torch.uint8, device="cuda")
    binding.linear_from_host(Xh, Wq, sw, None, 6.0, Yh, Xd, Yd, ws, bias=bd)
    torch.cuda.synchronize()
    assert torch.equal(Yh, Y_ref.cpu())
    layer = Linear8bitLt(W, bd, threshold=6.0, keep_fp16_weight=False)
    assert layer.W16 is None
    assert torch.equal(layer(torch.from_numpy(w.X).cuda()), Y_ref)
    Wq_o, sw_o = orc.quantize_weight(w.W)
    check_y(Y_ref.cpu().numpy(), orc.linear(w.X, Wq_o, sw_o, None, 6.0, bias=b)["Y"], "module")
