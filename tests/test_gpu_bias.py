"""The layer with a bias (bnb_int8_linear_bias) and the Linear8bitLt wrapper,
against the oracle, on every path: decode (T <= 16) and the tcgen05 GEMM
(the legacy mma GEMM in test_gpu_options.py) (GPU)."""

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


def _bias(N: int, seed: int) -> np.ndarray:
    """A seeded fp16 bias mixing tiny, O(1) and large entries."""
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(N) * rng.choice([1e-3, 0.5, 20.0], N)).astype(np.float16)


@pytest.mark.parametrize("T,K,N,ncols", [
    (1, 256, 64, 2), (16, 4096, 4096, 4), (11, 1040, 520, 9), (16, 1040, 96, 70),
    (17, 272, 129, 3), (300, 1024, 200, 4), (257, 2064, 1000, 7),
    (2, 512, 100, 2), (3, 2048, 300, 5), (6, 4096, 500, 3),
])
@pytest.mark.parametrize("tau", [6.0, 0.0, math.inf])
def test_bias_parity(orc, T, K, N, ncols, tau):
    import torch

    from int8_mixed_precision_04_b300 import binding
    w = inputs.random_small(T, K, N, ncols, seed=T + 3 * N + K, tau=tau)
    b = _bias(N, seed=N)
    X = torch.from_numpy(w.X).cuda()
    W = torch.from_numpy(w.W).cuda()
    Wq, sw = binding.quantize_weight(W)
    Y = binding.linear_bias(X, Wq, sw, W, torch.from_numpy(b).cuda(), tau).cpu().numpy()
    Wq_o, sw_o = orc.quantize_weight(w.W)
    ref = orc.linear(w.X, Wq_o, sw_o, w.W, tau, bias=b)
    check_y(Y, ref["Y"], f"bias T{T} K{K} N{N} tau{tau}")
    # a NULL bias is the plain layer, bit for bit
    Y0 = binding.linear_bias(X, Wq, sw, W, None, tau)
    assert torch.equal(Y0, binding.linear(X, Wq, sw, W, tau))


@pytest.mark.parametrize("T", [16, 48])
def test_bias_integer_exact(orc, T):
    """tau = inf, integer inputs and an integer bias: scales are 127, so the
    epilogue computes acc + b exactly and Y = fp16(X W^T + b) bit for bit."""
    import torch

    from int8_mixed_precision_04_b300 import binding
    X, W = inputs.int_valued(T, 64, 40, seed=T)
    b = (np.arange(40) * 211 - 4000).astype(np.float16)
    Wq, sw = binding.quantize_weight(torch.from_numpy(W).cuda())
    Y = binding.linear_bias(torch.from_numpy(X).cuda(), Wq, sw, torch.from_numpy(W).cuda(),
                            torch.from_numpy(b).cuda(), math.inf).cpu().numpy()
    Wq_o, sw_o = orc.quantize_weight(W)
    ref = orc.linear(X, Wq_o, sw_o, W, math.inf, bias=b)["Y"]
    exact = X.astype(np.int64) @ W.astype(np.int64).T + b.astype(np.int64)
    with np.errstate(over="ignore"):
        assert np.array_equal(ref.view(np.uint16), exact.astype(np.float16).view(np.uint16))
    assert np.array_equal(Y.view(np.uint16), ref.view(np.uint16))


def test_linear8bitlt(orc):
    """The wrapper over nn.Linear: leading batch dims, bias, threshold, an
    empty batch; its buffers are the library's weight codes."""
    import torch

    from int8_mixed_precision_04_b300 import Linear8bitLt
    torch.manual_seed(0)
    K, N = 512, 384
    lin = torch.nn.Linear(K, N, bias=True)
    layer = Linear8bitLt.from_linear(lin, threshold=6.0)
    w = inputs.random_small(2 * 3 * 5, K, N, 3, seed=8)
    x = torch.from_numpy(w.X).cuda().reshape(2, 3, 5, K)
    y = layer(x)
    assert y.shape == (2, 3, 5, N) and y.dtype == torch.float16
    W16 = lin.weight.detach().to(torch.float16).numpy()
    b16 = lin.bias.detach().to(torch.float16).numpy()
    Wq_o, sw_o = orc.quantize_weight(W16)
    assert np.array_equal(layer.Wq.cpu().numpy(), Wq_o)
    assert np.array_equal(layer.Wscale.cpu().numpy(), sw_o)
    ref = orc.linear(w.X, Wq_o, sw_o, W16, 6.0, bias=b16)
    check_y(y.reshape(-1, N).cpu().numpy(), ref["Y"], "Linear8bitLt")
    # decode-sized call (a different kernel) through the same module
    y1 = layer(x[0, 0, :4])
    check_y(y1.cpu().numpy(), orc.linear(w.X[:4], Wq_o, sw_o, W16, 6.0, bias=b16)["Y"], "decode")
    assert layer(torch.empty((0, K), dtype=torch.float16, device="cuda")).shape == (0, N)
    nobias = Linear8bitLt(torch.from_numpy(W16).cuda(), None, threshold=math.inf)
    ref_nb = orc.linear(w.X, Wq_o, sw_o, W16, math.inf)
    check_y(nobias(torch.from_numpy(w.X).cuda()).cpu().numpy(), ref_nb["Y"], "no bias")
