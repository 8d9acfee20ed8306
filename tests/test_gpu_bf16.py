"""The layer with bf16 X, W16, bias and Y (bnb_int8_linear_ex, dtype bf16)
against the oracle's bf16 leg, on every path (GPU).

Bit-exact: outlier list, row scales, activation and weight codes, weight
scales and the int32 accumulators.  Y: bf16 keeps 8 significant bits, so an
fp32 evaluation and the oracle's exact one may round to neighbouring bf16
values whenever the exact value lies near a rounding boundary; the bound is
therefore per element, from the arithmetic: |Y - v| <= ulp_bf16(v) +
2^-20 max_row |v|, with v the oracle's exact (double) pre-rounding value and
the second term the fp32 accumulation error.
"""

import math
import numpy as np
import pytest

import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from int8_mixed_precision_04_b300 import binding, build
    build.build()
    binding.load()


def _bf16_bits(x) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def _bits_f64(b) -> np.ndarray:
    return (np.asarray(b, np.uint32) << 16).view(np.float32).astype(np.float64)


def _dev(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _host_bits(t) -> np.ndarray:
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def check_y_bf16(y_bits, ref, sw, bias_bits, what):
    """Per element: |Y - v| <= ulp_bf16(v) + 2^-20 max_row |v|."""
    sx = ref["sx"][ref["rows"]].astype(np.float64)
    v = ref["acc"].astype(np.float64) * sx[:, None] * sw.astype(np.float64)[None, :] / 16129.0
    v += ref["out"]
    if bias_bits is not None:
        v += _bits_f64(bias_bits)[None, :]
    y = _bits_f64(y_bits)
    assert not np.isnan(y).any(), f"{what}: NaN"
    big = np.abs(v) >= 3.3961775292304e38  # rounds to inf in bf16
    assert np.array_equal(np.isinf(y), big), f"{what}: infinities"
    fin = ~big
    av = np.abs(np.where(fin, v, 0.0))
    e = np.floor(np.log2(np.maximum(av, 2.0 ** -133)))
    ulp = 2.0 ** (np.maximum(e, -126) - 7)
    row = av.max(axis=1, keepdims=True)
    err = np.abs(np.where(fin, y - v, 0.0))
    bad = np.argwhere(err > ulp + 2.0 ** -20 * row)
    assert len(bad) == 0, (f"{what}: {len(bad)} outputs beyond one bf16 ulp, first "
                           f"{bad[0].tolist()}: {y[tuple(bad[0])]} vs {v[tuple(bad[0])]}")


def run_bf16(orc, Xb, Wb, tau, bias=None, wq_only=False, rows=None, what="", opts=0):
    import torch

    from int8_mixed_precision_04_b300 import binding
    W = _dev(Wb)
    Wq, sw = binding.quantize_weight(W)
    if opts:
        r = binding.linear_opts(_dev(Xb), Wq, sw, None if wq_only else W, tau, opts,
                                bias=None if bias is None else _dev(bias), debug=True)
    else:
        r = binding.linear_debug(_dev(Xb), Wq, sw, None if wq_only else W, tau,
                                 bias=None if bias is None else _dev(bias))
    torch.cuda.synchronize()
    assert binding.last_device_status(r["workspace"]) == 0
    Wq_o, sw_o = orc.quantize_weight(Wb, fmt="bf16")
    assert np.array_equal(Wq.cpu().numpy(), Wq_o), f"{what}: weight codes"
    assert np.array_equal(sw.cpu().numpy(), sw_o), f"{what}: weight scales"
    ref = orc.linear(Xb, Wq_o, sw_o, None if wq_only else Wb, tau, rows=rows, bias=bias,
                     fmt="bf16")
    nO = int(r["nO"].item())
    assert np.array_equal(r["O"][:nO].cpu().numpy(), ref["O"]), f"{what}: outlier list"
    assert np.array_equal(r["sx"].cpu().numpy(), ref["sx"]), f"{what}: row scales"
    assert np.array_equal(r["Xq"].cpu().numpy(), ref["Xq"]), f"{what}: activation codes"
    rows_t = torch.from_numpy(ref["rows"]).cuda()
    acc = r["acc"].index_select(0, rows_t).cpu().numpy()
    assert np.array_equal(acc, ref["acc"]), f"{what}: int32 accumulators"
    y = _host_bits(r["Y"].index_select(0, rows_t))
    check_y_bf16(y, ref, sw_o, bias, what)
    return r, ref


def _workload(T, K, N, ncols, seed, tau):
    w = inputs.random_small(T, K, N, ncols, seed=seed, tau=tau)
    return _bf16_bits(w.X.astype(np.float32)), _bf16_bits(w.W.astype(np.float32))


@pytest.mark.parametrize("T,K,N,ncols", [
    (1, 256, 64, 2), (16, 4096, 4096, 4), (11, 1040, 520, 9), (16, 1040, 96, 70),
    (17, 272, 129, 3), (300, 1024, 200, 4), (257, 2064, 1000, 7), (130, 512, 257, 40),
    (2, 512, 100, 2), (3, 2048, 300, 5), (6, 4096, 500, 3),
])
@pytest.mark.parametrize("tau", [6.0, 0.0, math.inf])
@pytest.mark.parametrize("form", ["w16", "bias", "wq_only"])
def test_bf16_parity(orc, T, K, N, ncols, tau, form):
    Xb, Wb = _workload(T, K, N, ncols, seed=T + 7 * N + K, tau=tau)
    bias = _bf16_bits(inputs.bias(N, K, seed=N).astype(np.float32)) if form != "w16" else None
    run_bf16(orc, Xb, Wb, tau, bias=bias, wq_only=form == "wq_only",
             what=f"bf16 {form} T{T} K{K} N{N} tau{tau}")


@pytest.mark.parametrize("T", [16, 48])
def test_bf16_integer_exact(orc, T):
    """tau = inf, integer inputs: Y = bf16(X W^T) bit for bit."""
    from int8_mixed_precision_04_b300 import binding
    X16, W16 = inputs.int_valued(T, 64, 40, seed=T)
    Xb, Wb = _bf16_bits(X16.astype(np.float32)), _bf16_bits(W16.astype(np.float32))
    W = _dev(Wb)
    Wq, sw = binding.quantize_weight(W)
    Y = _host_bits(binding.linear_ex(_dev(Xb), Wq, sw, W, None, math.inf))
    exact = X16.astype(np.int64) @ W16.astype(np.int64).T
    assert np.array_equal(Y, _bf16_bits(exact.astype(np.float32)))


@pytest.mark.parametrize("T,K,N", [(16, 1024, 256), (64, 1024, 256)])
@pytest.mark.parametrize("scale_exp", [124, -126, -100, 100])
def test_bf16_extreme_magnitudes(orc, T, K, N, scale_exp):
    """Rows scaled to bf16's range ends, where 127 x (or 127 / a) leaves fp32's
    range without the power-of-two rescaling: codes, scales, outliers and
    accumulators stay bit-exact (Y is checked where it is representable)."""
    rng = np.random.default_rng(scale_exp + 300)
    # X scaled; W too at the range ends (Y is then out of range and unchecked)
    X = rng.standard_normal((T, K)).astype(np.float32) * np.float32(2.0 ** scale_exp)
    W = (rng.standard_normal((N, K)) * 0.05).astype(np.float32)
    if abs(scale_exp) >= 120:
        W *= np.float32(2.0 ** scale_exp)
    Xb, Wb = _bf16_bits(X), _bf16_bits(W)
    tau = float(3.0 * 2.0 ** scale_exp) if abs(scale_exp) < 120 else math.inf
    if abs(scale_exp) < 120:
        run_bf16(orc, Xb, Wb, tau, what=f"bf16 scale 2^{scale_exp}")
        return
    import torch

    from int8_mixed_precision_04_b300 import binding
    Wd = _dev(Wb)
    Wq, sw = binding.quantize_weight(Wd)
    r = binding.linear_debug(_dev(Xb), Wq, sw, Wd, tau)
    torch.cuda.synchronize()
    Wq_o, sw_o = orc.quantize_weight(Wb, fmt="bf16")
    assert np.array_equal(Wq.cpu().numpy(), Wq_o) and np.array_equal(sw.cpu().numpy(), sw_o)
    ref = orc.linear(Xb, Wq_o, sw_o, Wb, tau, fmt="bf16")
    assert np.array_equal(r["sx"].cpu().numpy(), ref["sx"])
    assert np.array_equal(r["Xq"].cpu().numpy(), ref["Xq"])
    assert np.array_equal(r["acc"].cpu().numpy(), ref["acc"])


def test_bf16_module_and_from_host(orc):
    """Linear8bitLt in bf16 (with and without its 16-bit weight) and
    bnb_int8_linear_from_host_ex give bnb_int8_linear_ex's Y exactly."""
    import torch

    from int8_mixed_precision_04_b300 import Linear8bitLt, binding
    torch.manual_seed(1)
    K, N, T = 512, 384, 30
    lin = torch.nn.Linear(K, N, bias=True)
    Xb, _ = _workload(T, K, N, 3, seed=9, tau=6.0)
    x = _dev(Xb)
    for keep in (True, False):
        layer = Linear8bitLt.from_linear(lin, threshold=6.0, keep_fp16_weight=keep,
                                         dtype=torch.bfloat16)
        y = layer(x.reshape(2, 15, K))
        assert y.dtype == torch.bfloat16 and y.shape == (2, 15, N)
        Y_ref = binding.linear_ex(x, layer.Wq, layer.Wscale, layer.W16, layer.bias, 6.0)
        assert torch.equal(y.reshape(T, N), Y_ref)
        Xh = x.cpu().pin_memory()
        Yh = torch.empty((T, N), dtype=torch.bfloat16).pin_memory()
        Xd = torch.empty_like(x)
        Yd = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(binding.workspace_bytes(T, N, K), dtype=torch.uint8, device="cuda")
        binding.linear_from_host(Xh, layer.Wq, layer.Wscale, layer.W16, 6.0, Yh, Xd, Yd, ws,
                                 bias=layer.bias)
        torch.cuda.synchronize()
        assert torch.equal(Yh, Y_ref.cpu())
        Wb = _host_bits(lin.weight.detach().to(torch.bfloat16))
        Wq_o, sw_o = orc.quantize_weight(Wb, fmt="bf16")
        bias_b = _host_bits(lin.bias.detach().to(torch.bfloat16))
        ref = orc.linear(Xb, Wq_o, sw_o, Wb if keep else None, 6.0, bias=bias_b, fmt="bf16")
        check_y_bf16(_host_bits(Y_ref), ref, sw_o, bias_b, f"module keep={keep}")
